// decode_hq2b.cu -- split-K decode attention that reads the 2-bit pages directly.
//
// "KV at 9 KB a token" ("How it works"): attention reads the compressed cache itself; no
// decompressed copy exists in HBM.  "Half the Cache, Twice the Context" ("The cliff is in
// the accumulator"): partial sums live in FP32 registers, per page and per warp, and are
// merged once at the end (two-level accumulation).
//
// Work split.  Every (lane, KV head) contributes the pages before its exact tail (the open
// page and the recent-key window, handled by the combine kernel).  All those pages form one
// list ordered (lane, head, page); a persistent grid of 2 CTAs x 4 warps per SM cuts it into
// equal contiguous ranges, one per warp, so ragged lanes cost nothing in balance.  A warp
// writes one FP32 partial (m, l, acc[256]) for each (lane, head) segment its range touches.
//
// Per warp, pages stream through a STAGES-deep shared-memory ring filled by 1-D TMA bulk
// copies (cp.async.bulk, one 9,216 B copy = the page's K and V blocks of this layer/head),
// completion tracked by an mbarrier per stage; every wait is bounded.
//
// Per page (64 tokens, the G <= 8 query heads of the group padded to n = 8):
//   S^T = K^ . Q~^T on mma.sync m16n8k16 (fp16 in, fp32 accumulate): A = 2-bit K codes
//     unpacked straight into fragments as fp16 (4 + c) with one shift + one LOP3 per pair,
//     B = q (.) s_page (the per-channel K scales folded into the query, one HMUL2 per pair).
//     k^ = s (2c - 3) = s (2 (4 + c) - 11), so the score is 2 raw - 11 sum(q~); sum(q~) comes
//     from one more MMA chain with an all-ones A, so it uses exactly the rounded q~.
//     The contraction order over the 256 dims is permuted so each thread's A and B come
//     from 16 contiguous code bytes; any permutation of a dot product is the same sum.
//   online softmax in FP32 (log2 domain), one max per page per head.
//   O^T += V^ . P^T on the same MMA: A = V codes (4 + c) of two tokens per fp16 pair
//     (byte permute + shift + LOP3), B = P (.) s_v (per-token V scale folded into P) moved
//     from the S^T accumulator layout to the B layout with movmatrix.trans; the z offsets
//     and the "+4" are added back with sum(P z) (FP32) and one all-ones MMA per k-step.
#include "kvq_internal.cuh"
#include "attn_args.cuh"

namespace kvq {

constexpr int DEC_WARPS = 4;
#ifndef KVQ_DEC_CTAS_PER_SM
#define KVQ_DEC_CTAS_PER_SM 2
#endif
#ifndef KVQ_DEC_STAGES
#define KVQ_DEC_STAGES 2
#endif
constexpr int DEC_CTAS_PER_SM = KVQ_DEC_CTAS_PER_SM;  // resident CTAs per SM the grid is sized for
constexpr int DEC_STAGES = KVQ_DEC_STAGES;            // pages in flight per warp
constexpr int STAGE_BYTES = 2 * HQ2B_BLOCK;  // K block + V block of one page, one layer/head
constexpr int V_OFF = HQ2B_BLOCK;
constexpr int MIN_PAGES_PER_WARP = 2;
constexpr int DEC_MAX_SLOTS = 96;            // partial records per (lane, query head), at most
constexpr int SPIN_LIMIT = 1 << 16;          // bounded mbarrier waits (x ~1 us hint)

// pages of lane b handled by the MMA path (everything before its exact tail)
__device__ __forceinline__ int main_pages(const CacheView& c, const int32_t* seq_len, int b, bool* bad = nullptr) {
  const int len = seq_len[b];
  if (len < 0 || len > c.max_pages * P) {
    if (bad) *bad = true;
    return 0;
  }
  const int ef = exact_from(len, c.window);
  return ef <= 0 ? 0 : ef / P;
}

// pages per warp: an even share of all pages, but never so few that one (lane, head) segment
// spans more than DEC_MAX_SLOTS warps (min_wp is set from max_seq_len by the host)
__device__ __forceinline__ int units_per_warp(int units, int nwarps, int min_wp) {
  const int w = (units + nwarps - 1) / nwarps;
  return w < min_wp ? min_wp : w;
}

// ----------------------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t h2mul(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 r = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&r);
}

// A-operand pairs straight from a code word.  x << 2 brings codes 0..3 of the low byte of each
// 16-bit half to mantissa bits 2-3, 4-5, 6-7, 8-9; x >> 6 does the same for the high byte.
// OR-ing in the exponent of 256, 64, 16 or 4 makes each half read exactly M + c; one HFMA2
// (on the FMA pipe) then yields 2c - 3 (keys) or c (values) exactly.
__device__ __forceinline__ uint32_t code_raw(uint32_t x, int pos) {
  const uint32_t mask = pos == 0 ? 0x000C000Cu : pos == 1 ? 0x00300030u : pos == 2 ? 0x00C000C0u : 0x03000300u;
  const uint32_t magic = pos == 0 ? 0x5C005C00u : pos == 1 ? 0x54005400u : pos == 2 ? 0x4C004C00u : 0x44004400u;
  return (x & mask) | magic;
}
__device__ __forceinline__ uint32_t h2fma(uint32_t a, uint32_t b, uint32_t c) {
  __half2 r = __hfma2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b), *reinterpret_cast<__half2*>(&c));
  return *reinterpret_cast<uint32_t*>(&r);
}
// key code as 2c - 3: (M + c) * 2 - (2M + 3)
__device__ __forceinline__ uint32_t code_k(uint32_t x, int pos) {
  const uint32_t neg = pos == 0 ? 0xE006E006u : pos == 1 ? 0xD818D818u : pos == 2 ? 0xD060D060u : 0xC980C980u;
  return h2fma(code_raw(x, pos), 0x40004000u, neg);
}
// value code as c: (M + c) * 1 - M
__device__ __forceinline__ uint32_t code_v(uint32_t x, int pos) {
  const uint32_t neg = pos == 0 ? 0xDC00DC00u : pos == 1 ? 0xD400D400u : pos == 2 ? 0xCC00CC00u : 0xC400C400u;
  return h2fma(code_raw(x, pos), 0x3C003C00u, neg);
}

// 2^x for the softmax (x <= 0 or -inf); one MUFU.EX2, relative error ~2^-22
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void tma_page(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// true once the barrier's phase with this parity completed; false after SPIN_LIMIT tries
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (int i = 0; i < SPIN_LIMIT; i++) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(1000u)
        : "memory");
    if (ok) return true;
  }
  return false;
}

// QK row i of an m-tile holds token pi(i): swapping the two middle tokens of every group of
// four makes the V-code loads of the P.V step hit shared-memory banks at most 2-way.
__device__ __forceinline__ int perm_row(int i) { return i ^ ((i >> 1) & 1); }

// ----------------------------------------------------------------------------- main kernel
struct Cursor {
  int b, h, p, n;  // lane, head, page within the lane's main pages, main pages of the lane
};

__device__ __forceinline__ void cursor_next(Cursor& cu, const int* pre, int H) {
  if (++cu.p < cu.n) return;
  cu.p = 0;
  if (++cu.h < H) return;
  cu.h = 0;
  do {
    ++cu.b;
    cu.n = pre[cu.b + 1] - pre[cu.b];
  } while (cu.n == 0);
}

template <int STAGES>
__global__ void __launch_bounds__(DEC_WARPS * 32, DEC_CTAS_PER_SM) decode_hq2b_main(AttnArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const CacheView& c = a.c;
  const int H = c.num_kv_heads, G = c.group, Hq = c.num_q_heads;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, cq = lane & 3;
  uint8_t* ring_smem = smem + warp * STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + DEC_WARPS * STAGES * STAGE_BYTES) + warp * STAGES;
  int* pre = reinterpret_cast<int*>(smem + DEC_WARPS * STAGES * STAGE_BYTES + DEC_WARPS * STAGES * 8);

  // exclusive prefix of main pages over lanes
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < a.lanes; base += 32) {
      const int b = base + lane;
      bool bad = false;
      int n = b < a.lanes ? main_pages(c, a.seq_len, b, &bad) : 0;
      if (bad && blockIdx.x == 0) flag(c.status, KVQ_STATUS_LEN_GT_TABLE);
      int incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t;
      }
      if (b < a.lanes) pre[b + 1] = carry + incl;
      carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (lane == 0) pre[0] = 0;
  }
  if (lane == 0) {
    for (int s = 0; s < STAGES; s++) mbar_init(smem_u32(&bars[s]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();

  const int units = H * pre[a.lanes];
  const int Wp = units_per_warp(units, a.grid_warps, a.min_wp);
  const int gw = blockIdx.x * DEC_WARPS + warp;
  const int u0 = gw * Wp;
  const int u1 = min(u0 + Wp, units);
  if (u0 >= u1) return;

  // locate u0: lane b with H*pre[b] <= u0 < H*pre[b+1]
  Cursor cu;
  {
    int lo = 0, hi = a.lanes;  // invariant: H*pre[lo] <= u0 < H*pre[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (H * pre[mid] <= u0) lo = mid;
      else hi = mid;
    }
    cu.b = lo;
    cu.n = pre[lo + 1] - pre[lo];
    const int off = u0 - H * pre[lo];
    cu.h = off / cu.n;
    cu.p = off - cu.h * cu.n;
  }
  Cursor pc = cu;  // producer cursor, runs STAGES pages ahead
  const int64_t pool_pages = c.pool_pages;
  uint32_t valid = 0, phase = 0;
  int produced = u0;

  auto produce = [&](int slot) {
    const int32_t phys = c.page_table[(int64_t)pc.b * c.max_pages + pc.p];
    const bool ok = phys >= 0 && phys < pool_pages;
    if (ok) {
      if (lane == 0) {
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        const uint8_t* src = c.pool + (int64_t)phys * c.page_bytes + block_offset(KVQ_FMT_HQ2B, H, c.layer, pc.h, 0);
        tma_page(smem_u32(ring_smem + slot * STAGE_BYTES), src, STAGE_BYTES, smem_u32(&bars[slot]));
      }
      valid |= 1u << slot;
    } else {
      valid &= ~(1u << slot);
      if (lane == 0) flag(c.status, KVQ_STATUS_PAGE_OOB);
    }
    ++produced;
    if (produced < u1) cursor_next(pc, pre, H);
  };
#pragma unroll
  for (int s = 0; s < STAGES; s++)
    if (u0 + s < u1) produce(s);

  // per-thread state: heads e0 = 2*cq, e1 = 2*cq + 1 of the group
  float O[16][4];
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f, Z00 = 0.f, Z01 = 0.f, Z10 = 0.f, Z11 = 0.f;
  uint32_t qh[16][2];
  const float sl2 = a.scale_log2;

  auto reset = [&]() {
#pragma unroll
    for (int i = 0; i < 16; i++)
#pragma unroll
      for (int e = 0; e < 4; e++) O[i][e] = 0.f;
    m0 = m1 = -INFINITY;
    l0 = l1 = Z00 = Z01 = Z10 = Z11 = 0.f;
  };
  // q of head r of the group, dims 64cq .. 64cq+63, as fp16 pairs in the contraction order
  auto load_q = [&](int b, int h) {
    uint32_t w[32];
    if (r < G) {
      const uint4* src = reinterpret_cast<const uint4*>(a.q + ((int64_t)b * Hq + h * G + r) * D + 64 * cq);
#pragma unroll
      for (int i = 0; i < 8; i++) {
        const uint4 v = src[i];
        w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; i++) w[i] = 0u;
    }
    auto qf = [&](int e) { return (e & 1) ? bf16_hi(w[e >> 1]) : bf16_lo(w[e >> 1]); };
#pragma unroll
    for (int j = 0; j < 4; j++)
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const int d0 = 16 * j + i;
        qh[4 * j + i][0] = pack_h2(qf(d0), qf(d0 + 8));
        qh[4 * j + i][1] = pack_h2(qf(d0 + 4), qf(d0 + 12));
      }
  };
  auto flush = [&](int b, int h) {
    // complete the per-thread partial sums over the 8 row groups
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, o);
      l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, o);
      Z00 += __shfl_xor_sync(0xFFFFFFFFu, Z00, o);
      Z01 += __shfl_xor_sync(0xFFFFFFFFu, Z01, o);
      Z10 += __shfl_xor_sync(0xFFFFFFFFu, Z10, o);
      Z11 += __shfl_xor_sync(0xFFFFFFFFu, Z11, o);
    }
    const int segstart = H * pre[b] + h * (pre[b + 1] - pre[b]);
    const int k = gw - segstart / Wp;
#pragma unroll
    for (int e = 0; e < 2; e++) {
      const int head = 2 * cq + e;
      if (head < G) {
        const int64_t pidx = ((int64_t)b * Hq + h * G + head) * a.max_splits + k;
        float* dst = a.ws_o + pidx * D;
#pragma unroll
        for (int hf = 0; hf < 2; hf++) {
          const float z = hf == 0 ? (e == 0 ? Z00 : Z01) : (e == 0 ? Z10 : Z11);
          float v[16];
#pragma unroll
          for (int i = 0; i < 8; i++) {
            v[i] = O[8 * hf + i][e] + z;
            v[8 + i] = O[8 * hf + i][2 + e] + z;
          }
          float4* d4 = reinterpret_cast<float4*>(dst + 128 * hf + 16 * r);
#pragma unroll
          for (int i = 0; i < 4; i++) d4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
        if (r == 0)
          reinterpret_cast<float2*>(a.ws_ml)[pidx] = e == 0 ? make_float2(m0, l0) : make_float2(m1, l1);
      }
    }
  };

  reset();
  load_q(cu.b, cu.h);
  bool timed_out = false;
  for (int u = u0; u < u1; u++) {
    const int slot = (u - u0) % STAGES;
    if (valid & (1u << slot)) {
      // every lane waits; the warp gives up together if any lane ran out of tries
      const bool ok = mbar_wait(smem_u32(&bars[slot]), (phase >> slot) & 1u);
      if (!__all_sync(0xFFFFFFFFu, ok)) {
        timed_out = true;
        break;
      }
      phase ^= 1u << slot;
      const uint8_t* st = ring_smem + slot * STAGE_BYTES;

      // ---- S^T for the four 16-token m-tiles.  k-step ks = 4j + i of thread column cq covers
      // dims 64cq + 16j + {i, i+8} (A regs 0/1: codes of bytes 0/2 of word j) and
      // {i+4, i+12} (A regs 2/3: bytes 1/3); q~ = q (.) s_page is formed per word j from the
      // natural-order scale pairs.
      float S[4][4];
#pragma unroll
      for (int mt = 0; mt < 4; mt++)
#pragma unroll
        for (int e = 0; e < 4; e++) S[mt][e] = 0.f;
      const uint8_t* krow_a = st + perm_row(r) * HQ2B_ROW + 16 * cq;
      const uint8_t* krow_b = st + (8 + perm_row(r)) * HQ2B_ROW + 16 * cq;
      const uint8_t* kscale = st + HQ2B_META_OFF + 128 * cq;
#pragma unroll
      for (int j = 0; j < 4; j++) {
        const uint4 s_lo = *reinterpret_cast<const uint4*>(kscale + 32 * j);       // dims 16j .. 16j+7
        const uint4 s_hi = *reinterpret_cast<const uint4*>(kscale + 32 * j + 16);  // dims 16j+8 .. 16j+15
        const uint32_t slo[4] = {s_lo.x, s_lo.y, s_lo.z, s_lo.w};
        const uint32_t shi[4] = {s_hi.x, s_hi.y, s_hi.z, s_hi.w};
        uint32_t bq[4][2];
#pragma unroll
        for (int i = 0; i < 4; i++) {
          const uint32_t sel = (i & 1) ? 0x7632u : 0x5410u;
          bq[i][0] = h2mul(qh[4 * j + i][0], __byte_perm(slo[i >> 1], shi[i >> 1], sel));
          bq[i][1] = h2mul(qh[4 * j + i][1], __byte_perm(slo[2 + (i >> 1)], shi[2 + (i >> 1)], sel));
        }
#pragma unroll
        for (int mt = 0; mt < 4; mt++) {
          const uint32_t wa = *reinterpret_cast<const uint32_t*>(krow_a + 16 * mt * HQ2B_ROW + 4 * j);
          const uint32_t wb = *reinterpret_cast<const uint32_t*>(krow_b + 16 * mt * HQ2B_ROW + 4 * j);
          const uint32_t la = wa << 2, ra = wa >> 6, lb = wb << 2, rb = wb >> 6;
#pragma unroll
          for (int i = 0; i < 4; i++)
            mma16816(S[mt], code_k(la, i), code_k(lb, i), code_k(ra, i), code_k(rb, i), bq[i][0], bq[i][1]);
        }
      }
      // ---- online softmax (log2 domain)
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int mt = 0; mt < 4; mt++) {
        S[mt][0] *= sl2;
        S[mt][1] *= sl2;
        S[mt][2] *= sl2;
        S[mt][3] *= sl2;
        mx0 = fmaxf(mx0, fmaxf(S[mt][0], S[mt][2]));
        mx1 = fmaxf(mx1, fmaxf(S[mt][1], S[mt][3]));
      }
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, o));
      }
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float al0 = ex2(m0 - mn0), al1 = ex2(m1 - mn1);
      m0 = mn0;
      m1 = mn1;
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int mt = 0; mt < 4; mt++) {
        S[mt][0] = ex2(S[mt][0] - mn0);
        S[mt][1] = ex2(S[mt][1] - mn1);
        S[mt][2] = ex2(S[mt][2] - mn0);
        S[mt][3] = ex2(S[mt][3] - mn1);
        ps0 += S[mt][0] + S[mt][2];
        ps1 += S[mt][1] + S[mt][3];
      }
      l0 = fmaf(l0, al0, ps0);
      l1 = fmaf(l1, al1, ps1);
      Z00 *= al0; Z10 *= al0; Z01 *= al1; Z11 *= al1;
      if (__any_sync(0xFFFFFFFFu, al0 != 1.0f || al1 != 1.0f)) {
#pragma unroll
        for (int i = 0; i < 16; i++) {
          O[i][0] *= al0; O[i][1] *= al1; O[i][2] *= al0; O[i][3] *= al1;
        }
      }
      // ---- P (.) s_v per half, sum(P z), and the B fragments of P.V
      uint32_t Bv[2][4][2];
#pragma unroll
      for (int mt = 0; mt < 4; mt++) {
#pragma unroll
        for (int rr = 0; rr < 2; rr++) {
          const int tok = 16 * mt + 8 * rr + perm_row(r);
          const uint2 mw = *reinterpret_cast<const uint2*>(st + V_OFF + HQ2B_META_OFF + tok * 8);
          const float s0 = half_bits_to_float((uint16_t)(mw.x & 0xFFFFu));
          const float z0 = half_bits_to_float((uint16_t)(mw.x >> 16));
          const float s1 = half_bits_to_float((uint16_t)(mw.y & 0xFFFFu));
          const float z1 = half_bits_to_float((uint16_t)(mw.y >> 16));
          const float pa = S[mt][2 * rr], pb = S[mt][2 * rr + 1];
          Z00 = fmaf(pa, z0, Z00);
          Z01 = fmaf(pb, z0, Z01);
          Z10 = fmaf(pa, z1, Z10);
          Z11 = fmaf(pb, z1, Z11);
          Bv[0][mt][rr] = movmatrix_t(pack_h2(pa * s0, pb * s0));
          Bv[1][mt][rr] = movmatrix_t(pack_h2(pa * s1, pb * s1));
        }
      }
      // ---- O^T += V^ . P'^T: a fp16 pair holds one dim of two tokens (bytes permuted so each
      // half of a word is one token) as the exact code c
      const int t0 = perm_row(2 * cq), t1 = perm_row(2 * cq + 1);
#pragma unroll
      for (int mt = 0; mt < 4; mt++) {
#pragma unroll
        for (int hf = 0; hf < 2; hf++) {
          const uint8_t* vb = st + V_OFF + 32 * hf + 4 * r;
          const uint32_t w0 = *reinterpret_cast<const uint32_t*>(vb + (16 * mt + t0) * HQ2B_ROW);
          const uint32_t w1 = *reinterpret_cast<const uint32_t*>(vb + (16 * mt + t1) * HQ2B_ROW);
          const uint32_t w2 = *reinterpret_cast<const uint32_t*>(vb + (16 * mt + 8 + t0) * HQ2B_ROW);
          const uint32_t w3 = *reinterpret_cast<const uint32_t*>(vb + (16 * mt + 8 + t1) * HQ2B_ROW);
          // [tok_a byte k, tok_a byte k+1, tok_b byte k, tok_b byte k+1], k = 0 (dims 16r..16r+7) or 2 (+8)
          const uint32_t x[4] = {__byte_perm(w0, w1, 0x5410u), __byte_perm(w0, w1, 0x7632u),
                                 __byte_perm(w2, w3, 0x5410u), __byte_perm(w2, w3, 0x7632u)};
          uint32_t lo[4], hi[4];
#pragma unroll
          for (int k = 0; k < 4; k++) {
            lo[k] = x[k] << 2;  // codes of the first byte of each half
            hi[k] = x[k] >> 6;  // codes of the second byte
          }
#pragma unroll
          for (int i8 = 0; i8 < 8; i8++) {
            const int pos = i8 & 3;
            const uint32_t* src = i8 < 4 ? lo : hi;
            mma16816(O[8 * hf + i8], code_v(src[0], pos), code_v(src[1], pos), code_v(src[2], pos),
                     code_v(src[3], pos), Bv[hf][mt][0], Bv[hf][mt][1]);
          }
        }
      }
      __syncwarp();
    }
    // refill this slot with the page STAGES ahead
    if (produced < u1) produce(slot);
    // segment boundary: flush and start the next (lane, head)
    const bool last = (u + 1 == u1);
    if (last || cu.p + 1 == cu.n) {
      flush(cu.b, cu.h);
      if (!last) {
        cursor_next(cu, pre, H);
        reset();
        load_q(cu.b, cu.h);
      }
    } else {
      cursor_next(cu, pre, H);
    }
  }
  if (timed_out) {
    if (lane == 0) flag(c.status, KVQ_STATUS_TIMEOUT);
    // let copies still in flight land before the CTA's shared memory is released
    for (int s = 0; s < STAGES; s++)
      if (valid & (1u << s)) mbar_wait(smem_u32(&bars[s]), (phase >> s) & 1u);
  }
}

// ----------------------------------------------------------------------------- combine + tail
// One CTA per (lane, query head): attends the exact tail [tail_start, len) on CUDA cores
// (keys from the ring past exact_from, else from the page codes) and merges it with the
// main-path partials of this (lane, head) in FP32.
__global__ void __launch_bounds__(256) decode_hq2b_combine(AttnArgs a) {
  const CacheView& c = a.c;
  const int H = c.num_kv_heads, G = c.group, Hq = c.num_q_heads;
  const int b = blockIdx.x, j = blockIdx.y, h = j / G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ int s_sum[2][8];
  __shared__ float wm[8], wl[8];
  __shared__ __align__(16) float wacc[8][D];

  // main pages of lanes before b, and of all lanes
  int before = 0, total = 0;
  for (int i = threadIdx.x; i < a.lanes; i += blockDim.x) {
    const int n = main_pages(c, a.seq_len, i);
    total += n;
    if (i < b) before += n;
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    before += __shfl_xor_sync(0xFFFFFFFFu, before, o);
    total += __shfl_xor_sync(0xFFFFFFFFu, total, o);
  }
  if (lane == 0) {
    s_sum[0][warp] = before;
    s_sum[1][warp] = total;
  }
  __syncthreads();
  before = 0;
  total = 0;
#pragma unroll
  for (int w = 0; w < 8; w++) {
    before += s_sum[0][w];
    total += s_sum[1][w];
  }
  float* out = a.out + ((int64_t)b * Hq + j) * D;
  const int len = a.seq_len[b];
  if (len < 0 || len > c.max_pages * P) {
    out[threadIdx.x] = 0.f;
    return;
  }
  const int npg = main_pages(c, a.seq_len, b);
  const int ef = exact_from(len, c.window);
  const int tail_start = npg * P;

  // ---- tail on CUDA cores: warp w takes tokens tail_start + w, + 8, ...
  float q[8];
  {
    const uint4 w4 = reinterpret_cast<const uint4*>(a.q + ((int64_t)b * Hq + j) * D)[lane];
    const uint32_t u[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
      q[2 * i] = bf16_lo(u[i]) * a.scale_log2;
      q[2 * i + 1] = bf16_hi(u[i]) * a.scale_log2;
    }
  }
  float m = -INFINITY, l = 0.f, acc[8];
#pragma unroll
  for (int i = 0; i < 8; i++) acc[i] = 0.f;
  bool oob = false;
  for (int t = tail_start + warp; t < len; t += 8) {
    const int32_t phys = c.page_table[(int64_t)b * c.max_pages + t / P];
    if (phys < 0 || phys >= c.pool_pages) {
      oob = true;
      continue;
    }
    const uint8_t* page = c.pool + (int64_t)phys * c.page_bytes;
    const uint8_t* kblk = page + block_offset(KVQ_FMT_HQ2B, H, c.layer, h, 0);
    const uint8_t* vblk = kblk + HQ2B_BLOCK;
    const int slot = t % P;
    float kx[8];
    if (t >= ef) {
      const uint4 w4 = reinterpret_cast<const uint4*>(c.ring + ring_row_offset(c, b, h, slot))[lane];
      const uint32_t u[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
      for (int i = 0; i < 4; i++) {
        kx[2 * i] = bf16_lo(u[i]);
        kx[2 * i + 1] = bf16_hi(u[i]);
      }
    } else {
      const uint32_t codes = reinterpret_cast<const uint16_t*>(kblk + slot * HQ2B_ROW)[lane];
      const uint4 sw = reinterpret_cast<const uint4*>(kblk + HQ2B_META_OFF)[lane];
      const __half2* sc = reinterpret_cast<const __half2*>(&sw);
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const float2 sp = __half22float2(sc[i]);
        kx[2 * i] = sp.x * (float)(2 * (int)((codes >> (4 * i)) & 3) - 3);
        kx[2 * i + 1] = sp.y * (float)(2 * (int)((codes >> (4 * i + 2)) & 3) - 3);
      }
    }
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < 8; i++) dot = fmaf(q[i], kx[i], dot);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, o);
    const uint32_t codes = reinterpret_cast<const uint16_t*>(vblk + slot * HQ2B_ROW)[lane];
    const uint32_t meta = reinterpret_cast<const uint32_t*>(vblk + HQ2B_META_OFF + slot * 8)[lane >> 4];
    const float sv = half_bits_to_float((uint16_t)(meta & 0xFFFFu));
    const float zv = half_bits_to_float((uint16_t)(meta >> 16));
    const float mn = fmaxf(m, dot);
    const float al = exp2f(m - mn), p = exp2f(dot - mn);
    m = mn;
    l = fmaf(l, al, p);
#pragma unroll
    for (int i = 0; i < 8; i++) acc[i] = fmaf(acc[i], al, p * (zv + (float)((codes >> (2 * i)) & 3) * sv));
  }
  if (oob && lane == 0) flag(c.status, KVQ_STATUS_PAGE_OOB);
  if (lane == 0) {
    wm[warp] = m;
    wl[warp] = l;
  }
  reinterpret_cast<float4*>(&wacc[warp][8 * lane])[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  reinterpret_cast<float4*>(&wacc[warp][8 * lane])[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  __syncthreads();

  // ---- merge: main partials of this (lane, head) + the 8 tail warps
  const int d = threadIdx.x;
  int nk = 0;
  int64_t p0 = 0;
  if (npg > 0) {
    const int units = H * total;
    const int Wp = units_per_warp(units, a.grid_warps, a.min_wp);
    const int segstart = H * before + h * npg;
    nk = (segstart + npg - 1) / Wp - segstart / Wp + 1;
    p0 = ((int64_t)b * Hq + j) * a.max_splits;
  }
  const float2* ml = reinterpret_cast<const float2*>(a.ws_ml) + p0;
  float M = -INFINITY;
#pragma unroll 8
  for (int k = 0; k < nk; k++) M = fmaxf(M, ml[k].x);
#pragma unroll
  for (int w = 0; w < 8; w++) M = fmaxf(M, wm[w]);
  float num = 0.f, den = 0.f;
#pragma unroll 8
  for (int k = 0; k < nk; k++) {
    const float2 e = ml[k];
    const float w = e.x == -INFINITY ? 0.f : exp2f(e.x - M);
    den = fmaf(e.y, w, den);
    num = fmaf(a.ws_o[(p0 + k) * D + d], w, num);
  }
#pragma unroll
  for (int w = 0; w < 8; w++) {
    const float e = wm[w] == -INFINITY ? 0.f : exp2f(wm[w] - M);
    den = fmaf(wl[w], e, den);
    num = fmaf(wacc[w][d], e, num);
  }
  out[d] = den > 0.f ? num / den : 0.f;
}

// ----------------------------------------------------------------------------- host side
// A segment of npg pages cut into ranges of Wp pages touches at most floor((npg-1)/Wp) + 2
// warps; slots - 2 >= ceil(npg / Wp) keeps that within `slots`.
int decode_hq2b_slots(int max_seq_len) {
  const int max_npg = max_seq_len / P;
  const int s = max_npg / MIN_PAGES_PER_WARP + 2;
  return s < DEC_MAX_SLOTS ? s : DEC_MAX_SLOTS;
}

static int decode_hq2b_min_wp(int max_seq_len) {
  const int max_npg = max_seq_len / P;
  const int slots = decode_hq2b_slots(max_seq_len);
  const int w = (max_npg + slots - 3) / (slots - 2);
  return w > MIN_PAGES_PER_WARP ? w : MIN_PAGES_PER_WARP;
}

static int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 1;
  }
  return cached[dev];
}

constexpr int MAX_LANES_FAST = 8192;

int launch_attn_generic(int fmt, const AttnArgs& a, int decode, cudaStream_t stream);

int launch_decode_hq2b(const AttnArgs& a_in, cudaStream_t stream) {
  AttnArgs a = a_in;
  if (a.lanes > MAX_LANES_FAST) return KVQ_ERR_UNSUPPORTED;
  const int grid = sm_count() * DEC_CTAS_PER_SM;
  a.grid_warps = grid * DEC_WARPS;
  a.min_wp = decode_hq2b_min_wp(a.max_seq_len);
  const size_t smem = (size_t)DEC_WARPS * DEC_STAGES * STAGE_BYTES + DEC_WARPS * DEC_STAGES * 8 +
                      (size_t)(a.lanes + 1) * sizeof(int);
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!attr_set[dev]) {
    cudaFuncSetAttribute(decode_hq2b_main<DEC_STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         DEC_WARPS * DEC_STAGES * STAGE_BYTES + DEC_WARPS * DEC_STAGES * 8 +
                             (MAX_LANES_FAST + 1) * (int)sizeof(int));
    attr_set[dev] = true;
  }
  decode_hq2b_main<DEC_STAGES><<<grid, DEC_WARPS * 32, smem, stream>>>(a);
  decode_hq2b_combine<<<dim3(a.lanes, a.c.num_q_heads), 256, 0, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq

// decode_hq2b.cu -- split-K decode attention that reads the 2-bit pages directly.
//
// "KV at 9 KB a token" ("How it works"): attention reads the compressed cache itself; no
// decompressed copy exists in HBM.  "Half the Cache, Twice the Context" ("The cliff is in
// the accumulator"): partial sums live in FP32 registers, per page and per warp, and are
// merged once at the end (two-level accumulation).
//
// Work split.  Every (lane, KV head) contributes the pages before its exact tail (the open
// page and the recent-key window, handled by the combine kernel).  All those pages form one
// list ordered (lane, head, page); a persistent grid of 2 CTAs per SM, each of DEC_PAIRS warp
// pairs, cuts it into equal contiguous ranges, one per pair, so ragged lanes cost nothing in
// balance.  A pair writes one FP32 partial (m, l, acc[256]) for each (lane, head) segment its
// range touches; decode_hq2b_combine merges them with the tail.
//
// Warp pair.  The Q.K^T warp streams each page's K block (4,608 B) and the P.V warp its V block
// through their own 2-slot rings of 1-D bulk copies (cp.async.bulk), completion tracked by an
// mbarrier per slot; P and the rescale factors pass from the first to the second through a
// double-buffered shared-memory slot.  Every wait is bounded.
//
// Per page (64 tokens, the G <= 8 query heads of the group padded to n = 8), on mma.sync
// m16n8k16 (fp16 in, fp32 accumulate):
//   S^T = K^ . Q~^T: A = the 2-bit K codes read straight as the fp16 numbers M + c (one LOP3 per
//     register, see the A-operand notes below), B = q (.) s_page (the per-channel K scales
//     folded into the query, one HMUL2 per pair); one more MMA chain with A = M + 1.5 gives
//     sum q~ (M + 1.5), so q~ . k^ = 2 (sum q~ (M + c) - sum q~ (M + 1.5)) with exactly the
//     rounded q~.  The per-token-K instance keeps q as B and applies each token's (s, z) to
//     per-half sums instead.  The contraction order over the 256 dims is permuted so that each
//     thread's A and B come from contiguous code bytes; a dot product does not depend on it.
//   online softmax in FP32 (log2 domain) with a lazy rescale.
//   O^T += V^ . P'^T: A = V codes of two tokens per fp16 pair (byte permute, one AND: the code
//     c at mantissa bits 2k, 2k + 1 with a zero exponent field is the fp16 subnormal c 2^(2k-24),
//     exact, and the power of two comes off once at the end), B = P' = P (.) s_v (the per-token V
//     scale folded into P, fp16).  P reaches the P.V warp already in the B layout (fp16, moved
//     from the S^T accumulator layout with movmatrix.trans by the Q.K^T warp); one more MMA per
//     16 tokens with A rows (z0, z1, s0, s1, 1) of the tokens' metadata and B = P gives
//     sum P z per half, sum P s per half and sum P in FP32.
#include "kvq_internal.cuh"
#include "attn_args.cuh"
#include "append_ops.cuh"
#include "mma_tma.cuh"

namespace kvq {

#ifndef KVQ_DEC_CTAS_PER_SM
#define KVQ_DEC_CTAS_PER_SM 2
#endif
#ifndef KVQ_DEC_PAIRS
#define KVQ_DEC_PAIRS 4
#endif
constexpr int DEC_PAIRS = KVQ_DEC_PAIRS;               // warp pairs per CTA
constexpr int DEC_CTAS_PER_SM = KVQ_DEC_CTAS_PER_SM;  // resident CTAs per SM the grid is sized for
// A pair takes at least MIN_PAGES_PER_WARP pages, and a (lane, head) segment writes at most
// DEC_MAX_SLOTS partial records: a single long lane (131,072 tokens, 2,048 pages a head) is still
// cut into ranges of 9 pages, enough to keep every pair of the grid busy, while 8 lanes of 40,960
// tokens need 162 records a (lane, query head), 32 MB of workspace.
constexpr int MIN_PAGES_PER_WARP = 4;
constexpr int DEC_MAX_SLOTS = 256;           // partial records per (lane, query head), at most

// pages of lane b handled by the MMA path (everything before its exact tail); a lane whose
// length is unusable has none, and *err (if given) receives its status bits
__device__ __forceinline__ int main_pages(const AttnArgs& a, int b, int* err = nullptr) {
  const int len = a.seq_len[b];
  if (const int e = lane_len_error(a, len)) {
    if (err) *err = e;
    return 0;
  }
  const int ef = exact_from(len, a.c.window, a.c.ktok);
  return ef <= 0 ? 0 : ef / P;
}

// pages per warp: an even share of all pages, but never so few that one (lane, head) segment
// spans more than DEC_MAX_SLOTS warps (min_wp is set from max_seq_len by the host)
__device__ __forceinline__ int units_per_warp(int units, int nwarps, int min_wp) {
  const int w = (units + nwarps - 1) / nwarps;
  return w < min_wp ? min_wp : w;
}

// ----------------------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t h2mul(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

// A-operand pairs straight from a code word.  A 16-bit half holding code byte(s) with the code
// of position i at bits e + 2i, e + 2i + 1 reads as the fp16 number M + c once every other bit
// is masked off and the exponent of M = 2^(10 - e - 2i) is OR-ed in (one LOP3); M + c is exact.
//   keys:   e = 2 (the word shifted left by 2, or right by 6 for its high byte): M = 256, 64, 16,
//           4; the MMA takes M + c as is and a per-page correction removes the M + 1.5 part.
//   values: no exponent at all.  The word as is (low byte) or shifted right by 8 (high byte)
//           leaves the code of position k at bits 2k, 2k + 1 of each half; masked (one AND) the
//           half is the fp16 subnormal c 2^(2k - 24), exact, and the tensor core multiplies
//           subnormals exactly.  Each O accumulator takes one position only, so its factor
//           2^(2k - 24) comes off with one multiply when the partial is written.
//           The rotated format subtracts 1.5 sum P' per half at the end (sum P' from one MMA
//           with A = 1), which centres the codes: the fp16 rounding of P (.) s_v scales a whole
//           code row, whose mean is 1.5, and the inverse rotation gathers that common part
//           onto output dims 0 and 128; on centred rows it has mean ~0.
__device__ __forceinline__ uint32_t lop_and_or(uint32_t x, uint32_t mask, uint32_t magic) {
  return (x & mask) | magic;
}
constexpr uint32_t KMASK0 = 0x000C000Cu;   // key code position i: KMASK0 << 2i after the shift
constexpr uint32_t VMASK = 0x00030003u;    // value code position i: VMASK << 2i
// fp16x2 bit patterns: M + 0 for keys (256, 64, 16, 4) and the key correction M + 1.5 (257.5,
// 65.5, 17.5, 5.5), all exact in fp16
__constant__ uint32_t c_kmag[4] = {0x5C005C00u, 0x54005400u, 0x4C004C00u, 0x44004400u};
__constant__ uint32_t c_kcor[4] = {0x5C065C06u, 0x54185418u, 0x4C604C60u, 0x45804580u};
// 2^(24 - 2k): the factor that turns an accumulator of subnormal codes at position k back into
// codes
__device__ __forceinline__ constexpr float vpos_scale(int k) {
  return k == 0 ? 16777216.0f : k == 1 ? 4194304.0f : k == 2 ? 1048576.0f : 262144.0f;
}

__device__ __forceinline__ uint32_t shl2(uint32_t x) { return x << 2; }
__device__ __forceinline__ uint32_t shr6(uint32_t x) { return x >> 6; }
__device__ __forceinline__ uint32_t shr8(uint32_t x) { return x >> 8; }

// lazy rescale: the running max of a head moves only when a page max exceeds it by more than
// RESCALE_LOG2 (log2 domain), so P <= 2^0.5 and P * s_v stays below 65,504 for any finite V
constexpr float RESCALE_LOG2 = 0.5f;

// Dims of word jw (16 dims) of thread column cq in the Q.K^T contraction.  The plain layout
// gives each thread 64 contiguous dims; the per-token-K layout keeps every k-step inside one
// 128-dim half (jw 0-1: dims 0-127, jw 2-3: dims 128-255), since its keys scale per half.
template <bool KTOK>
__device__ __forceinline__ constexpr int dim_base(int cq, int jw) {
  return KTOK ? 128 * (jw >> 1) + 32 * cq + 16 * (jw & 1) : 64 * cq + 16 * jw;
}
constexpr uint32_t H2_ONE = 0x3C003C00u;   // 1.0 in both fp16 lanes

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

// Exchange slot written by the Q.K warp and read by the P.V warp of a pair, one page each:
// per thread P of 4 m-tiles as fp16 B fragments (2 registers per m-tile: tokens 0-7 and 8-15
// of the tile, for head r), then (alpha0, alpha1, m0, m1).  Stored as [3 uint4][32 lanes] so
// both sides access it without bank conflicts.
constexpr int X_F4 = 3;
constexpr int X_BYTES = X_F4 * 32 * 16;
constexpr int QS_BYTES = 8 * 32 * 16;   // the Q.K warp's query pairs: [8 uint4][32 lanes]
constexpr int PAIR_BYTES = 4 * HQ2B_BLOCK + 2 * X_BYTES + QS_BYTES;  // K ring 2, V ring 2, exchange 2, q
enum { PB_KFULL = 0, PB_VFULL = 2, PB_XFULL = 4, PB_XEMPTY = 6, PB_COUNT = 8 };

__device__ __forceinline__ void locate(int u0, const int* pre, int lanes, int H, Cursor& cu) {
  int lo = 0, hi = lanes;  // invariant: H*pre[lo] <= u0 < H*pre[hi]
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

// Warp pairs: warp w < DEC_PAIRS runs Q.K^T + softmax of a page, warp w + DEC_PAIRS runs its
// P.V one page behind; both walk the same range of pages.  Each warp streams its own half of
// every page (K block / V block, 4,608 B each) through a 2-slot TMA ring.
template <bool CENTRED, bool KTOK>
__global__ void __launch_bounds__(DEC_PAIRS * 64, DEC_CTAS_PER_SM) decode_hq2b_main(AttnArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const CacheView& c = a.c;
  const int H = c.num_kv_heads, G = c.group, Hq = c.num_q_heads;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, cq = lane & 3;
  const int pair = warp % DEC_PAIRS;
  const bool is_qk = warp < DEC_PAIRS;
  uint8_t* pbase = smem + pair * PAIR_BYTES;
  uint8_t* kring = pbase;                            // 2 x K block
  uint8_t* vring = pbase + 2 * HQ2B_BLOCK;           // 2 x V block
  float4* xring = reinterpret_cast<float4*>(pbase + 4 * HQ2B_BLOCK);
  uint4* qsm = reinterpret_cast<uint4*>(pbase + 4 * HQ2B_BLOCK + 2 * X_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + DEC_PAIRS * PAIR_BYTES) + pair * PB_COUNT;
  int* pre = reinterpret_cast<int*>(smem + DEC_PAIRS * PAIR_BYTES + DEC_PAIRS * PB_COUNT * 8);

  auto BAR = [&](int i) { return smem_u32(&bars[i]); };
  // the combine kernel may be scheduled now: it does its own tail work first and waits for
  // this grid's completion before it reads any partial
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

  // exclusive prefix of main pages over lanes
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < a.lanes; base += 32) {
      const int b = base + lane;
      int err = 0;
      int n = b < a.lanes ? main_pages(a, b, &err) : 0;
      if (err && blockIdx.x == 0) flag(c.status, err);
      int incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t;
      }
      if (b < a.lanes) {
        pre[b + 1] = carry + incl;
        int cp = -1;
        if (a.step.active && a.step.n_new[b] == 1) {
          const int st = a.step.start_pos[b];
          if (st >= 0 && (st + 1) % P == 0) cp = st / P;
        }
        pre[a.lanes + 1 + b] = cp;   // fused decode step: the page the step's token closes, or -1
      }
      carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (lane == 0) pre[0] = 0;
  }
  if (lane == 0 && is_qk) {
    for (int i = 0; i < 2; i++) {
      mbar_init(BAR(PB_KFULL + i), 1);
      mbar_init(BAR(PB_VFULL + i), 1);
      mbar_init(BAR(PB_XFULL + i), 1);
      mbar_init(BAR(PB_XEMPTY + i), 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  const int units = H * pre[a.lanes];
  const int Wp = units_per_warp(units, a.grid_warps, a.min_wp);
  const int gp = blockIdx.x * DEC_PAIRS + pair;
  const int u0 = gp * Wp;
  const int u1 = min(u0 + Wp, units);
  if (u0 >= u1) {
    asm volatile("griddepcontrol.wait;\n" ::: "memory");   // see the end of the kernel
    return;
  }
  const int n_units = u1 - u0;

  Cursor cu;
  locate(u0, pre, a.lanes, H, cu);
  // producer cursor (this warp's own ring), two pages ahead at most
  Cursor pc = cu;
  int produced = 0;
  uint32_t valid = 0;
  uint8_t* ring = is_qk ? kring : vring;
  const int kv = is_qk ? 0 : 1;
  const int full_bar = is_qk ? PB_KFULL : PB_VFULL;
  // physical pages of this warp's units, 32 at a time: lane l of chunk k holds the page of unit
  // u0 + 32k + l (-1 past the range), so a page's copy waits on a page-table load only once per
  // 32 pages
  auto phys_chunk = [&](int k) -> int32_t {
    const int u = u0 + 32 * k + lane;
    int32_t ph = -1;
    if (u < u1) {
      Cursor t;
      locate(u, pre, a.lanes, H, t);
      ph = c.page_table[(int64_t)t.b * c.max_pages + t.p];
    }
    return ph;
  };
  int32_t ph_cur = phys_chunk(0);
  auto produce = [&]() {
    const int slot = produced & 1;
    if ((produced & 31) == 0 && produced > 0) ph_cur = phys_chunk(produced >> 5);
    const int32_t phys = __shfl_sync(0xFFFFFFFFu, ph_cur, produced & 31);
    const bool ok = phys >= 0 && phys < c.pool_pages;
    if (ok) {
      // fused decode step: a page that the step's token closes (a main page only with window 0)
      // gets its K block and last V row from the append kernel this grid overlaps: wait for it
      if (a.step.active && pre[a.lanes + 1 + pc.b] == pc.p) asm volatile("griddepcontrol.wait;\n" ::: "memory");
      if (lane == 0) {
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        const uint8_t* src = c.pool + (int64_t)phys * c.page_bytes + block_offset(KVQ_FMT_HQ2B, H, c.layer, pc.h, kv);
        tma_page(smem_u32(ring + slot * HQ2B_BLOCK), src, HQ2B_BLOCK, BAR(full_bar + slot));
      }
      valid |= 1u << slot;
    } else {
      valid &= ~(1u << slot);
      if (lane == 0 && is_qk) flag(c.status, KVQ_STATUS_PAGE_OOB);
    }
    if (++produced < n_units) cursor_next(pc, pre, H);
  };
  produce();
  if (n_units > 1) produce();

  bool timed_out = false;
  if (is_qk) {
    // =========================================================== Q.K^T + softmax warp
    float m0 = -INFINITY, m1 = -INFINITY;
    const float sl2 = a.scale_log2;
    uint32_t kmag[4], kcor[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
      kmag[i] = c_kmag[i];
      kcor[i] = KTOK ? 0u : c_kcor[i];
    }
    float tk_mq[2][2], tk_q[2][2];   // per-token-K: sum_half q M and sum_half q, heads 2cq, 2cq+1
    // q of head r of the group, the 64 dims dim_base(cq, jw) + 0..15 (jw = 0..3), as the fp16
    // B-fragment pairs of k-steps 4jw + i: (d, d+8) and (d+4, d+12) with d = 16jw + i; kept in
    // shared memory, one uint4 = the 4 k-steps' first pairs or second pairs of one jw
    auto load_q = [&](int b, int h) {
      uint32_t w[32];
      if (r < G) {
        // rotated format: H q (fp16, written by rotate_q_kernel), else q (bf16)
        const int64_t qo = ((int64_t)b * Hq + h * G + r) * D;
        const uint4* src = a.c.rotated ? reinterpret_cast<const uint4*>(a.q_rot + qo)
                                       : reinterpret_cast<const uint4*>(a.q + qo);
#pragma unroll
        for (int i = 0; i < 8; i++) {
          const uint4 v = src[(dim_base<KTOK>(cq, i >> 1) + 8 * (i & 1)) / 8];
          w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; i++) w[i] = 0u;
      }
      auto qf = [&](int e) {
        if (a.c.rotated) return half_bits_to_float((uint16_t)((e & 1) ? w[e >> 1] >> 16 : w[e >> 1] & 0xFFFFu));
        return (e & 1) ? bf16_hi(w[e >> 1]) : bf16_lo(w[e >> 1]);
      };
#pragma unroll
      for (int jw = 0; jw < 4; jw++) {
        uint32_t p0[4], p1[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
          const int d0 = 16 * jw + i;
          p0[i] = pack_h2(qf(d0), qf(d0 + 8));
          p1[i] = pack_h2(qf(d0 + 4), qf(d0 + 12));
        }
        qsm[(2 * jw) * 32 + lane] = make_uint4(p0[0], p0[1], p0[2], p0[3]);
        qsm[(2 * jw + 1) * 32 + lane] = make_uint4(p1[0], p1[1], p1[2], p1[3]);
      }
      __syncwarp();
      if constexpr (KTOK) {
        // per (lane, head) segment: sum over each half of q M and of q, per head of the thread's
        // columns, from MMAs with constant A (every row the same)
        float mq[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        float qq[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int jw = 0; jw < 4; jw++) {
          const uint4 qa = qsm[(2 * jw) * 32 + lane], qb = qsm[(2 * jw + 1) * 32 + lane];
          const uint32_t q0[4] = {qa.x, qa.y, qa.z, qa.w}, q1[4] = {qb.x, qb.y, qb.z, qb.w};
#pragma unroll
          for (int i = 0; i < 4; i++) {
            mma16816(mq[jw >> 1], kmag[i], kmag[i], kmag[i], kmag[i], q0[i], q1[i]);
            mma16816(qq[jw >> 1], H2_ONE, H2_ONE, H2_ONE, H2_ONE, q0[i], q1[i]);
          }
        }
#pragma unroll
        for (int e = 0; e < 2; e++) {
          tk_mq[0][e] = mq[0][e];
          tk_mq[1][e] = mq[1][e];
          tk_q[0][e] = qq[0][e];
          tk_q[1][e] = qq[1][e];
        }
      }
    };
    load_q(cu.b, cu.h);
    for (int j = 0; j < n_units; j++) {
      const int slot = j & 1;
      const uint32_t par = (j >> 1) & 1;
      float S[4][4];
#pragma unroll
      for (int mt = 0; mt < 4; mt++)
#pragma unroll
        for (int e = 0; e < 4; e++) S[mt][e] = -INFINITY;
      if (valid & (1u << slot)) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(BAR(PB_KFULL + slot), par))) { timed_out = true; break; }
        const uint8_t* st = kring + slot * HQ2B_BLOCK;
        float Cc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};   // sum over dims of q~ (M + 1.5), in two chains
        float S1[4][4];                       // per-token-K: the second half's sums (S: the first)
#pragma unroll
        for (int mt = 0; mt < 4; mt++)
#pragma unroll
          for (int e = 0; e < 4; e++) S[mt][e] = S1[mt][e] = 0.f;
        const uint8_t* krow_a = st + perm_row(r) * HQ2B_ROW;
        const uint8_t* krow_b = st + (8 + perm_row(r)) * HQ2B_ROW;
        // k-step ks = 4j + i of thread column cq covers dims dim_base(cq, j) + {i, i+8} (A regs
        // 0/1: codes of bytes 0/2 of word j) and {i+4, i+12} (A regs 2/3: bytes 1/3)
#pragma unroll
        for (int jw = 0; jw < 4; jw++) {
          const uint4 qa = qsm[(2 * jw) * 32 + lane], qb = qsm[(2 * jw + 1) * 32 + lane];
          const uint32_t q0[4] = {qa.x, qa.y, qa.z, qa.w}, q1[4] = {qb.x, qb.y, qb.z, qb.w};
          uint32_t bq[4][2];
          if constexpr (KTOK) {
            // keys scaled per token: the B operand is q itself
#pragma unroll
            for (int i = 0; i < 4; i++) {
              bq[i][0] = q0[i];
              bq[i][1] = q1[i];
            }
          } else {
            const uint8_t* kscale = st + HQ2B_META_OFF + 2 * dim_base<KTOK>(cq, jw);
            const uint4 s_lo = *reinterpret_cast<const uint4*>(kscale);
            const uint4 s_hi = *reinterpret_cast<const uint4*>(kscale + 16);
            const uint32_t slo[4] = {s_lo.x, s_lo.y, s_lo.z, s_lo.w};
            const uint32_t shi[4] = {s_hi.x, s_hi.y, s_hi.z, s_hi.w};
#pragma unroll
            for (int i = 0; i < 4; i++) {
              const uint32_t sel = (i & 1) ? 0x7632u : 0x5410u;
              bq[i][0] = h2mul(q0[i], __byte_perm(slo[i >> 1], shi[i >> 1], sel));
              bq[i][1] = h2mul(q1[i], __byte_perm(slo[2 + (i >> 1)], shi[2 + (i >> 1)], sel));
              mma16816(Cc[i & 1], kcor[i], kcor[i], kcor[i], kcor[i], bq[i][0], bq[i][1]);
            }
          }
          // the code word of word jw (16 dims) of the thread's two key rows in every m-tile
          const int wbyte = dim_base<KTOK>(cq, jw) / 4;
          uint32_t la[4], ra[4], lb[4], rb[4];
#pragma unroll
          for (int mt = 0; mt < 4; mt++) {
            const uint32_t wa = *reinterpret_cast<const uint32_t*>(krow_a + 16 * mt * HQ2B_ROW + wbyte);
            const uint32_t wb = *reinterpret_cast<const uint32_t*>(krow_b + 16 * mt * HQ2B_ROW + wbyte);
            la[mt] = shl2(wa);
            ra[mt] = shr6(wa);
            lb[mt] = shl2(wb);
            rb[mt] = shr6(wb);
          }
          // the four m-tiles' accumulators in turn, so that no MMA waits on the one before it
#pragma unroll
          for (int i = 0; i < 4; i++) {
            const uint32_t mk = KMASK0 << (2 * i);
#pragma unroll
            for (int mt = 0; mt < 4; mt++) {
              float(&acc)[4] = (KTOK && jw >= 2) ? S1[mt] : S[mt];
              mma16816(acc, lop_and_or(la[mt], mk, kmag[i]), lop_and_or(lb[mt], mk, kmag[i]),
                       lop_and_or(ra[mt], mk, kmag[i]), lop_and_or(rb[mt], mk, kmag[i]), bq[i][0], bq[i][1]);
            }
          }
        }
#pragma unroll
        for (int e = 0; e < 4; e++) Cc[0][e] += Cc[1][e];
        if constexpr (KTOK) {
          // q . k^ = sum over halves of s (sum q (M + c) - sum q M) + z sum q, with the token's
          // own (s, z) per half, then the softmax scale (log2 domain)
#pragma unroll
          for (int mt = 0; mt < 4; mt++)
#pragma unroll
            for (int rr = 0; rr < 2; rr++) {
              const uint2 mw = *reinterpret_cast<const uint2*>(st + HQ2B_META_OFF + (16 * mt + 8 * rr + perm_row(r)) * 8);
              const float s0 = half_bits_to_float((uint16_t)(mw.x & 0xFFFFu)) * sl2;
              const float z0 = half_bits_to_float((uint16_t)(mw.x >> 16)) * sl2;
              const float s1 = half_bits_to_float((uint16_t)(mw.y & 0xFFFFu)) * sl2;
              const float z1 = half_bits_to_float((uint16_t)(mw.y >> 16)) * sl2;
#pragma unroll
              for (int e = 0; e < 2; e++) {
                const float c0 = fmaf(z0, tk_q[0][e], z1 * tk_q[1][e]);
                S[mt][2 * rr + e] = fmaf(s0, S[mt][2 * rr + e] - tk_mq[0][e],
                                         fmaf(s1, S1[mt][2 * rr + e] - tk_mq[1][e], c0));
              }
            }
        } else {
          // q~ . k^ = 2 (sum q~ (M + c) - sum q~ (M + 1.5)), then the softmax scale (log2 domain)
          const float k2 = 2.f * sl2;
          const float cn0 = -Cc[0][0] * k2, cn1 = -Cc[0][1] * k2;
#pragma unroll
          for (int mt = 0; mt < 4; mt++) {
            S[mt][0] = fmaf(S[mt][0], k2, cn0);
            S[mt][1] = fmaf(S[mt][1], k2, cn1);
            S[mt][2] = fmaf(S[mt][2], k2, cn0);
            S[mt][3] = fmaf(S[mt][3], k2, cn1);
          }
        }
      }
      __syncwarp();
      // the K slot is free: refill it two pages ahead
      if (produced < n_units) produce();
      // ---- online softmax (log2 domain): page max per head, P relative to the running max
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int mt = 0; mt < 4; mt++) {
        mx0 = fmaxf(mx0, fmaxf(S[mt][0], S[mt][2]));
        mx1 = fmaxf(mx1, fmaxf(S[mt][1], S[mt][3]));
      }
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, o));
      }
      // lazy rescale: move a head's max only when the page max passes it by RESCALE_LOG2
      float al0 = 1.f, al1 = 1.f;
      if (mx0 > m0 + RESCALE_LOG2) {
        if (m0 != -INFINITY) al0 = ex2(m0 - mx0);
        m0 = mx0;
      }
      if (mx1 > m1 + RESCALE_LOG2) {
        if (m1 != -INFINITY) al1 = ex2(m1 - mx1);
        m1 = mx1;
      }
      const float mu0 = m0 == -INFINITY ? 0.f : m0, mu1 = m1 == -INFINITY ? 0.f : m1;
      // P in fp16, moved from the S^T accumulator layout (token rows, head columns) to the B
      // layout of the P.V step: thread (r, cq) gets head r of tokens 2cq, 2cq + 1 (QK rows) of
      // each 8-token half of the m-tile
      uint32_t pb[4][2];
#pragma unroll
      for (int mt = 0; mt < 4; mt++) {
        pb[mt][0] = movmatrix_t(pack_h2(ex2(S[mt][0] - mu0), ex2(S[mt][1] - mu1)));
        pb[mt][1] = movmatrix_t(pack_h2(ex2(S[mt][2] - mu0), ex2(S[mt][3] - mu1)));
      }
      // ---- hand P, alpha and m to the P.V warp
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(BAR(PB_XEMPTY + slot), par ^ 1u))) { timed_out = true; break; }
      uint4* xs = reinterpret_cast<uint4*>(xring + slot * (X_F4 * 32));
      xs[lane] = make_uint4(pb[0][0], pb[0][1], pb[1][0], pb[1][1]);
      xs[32 + lane] = make_uint4(pb[2][0], pb[2][1], pb[3][0], pb[3][1]);
      reinterpret_cast<float4*>(xs)[64 + lane] = make_float4(al0, al1, m0, m1);
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];\n" ::"r"(BAR(PB_XFULL + slot)) : "memory");
      // next (lane, head) segment: fresh max, new query
      if (j + 1 < n_units) {
        if (cu.p + 1 == cu.n) {
          cursor_next(cu, pre, H);
          m0 = m1 = -INFINITY;
          load_q(cu.b, cu.h);
        } else {
          cursor_next(cu, pre, H);
        }
      }
    }
  } else {
    // =========================================================== P.V warp
    // O[8hf + i8]: rows = dims 128hf + 16r + 4(i8 >= 4) + (i8 & 3) and + 8, columns = heads
    // 2cq, 2cq+1; accumulates subnormal codes of position i8 & 3 (factor 2^(2(i8&3) - 24)).
    // Zm: rows (z0, z1, s0, s1, 1) x heads of the metadata MMA (thread row r holds row r);
    // Cp[hf] (rotated format): row 0 = sum P' of half hf.
    float O[16][4];
    float Zm[4] = {0.f, 0.f, 0.f, 0.f};
    float Cp[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int i = 0; i < 16; i++)
#pragma unroll
      for (int e = 0; e < 4; e++) O[i][e] = 0.f;
    const int t0 = perm_row(2 * cq), t1 = perm_row(2 * cq + 1);
    // metadata pairs in the B layout: tokens (t0, t1) are the memory pair (2cq, 2cq+1), swapped
    // for odd cq; low halves = s, high halves = z of a meta word
    const uint32_t sel_s = (cq & 1) ? 0x1054u : 0x5410u, sel_z = (cq & 1) ? 0x3276u : 0x7632u;
    // A of the metadata MMA, row r: z0 (r = 0), z1 (1), s0 (2), s1 (3), 1.0 (4), 0 (5-7)
    const bool zy = r & 1;
    const uint32_t zsel = r < 2 ? sel_z : sel_s;
    const uint32_t zand = r < 4 ? 0xFFFFFFFFu : 0u, zor = r == 4 ? 0x3C003C00u : 0u;
    const uint32_t ones_a = r == 0 ? 0x3C003C00u : 0u;   // A = 1 in row 0 (sum P', rotated format)
    for (int j = 0; j < n_units; j++) {
      const int slot = j & 1;
      const uint32_t par = (j >> 1) & 1;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(BAR(PB_XFULL + slot), par))) { timed_out = true; break; }
      // P of the page is read per m-tile below; the slot is released after the page
      const uint4* xs = reinterpret_cast<const uint4*>(xring + slot * (X_F4 * 32));
      const float4 am = reinterpret_cast<const float4*>(xs)[64 + lane];
      const float al0 = am.x, al1 = am.y;
      if (__any_sync(0xFFFFFFFFu, al0 != 1.0f || al1 != 1.0f)) {
#pragma unroll
        for (int i = 0; i < 16; i++) {
          O[i][0] *= al0; O[i][1] *= al1; O[i][2] *= al0; O[i][3] *= al1;
        }
        Zm[0] *= al0; Zm[1] *= al1;
        if (CENTRED) {
          Cp[0][0] *= al0; Cp[0][1] *= al1;
          Cp[1][0] *= al0; Cp[1][1] *= al1;
        }
      }
      if (valid & (1u << slot)) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(BAR(PB_VFULL + slot), par))) { timed_out = true; break; }
        const uint8_t* st = vring + slot * HQ2B_BLOCK;
        const uint4 pw0 = xs[lane], pw1 = xs[32 + lane];
        const uint32_t pbs[4][2] = {{pw0.x, pw0.y}, {pw0.z, pw0.w}, {pw1.x, pw1.y}, {pw1.z, pw1.w}};
#pragma unroll
        for (int mt = 0; mt < 4; mt++) {
          // per 8-token half rr: the tokens' metadata, P' = P (.) s per half (fp16, B layout),
          // and the metadata MMA's A row
          uint32_t Bv[2][2], za[2];
#pragma unroll
          for (int rr = 0; rr < 2; rr++) {
            const uint4 u = *reinterpret_cast<const uint4*>(st + HQ2B_META_OFF + (16 * mt + 8 * rr + 2 * cq) * 8);
            const uint32_t s0p = __byte_perm(u.x, u.z, sel_s), s1p = __byte_perm(u.y, u.w, sel_s);
            Bv[0][rr] = h2mul(pbs[mt][rr], s0p);
            Bv[1][rr] = h2mul(pbs[mt][rr], s1p);
            za[rr] = (__byte_perm(zy ? u.y : u.x, zy ? u.w : u.z, zsel) & zand) | zor;
          }
          mma16816(Zm, za[0], 0u, za[1], 0u, pbs[mt][0], pbs[mt][1]);
          if (CENTRED) {
            mma16816(Cp[0], ones_a, 0u, ones_a, 0u, Bv[0][0], Bv[0][1]);
            mma16816(Cp[1], ones_a, 0u, ones_a, 0u, Bv[1][0], Bv[1][1]);
          }
          // O^T += V^ . P'^T, a fp16 pair holding one dim of two tokens as a subnormal code
#pragma unroll
          for (int hf = 0; hf < 2; hf++) {
            const uint8_t* vb = st + 32 * hf + 4 * r;
            const uint32_t w0 = *reinterpret_cast<const uint32_t*>(vb + (16 * mt + t0) * HQ2B_ROW);
            const uint32_t w1 = *reinterpret_cast<const uint32_t*>(vb + (16 * mt + t1) * HQ2B_ROW);
            const uint32_t w2 = *reinterpret_cast<const uint32_t*>(vb + (16 * mt + 8 + t0) * HQ2B_ROW);
            const uint32_t w3 = *reinterpret_cast<const uint32_t*>(vb + (16 * mt + 8 + t1) * HQ2B_ROW);
            const uint32_t x[4] = {__byte_perm(w0, w1, 0x5410u), __byte_perm(w0, w1, 0x7632u),
                                   __byte_perm(w2, w3, 0x5410u), __byte_perm(w2, w3, 0x7632u)};
            uint32_t hi[4];
#pragma unroll
            for (int k = 0; k < 4; k++) hi[k] = shr8(x[k]);
#pragma unroll
            for (int i8 = 0; i8 < 8; i8++) {
              const uint32_t* src = i8 < 4 ? x : hi;
              const uint32_t mk = VMASK << (2 * (i8 & 3));
              mma16816(O[8 * hf + i8], src[0] & mk, src[1] & mk, src[2] & mk, src[3] & mk, Bv[hf][0], Bv[hf][1]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];\n" ::"r"(BAR(PB_XEMPTY + slot)) : "memory");
      if (produced < n_units) produce();
      // segment end: write this pair's partial (m, l, O + z-term) and start afresh
      const bool last = (j + 1 == n_units);
      if (last || cu.p + 1 == cu.n) {
        // the metadata sums of heads 2cq, 2cq+1 live in thread rows 0-4 of this column
        float zz[2][2], zs[2][2], ll[2], cp[2][2];
#pragma unroll
        for (int e = 0; e < 2; e++) {
          zz[0][e] = __shfl_sync(0xFFFFFFFFu, Zm[e], cq);
          zz[1][e] = __shfl_sync(0xFFFFFFFFu, Zm[e], 4 + cq);
          zs[0][e] = __shfl_sync(0xFFFFFFFFu, Zm[e], 8 + cq);
          zs[1][e] = __shfl_sync(0xFFFFFFFFu, Zm[e], 12 + cq);
          ll[e] = __shfl_sync(0xFFFFFFFFu, Zm[e], 16 + cq);
          cp[0][e] = __shfl_sync(0xFFFFFFFFu, Cp[0][e], cq);
          cp[1][e] = __shfl_sync(0xFFFFFFFFu, Cp[1][e], cq);
        }
        const int segstart = H * pre[cu.b] + cu.h * (pre[cu.b + 1] - pre[cu.b]);
        const int k = gp - segstart / Wp;
#pragma unroll
        for (int e = 0; e < 2; e++) {
          const int head = 2 * cq + e;
          if (head < G) {
            const int64_t pidx = ((int64_t)cu.b * Hq + cu.h * G + head) * a.max_splits + k;
            float* dst = a.ws_o + pidx * D;
#pragma unroll
            for (int hf = 0; hf < 2; hf++) {
              // the zero points: sum P z (plain); sum P (z + 1.5 s) - 1.5 sum P' (centred codes)
              const float z = CENTRED ? fmaf(1.5f, zs[hf][e] - cp[hf][e], zz[hf][e]) : zz[hf][e];
              float v[16];
#pragma unroll
              for (int i = 0; i < 8; i++) {
                v[i] = fmaf(O[8 * hf + i][e], vpos_scale(i & 3), z);
                v[8 + i] = fmaf(O[8 * hf + i][2 + e], vpos_scale(i & 3), z);
              }
              float4* d4 = reinterpret_cast<float4*>(dst + 128 * hf + 16 * r);
#pragma unroll
              for (int i = 0; i < 4; i++) d4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
            }
            if (r == 0)
              reinterpret_cast<float2*>(a.ws_ml)[pidx] = e == 0 ? make_float2(am.z, ll[0]) : make_float2(am.w, ll[1]);
          }
        }
        if (!last) {
          cursor_next(cu, pre, H);
#pragma unroll
          for (int i = 0; i < 16; i++)
#pragma unroll
            for (int e = 0; e < 4; e++) O[i][e] = 0.f;
#pragma unroll
          for (int e = 0; e < 4; e++) {
            Zm[e] = 0.f;
            Cp[0][e] = Cp[1][e] = 0.f;
          }
        }
      } else {
        cursor_next(cu, pre, H);
      }
    }
  }
  if (timed_out && lane == 0) flag(c.status, KVQ_STATUS_TIMEOUT);
  // copies still in flight into this warp's ring must land before the CTA's smem is released
  for (int q = max(0, produced - 2); q < produced; q++)
    if (valid & (1u << (q & 1))) mbar_wait(BAR(full_bar + (q & 1)), (q >> 1) & 1u);
  // in a fused decode step this grid completes only after the append it overlaps, so the
  // combine kernel's wait for this grid covers the append as well (a no-op otherwise)
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

// ----------------------------------------------------------------------------- combine + tail
// One CTA per (lane, query head).  Part 1 attends the exact tail [tail_start, len) on CUDA
// cores -- keys from the ring past exact_from, else from the closed page's codes; values from
// the page codes -- and needs nothing from the main kernel, so it runs while the main grid
// drains (programmatic dependent launch).  Part 2 waits for the main grid and merges its
// partials of this (lane, head) with the tail in FP32.
constexpr int TAIL_MAX = 2 * P;   // len - tail_start < 2 pages, since the window is at most a page

__global__ void __launch_bounds__(256, 1) decode_hq2b_combine(AttnArgs a) {
  // fused decode step whose append runs last: that kernel may be scheduled now (it touches
  // nothing this kernel reads, and waits for this grid before it exits)
  if (a.step.append_last) asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const CacheView& c = a.c;
  const int H = c.num_kv_heads, G = c.group, Hq = c.num_q_heads;
  const int b = blockIdx.x, j = blockIdx.y, h = j / G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  __shared__ __align__(16) float s_p[TAIL_MAX];                // tail scores, then probabilities
  __shared__ __align__(16) uint8_t s_vc[TAIL_MAX][HQ2B_ROW];  // tail V codes
  __shared__ __align__(16) uint32_t s_vm[TAIL_MAX][2];        // tail V meta (s0 z0, s1 z1)
  __shared__ __align__(16) float s_red[4][D];
  __shared__ float s_w[DEC_MAX_SLOTS];
  __shared__ float s_tail[2], s_fin[2];
  __shared__ int32_t s_phys[2];
  __shared__ int s_sum[2][8];

  // main pages of lanes before b, and of all lanes
  int before = 0, total = 0;
  for (int i = tid; i < a.lanes; i += blockDim.x) {
    const int n = main_pages(a, i);
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
  const int len = a.seq_len[b];
  const bool bad = lane_len_error(a, len) != 0;
  const int npg = bad ? 0 : main_pages(a, b);
  const int ef = bad ? 0 : exact_from(len, c.window, c.ktok);
  const int tail_start = npg * P;
  const int ntail = bad ? 0 : len - tail_start;
  // fused decode step: this step's token (position len - 1) may still be being appended while
  // this part runs, so the tail takes its key and value from the step inputs, never from the
  // ring or the page
  int st_start = 0, st_n = 0, st_off = 0;
  if (a.step.active && !bad) {
    st_start = a.step.start_pos[b];
    st_n = a.step.n_new[b];
    st_off = a.step.tok_offset[b];
    if (st_n < 0 || st_n > 1 || st_start < 0 || st_off < 0 || st_off + st_n > a.step.n_rows ||
        (st_n == 1 && st_start != len - 1) || (st_n == 0 && st_start != len)) {
      if (tid == 0 && j % G == 0) flag(c.status, KVQ_STATUS_BAD_LEN);
      st_n = 0;
    }
  }
  const int t_new = st_n ? st_start - tail_start : -1;   // tail index of the step token, or -1
  // the tail reads K codes of a page this step closes only for 0 < window < 64 (the close then
  // leaves keys below exact_from in that page): then wait for the step's append to be complete
  // (the main grid waits for it before it exits)
  if (st_n == 1 && (st_start + 1) % P == 0 && tail_start < ef) asm volatile("griddepcontrol.wait;\n" ::: "memory");
  if (tid < 2) {
    const int p = tail_start / P + tid;
    int32_t phys = -1;
    if (!bad && p * P < len) {
      phys = c.page_table[(int64_t)b * c.max_pages + p];
      if (phys < 0 || phys >= c.pool_pages) {
        if (j % G == 0) flag(c.status, KVQ_STATUS_PAGE_OOB);
        phys = -1;
      }
    }
    s_phys[tid] = phys;
  }
  __syncthreads();
  before = 0;
  total = 0;
#pragma unroll
  for (int w = 0; w < 8; w++) {
    before += s_sum[0][w];
    total += s_sum[1][w];
  }

  // ---- part 1a: tail V rows to shared memory (64 B codes + 8 B meta each)
  for (int i = tid; i < ntail * 4; i += blockDim.x) {
    const int t = i >> 2, pos = tail_start + t;
    if (t == t_new) continue;
    const int32_t phys = s_phys[pos / P - tail_start / P];
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (phys >= 0) {
      const uint8_t* vblk = c.pool + (int64_t)phys * c.page_bytes + block_offset(KVQ_FMT_HQ2B, H, c.layer, h, 1);
      w = reinterpret_cast<const uint4*>(vblk + (pos % P) * HQ2B_ROW)[i & 3];
      if ((i & 3) == 0) {
        const uint2 m = *reinterpret_cast<const uint2*>(vblk + HQ2B_META_OFF + (pos % P) * 8);
        s_vm[t][0] = m.x;
        s_vm[t][1] = m.y;
      }
    } else if ((i & 3) == 0) {
      s_vm[t][0] = s_vm[t][1] = 0u;
    }
    reinterpret_cast<uint4*>(s_vc[t])[i & 3] = w;
  }
  if (t_new >= 0 && warp == 0) {       // the step token's V row, quantized exactly as the append does
    const uint4 vx = reinterpret_cast<const uint4*>(a.step.v + ((int64_t)st_off * H + h) * D)[lane];
    uint32_t packed, meta;
    quant_v_row(vx, packed, meta);
    reinterpret_cast<uint16_t*>(s_vc[t_new])[lane] = (uint16_t)packed;
    if ((lane & 15) == 0) s_vm[t_new][lane >> 4] = meta;
  }
  // ---- part 1b: tail scores; warp w takes keys w, w + 8, ..., four at a time, lanes over dims
  float q[8], qc[8];   // q for keys from the ring; qc for keys from the codes (H q in the rotated format)
  {
    const uint4 w4 = reinterpret_cast<const uint4*>(a.q + ((int64_t)b * Hq + j) * D)[lane];
    const uint32_t u[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
      q[2 * i] = bf16_lo(u[i]) * a.scale_log2;
      q[2 * i + 1] = bf16_hi(u[i]) * a.scale_log2;
    }
    if (c.rotated) {
      const uint4 r4 = reinterpret_cast<const uint4*>(a.q_rot + ((int64_t)b * Hq + j) * D)[lane];
      const uint32_t ru[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
      for (int i = 0; i < 4; i++) {
        qc[2 * i] = half_bits_to_float((uint16_t)(ru[i] & 0xFFFFu)) * a.scale_log2;
        qc[2 * i + 1] = half_bits_to_float((uint16_t)(ru[i] >> 16)) * a.scale_log2;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; i++) qc[i] = q[i];
    }
  }
  // K channel scales of the closed page the tail starts in (dims 8 lane .. 8 lane + 7); in the
  // per-token-K format each code key brings its own (s, z) instead
  float ks[8];
  const uint8_t* kblk0 = nullptr;
  {
    uint4 sw = make_uint4(0u, 0u, 0u, 0u);
    if (tail_start < ef && s_phys[0] >= 0) {
      kblk0 = c.pool + (int64_t)s_phys[0] * c.page_bytes + block_offset(KVQ_FMT_HQ2B, H, c.layer, h, 0);
      if (!c.ktok) sw = reinterpret_cast<const uint4*>(kblk0 + HQ2B_META_OFF)[lane];
    }
    const __half2* sc = reinterpret_cast<const __half2*>(&sw);
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const float2 f = __half22float2(sc[i]);
      ks[2 * i] = f.x;
      ks[2 * i + 1] = f.y;
    }
  }
  for (int t0 = warp; t0 < ntail; t0 += 32) {
    float dot[4];
    uint4 kw[4];
#pragma unroll
    for (int u = 0; u < 4; u++) {             // loads of four keys in flight
      const int t = t0 + 8 * u, pos = tail_start + t;
      kw[u] = make_uint4(0u, 0u, 0u, 0u);
      if (t < ntail) {
        if (t == t_new && pos >= ef)   // (below exact_from it is read from the codes, like any key)
          kw[u] = reinterpret_cast<const uint4*>(a.step.k + ((int64_t)st_off * H + h) * D)[lane];
        else if (pos >= ef)
          kw[u] = reinterpret_cast<const uint4*>(c.ring + ring_row_offset(c, b, h, pos % P))[lane];
        else if (kblk0) {
          kw[u].x = reinterpret_cast<const uint16_t*>(kblk0 + (pos % P) * HQ2B_ROW)[lane];
          if (c.ktok) kw[u].y = reinterpret_cast<const uint32_t*>(kblk0 + HQ2B_META_OFF + (pos % P) * 8)[lane >> 4];
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const int pos = tail_start + t0 + 8 * u;
      float kx[8];
      if (pos >= ef) {
        const uint32_t w[4] = {kw[u].x, kw[u].y, kw[u].z, kw[u].w};
#pragma unroll
        for (int i = 0; i < 4; i++) {
          kx[2 * i] = bf16_lo(w[i]);
          kx[2 * i + 1] = bf16_hi(w[i]);
        }
      } else if (c.ktok) {
        const float sk = half_bits_to_float((uint16_t)(kw[u].y & 0xFFFFu));
        const float zk = half_bits_to_float((uint16_t)(kw[u].y >> 16));
#pragma unroll
        for (int i = 0; i < 8; i++) kx[i] = zk + (float)((kw[u].x >> (2 * i)) & 3u) * sk;
      } else {
#pragma unroll
        for (int i = 0; i < 8; i++) kx[i] = ks[i] * (float)(2 * (int)((kw[u].x >> (2 * i)) & 3u) - 3);
      }
      float d = 0.f;
#pragma unroll
      for (int i = 0; i < 8; i++) d = fmaf(pos >= ef ? q[i] : qc[i], kx[i], d);
      dot[u] = d;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
      for (int u = 0; u < 4; u++) dot[u] += __shfl_xor_sync(0xFFFFFFFFu, dot[u], o);
    if (lane < 4 && t0 + 8 * lane < ntail) {
      float v = dot[0];
#pragma unroll
      for (int u = 1; u < 4; u++) v = lane == u ? dot[u] : v;
      s_p[t0 + 8 * lane] = v;
    }
  }
  __syncthreads();
  // ---- part 1c: tail softmax (log2 domain), warp 0
  if (warp == 0) {
    float x[TAIL_MAX / 32];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < TAIL_MAX / 32; i++) {
      const int t = lane + 32 * i;
      x[i] = t < ntail ? s_p[t] : -INFINITY;
      m = fmaxf(m, x[i]);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    float l = 0.f;
#pragma unroll
    for (int i = 0; i < TAIL_MAX / 32; i++) {
      const float p = x[i] == -INFINITY ? 0.f : exp2f(x[i] - m);
      s_p[lane + 32 * i] = p;
      l += p;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, o);
    if (lane == 0) {
      s_tail[0] = m;
      s_tail[1] = l;
    }
  }
  __syncthreads();
  // ---- part 1d: tail P.V, thread = dim
  const int d = tid;
  float acc = 0.f;
  {
    const int hf = d >> 7, shift = 2 * (d & 3), byte = d >> 2;
#pragma unroll 8
    for (int t = 0; t < ntail; t++) {
      const uint32_t mw = s_vm[t][hf];
      const float sv = half_bits_to_float((uint16_t)(mw & 0xFFFFu));
      const float zv = half_bits_to_float((uint16_t)(mw >> 16));
      acc = fmaf(s_p[t], fmaf((float)((s_vc[t][byte] >> shift) & 3u), sv, zv), acc);
    }
  }

  // ---- part 2: the main partials are complete once the main grid is
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  int nk = 0;
  if (npg > 0) {
    const int units = H * total;
    const int Wp = units_per_warp(units, a.grid_warps, a.min_wp);
    const int segstart = H * before + h * npg;
    nk = (segstart + npg - 1) / Wp - segstart / Wp + 1;
  }
  const int64_t pbase = ((int64_t)b * Hq + j) * a.max_splits;
  // partial k goes to thread group k % 4; each thread sums 4 dims of its group's partials.  The
  // partials were written by the main grid moments ago and sit in L2, so the merge is
  // latency-bound: the loads of the first COMB_PRE partials of every group go out before warp 0
  // reads the (m, l) pairs, and the weights meet them after one round trip
  constexpr int COMB_PRE = 12;
  const int dq = tid & 63, kg = tid >> 6;
  const float4* part = reinterpret_cast<const float4*>(a.ws_o + pbase * D) + dq;
  float4 v0[COMB_PRE];
#pragma unroll
  for (int u = 0; u < COMB_PRE; u++) {
    const int k = kg + 4 * u;
    v0[u] = k < nk ? part[(int64_t)k * (D / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (warp == 0) {
    const float2* ml = reinterpret_cast<const float2*>(a.ws_ml) + pbase;
    float mk[DEC_MAX_SLOTS / 32], lk[DEC_MAX_SLOTS / 32];
    float M = s_tail[0];
#pragma unroll
    for (int i = 0; i < DEC_MAX_SLOTS / 32; i++) {
      const int k = lane + 32 * i;
      mk[i] = -INFINITY;
      lk[i] = 0.f;
      if (k < nk) {
        const float2 e = ml[k];
        mk[i] = e.x;
        lk[i] = e.y;
      }
      M = fmaxf(M, mk[i]);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
    float den = 0.f;
#pragma unroll
    for (int i = 0; i < DEC_MAX_SLOTS / 32; i++) {
      const int k = lane + 32 * i;
      const float w = mk[i] == -INFINITY ? 0.f : exp2f(mk[i] - M);
      if (k < nk) s_w[k] = w;
      den = fmaf(lk[i], w, den);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) den += __shfl_xor_sync(0xFFFFFFFFu, den, o);
    if (lane == 0) {
      const float wt = s_tail[0] == -INFINITY ? 0.f : exp2f(s_tail[0] - M);
      s_fin[0] = wt;
      s_fin[1] = fmaf(s_tail[1], wt, den);
    }
  }
  __syncthreads();
  {
    float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < COMB_PRE; u++) {
      const int k = kg + 4 * u;
      const float w = k < nk ? s_w[k] : 0.f;
      s4.x = fmaf(v0[u].x, w, s4.x);
      s4.y = fmaf(v0[u].y, w, s4.y);
      s4.z = fmaf(v0[u].z, w, s4.z);
      s4.w = fmaf(v0[u].w, w, s4.w);
    }
    for (int k0 = kg + 4 * COMB_PRE; k0 < nk; k0 += 32) {   // the rest, eight loads in flight at a time
      float4 v[8];
      float w[8];
#pragma unroll
      for (int u = 0; u < 8; u++) {
        const int k = k0 + 4 * u;
        v[u] = k < nk ? part[(int64_t)k * (D / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
        w[u] = k < nk ? s_w[k] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 8; u++) {
        s4.x = fmaf(v[u].x, w[u], s4.x);
        s4.y = fmaf(v[u].y, w[u], s4.y);
        s4.z = fmaf(v[u].z, w[u], s4.z);
        s4.w = fmaf(v[u].w, w[u], s4.w);
      }
    }
    reinterpret_cast<float4*>(s_red[kg])[dq] = s4;
  }
  __syncthreads();
  const float num = fmaf(acc, s_fin[0], s_red[0][d] + s_red[1][d] + s_red[2][d] + s_red[3][d]);
  const float den = s_fin[1];
  const float o = den > 0.f ? num / den : 0.f;
  if (!c.rotated) {
    a.out[((int64_t)b * Hq + j) * D + d] = o;
  } else {
    // the pages hold H v: the merged output is H o, and H H = I turns it back
    __syncthreads();
    s_red[0][d] = o;
    __syncthreads();
    if (warp == 0) {
      float x[8];
#pragma unroll
      for (int i = 0; i < 8; i++) x[i] = s_red[0][8 * lane + i];
      warp_fwht256(x);
      float4* dst = reinterpret_cast<float4*>(a.out + ((int64_t)b * Hq + j) * D + 8 * lane);
      dst[0] = make_float4(x[0], x[1], x[2], x[3]);
      dst[1] = make_float4(x[4], x[5], x[6], x[7]);
    }
  }
}

// ----------------------------------------------------------------------------- rotated query
// Rotated format: H q of every (lane, query head) in fp16, one warp per row.
__global__ void __launch_bounds__(256) rotate_q_kernel(AttnArgs a) {
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= a.lanes * a.c.num_q_heads) return;
  const uint4 w4 = reinterpret_cast<const uint4*>(a.q + (int64_t)row * D)[lane];
  const uint32_t u[4] = {w4.x, w4.y, w4.z, w4.w};
  float x[8];
#pragma unroll
  for (int i = 0; i < 4; i++) {
    x[2 * i] = bf16_lo(u[i]);
    x[2 * i + 1] = bf16_hi(u[i]);
  }
  warp_fwht256(x);
  uint4 o;
  o.x = pack_h2(x[0], x[1]);
  o.y = pack_h2(x[2], x[3]);
  o.z = pack_h2(x[4], x[5]);
  o.w = pack_h2(x[6], x[7]);
  reinterpret_cast<uint4*>(a.q_rot + (int64_t)row * D)[lane] = o;
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
  a.grid_warps = grid * DEC_PAIRS;     // work is split over warp pairs
  a.min_wp = decode_hq2b_min_wp(a.max_seq_len);
  const size_t fixed = (size_t)DEC_PAIRS * PAIR_BYTES + DEC_PAIRS * PB_COUNT * 8;
  const size_t smem = fixed + (size_t)(2 * a.lanes + 1) * sizeof(int);
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!attr_set[dev]) {
    const int max_smem = (int)(fixed + (2 * MAX_LANES_FAST + 1) * sizeof(int));
    cudaFuncSetAttribute(decode_hq2b_main<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    cudaFuncSetAttribute(decode_hq2b_main<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    cudaFuncSetAttribute(decode_hq2b_main<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    attr_set[dev] = true;
  }
  // the rotated format takes the centred value codes (see the A-operand notes above)
  // and the per-token-K format its own Q.K^T step
  void (*const main_kernel)(AttnArgs) = a.c.rotated ? decode_hq2b_main<true, false>
                                        : a.c.ktok   ? decode_hq2b_main<false, true>
                                                     : decode_hq2b_main<false, false>;
  if (a.c.rotated) {
    const int rows = a.lanes * a.c.num_q_heads;
    rotate_q_kernel<<<(rows + 7) / 8, 256, 0, stream>>>(a);
  }
  if (a.step.active && !a.step.append_last) {
    // fused decode step: overlap the append kernel launched just before
    cudaLaunchConfig_t mc = {};
    mc.gridDim = dim3(grid);
    mc.blockDim = dim3(DEC_PAIRS * 64);
    mc.dynamicSmemBytes = smem;
    mc.stream = stream;
    cudaLaunchAttribute mattr[1];
    mattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    mattr[0].val.programmaticStreamSerializationAllowed = 1;
    mc.attrs = mattr;
    mc.numAttrs = 1;
    if (cudaLaunchKernelEx(&mc, main_kernel, a) != cudaSuccess) return KVQ_ERR_CUDA;
  } else {
    main_kernel<<<grid, DEC_PAIRS * 64, smem, stream>>>(a);
  }
  // the combine may start while the main grid drains; it waits for it before reading partials
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.lanes, a.c.num_q_heads);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, decode_hq2b_combine, a) != cudaSuccess) return KVQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq

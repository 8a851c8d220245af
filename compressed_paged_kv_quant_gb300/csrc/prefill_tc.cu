// prefill_tc.cu -- chunked-prefill attention over the 2-bit pages on the 5th-generation
// tensor cores (tcgen05, TMEM accumulators), sm_103a.
//
// "KV at 9 KB a token" ("How it works"): since 0.7.3 prefill attention reads the compressed
// cache directly -- no decompressed copy of the prompt exists in HBM.  Here each 64-token page
// is dequantised once into shared memory, where it feeds the MMAs of 128 query rows.  The
// split partials are written before they are read, so the workspace is never zeroed ("One
// cleanup came free with the format").
//
// CTA = up to 128 rows of (query, head) pairs of one GQA group (row = qi * G + g) x one key
// split of `split_tokens` keys.
//   TMEM (512 columns):  Q [0,128) as fp16 pairs (A operand of S = Q K^T);
//                        S/P double buffer [128,192) [192,256): S lands in fp32, P is written
//                        back over its first 32 columns as fp16 pairs (A operand of O += P V);
//                        O [256,512) fp32 accumulator of the split.
//   Shared memory:       K tile x2 (64 keys x 256 dims fp16, 128B-swizzled, K-major B of S),
//                        V tile x2 (the same [key][dim] layout, read as the MN-major B of PV),
//                        compressed-page staging x PT_NSTG (one 9,216 B TMA bulk copy per page).
//   Warps 0-3: softmax, one row per thread (= TMEM lane): S from TMEM, causal mask, online
//              max with lazy O rescale (only when a row max grows by more than 2^8), P to
//              TMEM, l in FP32; the epilogue writes (m, l, O) of the split.
//   Warps 4-10: page TMA (one elected thread) and dequantisation into the swizzled tiles.
//   Warp 11:   one thread issues every tcgen05.mma (S(j+1) ahead of PV(j)) and commits
//              their completion to mbarriers.
// Every mbarrier wait is bounded; on a timeout the CTA flags KVQ_STATUS_TIMEOUT, stops, waits
// (bounded) for its copies and MMAs in flight, and still releases its TMEM.
#include "kvq_internal.cuh"
#include "attn_args.cuh"

namespace kvq {

constexpr int PT_ROWS = 128;
constexpr int PT_DQ_WARPS = 7;                    // TMA + dequantisation warps (12 warps: <= 168 regs)
constexpr int PT_MMA_WARP = 4 + PT_DQ_WARPS;      // the warp whose lane 0 issues the MMAs
constexpr int PT_THREADS = (PT_MMA_WARP + 1) * 32;
constexpr int SM_K = 0;                   // 2 K tile buffers
constexpr int PT_MAX_TILES = PREFILL_SPLIT / P;   // 64-key tiles of one split (a CTA's keys)

// Per page format.  The staging ring holds a page's K and V blocks of one (layer, head) as one
// bulk copy a stage: 9,216 B for the 2-bit layouts (6 stages), 32 KB for FP8 (2 stages).  Two
// formats keep the K tile as two fp16 parts (hi, lo), 64 KB a buffer (3 stages): the per-token-K
// format (its keys z + c s sit on a grid set by the token's largest values, too coarse for one
// fp16) and the rotated format (its keys are turned back by H in the dequantisation, so every
// element is a sum that one fp16 would round).  The rotated format turns its value rows back
// as well, so q and the output stay in the original basis.
template <int FMT>
struct PfLayout {
  static constexpr int LFMT = FMT == KVQ_FMT_FP8 ? KVQ_FMT_FP8 : KVQ_FMT_HQ2B;   // byte layout
  static constexpr bool KSPLIT = FMT == KVQ_FMT_HQ2B_TOK || FMT == KVQ_FMT_HQ2B_HAD;
  static constexpr int K_BUF = KSPLIT ? 65536 : 32768;   // one K tile buffer (hi, then lo)
  static constexpr int V_BUF = 32768;                     // one V tile buffer
  static constexpr int SM_V = 2 * K_BUF;
  static constexpr int SM_STG = SM_V + 2 * V_BUF;
  static constexpr int STAGE = 2 * block_bytes(LFMT);
  static constexpr int NSTG = LFMT == KVQ_FMT_FP8 ? 2 : KSPLIT ? 3 : 6;
  static constexpr int SM_BAR = SM_STG + NSTG * STAGE;
  static constexpr int NUM_BARS = 13 + 2 * NSTG;
  static constexpr int SM_ABORT = SM_BAR + NUM_BARS * 8;
  static constexpr int SM_TMEM = SM_ABORT + 4;
  static constexpr int SM_PAGES = SM_TMEM + 16;       // the CTA's page ids, PT_MAX_TILES int32
  static constexpr int SMEM = SM_PAGES + 4 * PT_MAX_TILES + 1024;   // + slack to align the base to 1,024 B
};
constexpr int TM_Q = 0, TM_S0 = 128, TM_O = 256;
constexpr int PT_SPIN = 1 << 16;
constexpr float RESCALE_LOG2 = 8.0f;

enum {
  B_K_FULL = 0, B_K_EMPTY = 2, B_V_FULL = 4, B_S_FULL = 6, B_P_FULL = 8, B_PV_DONE = 10, B_Q_READY = 12,
  B_STG_FULL = 13   // then NSTG "full" and NSTG "empty" barriers of the staging ring
};

__device__ __forceinline__ uint32_t sm_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void bar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity) {
  for (int i = 0; i < PT_SPIN; i++) {
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

// ---------------------------------------------------------------------------- tcgen05 wrappers
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

// D(tmem) (+)= A(tmem) . B(smem descriptor)^T
__device__ __forceinline__ void tc_mma_ts(uint32_t d, uint32_t a, uint64_t b_desc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a), "l"(b_desc), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar) : "memory");
}

#define TC_LD32(taddr, r)                                                                                        \
  asm volatile(                                                                                                  \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"   \
      "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"                                       \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),           \
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),     \
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),   \
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])    \
      : "r"(taddr))

#define TC_ST32(taddr, r)                                                                                        \
  asm volatile(                                                                                                  \
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"    \
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),                       \
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),         \
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), \
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]),            \
      "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])                                      \
      : "memory")

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
// Registers written by tcgen05.ld hold their values only after tcgen05.wait::ld: after the wait,
// each passes through an empty volatile asm, so that no read of it is scheduled above the wait.
template <int N>
__device__ __forceinline__ void tc_regs_ready(uint32_t* r) {
#pragma unroll
  for (int i = 0; i < N; i++) asm volatile("" : "+r"(r[i]));
}
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

// shared-memory matrix descriptor: 128B swizzle, K-major, 8-row groups 1,024 B apart
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;             // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;   // stride byte offset
  d |= (uint64_t)1 << 46;             // descriptor version of the sm_100 family
  d |= (uint64_t)2 << 61;             // 128-byte swizzle
  return d;
}

// shared-memory matrix descriptor: 128B swizzle, MN-major (the N index runs along the 128 B rows):
// 64-element N blocks `lbo` bytes apart, 8-row K groups `sbo` bytes apart
constexpr uint32_t PV_LBO = 8192, PV_SBO = 1024;
__device__ __forceinline__ uint64_t sw128_mn_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(PV_LBO >> 4) << 16;
  d |= (uint64_t)(PV_SBO >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// instruction descriptor: D f32, A f16, B f16, A K-major, B K-major (or MN-major), M x N
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool b_mn_major = false) {
  return (1u << 4) | (b_mn_major ? (1u << 16) : 0u) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// byte offset of 16 B chunk `chunk` (0..7) of `row` in a 128B-swizzled region (1,024 B atoms)
__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t chunk) {
  return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

__device__ __forceinline__ float ex2f(float x) {  // 2^x, one MUFU.EX2
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// Blackwell's three-input max and paired FP32 arithmetic (two lanes of one 64-bit register, each
// an IEEE operation): half the softmax's max, FMA and add instructions
__device__ __forceinline__ float fmax3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;\n" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2(float a, float b) {
  uint64_t p;
  asm("mov.b64 %0, {%1, %2};\n" : "=l"(p) : "f"(a), "f"(b));
  return p;
}
__device__ __forceinline__ void f2split(uint64_t p, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;\n" : "=f"(a), "=f"(b) : "l"(p));
}
__device__ __forceinline__ uint64_t fma_f2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;\n" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add_f2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;\n" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ uint32_t h2u(__half2 x) { return *reinterpret_cast<uint32_t*>(&x); }
__device__ __forceinline__ __half2 u2h(uint32_t x) { return *reinterpret_cast<__half2*>(&x); }

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];\n" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t ld_shared_u8(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u8 %0, [%1];\n" : "=h"(v) : "r"(addr));
  return v;
}

// Two code bytes (dims 4k + j of byte k at bits 2j) -> four fp16 pairs holding 4 + c for dims
// (0,1), (2,3), (4,5), (6,7): each multiply spreads a byte to two places (no overlap, so it is an
// OR), the mask keeps one code per half at mantissa bits 8-9, the exponent of 4 makes it 4 + c.
__device__ __forceinline__ void dq_pairs(uint32_t lo, uint32_t hi, uint32_t (&x)[4]) {
  x[0] = ((lo * 0x00400100u) & 0x03000300u) | 0x44004400u;
  x[1] = ((lo * 0x00040010u) & 0x03000300u) | 0x44004400u;
  x[2] = ((hi * 0x00400100u) & 0x03000300u) | 0x44004400u;
  x[3] = ((hi * 0x00040010u) & 0x03000300u) | 0x44004400u;
}

// two E4M3 bytes (low 16 bits) -> fp16 pair, exact
__device__ __forceinline__ uint32_t e4m3x2_h2(uint32_t x) {
  uint32_t y;
  asm("{\n .reg .b16 t;\n cvt.u16.u32 t, %1;\n cvt.rn.f16x2.e4m3x2 %0, t;\n}\n" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// ---------------------------------------------------------------------------- kernel
// grid (splits, ceil(max_n_q / QT), lanes * H); PT_THREADS threads; PfLayout<FMT>::SMEM dynamic smem
template <int FMT>
__global__ void __launch_bounds__(PT_THREADS, 1) prefill_tc(AttnArgs a) {
  using LY = PfLayout<FMT>;
  constexpr int PT_STAGE = LY::STAGE, PT_NSTG = LY::NSTG;
  constexpr int B_STG_EMPTY = B_STG_FULL + PT_NSTG;
  constexpr bool FP8 = LY::LFMT == KVQ_FMT_FP8;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const CacheView& c = a.c;
  const int H = c.num_kv_heads, G = c.group, Hq = c.num_q_heads;
  const int QT = PT_ROWS / G;
  const int b = blockIdx.z / H, h = blockIdx.z % H, qt = blockIdx.y, s = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- rows and keys of this CTA (uniform: early exits happen before any barrier)
  const int len = a.seq_len[b];
  const int nq = a.n_q[b], qoff = a.q_offset[b], qpos0 = a.q_pos0[b];
  if (lane_len_error(a, len) || nq < 0 || nq > a.max_n_q || qoff < 0 || (int64_t)qoff + nq > a.n_q_rows ||
      qpos0 < 0 || (int64_t)qpos0 + nq > len) {
    if (threadIdx.x == 0 && s == 0 && qt == 0 && h == 0) flag(c.status, KVQ_STATUS_BAD_LEN);
    return;
  }
  const int q_first = qt * QT;
  if (q_first >= nq) return;
  const int q_last = min(nq, q_first + QT) - 1;
  const int kmax = qpos0 + q_last + 1;
  const int k0 = s * a.split_tokens;
  if (k0 >= kmax) return;
  const int k1 = min(k0 + a.split_tokens, kmax);
  const int p0 = k0 / P;
  const int ntiles = (k1 + P - 1) / P - p0;
  // first key read exact from the ring (FP8 pages have no ring: every key from its page)
  const int ef = FP8 ? len : exact_from(len, c.window, c.ktok);

  uint8_t* smem = smem_raw + ((1024u - (sm_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + LY::SM_BAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + LY::SM_ABORT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + LY::SM_TMEM);
  auto BAR = [&](int i) { return sm_u32(&bars[i]); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < PT_NSTG; i++) {
      bar_init(BAR(B_STG_FULL + i), 1);
      bar_init(BAR(B_STG_EMPTY + i), PT_DQ_WARPS);
    }
    for (int i = 0; i < 2; i++) {
      bar_init(BAR(B_K_FULL + i), PT_DQ_WARPS);
      bar_init(BAR(B_K_EMPTY + i), 1);
      bar_init(BAR(B_V_FULL + i), PT_DQ_WARPS);
      bar_init(BAR(B_S_FULL + i), 1);
      bar_init(BAR(B_P_FULL + i), 4);
      bar_init(BAR(B_PV_DONE + i), 1);
    }
    bar_init(BAR(B_Q_READY), 4);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(sm_u32(tmem_slot)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool timed_out = false;

  if (warp < 4) {
    // =============================================================== softmax warps
    const int row = 32 * warp + lane;
    const int qi = row / G, g = row - (row / G) * G;
    const bool row_valid = row < QT * G && q_first + qi < nq;
    const int qpos = qpos0 + q_first + qi;
    const uint32_t tl = tmem + ((uint32_t)(32 * warp) << 16);
    // softmax scale (log2 domain); FP8 pages: times the K scale, E4M3 values being unscaled in the tile
    const float sl2 = FP8 ? a.scale_log2 * c.k_scale : a.scale_log2;
    // Q row -> TMEM columns [0,128) as fp16 pairs
    for (int ch = 0; ch < 4; ch++) {
      uint32_t r[32];
      if (row_valid) {
        const uint4* src =
            reinterpret_cast<const uint4*>(a.q + ((int64_t)(qoff + q_first + qi) * Hq + h * G + g) * D + 64 * ch);
#pragma unroll
        for (int i = 0; i < 8; i++) {
          const uint4 w = src[i];
          r[4 * i + 0] = h2u(__floats2half2_rn(bf16_lo(w.x), bf16_hi(w.x)));
          r[4 * i + 1] = h2u(__floats2half2_rn(bf16_lo(w.y), bf16_hi(w.y)));
          r[4 * i + 2] = h2u(__floats2half2_rn(bf16_lo(w.z), bf16_hi(w.z)));
          r[4 * i + 3] = h2u(__floats2half2_rn(bf16_lo(w.w), bf16_hi(w.w)));
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; i++) r[i] = 0u;
      }
      TC_ST32(tl + TM_Q + 32 * ch, r);
    }
    tc_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) bar_arrive(BAR(B_Q_READY));

    float m_run = -INFINITY, l_run = 0.f;
    for (int j = 0; j < ntiles; j++) {
      const int buf = j & 1;
      const uint32_t par = (j >> 1) & 1;
      if (__any_sync(0xFFFFFFFFu, *abort_flag != 0)) { timed_out = true; break; }
      if (!__all_sync(0xFFFFFFFFu, bar_wait(BAR(B_S_FULL + buf), par))) { timed_out = true; break; }
      tc_fence_after();
      uint32_t sv[64];
      TC_LD32(tl + TM_S0 + 64 * buf, sv);
      TC_LD32(tl + TM_S0 + 64 * buf + 32, (sv + 32));
      tc_wait_ld();
      tc_regs_ready<64>(sv);
      const int key0 = (p0 + j) * P;
      // a tile entirely below the causal diagonal of every row of the CTA needs no mask (rows
      // past the last query hold Q = 0 and are never written)
      const bool full = key0 + P - 1 <= qpos0 + q_first;
      // row max and (below) row sum as independent chains (the softmax sits between S and P.V on
      // the tensor pipe, so its latency matters), on three-input max and paired FP32 operations
      // (the warps share their SM sub-partitions' issue slots with the dequantisation)
      float t4[4];
#pragma unroll
      for (int i = 0; i < 4; i++) t4[i] = -INFINITY;
      if (full) {
#pragma unroll
        for (int cidx = 0; cidx < 64; cidx += 2)
          t4[(cidx >> 1) & 3] = fmax3f(t4[(cidx >> 1) & 3], __uint_as_float(sv[cidx]), __uint_as_float(sv[cidx + 1]));
      } else {
#pragma unroll
        for (int cidx = 0; cidx < 64; cidx += 2) {
          const bool ok0 = row_valid && key0 + cidx <= qpos, ok1 = row_valid && key0 + cidx + 1 <= qpos;
          const float x0 = ok0 ? __uint_as_float(sv[cidx]) * sl2 : -INFINITY;
          const float x1 = ok1 ? __uint_as_float(sv[cidx + 1]) * sl2 : -INFINITY;
          sv[cidx] = __float_as_uint(x0);
          sv[cidx + 1] = __float_as_uint(x1);
          t4[(cidx >> 1) & 3] = fmax3f(t4[(cidx >> 1) & 3], x0, x1);
        }
      }
      float tmax = fmaxf(fmax3f(t4[0], t4[1], t4[2]), t4[3]);
      if (full) tmax *= sl2;
      const float m_new = fmaxf(m_run, tmax);
      const bool first = (j == 0) || (m_run == -INFINITY);
      const bool need = !first && (m_new > m_run + RESCALE_LOG2);
      if (__any_sync(0xFFFFFFFFu, need)) {
        // O must be stable: PV(j-1) complete
        if (!__all_sync(0xFFFFFFFFu, bar_wait(BAR(B_PV_DONE + ((j - 1) & 1)), ((j - 1) >> 1) & 1))) {
          timed_out = true;
          break;
        }
        tc_fence_after();
        const float alpha = need ? ex2f(m_run - m_new) : 1.0f;
        for (int ch = 0; ch < 8; ch++) {
          uint32_t o[32];
          TC_LD32(tl + TM_O + 32 * ch, o);
          tc_wait_ld();
          tc_regs_ready<32>(o);
#pragma unroll
          for (int i = 0; i < 32; i++) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          TC_ST32(tl + TM_O + 32 * ch, o);
        }
        tc_wait_st();
        if (need) {
          l_run *= alpha;
          m_run = m_new;
        }
      }
      if (first) m_run = m_new;
      const float m_use = m_run == -INFINITY ? 0.f : m_run;
      uint32_t pr[32];
      uint64_t ps2[4];   // row sum: 4 chains of key pairs
#pragma unroll
      for (int i = 0; i < 4; i++) ps2[i] = 0ull;   // (+0, +0)
      {
        // 2^(x sc - m) for the pair of keys 2i, 2i + 1; masked keys hold -inf (2^-inf = 0)
        const uint64_t sc2 = full ? f2(sl2, sl2) : f2(1.0f, 1.0f), nm2 = f2(-m_use, -m_use);
#pragma unroll
        for (int i = 0; i < 32; i++) {
          float a0, a1;
          f2split(fma_f2(f2(__uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1])), sc2, nm2), a0, a1);
          const float e0 = ex2f(a0), e1 = ex2f(a1);
          ps2[i & 3] = add_f2(ps2[i & 3], f2(e0, e1));
          pr[i] = h2u(__floats2half2_rn(e0, e1));
        }
      }
      {
        float q[8];
#pragma unroll
        for (int i = 0; i < 4; i++) f2split(ps2[i], q[2 * i], q[2 * i + 1]);
        l_run += ((q[0] + q[1]) + (q[2] + q[3])) + ((q[4] + q[5]) + (q[6] + q[7]));
      }
      TC_ST32(tl + TM_S0 + 64 * buf, pr);
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) bar_arrive(BAR(B_P_FULL + buf));
    }
    // ---- epilogue: (m, l, O) of this split
    if (!timed_out && ntiles > 0) {
      const int jl = ntiles - 1;
      if (!__all_sync(0xFFFFFFFFu, bar_wait(BAR(B_PV_DONE + (jl & 1)), (jl >> 1) & 1))) timed_out = true;
    }
    if (!timed_out) {
      tc_fence_after();
      const int64_t pidx = ((int64_t)(qoff + q_first + qi) * Hq + h * G + g) * a.max_splits + s;
      const float vsc = FP8 ? c.v_scale : 1.0f;   // FP8 pages: the V scale, E4M3 values being unscaled
      for (int ch = 0; ch < 8; ch++) {
        uint32_t o[32];
        TC_LD32(tl + TM_O + 32 * ch, o);
        tc_wait_ld();
        tc_regs_ready<32>(o);
        if (row_valid) {
          float4* dst = reinterpret_cast<float4*>(a.ws_o + pidx * D + 32 * ch);
#pragma unroll
          for (int i = 0; i < 8; i++)
            dst[i] = make_float4(__uint_as_float(o[4 * i]) * vsc, __uint_as_float(o[4 * i + 1]) * vsc,
                                 __uint_as_float(o[4 * i + 2]) * vsc, __uint_as_float(o[4 * i + 3]) * vsc);
        }
      }
      if (row_valid) reinterpret_cast<float2*>(a.ws_ml)[pidx] = make_float2(m_run, l_run);
    }
  } else if (warp < PT_MMA_WARP) {
    // =============================================================== TMA + dequant warps
    const int tid = threadIdx.x - 128;             // 0 .. 32 * PT_DQ_WARPS - 1
    constexpr int DQ_T = 32 * PT_DQ_WARPS;
    const int64_t lane_row = (int64_t)b * c.max_pages;
    // the page ids of the CTA's tiles, read once into shared memory by the copier's warp (the
    // copies then wait on no global load)
    int32_t* s_pages = reinterpret_cast<int32_t*>(smem + LY::SM_PAGES);
    auto issue = [&](int j) -> bool {
      const int buf = j % PT_NSTG;
      if (!bar_wait(BAR(B_STG_EMPTY + buf), ((j / PT_NSTG) & 1) ^ 1)) return false;
      const int32_t phys = s_pages[j];
      if (phys < 0 || phys >= c.pool_pages) {
        flag(c.status, KVQ_STATUS_PAGE_OOB);
        bar_arrive(BAR(B_STG_FULL + buf));
        return true;
      }
      const uint8_t* src = c.pool + (int64_t)phys * c.page_bytes + block_offset(LY::LFMT, H, c.layer, h, 0);
      const uint32_t dst = sm_u32(smem + LY::SM_STG + buf * PT_STAGE);
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(BAR(B_STG_FULL + buf)),
                   "r"((uint32_t)PT_STAGE)
                   : "memory");
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
          "l"(src), "r"((uint32_t)PT_STAGE), "r"(BAR(B_STG_FULL + buf))
          : "memory");
      return true;
    };
    if (tid < 32) {
      for (int jj = tid; jj < ntiles; jj += 32) s_pages[jj] = c.page_table[lane_row + p0 + jj];
      __syncwarp();
    }
    int issued = 0;
    if (tid == 0) {
      for (; issued < PT_NSTG && issued < ntiles; issued++)
        if (!issue(issued)) { timed_out = true; break; }
    }
    const __half2 two = __float2half2_rn(2.0f), m11 = __float2half2_rn(-11.0f);
    const __half2 one2 = __float2half2_rn(1.0f), m4 = __float2half2_rn(-4.0f);
    // Item = (key t, chunk cc = dims 8cc .. 8cc+7); DQ_T is a multiple of 32, so a thread keeps
    // its chunk for the whole tile and walks keys t0, t0 + KSTEP, ...  Both tiles are stored
    // [dim block cc/8][key t][chunk cc%8 ^ t%8]: a warp writes one key row, 512 contiguous
    // bytes of swizzled chunks, free of bank conflicts.
    const int cc = tid & 31, t0 = tid >> 5;
    constexpr int KSTEP = DQ_T / 32;
    constexpr int DQ_MAXI = (P + KSTEP - 1) / KSTEP;   // keys a thread takes of a tile, at most
    constexpr bool DQ_BATCH = FMT != KVQ_FMT_HQ2B_HAD;     // all of a tile's loads first
    const uint32_t tile_off = (uint32_t)(cc >> 3) * 8192u;
    for (int j = 0; j < ntiles && !timed_out; j++) {
      const int buf = j & 1;
      const uint32_t par = (j >> 1) & 1;
      if (__any_sync(0xFFFFFFFFu, *abort_flag != 0)) { timed_out = true; break; }
      const int sbuf = j % PT_NSTG;
      if (!__all_sync(0xFFFFFFFFu, bar_wait(BAR(B_STG_FULL + sbuf), (j / PT_NSTG) & 1))) { timed_out = true; break; }
      const uint32_t stg = sm_u32(smem + LY::SM_STG + sbuf * PT_STAGE);
      const int key0 = (p0 + j) * P;
      // ---- K tile (B of S, K-major): k^ = s_d (2c - 3) (per channel), z + c s (per-token-K
      // format), the E4M3 value (FP8; its scale multiplies the scores); keys from the ring as
      // they are, turned by H in the rotated format (a warp holds one key row, 8 dims a lane)
      if (!__all_sync(0xFFFFFFFFu, bar_wait(BAR(B_K_EMPTY + buf), par ^ 1))) { timed_out = true; break; }
      const uint32_t kb = sm_u32(smem + SM_K + buf * LY::K_BUF) + tile_off;
      {
        uint32_t scs[4] = {0u, 0u, 0u, 0u};
        if constexpr (!FP8 && FMT != KVQ_FMT_HQ2B_TOK) {
          const uint4 sc = ld_shared_v4(stg + HQ2B_META_OFF + 16 * cc);
          scs[0] = sc.x; scs[1] = sc.y; scs[2] = sc.z; scs[3] = sc.w;
        }
        // The raw words of key t (dims 8cc .. 8cc + 7): ra, rb = its two code bytes (2-bit
        // layouts) or its two E4M3 words (FP8); rm = its metadata word (per-token-K format).
        auto key_raw = [&](int t, uint32_t& ra, uint32_t& rb, uint32_t& rm) {
          if constexpr (FP8) {
            ra = ld_shared_u32(stg + t * D + 8 * cc);
            rb = ld_shared_u32(stg + t * D + 8 * cc + 4);
          } else {
            ra = ld_shared_u8(stg + t * HQ2B_ROW + 2 * cc);
            rb = ld_shared_u8(stg + t * HQ2B_ROW + 2 * cc + 1);
            if constexpr (FMT == KVQ_FMT_HQ2B_TOK) rm = ld_shared_u32(stg + HQ2B_META_OFF + t * 8 + 4 * (cc >> 4));
          }
        };
        // raw words -> 4 fp16 pairs of k^ (plain 2-bit and FP8 layouts)
        auto key_code = [&](uint32_t ra, uint32_t rb) -> uint4 {
          uint32_t res[4];
          if constexpr (FP8) {
            res[0] = e4m3x2_h2(ra); res[1] = e4m3x2_h2(ra >> 16); res[2] = e4m3x2_h2(rb); res[3] = e4m3x2_h2(rb >> 16);
          } else {
            dq_pairs(ra, rb, res);
#pragma unroll
            for (int p = 0; p < 4; p++) res[p] = h2u(__hmul2(__hfma2(u2h(res[p]), two, m11), u2h(scs[p])));
          }
          return make_uint4(res[0], res[1], res[2], res[3]);
        };
        // per-token-K format: k^ = z + c s exactly in fp32 (one rounding at most), stored as the fp16
        // pair hi = fp16(k^), lo = fp16(k^ - hi), in the two halves of the K buffer
        // (rotated format: the key's rotated coordinates s_d (2c - 3) turned back by H, a warp per
        // key row, lane cc holding dims 8cc .. 8cc + 7)
        auto key_split = [&](uint32_t ra, uint32_t rb, uint32_t rm, uint4& hi, uint4& lo) {
          const uint32_t code = ra | (rb << 8);
          float v[8];
          if constexpr (FMT == KVQ_FMT_HQ2B_HAD) {
#pragma unroll
            for (int p = 0; p < 4; p++) {
              const float2 sp = __half22float2(u2h(scs[p]));
              v[2 * p] = sp.x * (float)(2 * (int)((code >> (4 * p)) & 3u) - 3);
              v[2 * p + 1] = sp.y * (float)(2 * (int)((code >> (4 * p + 2)) & 3u) - 3);
            }
            warp_fwht256(v);
          } else {
            const float sf = half_bits_to_float((uint16_t)(rm & 0xFFFFu)), zf = half_bits_to_float((uint16_t)(rm >> 16));
#pragma unroll
            for (int e = 0; e < 8; e++) v[e] = fmaf((float)((code >> (2 * e)) & 3u), sf, zf);
          }
          uint32_t h[4], l[4];
#pragma unroll
          for (int p = 0; p < 4; p++) {
            const __half2 hh = __floats2half2_rn(v[2 * p], v[2 * p + 1]);
            const float2 hf = __half22float2(hh);
            h[p] = h2u(hh);
            l[p] = h2u(__floats2half2_rn(v[2 * p] - hf.x, v[2 * p + 1] - hf.y));
          }
          hi = make_uint4(h[0], h[1], h[2], h[3]);
          lo = make_uint4(l[0], l[1], l[2], l[3]);
        };
        if (!DQ_BATCH && key0 + P <= ef) {
          // rotated format: a key row at a time (each row's transform is a long run of shuffles;
          // a loop unrolled over all of a thread's rows is too much code)
#pragma unroll 2
          for (int t = t0; t < P; t += KSTEP) {
            uint32_t ra = 0u, rb = 0u, rm = 0u;
            key_raw(t, ra, rb, rm);
            uint4 hi, lo;
            key_split(ra, rb, rm, hi, lo);
            st_shared_v4(kb + swz(t, cc & 7), hi);
            st_shared_v4(kb + 32768 + swz(t, cc & 7), lo);
          }
        } else if (key0 + P <= ef) {   // every key of the tile comes from the page (ef <= len)
          // every raw word of the thread's keys first (the loads overlap), then convert and store
          uint32_t ra[DQ_MAXI], rb[DQ_MAXI], rm[DQ_MAXI];
#pragma unroll
          for (int k = 0; k < DQ_MAXI; k++)
            if (t0 + KSTEP * k < P) key_raw(t0 + KSTEP * k, ra[k], rb[k], rm[k]);
#pragma unroll
          for (int k = 0; k < DQ_MAXI; k++) {
            const int t = t0 + KSTEP * k;
            if (t < P) {
              if constexpr (LY::KSPLIT) {
                uint4 hi, lo;
                key_split(ra[k], rb[k], rm[k], hi, lo);
                st_shared_v4(kb + swz(t, cc & 7), hi);
                st_shared_v4(kb + 32768 + swz(t, cc & 7), lo);
              } else {
                st_shared_v4(kb + swz(t, cc & 7), key_code(ra[k], rb[k]));
              }
            }
          }
        } else
#pragma unroll 4
        for (int t = t0; t < P; t += KSTEP) {
          const int kp = key0 + t;
          uint4 o = make_uint4(0u, 0u, 0u, 0u), olo = make_uint4(0u, 0u, 0u, 0u);
          if (kp < len) {
            if (kp >= ef) {
              const uint4 w = reinterpret_cast<const uint4*>(
                  c.ring + ((((int64_t)b * c.num_layers + c.layer) * H + h) * P + (kp % P)) * D)[cc];
              o.x = h2u(__floats2half2_rn(bf16_lo(w.x), bf16_hi(w.x)));
              o.y = h2u(__floats2half2_rn(bf16_lo(w.y), bf16_hi(w.y)));
              o.z = h2u(__floats2half2_rn(bf16_lo(w.z), bf16_hi(w.z)));
              o.w = h2u(__floats2half2_rn(bf16_lo(w.w), bf16_hi(w.w)));
            } else {
              uint32_t ra = 0u, rb = 0u, rm = 0u;
              key_raw(t, ra, rb, rm);
              if constexpr (LY::KSPLIT) key_split(ra, rb, rm, o, olo);
              else o = key_code(ra, rb);
            }
          }
          st_shared_v4(kb + swz(t, cc & 7), o);
          if constexpr (LY::KSPLIT) st_shared_v4(kb + 32768 + swz(t, cc & 7), olo);
        }
      }
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      __syncwarp();
      if (lane == 0) bar_arrive(BAR(B_K_FULL + buf));
      // ---- V tile (B of PV, MN-major): v^ = z + c s, one rounding, per token and 128-dim half
      if (!__all_sync(0xFFFFFFFFu, bar_wait(BAR(B_PV_DONE + buf), par ^ 1))) { timed_out = true; break; }
      const uint32_t vb = sm_u32(smem + LY::SM_V + buf * LY::V_BUF) + tile_off;
      const uint32_t vst = stg + block_bytes(LY::LFMT);
      const bool vall = key0 + P <= len;
      if constexpr (!DQ_BATCH) {
        // rotated format: v^ = H (z + c s), a row at a time (the transform is a long run of
        // shuffles): the rotated row dequantized in fp32, turned back by the warp
#pragma unroll 2
        for (int t = t0; t < P; t += KSTEP) {
          uint4 o = make_uint4(0u, 0u, 0u, 0u);
          if (vall || key0 + t < len) {   // (the same for the whole warp: one row a warp)
            const uint32_t meta = ld_shared_u32(vst + HQ2B_META_OFF + t * 8 + 4 * (cc >> 4));
            const uint32_t code =
                ld_shared_u8(vst + t * HQ2B_ROW + 2 * cc) | (ld_shared_u8(vst + t * HQ2B_ROW + 2 * cc + 1) << 8);
            const float sf = half_bits_to_float((uint16_t)(meta & 0xFFFFu));
            const float zf = half_bits_to_float((uint16_t)(meta >> 16));
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; e++) v[e] = fmaf((float)((code >> (2 * e)) & 3u), sf, zf);
            warp_fwht256(v);
            o = make_uint4(h2u(__floats2half2_rn(v[0], v[1])), h2u(__floats2half2_rn(v[2], v[3])),
                           h2u(__floats2half2_rn(v[4], v[5])), h2u(__floats2half2_rn(v[6], v[7])));
          }
          st_shared_v4(vb + swz(t, cc & 7), o);
        }
      } else {
        // raw words of the thread's value rows first (codes or E4M3 words, and the meta word),
        // then convert and store; rows past the sequence are stored as zeros (only the last
        // tile has such rows: the others take a path without a per-row test)
        uint32_t ra[DQ_MAXI], rb[DQ_MAXI], rm[DQ_MAXI];
        auto v_load = [&](int k, int t) {
          if constexpr (FP8) {
            ra[k] = ld_shared_u32(vst + t * D + 8 * cc);
            rb[k] = ld_shared_u32(vst + t * D + 8 * cc + 4);
          } else {
            rm[k] = ld_shared_u32(vst + HQ2B_META_OFF + t * 8 + 4 * (cc >> 4));
            ra[k] = ld_shared_u8(vst + t * HQ2B_ROW + 2 * cc);
            rb[k] = ld_shared_u8(vst + t * HQ2B_ROW + 2 * cc + 1);
          }
        };
        auto v_conv = [&](int k) -> uint4 {
          if constexpr (FP8) {
            return make_uint4(e4m3x2_h2(ra[k]), e4m3x2_h2(ra[k] >> 16), e4m3x2_h2(rb[k]), e4m3x2_h2(rb[k] >> 16));
          } else {
            const __half2 s2 = u2h(__byte_perm(rm[k], 0u, 0x1010u)), z2 = u2h(__byte_perm(rm[k], 0u, 0x3232u));
            uint32_t res[4];
            dq_pairs(ra[k], rb[k], res);
#pragma unroll
            for (int p = 0; p < 4; p++) res[p] = h2u(__hfma2(__hfma2(u2h(res[p]), one2, m4), s2, z2));
            return make_uint4(res[0], res[1], res[2], res[3]);
          }
        };
        if (vall) {
#pragma unroll
          for (int k = 0; k < DQ_MAXI; k++)
            if (t0 + KSTEP * k < P) v_load(k, t0 + KSTEP * k);
#pragma unroll
          for (int k = 0; k < DQ_MAXI; k++)
            if (t0 + KSTEP * k < P) st_shared_v4(vb + swz(t0 + KSTEP * k, cc & 7), v_conv(k));
        } else {
#pragma unroll
          for (int k = 0; k < DQ_MAXI; k++) {
            const int t = t0 + KSTEP * k;
            if (t < P && key0 + t < len) v_load(k, t);
          }
#pragma unroll
          for (int k = 0; k < DQ_MAXI; k++) {
            const int t = t0 + KSTEP * k;
            if (t < P) st_shared_v4(vb + swz(t, cc & 7), key0 + t < len ? v_conv(k) : make_uint4(0u, 0u, 0u, 0u));
          }
        }
      }
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      __syncwarp();
      if (lane == 0) {
        bar_arrive(BAR(B_V_FULL + buf));
        bar_arrive(BAR(B_STG_EMPTY + sbuf));
      }
      // the copier refills the stage of tile j - 1 (not of tile j, which the other warps may
      // still be reading), so its wait rarely holds up its own warp
      if (tid == 0 && j >= 1 && issued < ntiles) {
        if (!issue(issued)) timed_out = true;
        issued++;
      }
      timed_out = __shfl_sync(0xFFFFFFFFu, timed_out, 0);
    }
    // copies still in flight must land before the CTA exits
    if (tid == 0) {
      for (int j = max(0, issued - PT_NSTG); j < issued; j++) bar_wait(BAR(B_STG_FULL + j % PT_NSTG), (j / PT_NSTG) & 1);
    }
  } else {
    // =============================================================== MMA warp (one thread)
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_f16(128, 64);
      constexpr uint32_t IDESC_PV = idesc_f16(128, 256, true);
      bool ok = bar_wait(BAR(B_Q_READY), 0);
      tc_fence_after();
      auto issue_s = [&](int j) {
        const int buf = j & 1;
        tc_fence_after();
        const uint32_t kb = sm_u32(smem + SM_K + buf * LY::K_BUF);
#pragma unroll
        for (int ks = 0; ks < 16; ks++)
          tc_mma_ts(tmem + TM_S0 + 64 * buf, tmem + TM_Q + 8 * ks, sw128_desc(kb + (ks >> 2) * 8192 + (ks & 3) * 32),
                    IDESC_S, ks > 0);
        if constexpr (LY::KSPLIT) {   // + Q . K_lo^T: the low parts of the keys
#pragma unroll
          for (int ks = 0; ks < 16; ks++)
            tc_mma_ts(tmem + TM_S0 + 64 * buf, tmem + TM_Q + 8 * ks,
                      sw128_desc(kb + 32768 + (ks >> 2) * 8192 + (ks & 3) * 32), IDESC_S, 1u);
        }
        tc_commit(BAR(B_S_FULL + buf));
        tc_commit(BAR(B_K_EMPTY + buf));
      };
      auto issue_pv = [&](int j) {
        const int buf = j & 1;
        tc_fence_after();
        const uint32_t vb = sm_u32(smem + LY::SM_V + buf * LY::V_BUF);
#pragma unroll
        for (int ks = 0; ks < 4; ks++)
          tc_mma_ts(tmem + TM_O, tmem + TM_S0 + 64 * buf + 8 * ks, sw128_mn_desc(vb + 2048 * ks), IDESC_PV,
                    (j > 0 || ks > 0) ? 1u : 0u);
        tc_commit(BAR(B_PV_DONE + buf));
      };
      int last_pv = -1;
      if (ok && ntiles > 0) {
        ok = bar_wait(BAR(B_K_FULL), 0);
        if (ok) issue_s(0);
      }
      // Per tile j: S(j+1) once its K tile is ready, then PV(j) once P(j) and the V tile are.
      // S(j+1) reuses the S/P buffer of tile j-1, whose PV was issued in the previous round (the
      // MMAs run in issue order).  The waits suspend the thread (no polling), so the issuer takes
      // no issue slots from the dequantisation and softmax warps while it waits.
      for (int j = 0; j < ntiles && ok; j++) {
        const int buf = j & 1;
        const uint32_t par = (j >> 1) & 1;
        if (j + 1 < ntiles) {
          ok = bar_wait(BAR(B_K_FULL + ((j + 1) & 1)), ((j + 1) >> 1) & 1) && !*abort_flag;
          if (!ok) break;
          issue_s(j + 1);
        }
        ok = bar_wait(BAR(B_P_FULL + buf), par) && bar_wait(BAR(B_V_FULL + buf), par) && !*abort_flag;
        if (!ok) break;
        issue_pv(j);
        last_pv = j;
      }
      if (!ok) {
        timed_out = true;
        *abort_flag = 1;
      }
      // the MMAs issued must finish before TMEM is released
      if (last_pv >= 0) bar_wait(BAR(B_PV_DONE + (last_pv & 1)), (last_pv >> 1) & 1);
    }
    __syncwarp();
  }
  if (timed_out) {
    *abort_flag = 1;
    if (lane == 0) flag(c.status, KVQ_STATUS_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;\n" ::"r"(tmem));
  }
}

template <int FMT>
static int launch_prefill_fmt(const AttnArgs& a, cudaStream_t stream) {
  if (a.split_tokens > PREFILL_SPLIT || a.split_tokens % P) return KVQ_ERR_UNSUPPORTED;   // s_pages holds one split
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!attr_set[dev]) {
    cudaFuncSetAttribute(prefill_tc<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, PfLayout<FMT>::SMEM);
    attr_set[dev] = true;
  }
  const int QT = PT_ROWS / a.c.group;
  dim3 grid(a.max_splits, (a.max_n_q + QT - 1) / QT, a.lanes * a.c.num_kv_heads);
  prefill_tc<FMT><<<grid, PT_THREADS, PfLayout<FMT>::SMEM, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

// The tensor-core prefill of every compressed format: fmt is the geometry's format.
int launch_prefill_tc(int fmt, const AttnArgs& a, cudaStream_t stream) {
  switch (fmt) {
    case KVQ_FMT_HQ2B: return launch_prefill_fmt<KVQ_FMT_HQ2B>(a, stream);
    case KVQ_FMT_HQ2B_HAD: return launch_prefill_fmt<KVQ_FMT_HQ2B_HAD>(a, stream);
    case KVQ_FMT_HQ2B_TOK: return launch_prefill_fmt<KVQ_FMT_HQ2B_TOK>(a, stream);
    case KVQ_FMT_FP8: return launch_prefill_fmt<KVQ_FMT_FP8>(a, stream);
    default: return KVQ_ERR_UNSUPPORTED;
  }
}

}  // namespace kvq

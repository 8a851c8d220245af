// append_ops.cuh -- the quantize-and-append arithmetic, shared by the append kernels and by the
// fused decode step (whose combine kernel appends the step's token).
//
// Format: include/kvq.h ("KV at 9 KB a token", "How it works": 64 B of 2-bit code + an 8 B
// metadata row per head per token, 64-token pages).  Axes follow the KIVI rule quoted in
// "Half the Cache, Twice the Context", table "Two losses with one name": V per token, K per
// channel.  All quantizer arithmetic is IEEE fp32 round-to-nearest-even (__fdiv_rn, __fsub_rn,
// ..., never contracted into FMAs) so the bytes match a CPU implementation of the same steps.
#pragma once
#include "kvq_internal.cuh"

namespace kvq {

struct AppendArgs {
  CacheView c;
  uint8_t* pool;
  __nv_bfloat16* ring;
  const int32_t* start_pos;
  const int32_t* n_new;
  const int32_t* tok_offset;
  int max_new, n_rows, lanes;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
};

constexpr int ROWS_PER_CTA = 8;  // tokens per CTA of the rows kernel (x num_kv_heads items)

__device__ __forceinline__ bool read_lane(const AppendArgs& a, int b, int& start, int& n, int& off) {
  start = a.start_pos[b];
  n = a.n_new[b];
  off = a.tok_offset[b];
  if (n < 0 || n > a.max_new || start < 0 || off < 0 || (int64_t)off + n > a.n_rows) {
    if (threadIdx.x == 0) flag(a.c.status, KVQ_STATUS_BAD_LEN);
    return false;
  }
  return true;
}

__device__ __forceinline__ bool finite16(float x) { return fabsf(x) <= 65504.0f; }  // false for NaN

__device__ __forceinline__ bool row8_ok(uint4 w) {
  uint32_t u[4] = {w.x, w.y, w.z, w.w};
  bool ok = true;
#pragma unroll
  for (int i = 0; i < 4; i++) ok = ok && finite16(bf16_lo(u[i])) && finite16(bf16_hi(u[i]));
  return ok;
}

// V row quantization by one warp, per token and 128-dim half (lanes 0-15: dims 0..127, lanes
// 16-31: dims 128..255): lane l holds dims 8l..8l+7 of the row (bf16) in vx and gets their 2-bit
// codes (16 bits, dim 8l+j at bits 2j) and the meta word of its half (s | z << 16, fp16 each).
__device__ __forceinline__ void quant_v_row_f32(const float (&x)[8], uint32_t& packed, uint32_t& meta) {
  float mn = x[0], mx = x[0];
#pragma unroll
  for (int j = 1; j < 8; j++) {
    mn = fminf(mn, x[j]);
    mx = fmaxf(mx, x[j]);
  }
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  }
  const __half zh = __float2half_rn(mn);
  const __half sh = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), 3.0f));
  const float zf = __half2float(zh), sf = __half2float(sh);
  packed = 0;
#pragma unroll
  for (int j = 0; j < 8; j++) {
    int code = 0;
    if (sf != 0.0f) {
      float q = __fdiv_rn(__fsub_rn(x[j], zf), sf);
      q = fminf(fmaxf(rintf(q), 0.0f), 3.0f);
      code = (int)q;
    }
    packed |= (uint32_t)code << (2 * j);
  }
  meta = (uint32_t)__half_as_ushort(sh) | ((uint32_t)__half_as_ushort(zh) << 16);
}

__device__ __forceinline__ void bf16x8_to_f32(uint4 w, float (&x)[8]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int j = 0; j < 4; j++) {
    x[2 * j] = bf16_lo(u[j]);
    x[2 * j + 1] = bf16_hi(u[j]);
  }
}

__device__ __forceinline__ void quant_v_row(uint4 vx, uint32_t& packed, uint32_t& meta) {
  float x[8];
  bf16x8_to_f32(vx, x);
  quant_v_row_f32(x, packed, meta);
}

// The rotated format's V row: Walsh-Hadamard transform of the row (all 32 lanes), then the same
// quantizer; false (on every lane) when a rotated value is not finite in fp16.
__device__ __forceinline__ bool quant_v_row_rot(uint4 vx, uint32_t& packed, uint32_t& meta) {
  float x[8];
  bf16x8_to_f32(vx, x);
  warp_fwht256(x);
  bool ok = true;
#pragma unroll
  for (int j = 0; j < 8; j++) ok = ok && finite16(x[j]);
  if (!__all_sync(0xFFFFFFFFu, ok)) return false;
  quant_v_row_f32(x, packed, meta);
  return true;
}

// Page-close quantization of K, per channel over the page's 64 keys, by PARTS x 256 threads:
// thread (part, d) handles channel d = tid % 256 for keys (64 / PARTS) * part ...
constexpr int KCLOSE_PARTS = 4;
constexpr int KCLOSE_THREADS = KCLOSE_PARTS * D;

// Per-channel quantization of the K block of page p (lane b, head h) into shared memory:
// codes[64 keys][64 B] and scales[256] (fp16).  Keys before `start` come from the ring, the rest
// from k rows off + (pos - start).  Every thread of the CTA (PARTS x 256 of them) calls it;
// returns false on every thread when a key is not finite in fp16 (nothing usable written).
template <int PARTS = KCLOSE_PARTS>
__device__ __forceinline__ bool kclose_core(const AppendArgs& a, int b, int h, int p, int start, int off,
                                            uint8_t* codes, __half* scales) {
  const CacheView& c = a.c;
  const int d = threadIdx.x & (D - 1), part = threadIdx.x >> 8;
  const int H = c.num_kv_heads;
  constexpr int T = P / PARTS;
  // with few threads (many keys each) the keys are read twice instead of held in registers
  constexpr bool HOLD = T <= 16;
  auto key = [&](int i) {
    const int t = T * part + i;
    const int pos = p * P + t;
    return __bfloat162float(pos < start ? a.ring[ring_row_offset(c, b, h, t) + d]
                                        : a.k[((int64_t)(off + pos - start) * H + h) * D + d]);
  };
  float x[HOLD ? T : 1];
  float amax = 0.0f;
  bool bad = false;
  constexpr int UNROLL = HOLD ? T : 8;
#pragma unroll UNROLL
  for (int i = 0; i < T; i++) {
    const float xi = key(i);
    if (HOLD) x[i] = xi;
    bad |= !finite16(xi);
    amax = fmaxf(amax, fabsf(xi));
  }
  __shared__ float part_max[PARTS][D];
  part_max[part][d] = amax;
  if (__syncthreads_or(bad)) return false;
  amax = part_max[0][d];
#pragma unroll
  for (int i = 1; i < PARTS; i++) amax = fmaxf(amax, part_max[i][d]);
  const __half sh = __float2half_rn(__fdiv_rn(amax, 3.0f));
  const float sf = __half2float(sh);
#pragma unroll UNROLL
  for (int i = 0; i < T; i++) {
    const int t = T * part + i;
    int code = 2;
    if (sf != 0.0f) {
      float u = __fdiv_rn(HOLD ? x[HOLD ? i : 0] : key(i), sf);
      u = __fadd_rn(u, 3.0f);
      u = __fmul_rn(0.5f, u);
      u = fminf(fmaxf(rintf(u), 0.0f), 3.0f);
      code = (int)u;
    }
    uint32_t bits = (uint32_t)code << (2 * (d & 3));
    bits |= __shfl_xor_sync(0xFFFFFFFFu, bits, 1);
    bits |= __shfl_xor_sync(0xFFFFFFFFu, bits, 2);
    if ((d & 3) == 0) codes[t * HQ2B_ROW + d / 4] = (uint8_t)bits;
  }
  if (part == 0) scales[d] = sh;
  __syncthreads();
  return true;
}

// kclose_core for the rotated format, by exactly 1,024 threads: warp w rotates keys w and w + 32
// (lane l holds channels 8l .. 8l+7 of the rotated key), the channel maxima meet in shared
// memory, and each lane writes the 2 code bytes of its channels for both keys.  The per-element
// arithmetic is kclose_core's, on the rotated values.
__device__ __forceinline__ bool kclose_core_rot(const AppendArgs& a, int b, int h, int p, int start, int off,
                                                uint8_t* codes, __half* scales) {
  const CacheView& c = a.c;
  const int H = c.num_kv_heads;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  float x[2][8];
  bool bad = false;
#pragma unroll
  for (int i = 0; i < 2; i++) {
    const int t = w + 32 * i, pos = p * P + t;
    const uint4 kw = pos < start ? reinterpret_cast<const uint4*>(a.ring + ring_row_offset(c, b, h, t))[lane]
                                 : reinterpret_cast<const uint4*>(a.k + ((int64_t)(off + pos - start) * H + h) * D)[lane];
    bf16x8_to_f32(kw, x[i]);
#pragma unroll
    for (int e = 0; e < 8; e++) bad |= !finite16(x[i][e]);
    warp_fwht256(x[i]);
#pragma unroll
    for (int e = 0; e < 8; e++) bad |= !finite16(x[i][e]);
  }
  __shared__ float part_max[32][D];
#pragma unroll
  for (int e = 0; e < 8; e++) part_max[w][8 * lane + e] = fmaxf(fabsf(x[0][e]), fabsf(x[1][e]));
  if (__syncthreads_or(bad)) return false;
  if (threadIdx.x < D) {
    const int d = threadIdx.x;
    float m = part_max[0][d];
    for (int i = 1; i < 32; i++) m = fmaxf(m, part_max[i][d]);
    scales[d] = __float2half_rn(__fdiv_rn(m, 3.0f));
  }
  __syncthreads();
  float sf[8];
#pragma unroll
  for (int e = 0; e < 8; e++) sf[e] = __half2float(scales[8 * lane + e]);
#pragma unroll
  for (int i = 0; i < 2; i++) {
    uint32_t bits = 0;
#pragma unroll
    for (int e = 0; e < 8; e++) {
      int code = 2;
      if (sf[e] != 0.0f) {
        float q = __fdiv_rn(x[i][e], sf[e]);
        q = __fadd_rn(q, 3.0f);
        q = __fmul_rn(0.5f, q);
        q = fminf(fmaxf(rintf(q), 0.0f), 3.0f);
        code = (int)q;
      }
      bits |= (uint32_t)code << (2 * e);
    }
    reinterpret_cast<uint16_t*>(codes + (w + 32 * i) * HQ2B_ROW)[lane] = (uint16_t)bits;
  }
  __syncthreads();
  return true;
}

// Whether page p of lane b can take a K block: inside the table and mapped to a pool page
// (flags and returns false otherwise; the same answer on every thread).
__device__ __forceinline__ bool kblock_page_ok(const CacheView& c, int b, int p) {
  if (p >= c.max_pages) {
    if (threadIdx.x == 0) flag(c.status, KVQ_STATUS_LEN_GT_TABLE);
    return false;
  }
  const int32_t phys = c.page_table[(int64_t)b * c.max_pages + p];
  if (phys < 0 || phys >= c.pool_pages) {
    if (threadIdx.x == 0) flag(c.status, KVQ_STATUS_PAGE_OOB);
    return false;
  }
  return true;
}

// The K block of page p, quantized by kclose_core, stored into the page (threads 0..255 store).
__device__ __forceinline__ void kblock_store(const AppendArgs& a, int b, int h, int p, const uint8_t* codes,
                                             const __half* scales) {
  const CacheView& c = a.c;
  const int32_t phys = c.page_table[(int64_t)b * c.max_pages + p];
  if (threadIdx.x < D) {
    uint8_t* kblk = a.pool + (int64_t)phys * c.page_bytes + block_offset(KVQ_FMT_HQ2B, c.num_kv_heads, c.layer, h, 0);
    reinterpret_cast<uint4*>(kblk)[threadIdx.x] = reinterpret_cast<const uint4*>(codes)[threadIdx.x];
    reinterpret_cast<__half*>(kblk + HQ2B_META_OFF)[threadIdx.x] = scales[threadIdx.x];
  }
}

// Page close of one group of KGROUP_CH channels, for a decode step's append: a CTA of
// KGROUP_THREADS threads, thread (part, c) quantizing channel KGROUP_CH * grp + c for keys
// 16 part .. 16 part + 15 with kclose_core's arithmetic, then storing the group's 16 code bytes of
// every key row and its scales.  Four such CTAs close a page in a quarter of the time one
// 1,024-thread CTA takes, and each leaves room on its SM for a decode CTA beside it.
constexpr int KGROUP_CH = 64;
constexpr int KGROUP_THREADS = 256;
__device__ __forceinline__ void kclose_group(const AppendArgs& a, int b, int h, int p, int start, int off, int grp) {
  const CacheView& c = a.c;
  if (p >= c.max_pages) {
    if (threadIdx.x == 0) flag(c.status, KVQ_STATUS_LEN_GT_TABLE);
    return;
  }
  const int H = c.num_kv_heads;
  const int cl = threadIdx.x & (KGROUP_CH - 1), part = threadIdx.x / KGROUP_CH, d = KGROUP_CH * grp + cl;
  constexpr int PARTS = KGROUP_THREADS / KGROUP_CH;
  constexpr int T = P / PARTS;
  __shared__ __align__(16) uint8_t codes[P * (KGROUP_CH / 4)];   // 64 key rows x 16 B
  __shared__ __half scales[KGROUP_CH];
  __shared__ float part_max[PARTS][KGROUP_CH];
  // Every load of the close goes out before any is used (one round trip, not three): the page
  // id, the thread's T keys of channel d, and the first of its share of the input rows' values
  // for the finite check (every channel of the keys that come from this call's input rows; ring
  // rows were checked when they were appended: a bad value anywhere in them leaves the whole K
  // block unwritten, in all four group CTAs alike, as a whole-page close would).
  const int32_t phys = c.page_table[(int64_t)b * c.max_pages + p];
  __nv_bfloat16 xr[T];
#pragma unroll
  for (int i = 0; i < T; i++) {
    const int t = T * part + i;
    const int pos = p * P + t;
    xr[i] = pos < start ? a.ring[ring_row_offset(c, b, h, t) + d] : a.k[((int64_t)(off + pos - start) * H + h) * D + d];
  }
  const int first = max(0, start - p * P), n_in = (P - first) * D;
  const __nv_bfloat16 in0 = (int)threadIdx.x < n_in
                                ? a.k[((int64_t)(off + p * P + first + threadIdx.x / D - start) * H + h) * D + threadIdx.x % D]
                                : __float2bfloat16(0.0f);
  if (phys < 0 || phys >= c.pool_pages) {
    if (threadIdx.x == 0) flag(c.status, KVQ_STATUS_PAGE_OOB);
    return;
  }
  float x[T];
  float amax = 0.0f;
  bool bad = !finite16(__bfloat162float(in0));
#pragma unroll
  for (int i = 0; i < T; i++) {
    x[i] = __bfloat162float(xr[i]);
    bad |= !finite16(x[i]);
    amax = fmaxf(amax, fabsf(x[i]));
  }
  part_max[part][cl] = amax;
  for (int i = threadIdx.x + KGROUP_THREADS; i < n_in; i += KGROUP_THREADS) {   // more than one input row
    const int pos = p * P + first + i / D;
    bad |= !finite16(__bfloat162float(a.k[((int64_t)(off + pos - start) * H + h) * D + i % D]));
  }
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0) flag(c.status, KVQ_STATUS_BAD_INPUT);
    return;
  }
  amax = part_max[0][cl];
#pragma unroll
  for (int i = 1; i < PARTS; i++) amax = fmaxf(amax, part_max[i][cl]);
  const __half sh = __float2half_rn(__fdiv_rn(amax, 3.0f));
  const float sf = __half2float(sh);
#pragma unroll
  for (int i = 0; i < T; i++) {
    const int t = T * part + i;
    int code = 2;
    if (sf != 0.0f) {
      float u = __fdiv_rn(x[i], sf);
      u = __fadd_rn(u, 3.0f);
      u = __fmul_rn(0.5f, u);
      u = fminf(fmaxf(rintf(u), 0.0f), 3.0f);
      code = (int)u;
    }
    uint32_t bits = (uint32_t)code << (2 * (cl & 3));
    bits |= __shfl_xor_sync(0xFFFFFFFFu, bits, 1);
    bits |= __shfl_xor_sync(0xFFFFFFFFu, bits, 2);
    if ((cl & 3) == 0) codes[t * (KGROUP_CH / 4) + cl / 4] = (uint8_t)bits;
  }
  if (part == 0) scales[cl] = sh;
  __syncthreads();
  if (threadIdx.x < P) {
    uint8_t* kblk = a.pool + (int64_t)phys * c.page_bytes + block_offset(KVQ_FMT_HQ2B, H, c.layer, h, 0);
    *reinterpret_cast<uint4*>(kblk + threadIdx.x * HQ2B_ROW + (KGROUP_CH / 4) * grp) =
        reinterpret_cast<const uint4*>(codes)[threadIdx.x];
    if (threadIdx.x < KGROUP_CH)
      reinterpret_cast<__half*>(kblk + HQ2B_META_OFF)[KGROUP_CH * grp + threadIdx.x] = scales[threadIdx.x];
  }
}

// Page close: quantize page p's K block per channel and store it; every thread of the CTA
// (PARTS x 256) calls it.
template <int PARTS = KCLOSE_PARTS>
__device__ __forceinline__ void kclose_page(const AppendArgs& a, int b, int h, int p, int start, int off) {
  if (!kblock_page_ok(a.c, b, p)) return;
  __shared__ __align__(16) uint8_t codes[P * HQ2B_ROW];
  __shared__ __align__(16) __half scales[D];
  const bool ok = (PARTS == 4 && a.c.rotated) ? kclose_core_rot(a, b, h, p, start, off, codes, scales)
                                              : kclose_core<PARTS>(a, b, h, p, start, off, codes, scales);
  if (!ok) {
    if (threadIdx.x == 0) flag(a.c.status, KVQ_STATUS_BAD_INPUT);
    return;
  }
  kblock_store(a, b, h, p, codes, scales);
}

// One warp: token i of lane b, head h -- V row quantization (HQ2B; the K row too in the
// per-token-K format), plain stores (BF16) or E4M3 conversion (FP8), and the key into the ring (only the chunk's last 64 tokens: the ring keeps the newest key of each
// slot).  Returns after flagging when the token is past the table or its page is invalid.
template <int FMT>
__device__ __forceinline__ void append_row(const AppendArgs& a, int b, int h, int i, int start, int n, int off) {
  const CacheView& c = a.c;
  const int lane = threadIdx.x & 31;
  const int H = c.num_kv_heads;
  const int64_t t = (int64_t)start + i, row = (int64_t)off + i;
  if (t / P >= c.max_pages) {
    if (lane == 0) flag(c.status, KVQ_STATUS_LEN_GT_TABLE);
    return;
  }
  // the page id and the token's rows in one round trip (the rows are inside the inputs whatever
  // the page id)
  const int32_t phys = c.page_table[(int64_t)b * c.max_pages + t / P];
  const uint4 kx = reinterpret_cast<const uint4*>(a.k + (row * H + h) * D)[lane];
  const uint4 vx = reinterpret_cast<const uint4*>(a.v + (row * H + h) * D)[lane];
  if (phys < 0 || phys >= c.pool_pages) {
    if (lane == 0) flag(c.status, KVQ_STATUS_PAGE_OOB);
    return;
  }
  const int slot = (int)(t % P);
  if (__any_sync(0xFFFFFFFFu, !(row8_ok(kx) && row8_ok(vx)))) {
    if (lane == 0) flag(c.status, KVQ_STATUS_BAD_INPUT);
    return;
  }
  uint8_t* page = a.pool + (int64_t)phys * c.page_bytes;
  uint8_t* kblk = page + block_offset(FMT, H, c.layer, h, 0);
  uint8_t* vblk = page + block_offset(FMT, H, c.layer, h, 1);
  if (FMT == KVQ_FMT_BF16) {
    reinterpret_cast<uint4*>(kblk + slot * D * 2)[lane] = kx;
    reinterpret_cast<uint4*>(vblk + slot * D * 2)[lane] = vx;
    return;
  }
  if (FMT == KVQ_FMT_FP8) {
    reinterpret_cast<uint2*>(kblk + slot * D)[lane] = fp8_encode8(kx, c.k_scale);
    reinterpret_cast<uint2*>(vblk + slot * D)[lane] = fp8_encode8(vx, c.v_scale);
    return;
  }
  uint32_t packed, meta;
  if (c.rotated) {
    if (!quant_v_row_rot(vx, packed, meta)) {
      if (lane == 0) flag(c.status, KVQ_STATUS_BAD_INPUT);
      return;
    }
  } else {
    quant_v_row(vx, packed, meta);
  }
  reinterpret_cast<uint16_t*>(vblk + slot * HQ2B_ROW)[lane] = (uint16_t)packed;
  if ((lane & 15) == 0) reinterpret_cast<uint32_t*>(vblk + HQ2B_META_OFF + slot * 8)[lane >> 4] = meta;
  if (c.ktok) {   // per-token-K format: the key row is coded now, by the V rule, in the K block
    quant_v_row(kx, packed, meta);
    reinterpret_cast<uint16_t*>(kblk + slot * HQ2B_ROW)[lane] = (uint16_t)packed;
    if ((lane & 15) == 0) reinterpret_cast<uint32_t*>(kblk + HQ2B_META_OFF + slot * 8)[lane >> 4] = meta;
  }
  if (i >= n - P) reinterpret_cast<uint4*>(a.ring + ring_row_offset(c, b, h, slot))[lane] = kx;
}

}  // namespace kvq

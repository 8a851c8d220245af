// append.cu -- quantize-and-append of new tokens into the paged pool.
//
// Format: include/kvq.h ("KV at 9 KB a token", "How it works": 64 B of 2-bit code + an 8 B
// metadata row per head per token, 64-token pages).  Axes follow the KIVI rule quoted in
// "Half the Cache, Twice the Context", table "Two losses with one name": V per token, K per
// channel.  K per channel needs all 64 keys of a page, so a K row first lands in the exact
// bf16 ring (the "window of exact recent keys", "The KV cache and prompt reuse") and the
// page's K block is written when the page closes.
//
// Chunks (at most max_new > 1 tokens per lane): two launches, in stream order:
//   1. kclose: one CTA per (closing page, head, lane) quantizes the page's K block per channel,
//      reading keys appended by earlier calls from the ring and this call's keys from `k`.
//   2. rows:   one warp per (token, head) quantizes the V row, and stores the K row in the
//      ring (only the chunk's last 64 tokens -- the ring keeps the newest key of each slot).
// Launch 1 must read the ring before launch 2 overwrites it; stream order guarantees that.
// Decode steps (max_new == 1): one launch does both for each (lane, head).
// All quantizer arithmetic is IEEE fp32 round-to-nearest-even (__fdiv_rn, __fsub_rn, ...,
// never contracted into FMAs) so the bytes match a CPU implementation of the same steps.
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

// Page-close quantization of K, per channel over the page's 64 keys.  1,024 threads: thread
// (part, d) handles channel d = tid % 256 for keys 16*part .. 16*part + 15.
constexpr int KCLOSE_PARTS = 4;
constexpr int KCLOSE_THREADS = KCLOSE_PARTS * D;

// Quantize the K block of page p (lane b, head h) per channel; every thread of the CTA calls it.
__device__ __forceinline__ void kclose_page(const AppendArgs& a, int b, int h, int p, int start, int off) {
  const CacheView& c = a.c;
  if (p >= c.max_pages) {
    if (threadIdx.x == 0) flag(c.status, KVQ_STATUS_LEN_GT_TABLE);
    return;
  }
  const int32_t phys = c.page_table[(int64_t)b * c.max_pages + p];
  if (phys < 0 || phys >= c.pool_pages) {
    if (threadIdx.x == 0) flag(c.status, KVQ_STATUS_PAGE_OOB);
    return;
  }
  const int d = threadIdx.x & (D - 1), part = threadIdx.x >> 8;
  const int H = c.num_kv_heads;
  constexpr int T = P / KCLOSE_PARTS;
  float x[T];
  float amax = 0.0f;
  bool bad = false;
#pragma unroll
  for (int i = 0; i < T; i++) {
    const int t = T * part + i;
    const int pos = p * P + t;
    __nv_bfloat16 e = pos < start ? a.ring[ring_row_offset(c, b, h, t) + d]
                                  : a.k[((int64_t)(off + pos - start) * H + h) * D + d];
    x[i] = __bfloat162float(e);
    bad |= !finite16(x[i]);
    amax = fmaxf(amax, fabsf(x[i]));
  }
  __shared__ float part_max[KCLOSE_PARTS][D];
  __shared__ __align__(16) uint8_t codes[P * HQ2B_ROW];
  part_max[part][d] = amax;
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0) flag(c.status, KVQ_STATUS_BAD_INPUT);
    return;
  }
  amax = part_max[0][d];
#pragma unroll
  for (int i = 1; i < KCLOSE_PARTS; i++) amax = fmaxf(amax, part_max[i][d]);
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
    uint32_t bits = (uint32_t)code << (2 * (d & 3));
    bits |= __shfl_xor_sync(0xFFFFFFFFu, bits, 1);
    bits |= __shfl_xor_sync(0xFFFFFFFFu, bits, 2);
    if ((d & 3) == 0) codes[t * HQ2B_ROW + d / 4] = (uint8_t)bits;
  }
  __syncthreads();
  if (threadIdx.x < D) {
    uint8_t* kblk = a.pool + (int64_t)phys * c.page_bytes + block_offset(KVQ_FMT_HQ2B, H, c.layer, h, 0);
    reinterpret_cast<uint4*>(kblk)[threadIdx.x] = reinterpret_cast<const uint4*>(codes)[threadIdx.x];
    reinterpret_cast<__half*>(kblk + HQ2B_META_OFF)[d] = sh;
  }
}

__global__ void __launch_bounds__(KCLOSE_THREADS) append_kclose_kernel(AppendArgs a) {
  const int b = blockIdx.z, h = blockIdx.y;
  int start, n, off;
  if (!read_lane(a, b, start, n, off)) return;
  const int n_close = (start + n) / P - start / P;
  if ((int)blockIdx.x >= n_close) return;
  kclose_page(a, b, h, start / P + blockIdx.x, start, off);
}

// One warp: token i of lane b, head h -- V row quantization (HQ2B) or plain stores (BF16), and
// the key into the ring (only the chunk's last 64 tokens: the ring keeps the newest key of each
// slot).  Returns after flagging when the token is past the table or its page is invalid.
template <int FMT>
__device__ __forceinline__ void append_row(const AppendArgs& a, int b, int h, int i, int start, int n, int off) {
  const CacheView& c = a.c;
  const int lane = threadIdx.x & 31;
  const int H = c.num_kv_heads;
  {
    const int64_t t = (int64_t)start + i, row = (int64_t)off + i;
    if (t / P >= c.max_pages) {
      if (lane == 0) flag(c.status, KVQ_STATUS_LEN_GT_TABLE);
      return;
    }
    const int32_t phys = c.page_table[(int64_t)b * c.max_pages + t / P];
    if (phys < 0 || phys >= c.pool_pages) {
      if (lane == 0) flag(c.status, KVQ_STATUS_PAGE_OOB);
      return;
    }
    const int slot = (int)(t % P);
    const uint4 kx = reinterpret_cast<const uint4*>(a.k + (row * H + h) * D)[lane];
    const uint4 vx = reinterpret_cast<const uint4*>(a.v + (row * H + h) * D)[lane];
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
    // V, per token, per 128-dim half (lanes 0-15: dims 0..127, lanes 16-31: dims 128..255)
    const uint32_t u[4] = {vx.x, vx.y, vx.z, vx.w};
    float x[8];
#pragma unroll
    for (int j = 0; j < 4; j++) {
      x[2 * j] = bf16_lo(u[j]);
      x[2 * j + 1] = bf16_hi(u[j]);
    }
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
    uint32_t packed = 0;
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
    reinterpret_cast<uint16_t*>(vblk + slot * HQ2B_ROW)[lane] = (uint16_t)packed;
    if ((lane & 15) == 0) {
      const uint32_t meta = (uint32_t)__half_as_ushort(sh) | ((uint32_t)__half_as_ushort(zh) << 16);
      reinterpret_cast<uint32_t*>(vblk + HQ2B_META_OFF + slot * 8)[lane >> 4] = meta;
    }
    if (i >= n - P) reinterpret_cast<uint4*>(a.ring + ring_row_offset(c, b, h, slot))[lane] = kx;
  }
}

template <int FMT>
__global__ void __launch_bounds__(256) append_rows_kernel(AppendArgs a) {
  const int b = blockIdx.y;
  int start, n, off;
  if (!read_lane(a, b, start, n, off)) return;
  const int warp = threadIdx.x >> 5;
  const int H = a.c.num_kv_heads;
  const int i0 = blockIdx.x * ROWS_PER_CTA;
  for (int item = warp; item < ROWS_PER_CTA * H; item += 8) {
    const int i = i0 + item / H, h = item % H;
    if (i >= n) break;
    append_row<FMT>(a, b, h, i, start, n, off);
  }
}

// Decode-time append (at most one new token per lane) in one launch: CTA (lane b, head h); warp
// 0 writes the token's row, and when the token closes its page every thread quantizes the
// page's K block.  The page close reads ring slots 0..62 and this token's key from `k`; the row
// write touches slot 63 only, so the two never meet.
template <int FMT>
__global__ void __launch_bounds__(KCLOSE_THREADS) append_one_kernel(AppendArgs a) {
  const int b = blockIdx.x, h = blockIdx.y;
  int start, n, off;
  if (!read_lane(a, b, start, n, off) || n == 0) return;
  if (threadIdx.x < 32) append_row<FMT>(a, b, h, 0, start, n, off);
  if (FMT == KVQ_FMT_HQ2B && (start + 1) % P == 0) kclose_page(a, b, h, start / P, start, off);
}

int launch_append(int fmt, const CacheView& c, uint8_t* pool, __nv_bfloat16* ring, const int32_t* start_pos,
                  const int32_t* n_new, const int32_t* tok_offset, int max_new, int n_rows, int lanes,
                  const __nv_bfloat16* k, const __nv_bfloat16* v, cudaStream_t stream) {
  AppendArgs a{c, pool, ring, start_pos, n_new, tok_offset, max_new, n_rows, lanes, k, v};
  if (max_new == 1) {
    dim3 g1(lanes, c.num_kv_heads);
    if (fmt == KVQ_FMT_HQ2B) append_one_kernel<KVQ_FMT_HQ2B><<<g1, KCLOSE_THREADS, 0, stream>>>(a);
    else append_one_kernel<KVQ_FMT_BF16><<<g1, KCLOSE_THREADS, 0, stream>>>(a);
  } else if (fmt == KVQ_FMT_HQ2B) {
    dim3 gk(max_new / P + 1, c.num_kv_heads, lanes);
    append_kclose_kernel<<<gk, KCLOSE_THREADS, 0, stream>>>(a);
    dim3 gr((max_new + ROWS_PER_CTA - 1) / ROWS_PER_CTA, lanes);
    append_rows_kernel<KVQ_FMT_HQ2B><<<gr, 256, 0, stream>>>(a);
  } else {
    dim3 gr((max_new + ROWS_PER_CTA - 1) / ROWS_PER_CTA, lanes);
    append_rows_kernel<KVQ_FMT_BF16><<<gr, 256, 0, stream>>>(a);
  }
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq

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
// Decode steps (max_new == 1): one launch does both for each (lane, head), the page close split
// over four CTAs of 64 channels each.
// The per-token-K format (KVQ_FMT_HQ2B_TOK) codes the K row with the V rule in the rows pass and
// has no page close.
// All quantizer arithmetic is IEEE fp32 round-to-nearest-even (__fdiv_rn, __fsub_rn, ...,
// never contracted into FMAs) so the bytes match a CPU implementation of the same steps.
#include "append_ops.cuh"

namespace kvq {

__global__ void __launch_bounds__(KCLOSE_THREADS) append_kclose_kernel(AppendArgs a) {
  const int b = blockIdx.z, h = blockIdx.y;
  int start, n, off;
  if (!read_lane(a, b, start, n, off)) return;
  const int n_close = (start + n) / P - start / P;
  if ((int)blockIdx.x >= n_close) return;
  kclose_page(a, b, h, start / P + blockIdx.x, start, off);
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

// Decode-time append (at most one new token per lane) in one launch: CTA (lane b, head h,
// channel group z); warp 0 of group 0 writes the token's row, and when the token closes its
// page, each group's CTA quantizes its KGROUP_CH channels of the page's K block (THREADS =
// KGROUP_THREADS, 4 groups), or one 1,024-thread CTA the whole block (the rotated format, whose
// keys are rotated a row at a time).  The page close reads ring slots 0..62 and this token's key
// from `k`; the row write touches slot 63 only, so the two never meet.
// LAST: launched as the programmatic dependent of the decode step's combine kernel (nothing the
// step's attention reads is written here); every CTA waits for that grid before it exits, so the
// kernel after this one in the stream sees the whole step complete.
template <int FMT, int THREADS>
__device__ __forceinline__ void append_one(const AppendArgs& a) {
  const int b = blockIdx.x, h = blockIdx.y, grp = blockIdx.z;
  int start, n, off;
  if (!read_lane(a, b, start, n, off) || n == 0) return;
  if (grp == 0 && threadIdx.x < 32) append_row<FMT>(a, b, h, 0, start, n, off);
  if (FMT == KVQ_FMT_HQ2B && !a.c.ktok && (start + 1) % P == 0) {
    if constexpr (THREADS == KCLOSE_THREADS) kclose_page(a, b, h, start / P, start, off);
    else kclose_group(a, b, h, start / P, start, off, grp);
  }
}

template <int FMT, int THREADS, bool LAST>
__global__ void __launch_bounds__(THREADS) append_one_kernel(AppendArgs a) {
  // a decode kernel launched as this grid's programmatic dependent (kvq_decode_step) may start
  // now; it waits for this grid before it reads anything written here
  if (!LAST) asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  append_one<FMT, THREADS>(a);
  if (LAST) asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

// Decode-step append of the plain 2-bit format as the programmatic dependent of the kernel just
// launched on `stream` (see append_one_kernel's LAST).
int launch_append_last(const CacheView& c, uint8_t* pool, __nv_bfloat16* ring, const int32_t* start_pos,
                       const int32_t* n_new, const int32_t* tok_offset, int n_rows, int lanes,
                       const __nv_bfloat16* k, const __nv_bfloat16* v, cudaStream_t stream) {
  AppendArgs a{c, pool, ring, start_pos, n_new, tok_offset, 1, n_rows, lanes, k, v};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(lanes, c.num_kv_heads, D / KGROUP_CH);
  cfg.blockDim = dim3(KGROUP_THREADS);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, append_one_kernel<KVQ_FMT_HQ2B, KGROUP_THREADS, true>, a) != cudaSuccess)
    return KVQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

int launch_append(int fmt, const CacheView& c, uint8_t* pool, __nv_bfloat16* ring, const int32_t* start_pos,
                  const int32_t* n_new, const int32_t* tok_offset, int max_new, int n_rows, int lanes,
                  const __nv_bfloat16* k, const __nv_bfloat16* v, cudaStream_t stream) {
  AppendArgs a{c, pool, ring, start_pos, n_new, tok_offset, max_new, n_rows, lanes, k, v};
  if (max_new == 1) {
    dim3 g1(lanes, c.num_kv_heads);
    if (fmt == KVQ_FMT_HQ2B && c.rotated) {
      append_one_kernel<KVQ_FMT_HQ2B, KCLOSE_THREADS, false><<<g1, KCLOSE_THREADS, 0, stream>>>(a);
    } else if (fmt == KVQ_FMT_HQ2B) {
      const dim3 gg(lanes, c.num_kv_heads, c.ktok ? 1 : D / KGROUP_CH);
      append_one_kernel<KVQ_FMT_HQ2B, KGROUP_THREADS, false><<<gg, KGROUP_THREADS, 0, stream>>>(a);
    } else if (fmt == KVQ_FMT_FP8) {
      append_one_kernel<KVQ_FMT_FP8, KGROUP_THREADS, false><<<g1, KGROUP_THREADS, 0, stream>>>(a);
    } else {
      append_one_kernel<KVQ_FMT_BF16, KGROUP_THREADS, false><<<g1, KGROUP_THREADS, 0, stream>>>(a);
    }
  } else if (fmt == KVQ_FMT_HQ2B) {
    if (!c.ktok) {   // the per-token-K format has no page close
      dim3 gk(max_new / P + 1, c.num_kv_heads, lanes);
      append_kclose_kernel<<<gk, KCLOSE_THREADS, 0, stream>>>(a);
    }
    dim3 gr((max_new + ROWS_PER_CTA - 1) / ROWS_PER_CTA, lanes);
    append_rows_kernel<KVQ_FMT_HQ2B><<<gr, 256, 0, stream>>>(a);
  } else {
    dim3 gr((max_new + ROWS_PER_CTA - 1) / ROWS_PER_CTA, lanes);
    if (fmt == KVQ_FMT_FP8) append_rows_kernel<KVQ_FMT_FP8><<<gr, 256, 0, stream>>>(a);
    else append_rows_kernel<KVQ_FMT_BF16><<<gr, 256, 0, stream>>>(a);
  }
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq

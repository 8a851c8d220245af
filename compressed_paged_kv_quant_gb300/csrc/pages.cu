// pages.cu -- bit-exact page moves between the pool and a page arena (gather / scatter).
//
// "The KV cache and prompt reuse" ("What a sequence is made of"; the tiering and eviction of
// cached pages it describes) moves whole pages between device memory and a slower tier and
// back.  A page here is opaque bytes (every layer and head of 64 tokens), so a move is a copy:
// gather puts pool pages page_ids[0..n) into arena slots 0..n, scatter puts arena slots back
// into pool pages page_ids[0..n).  The arena is any memory the GPU can address: device memory,
// or pinned host memory, which a Grace host exposes to the GPU over NVLink-C2C, so one kernel
// moves the pages without a staging copy.
//
// Grid: (chunks of 16 KB per page, pages); 256 threads; each thread moves 4 x 16 B per chunk.
#include "kvq_internal.cuh"
#include "mma_tma.cuh"

namespace kvq {

constexpr int PAGE_CHUNK = 16384;

__global__ void __launch_bounds__(256) page_move_kernel(uint8_t* pool, uint8_t* arena, const int32_t* page_ids,
                                                        int64_t page_bytes, int64_t pool_pages, int gather,
                                                        int32_t* status) {
  const int i = blockIdx.y;
  const int32_t phys = page_ids[i];
  if (phys < 0 || phys >= pool_pages) {
    if (threadIdx.x == 0 && blockIdx.x == 0) flag(status, KVQ_STATUS_PAGE_OOB);
    return;
  }
  uint8_t* pp = pool + (int64_t)phys * page_bytes;
  uint8_t* ap = arena + (int64_t)i * page_bytes;
  const uint4* src = reinterpret_cast<const uint4*>(gather ? pp : ap);
  uint4* dst = reinterpret_cast<uint4*>(gather ? ap : pp);
  const int64_t n16 = page_bytes / 16;
  const int64_t c0 = (int64_t)blockIdx.x * (PAGE_CHUNK / 16);
  uint4 v[4];
#pragma unroll
  for (int u = 0; u < 4; u++) {
    const int64_t e = c0 + threadIdx.x + 256 * u;
    if (e < n16) v[u] = src[e];
  }
#pragma unroll
  for (int u = 0; u < 4; u++) {
    const int64_t e = c0 + threadIdx.x + 256 * u;
    if (e < n16) dst[e] = v[u];
  }
}

int launch_page_move(uint8_t* pool, uint8_t* arena, const int32_t* page_ids, int n_pages, int64_t page_bytes,
                     int64_t pool_pages, int gather, int32_t* status, cudaStream_t stream) {
  const int64_t chunks = (page_bytes + PAGE_CHUNK - 1) / PAGE_CHUNK;
  for (int p0 = 0; p0 < n_pages; p0 += 65535) {   // gridDim.y limit
    const int np = n_pages - p0 < 65535 ? n_pages - p0 : 65535;
    dim3 grid((unsigned)chunks, (unsigned)np);
    page_move_kernel<<<grid, 256, 0, stream>>>(pool, arena + (int64_t)p0 * page_bytes, page_ids + p0, page_bytes,
                                               pool_pages, gather, status);
  }
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq

// ----------------------------------------------------------------------------- failure path
namespace kvq {
// One warp waits, with the bounded wait every kernel of the library uses, on an mbarrier that
// nothing arrives at: the wait gives up after its iteration limit (tens of milliseconds), the
// kernel sets KVQ_STATUS_TIMEOUT and returns, and the context stays usable.
__global__ void wait_timeout_kernel(int32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(&bar)), "r"(1u) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  const bool done = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bar), 0u));
  if (!done && threadIdx.x == 0) flag(status, KVQ_STATUS_TIMEOUT);
}
}  // namespace kvq

extern "C" int kvq_selftest_wait_timeout(int32_t* d_status, kvq_stream_t stream) {
  if (!d_status) return KVQ_ERR_INVALID_ARG;
  kvq::wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(d_status);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

// decode_noalloc.cu -- paged_decode_attn for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: plugins of a serving engine whose allocator owns
// every byte of the GPU and hands out no scratch, hosts whose memory budget forbids any
// allocation after start-up, and latency-critical loops where an allocation (which may
// synchronise the device) is not allowed.  They still need the split-K decode, which keeps its
// per-split partials (m, l, acc[256] in FP32) in scratch memory.  This entry point takes that
// scratch from one file-scope device array of a fixed size instead of a caller-provided
// workspace; the caller still passes inputs and outputs.
//
// Set-up: the first call on a device looks up the array's device address with
// cudaGetSymbolAddress, once per device, with that device current; make that first call before
// any stream capture begins.
//
// The array lives in every GPU that loads the library, for as long as the process runs.
// Every call shares it: two calls whose kernels overlap on the GPU (different streams, no
// ordering between them) race on it and give undefined results.  Nothing in it has to start
// at zero -- the decode writes every partial it reads within the same call -- so the
// contents a previous call left behind are never observed.
#include <mutex>

#include "kvq_internal.cuh"

namespace kvq {
int check_attn_common(const kvq_geom* g, int layer, const void* pool, size_t pool_bytes, const void* ring,
                      int window, const int32_t* page_table, int max_pages, int lanes, const int32_t* seq_len,
                      int max_seq_len, const void* q, void* workspace, float* out, int32_t* d_status,
                      bool need_workspace);
}  // namespace kvq

namespace {

constexpr size_t SCRATCH_BYTES = (size_t)KVQ_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_decode_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
std::mutex g_lock;
void* g_scratch_addr[MAX_DEVICES] = {nullptr};

// Device address of the scratch array on the current device.  The host-side name of the
// array is only a stand-in for it: a kernel must be given this address, never the symbol.
int scratch_address(void** ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return KVQ_ERR_CUDA;
  std::lock_guard<std::mutex> guard(g_lock);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return KVQ_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *ptr = g_scratch_addr[dev];
  return KVQ_OK;
}

}  // namespace

extern "C" {

int paged_decode_attn_noalloc(const kvq_geom* geom, int layer, const void* pool, size_t pool_bytes,
                              const void* ring, int window, const int32_t* page_table, int max_pages, int lanes,
                              const int32_t* seq_len, int max_seq_len, const void* q, float sm_scale, float* out,
                              int32_t* d_status, kvq_stream_t stream) {
  // the arguments are checked exactly as paged_decode_attn checks them, before the limit
  const int crc = kvq::check_attn_common(geom, layer, pool, pool_bytes, ring, window, page_table, max_pages, lanes,
                                         seq_len, max_seq_len, q, nullptr, out, d_status, false);
  if (crc || lanes == 0) return crc;
  if (kvq_decode_workspace_bytes(geom, lanes, max_seq_len) > SCRATCH_BYTES) return KVQ_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc) return rc;
  return paged_decode_attn(geom, layer, pool, pool_bytes, ring, window, page_table, max_pages, lanes, seq_len,
                           max_seq_len, q, sm_scale, scratch, SCRATCH_BYTES, out, d_status, stream);
}

}  // extern "C"

// kvq_internal.cuh -- layout constants and small device helpers shared by the kernels of
// libkvq.  The format itself is specified in include/kvq.h.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq.h"

namespace kvq {

constexpr int D = 256;             // head_dim
constexpr int P = 64;              // tokens per page
constexpr int HQ2B_ROW = 64;       // bytes of 2-bit code per token row
constexpr int HQ2B_BLOCK = 4608;   // 64 rows x 72 B: codes[64][64] + 512 B of scales / meta
constexpr int HQ2B_META_OFF = 4096;
constexpr int BF16_BLOCK = P * D * 2;  // 32,768 B
constexpr int MAX_GROUP = 8;

// split-K granularity of the generic attention kernel (tokens per split)
constexpr int GENERIC_SPLIT = 1024;   // decode, generic kernel
constexpr int DECODE_SPLIT_HQ2B = 1024;
constexpr int PREFILL_SPLIT = 8192;

__host__ __device__ constexpr int block_bytes(int fmt) { return fmt == KVQ_FMT_HQ2B ? HQ2B_BLOCK : BF16_BLOCK; }

// Everything a kernel needs to address one layer of the cache.
struct CacheView {
  const uint8_t* pool;
  int64_t pool_pages;
  int64_t page_bytes;
  const __nv_bfloat16* ring;  // [lanes][L][H][64][256]; null for BF16
  const int32_t* page_table;
  int max_pages;
  int num_layers, num_kv_heads, num_q_heads, group;
  int layer;
  int window;
  int32_t* status;
};

__device__ __forceinline__ void flag(int32_t* status, int bits) {
  if (status) atomicOr(status, bits);
}

// Byte offset of the (layer, head, kv) block within a page: blocks ordered [layer][head][K,V].
__host__ __device__ __forceinline__ int64_t block_offset(int fmt, int num_kv_heads, int layer, int head, int kv) {
  return ((int64_t)(layer * num_kv_heads + head) * 2 + kv) * block_bytes(fmt);
}

__device__ __forceinline__ int64_t ring_row_offset(const CacheView& c, int lane, int head, int slot) {
  return ((((int64_t)lane * c.num_layers + c.layer) * c.num_kv_heads + head) * P + slot) * D;
}

// First position whose key attention reads exact from the ring: min(len - W, start of the
// page that is still open).
__device__ __forceinline__ int exact_from(int len, int window) {
  int open_start = (len / P) * P;
  int w = len - window;
  return w < open_start ? w : open_start;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float half_bits_to_float(uint16_t h) {
  return __half2float(__ushort_as_half(h));
}

}  // namespace kvq

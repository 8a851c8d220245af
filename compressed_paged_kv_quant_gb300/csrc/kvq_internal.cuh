// kvq_internal.cuh -- layout constants and small device helpers shared by the kernels of
// libkvq.  The format itself is specified in include/kvq.h.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
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
constexpr int FP8_BLOCK = P * D;       // 16,384 B: one E4M3 byte per value
constexpr int MAX_GROUP = 8;

// split-K granularity of the generic attention kernel (tokens per split)
constexpr int GENERIC_SPLIT = 1024;   // decode, generic kernel
constexpr int DECODE_SPLIT_HQ2B = 1024;
constexpr int DECODE_SPLIT_FP8 = 1024;    // tokens per CTA of the FP8 decode kernel
constexpr int DECODE_SPLIT_BF16 = 1024;   // tokens per CTA of the BF16 decode kernel
constexpr int PREFILL_SPLIT = 8192;

__host__ __device__ constexpr int block_bytes(int fmt) {
  return fmt == KVQ_FMT_BF16 ? BF16_BLOCK : fmt == KVQ_FMT_FP8 ? FP8_BLOCK : HQ2B_BLOCK;
}

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
  int rotated;                // KVQ_FMT_HQ2B_HAD: page rows hold Walsh-Hadamard-rotated K and V
  int ktok;                   // KVQ_FMT_HQ2B_TOK: K rows coded per token like V (no page close)
  float k_scale, v_scale;     // KVQ_FMT_FP8: per-tensor scales (1 when the geometry gives 0)
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
// page that is still open); len - W in the per-token-K format, whose keys all have codes.
__device__ __forceinline__ int exact_from(int len, int window, int ktok) {
  int open_start = (len / P) * P;
  int w = len - window;
  return ktok || w < open_start ? w : open_start;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float half_bits_to_float(uint16_t h) {
  return __half2float(__ushort_as_half(h));
}

// FP8 E4M3: eight bf16 values (one uint4) divided by `scale` in fp32 and converted with round to
// nearest even, saturating at +-448 (one byte each, in order), and eight bytes back to floats
// times `scale`.
__device__ __forceinline__ uint2 fp8_encode8(uint4 w, float scale) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
  uint32_t h[4];
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const float2 f = make_float2(__fdiv_rn(bf16_lo(u[i]), scale), __fdiv_rn(bf16_hi(u[i]), scale));
    h[i] = (uint32_t)__nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
  }
  return make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
}
__device__ __forceinline__ void fp8_decode8(uint2 b, float scale, float (&x)[8]) {
  const uint32_t u[2] = {b.x, b.y};
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(u[i >> 1] >> (16 * (i & 1))), __NV_E4M3);
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&r));
    x[2 * i] = f.x * scale;
    x[2 * i + 1] = f.y * scale;
  }
}

// In-place 256-point Walsh-Hadamard transform of one row held by a warp (lane l holds elements
// 8l .. 8l+7), normalized by 1/16 so that it is its own inverse.  Stages h = 1, 2, 4 inside a
// lane, h = 8 .. 128 between lanes l and l ^ (h / 8); every butterfly is (a + b, a - b) with one
// IEEE fp32 operation each, the lower index taking the sum.
__device__ __forceinline__ void warp_fwht256(float (&x)[8]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int h = 1; h < 8; h <<= 1)
#pragma unroll
    for (int i = 0; i < 8; i++)
      if ((i & h) == 0) {
        const float a = x[i], b = x[i + h];
        x[i] = __fadd_rn(a, b);
        x[i + h] = __fsub_rn(a, b);
      }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = lane & m;
#pragma unroll
    for (int i = 0; i < 8; i++) {
      const float o = __shfl_xor_sync(0xFFFFFFFFu, x[i], m);
      x[i] = upper ? __fsub_rn(o, x[i]) : __fadd_rn(x[i], o);
    }
  }
#pragma unroll
  for (int i = 0; i < 8; i++) x[i] = __fmul_rn(x[i], 0.0625f);
}

}  // namespace kvq

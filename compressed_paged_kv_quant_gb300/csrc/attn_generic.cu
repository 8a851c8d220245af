// attn_generic.cu -- split-K paged attention on CUDA cores, for either format, plus the
// log-sum-exp combine shared by every split kernel.
//
// One warp owns one (query row, KV head, key split): lane l holds dims 8l..8l+7 of the G
// query heads of the group and of the running output.  Keys are read straight from the
// compressed pages (no decompressed copy in HBM: "KV at 9 KB a token", "How it works"), the
// score of each key is a warp reduction, and the online softmax keeps the running max, sum
// and output in FP32 registers.  Each split writes its FP32 partial (m, l, acc[256]) once;
// the combine kernel merges the splits in FP32 and rounds once at the end -- the two-level
// accumulation of "Half the Cache, Twice the Context", "The cliff is in the accumulator".
// Scores are kept in the log2 domain (q is pre-scaled by sm_scale * log2 e; exp2 throughout).
#include "kvq_internal.cuh"
#include "attn_args.cuh"

namespace kvq {

template <int FMT>
__device__ __forceinline__ bool page_of(const CacheView& c, int b, int t, const uint8_t*& page) {
  const int pi = t / P;
  const int32_t phys = c.page_table[(int64_t)b * c.max_pages + pi];
  if (phys < 0 || phys >= c.pool_pages) return false;
  page = c.pool + (int64_t)phys * c.page_bytes;
  return true;
}

// grid (max_splits, ceil(max_n_q / warps), lanes * H); blockDim = 32 * warps
template <int FMT>
__global__ void __launch_bounds__(128) attn_split_generic(AttnArgs a, int decode) {
  const CacheView& c = a.c;
  const int H = c.num_kv_heads, G = c.group, Hq = c.num_q_heads;
  const int b = blockIdx.z / H, h = blockIdx.z % H, s = blockIdx.x;
  const int warps = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.y * warps + warp;
  int row, n_keys, len;
  if (!resolve_query(a, decode, b, i, row, n_keys, len, lane == 0 && s == 0 && h == 0)) return;
  const int t0 = s * a.split_tokens;
  if (t0 >= n_keys) return;
  const int t1 = min(t0 + a.split_tokens, n_keys);

  float qv[MAX_GROUP][8];
#pragma unroll
  for (int g = 0; g < MAX_GROUP; g++) {
    if (g < G) {
      const uint4 w = reinterpret_cast<const uint4*>(a.q + ((int64_t)row * Hq + h * G + g) * D)[lane];
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 4; j++) {
        qv[g][2 * j] = bf16_lo(u[j]) * a.scale_log2;
        qv[g][2 * j + 1] = bf16_hi(u[j]) * a.scale_log2;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; j++) qv[g][j] = 0.0f;
    }
  }
  float m[MAX_GROUP], l[MAX_GROUP], acc[MAX_GROUP][8];
#pragma unroll
  for (int g = 0; g < MAX_GROUP; g++) {
    m[g] = -INFINITY;
    l[g] = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; j++) acc[g][j] = 0.0f;
  }
  const int ef = FMT == KVQ_FMT_HQ2B ? exact_from(len, c.window, c.ktok) : len;
  bool oob = false;
  for (int t = t0; t < t1; t++) {
    const uint8_t* page;
    if (!page_of<FMT>(c, b, t, page)) {
      oob = true;
      continue;
    }
    const int slot = t % P;
    const uint8_t* kblk = page + block_offset(FMT, H, c.layer, h, 0);
    const uint8_t* vblk = page + block_offset(FMT, H, c.layer, h, 1);
    float kx[8], vx[8];
    if (FMT == KVQ_FMT_FP8) {
      fp8_decode8(reinterpret_cast<const uint2*>(kblk + slot * D)[lane], c.k_scale, kx);
    } else if (FMT == KVQ_FMT_BF16 || t >= ef) {
      const uint4 w = FMT == KVQ_FMT_BF16
                          ? reinterpret_cast<const uint4*>(kblk + slot * D * 2)[lane]
                          : reinterpret_cast<const uint4*>(c.ring + ring_row_offset(c, b, h, slot))[lane];
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 4; j++) {
        kx[2 * j] = bf16_lo(u[j]);
        kx[2 * j + 1] = bf16_hi(u[j]);
      }
    } else if (c.ktok) {
      // per-token-K format: the key row is coded like a value row
      const uint32_t codes = reinterpret_cast<const uint16_t*>(kblk + slot * HQ2B_ROW)[lane];
      const uint32_t meta = reinterpret_cast<const uint32_t*>(kblk + HQ2B_META_OFF + slot * 8)[lane >> 4];
      const float sk = half_bits_to_float((uint16_t)(meta & 0xFFFFu));
      const float zk = half_bits_to_float((uint16_t)(meta >> 16));
#pragma unroll
      for (int j = 0; j < 8; j++) kx[j] = zk + (float)((codes >> (2 * j)) & 3) * sk;
    } else {
      const uint32_t codes = reinterpret_cast<const uint16_t*>(kblk + slot * HQ2B_ROW)[lane];
      const uint4 sw = reinterpret_cast<const uint4*>(kblk + HQ2B_META_OFF)[lane];
      const __half2* sc = reinterpret_cast<const __half2*>(&sw);
#pragma unroll
      for (int j = 0; j < 4; j++) {
        const float2 sp = __half22float2(sc[j]);
        kx[2 * j] = sp.x * (float)(2 * (int)((codes >> (4 * j)) & 3) - 3);
        kx[2 * j + 1] = sp.y * (float)(2 * (int)((codes >> (4 * j + 2)) & 3) - 3);
      }
    }
    if (FMT == KVQ_FMT_FP8) {
      fp8_decode8(reinterpret_cast<const uint2*>(vblk + slot * D)[lane], c.v_scale, vx);
    } else if (FMT == KVQ_FMT_BF16) {
      const uint4 w = reinterpret_cast<const uint4*>(vblk + slot * D * 2)[lane];
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 4; j++) {
        vx[2 * j] = bf16_lo(u[j]);
        vx[2 * j + 1] = bf16_hi(u[j]);
      }
    } else {
      const uint32_t codes = reinterpret_cast<const uint16_t*>(vblk + slot * HQ2B_ROW)[lane];
      const uint32_t meta = reinterpret_cast<const uint32_t*>(vblk + HQ2B_META_OFF + slot * 8)[lane >> 4];
      const float sv = half_bits_to_float((uint16_t)(meta & 0xFFFFu));
      const float zv = half_bits_to_float((uint16_t)(meta >> 16));
#pragma unroll
      for (int j = 0; j < 8; j++) vx[j] = zv + (float)((codes >> (2 * j)) & 3) * sv;
    }
#pragma unroll
    for (int g = 0; g < MAX_GROUP; g++) {
      if (g < G) {
        float dot = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; j++) dot = fmaf(qv[g][j], kx[j], dot);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, o);
        const float mn = fmaxf(m[g], dot);
        const float alpha = exp2f(m[g] - mn);
        const float p = exp2f(dot - mn);
        m[g] = mn;
        l[g] = l[g] * alpha + p;
#pragma unroll
        for (int j = 0; j < 8; j++) acc[g][j] = fmaf(acc[g][j], alpha, p * vx[j]);
      }
    }
  }
  if (oob && lane == 0) flag(c.status, KVQ_STATUS_PAGE_OOB);
#pragma unroll
  for (int g = 0; g < MAX_GROUP; g++) {
    if (g < G) {
      const int64_t pidx = ((int64_t)row * Hq + h * G + g) * a.max_splits + s;
      float4* o = reinterpret_cast<float4*>(a.ws_o + pidx * D + lane * 8);
      o[0] = make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
      o[1] = make_float4(acc[g][4], acc[g][5], acc[g][6], acc[g][7]);
      if (lane == 0) reinterpret_cast<float2*>(a.ws_ml)[pidx] = make_float2(m[g], l[g]);
    }
  }
}

// Merge the split partials of one (query row, query head): FP32 LSE merge, one rounding.
// grid (lanes * (decode ? 1 : max_n_q), Hq), 256 threads (one per dim).
__global__ void __launch_bounds__(256) attn_combine(AttnArgs a, int decode, int split_tokens) {
  const int per_lane = decode ? 1 : a.max_n_q;
  const int b = blockIdx.x / per_lane, i = blockIdx.x % per_lane, j = blockIdx.y;
  int row, n_keys, len;
  if (!resolve_query(a, decode, b, i, row, n_keys, len, false)) return;
  const int d = threadIdx.x;
  const int Hq = a.c.num_q_heads;
  float* out = a.out + ((int64_t)row * Hq + j) * D;
  const int nsplit = (n_keys + split_tokens - 1) / split_tokens;
  if (nsplit == 0) {
    out[d] = 0.0f;
    return;
  }
  const int64_t p0 = ((int64_t)row * Hq + j) * a.max_splits;
  const float2* ml = reinterpret_cast<const float2*>(a.ws_ml) + p0;
  float mx = -INFINITY;
#pragma unroll 8
  for (int s = 0; s < nsplit; s++) mx = fmaxf(mx, ml[s].x);
  float den = 0.0f, num = 0.0f;
#pragma unroll 8
  for (int s = 0; s < nsplit; s++) {
    const float2 e = ml[s];
    const float w = e.x == -INFINITY ? 0.0f : exp2f(e.x - mx);
    den = fmaf(e.y, w, den);
    num = fmaf(a.ws_o[(p0 + s) * D + d], w, num);
  }
  out[d] = den > 0.0f ? num / den : 0.0f;
}

int decode_split_tokens(int fmt) {
  return fmt == KVQ_FMT_HQ2B ? DECODE_SPLIT_HQ2B
         : fmt == KVQ_FMT_FP8  ? DECODE_SPLIT_FP8
         : fmt == KVQ_FMT_BF16 ? DECODE_SPLIT_BF16
                               : GENERIC_SPLIT;
}
int prefill_split_tokens(int) { return PREFILL_SPLIT; }

int launch_attn_combine(const AttnArgs& a, int decode, cudaStream_t stream) {
  const int rows = decode ? 1 : a.max_n_q;
  dim3 cg(a.lanes * rows, a.c.num_q_heads);
  attn_combine<<<cg, 256, 0, stream>>>(a, decode, a.split_tokens);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

int launch_attn_generic(int fmt, const AttnArgs& a, int decode, cudaStream_t stream) {
  const int warps = decode ? 1 : 4;
  const int rows = decode ? 1 : a.max_n_q;
  dim3 grid(a.max_splits, (rows + warps - 1) / warps, a.lanes * a.c.num_kv_heads);
  if (fmt == KVQ_FMT_HQ2B)
    attn_split_generic<KVQ_FMT_HQ2B><<<grid, 32 * warps, 0, stream>>>(a, decode);
  else if (fmt == KVQ_FMT_FP8)
    attn_split_generic<KVQ_FMT_FP8><<<grid, 32 * warps, 0, stream>>>(a, decode);
  else
    attn_split_generic<KVQ_FMT_BF16><<<grid, 32 * warps, 0, stream>>>(a, decode);
  dim3 cg(a.lanes * rows, a.c.num_q_heads);
  attn_combine<<<cg, 256, 0, stream>>>(a, decode, a.split_tokens);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq

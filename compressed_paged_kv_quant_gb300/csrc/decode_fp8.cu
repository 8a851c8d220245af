// decode_fp8.cu -- split-K decode attention over FP8 E4M3 pages on the tensor cores.
//
// The FP8 format (include/kvq.h) keeps one E4M3 byte per value, 256 B per head per token for K
// and for V: the FP8 cache of the vLLM study that "Half the Cache, Twice the Context" quotes
// ("What the vendors actually measured").  Its decode reads 3.6x the bytes of the 2-bit
// format, so this kernel is built to stream pages at HBM rate with little work per byte.
//
// CTA = 4 warps = one (lane, KV head, split of F8_SPLIT tokens).  A page's K and V blocks of
// this layer and head are adjacent in the page (16 KB each), so one 1-D bulk copy
// (cp.async.bulk) moves both into a F8_STAGES-deep shared-memory ring; every wait is bounded.  Warp w
// takes tokens 16w .. 16w + 15 of every page and runs its own online softmax over them:
//   S = K^ . q^T on mma.sync m16n8k16 (fp16 in, fp32 accumulate): A = K bytes turned into fp16
//     pairs by one cvt.e4m3x2 each (E4M3 -> fp16 is exact), B = q (fp16) of the group's heads
//     (padded to 8).  The contraction order over the 256 dims is permuted so that a thread's A
//     bytes of a k-step are one 32-bit word of its token row; a dot product does not depend
//     on its order.  The K scale multiplies the fp32 score.
//   O^T += V^ . P^T on the same MMA: A = V bytes of two tokens per fp16 pair (one byte permute,
//     two cvt), B = P (fp16, P <= 2^0.5 under the lazy rescale) moved from the S accumulator
//     layout to the B layout with movmatrix.trans.  Rows of O^T are dims in the order
//     32 g + 2 j (+1) for thread row g, so a thread's V bytes are 32 contiguous bytes a token.
// At the end the 4 warps' (m, l, O) merge in FP32 in shared memory, times the V scale, into
// one partial record of the split; the log-sum-exp combine (attn_generic.cu) merges splits --
// the two-level accumulation of "Half the Cache", "The cliff is in the accumulator".
#include "kvq_internal.cuh"
#include "attn_args.cuh"
#include "mma_tma.cuh"

namespace kvq {

#ifndef KVQ_F8_STAGES
#define KVQ_F8_STAGES 2
#endif
#ifndef KVQ_F8_CTAS
#define KVQ_F8_CTAS 3
#endif
constexpr int F8_WARPS = 4;
constexpr int F8_STAGES = KVQ_F8_STAGES;        // pages in the shared-memory ring
constexpr int F8_CTAS = KVQ_F8_CTAS;            // resident CTAs per SM the launch bounds ask for
constexpr int F8_STAGE_BYTES = 2 * FP8_BLOCK;                 // K block + V block: 32 KB
constexpr int F8_Q_OFF = F8_STAGES * F8_STAGE_BYTES;          // q as B fragments: [8][32 lanes] uint4
constexpr int F8_BAR_OFF = F8_Q_OFF + MAX_GROUP * D * 2;      // full[S], empty[S], valid[S]
constexpr int F8_SMEM = F8_BAR_OFF + F8_STAGES * 20 + 16;
constexpr float F8_LAZY = 0.5f;   // lazy rescale: a head's max moves only past +0.5 (log2), P <= 2^0.5

// two E4M3 bytes (low 16 bits) -> fp16 pair, exact
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint32_t x) {
  uint32_t y;
  asm("{\n .reg .b16 t;\n cvt.u16.u32 t, %1;\n cvt.rn.f16x2.e4m3x2 %0, t;\n}\n" : "=r"(y) : "r"(x));
  return y;
}

// grid (lanes * H, splits); 128 threads
__global__ void __launch_bounds__(F8_WARPS * 32, F8_CTAS) decode_fp8_split(AttnArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const CacheView& c = a.c;
  const int H = c.num_kv_heads, G = c.group, Hq = c.num_q_heads;
  const int b = blockIdx.x / H, h = blockIdx.x % H, s = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, cq = lane & 3;
  const int len = a.seq_len[b];
  if (len < 0 || len > c.max_pages * P) {
    if (threadIdx.x == 0 && s == 0 && h == 0) flag(c.status, KVQ_STATUS_LEN_GT_TABLE);
    return;
  }
  const int t0 = s * a.split_tokens;
  if (t0 >= len) return;                      // the combine reads no record of this split
  const int t1 = min(t0 + a.split_tokens, len);
  const int p0 = t0 / P, np = (t1 - t0 + P - 1) / P;

  uint8_t* stage = smem;
  uint4* qf = reinterpret_cast<uint4*>(smem + F8_Q_OFF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + F8_BAR_OFF);
  volatile int* svalid = reinterpret_cast<volatile int*>(smem + F8_BAR_OFF + 16 * F8_STAGES);
  auto FULL = [&](int i) { return smem_u32(&bars[i]); };
  auto EMPTY = [&](int i) { return smem_u32(&bars[F8_STAGES + i]); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < F8_STAGES; i++) {
      mbar_init(FULL(i), 1);
      mbar_init(EMPTY(i), F8_WARPS);
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  // q of head g of the group (zero past G) as this lane's fp16 B fragments: dims 64cq + 8k .. + 7
  // in qf[k * 32 + lane], k = 0..7, so the loop's reads are lane-contiguous (no bank conflicts)
  if (warp == 0) {
#pragma unroll
    for (int k = 0; k < 8; k++) {
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (g < G) w = reinterpret_cast<const uint4*>(a.q + ((int64_t)b * Hq + h * G + g) * D + 64 * cq)[k];
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; j++) o[j] = pack_h2(bf16_lo(u[j]), bf16_hi(u[j]));
      qf[k * 32 + lane] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
  __syncthreads();

  // page j of the split into stage j % F8_STAGES (thread 0 only)
  int issued = 0;
  auto issue = [&](int j) {
    const int st = j % F8_STAGES;
    const int32_t phys = c.page_table[(int64_t)b * c.max_pages + p0 + j];
    const bool ok = phys >= 0 && phys < c.pool_pages;
    svalid[st] = ok ? 1 : 0;
    if (ok) {
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      const uint8_t* src = c.pool + (int64_t)phys * c.page_bytes + block_offset(KVQ_FMT_FP8, H, c.layer, h, 0);
      tma_page(smem_u32(stage + st * F8_STAGE_BYTES), src, F8_STAGE_BYTES, FULL(st));
    } else {
      flag(c.status, KVQ_STATUS_PAGE_OOB);
      asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];\n" ::"r"(FULL(st)) : "memory");
    }
    issued = j + 1;
  };
  if (threadIdx.x == 0)
    for (int j = 0; j < F8_STAGES && j < np; j++) issue(j);

  const float kscale = a.scale_log2 * c.k_scale;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // heads 2cq, 2cq+1
  float O[16][4];
#pragma unroll
  for (int i = 0; i < 16; i++)
#pragma unroll
    for (int e = 0; e < 4; e++) O[i][e] = 0.f;
  bool timed_out = false;
  for (int j = 0; j < np; j++) {
    const int st = j % F8_STAGES;
    const uint32_t par = (j / F8_STAGES) & 1;
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(FULL(st), par))) {
      timed_out = true;
      break;
    }
    if (svalid[st]) {
      const uint8_t* kb = stage + st * F8_STAGE_BYTES;
      const uint8_t* vb = kb + FP8_BLOCK;
      // ---- S = K^ . q^T for tokens 16 warp + g (+8); thread column cq owns dims 64cq .. 64cq+63,
      // k-step 4 c4 + i covering dims 64cq + 16c4 + 4i + {0,1} (A regs 0/1) and {2,3} (regs 2/3)
      const uint8_t* krA = kb + (16 * warp + g) * D + 64 * cq;
      const uint8_t* krB = krA + 8 * D;
      float S[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c4 = 0; c4 < 4; c4++) {
        const uint4 ka = *reinterpret_cast<const uint4*>(krA + 16 * c4);
        const uint4 kbw = *reinterpret_cast<const uint4*>(krB + 16 * c4);
        const uint4 q0 = qf[(2 * c4) * 32 + lane], q1 = qf[(2 * c4 + 1) * 32 + lane];
        const uint32_t wa[4] = {ka.x, ka.y, ka.z, ka.w}, wb[4] = {kbw.x, kbw.y, kbw.z, kbw.w};
        const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
        for (int i = 0; i < 4; i++)
          mma16816(S, e4m3x2_to_h2(wa[i]), e4m3x2_to_h2(wb[i]), e4m3x2_to_h2(wa[i] >> 16), e4m3x2_to_h2(wb[i] >> 16),
                   qw[2 * i], qw[2 * i + 1]);
      }
      // scores (log2 domain), keys past the lane's length masked
      const int tok = (p0 + j) * P + 16 * warp + g;
#pragma unroll
      for (int e = 0; e < 4; e++) S[e] = (tok + 8 * (e >> 1) < len) ? S[e] * kscale : -INFINITY;
      // ---- online softmax over the warp's 16 tokens, per head
      float mx0 = fmaxf(S[0], S[2]), mx1 = fmaxf(S[1], S[3]);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, o));
      }
      float al0 = 1.f, al1 = 1.f;
      if (mx0 > m0 + F8_LAZY) {
        if (m0 != -INFINITY) al0 = ex2(m0 - mx0);
        m0 = mx0;
      }
      if (mx1 > m1 + F8_LAZY) {
        if (m1 != -INFINITY) al1 = ex2(m1 - mx1);
        m1 = mx1;
      }
      if (__any_sync(0xFFFFFFFFu, al0 != 1.f || al1 != 1.f)) {
        l0 *= al0;
        l1 *= al1;
#pragma unroll
        for (int i = 0; i < 16; i++) {
          O[i][0] *= al0; O[i][1] *= al1; O[i][2] *= al0; O[i][3] *= al1;
        }
      }
      const float mu0 = m0 == -INFINITY ? 0.f : m0, mu1 = m1 == -INFINITY ? 0.f : m1;
      const float pa = ex2(S[0] - mu0), pb = ex2(S[1] - mu1), pc = ex2(S[2] - mu0), pd = ex2(S[3] - mu1);
      l0 += pa + pc;
      l1 += pb + pd;
      // P as the B operand (k = token, n = head): transpose the accumulator's 8x8 halves
      const uint32_t b0 = movmatrix_t(pack_h2(pa, pb)), b1 = movmatrix_t(pack_h2(pc, pd));
      // ---- O^T += V^ . P^T; thread row g owns dims 32g .. 32g+31, tokens 2cq, 2cq+1, 2cq+8, 2cq+9
      const uint8_t* vr = vb + (16 * warp + 2 * cq) * D + 32 * g;
#pragma unroll
      for (int hh = 0; hh < 2; hh++) {
        const uint4 r0 = *reinterpret_cast<const uint4*>(vr + 16 * hh);
        const uint4 r1 = *reinterpret_cast<const uint4*>(vr + D + 16 * hh);
        const uint4 r2 = *reinterpret_cast<const uint4*>(vr + 8 * D + 16 * hh);
        const uint4 r3 = *reinterpret_cast<const uint4*>(vr + 9 * D + 16 * hh);
        const uint32_t w0[4] = {r0.x, r0.y, r0.z, r0.w}, w1[4] = {r1.x, r1.y, r1.z, r1.w};
        const uint32_t w2[4] = {r2.x, r2.y, r2.z, r2.w}, w3[4] = {r3.x, r3.y, r3.z, r3.w};
#pragma unroll
        for (int dj = 0; dj < 8; dj++) {      // dims 32g + 16hh + 2dj, +1
          const uint32_t sel = (dj & 1) ? 0x7362u : 0x5140u;
          const uint32_t lo = __byte_perm(w0[dj >> 1], w1[dj >> 1], sel);   // tokens 2cq, 2cq+1
          const uint32_t hi = __byte_perm(w2[dj >> 1], w3[dj >> 1], sel);   // tokens 2cq+8, 2cq+9
          mma16816(O[8 * hh + dj], e4m3x2_to_h2(lo), e4m3x2_to_h2(lo >> 16), e4m3x2_to_h2(hi), e4m3x2_to_h2(hi >> 16),
                   b0, b1);
        }
      }
    }
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];\n" ::"r"(EMPTY(st)) : "memory");
    // refill this stage with page j + F8_STAGES once all four warps have released it
    if (threadIdx.x == 0 && j + F8_STAGES < np) {
      if (mbar_wait(EMPTY(st), par)) issue(j + F8_STAGES);
      else timed_out = true;
    }
    if (warp == 0 && __shfl_sync(0xFFFFFFFFu, (int)timed_out, 0)) {
      timed_out = true;
      break;
    }
  }
  if (timed_out && lane == 0) flag(c.status, KVQ_STATUS_TIMEOUT);
  // copies still in flight must land before the stages are reused (bounded waits)
  if (threadIdx.x == 0)
    for (int j = max(0, issued - F8_STAGES); j < issued; j++) mbar_wait(FULL(j % F8_STAGES), (j / F8_STAGES) & 1);
  __syncthreads();
  if (__syncthreads_or(timed_out)) return;   // the status word reports it; no partial is written

  // ---- merge the 4 warps: per head the largest m, weights 2^(m_w - m), O and l summed in FP32
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, o);
    l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, o);
  }
  float* sm_m = reinterpret_cast<float*>(smem);                 // [4][8]
  float* sm_l = sm_m + F8_WARPS * MAX_GROUP;                    // [4][8]
  float* sm_o = sm_l + F8_WARPS * MAX_GROUP;                    // [4][8 heads][256 dims]
  if (g == 0) {
    sm_m[warp * MAX_GROUP + 2 * cq] = m0;
    sm_m[warp * MAX_GROUP + 2 * cq + 1] = m1;
    sm_l[warp * MAX_GROUP + 2 * cq] = l0;
    sm_l[warp * MAX_GROUP + 2 * cq + 1] = l1;
  }
  __syncthreads();
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int w = 0; w < F8_WARPS; w++) {
    mx[0] = fmaxf(mx[0], sm_m[w * MAX_GROUP + 2 * cq]);
    mx[1] = fmaxf(mx[1], sm_m[w * MAX_GROUP + 2 * cq + 1]);
  }
  const float own[2] = {m0, m1};
  float wt[2];
#pragma unroll
  for (int e = 0; e < 2; e++) wt[e] = own[e] == -INFINITY ? 0.f : ex2(own[e] - mx[e]);
#pragma unroll
  for (int i = 0; i < 16; i++)
#pragma unroll
    for (int e = 0; e < 4; e++) {
      const int head = 2 * cq + (e & 1), dim = 32 * g + 2 * i + (e >> 1);
      sm_o[(warp * MAX_GROUP + head) * D + dim] = O[i][e] * wt[e & 1];
    }
  __syncthreads();
  const int64_t base = ((int64_t)b * Hq + h * G) * a.max_splits + s;
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int head = i / D, dim = i % D;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < F8_WARPS; w++) v += sm_o[(w * MAX_GROUP + head) * D + dim];
    a.ws_o[(base + (int64_t)head * a.max_splits) * D + dim] = v * c.v_scale;
  }
  if (threadIdx.x < G) {
    const int head = threadIdx.x;
    float m = -INFINITY, l = 0.f;
    for (int w = 0; w < F8_WARPS; w++) m = fmaxf(m, sm_m[w * MAX_GROUP + head]);
    for (int w = 0; w < F8_WARPS; w++) {
      const float mw = sm_m[w * MAX_GROUP + head];
      if (mw != -INFINITY) l += sm_l[w * MAX_GROUP + head] * ex2(mw - m);
    }
    reinterpret_cast<float2*>(a.ws_ml)[base + (int64_t)head * a.max_splits] = make_float2(m, l);
  }
}

int launch_attn_combine(const AttnArgs& a, int decode, cudaStream_t stream);

int launch_decode_fp8(const AttnArgs& a, cudaStream_t stream) {
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!attr_set[dev]) {
    cudaFuncSetAttribute(decode_fp8_split, cudaFuncAttributeMaxDynamicSharedMemorySize, F8_SMEM);
    attr_set[dev] = true;
  }
  const int splits = (int)((a.max_seq_len + a.split_tokens - 1) / a.split_tokens);
  if (splits > 0) {
    dim3 grid(a.lanes * a.c.num_kv_heads, splits);
    decode_fp8_split<<<grid, F8_WARPS * 32, F8_SMEM, stream>>>(a);
  }
  if (cudaGetLastError() != cudaSuccess) return KVQ_ERR_CUDA;
  return launch_attn_combine(a, 1, stream);
}

}  // namespace kvq

// decode_fp8.cu -- split-K decode attention over FP8 E4M3 pages on the tensor cores.
//
// The FP8 format (include/kvq.h) keeps one E4M3 byte per value, 256 B per head per token for K
// and for V: the FP8 cache of the vLLM study that "Half the Cache, Twice the Context" quotes
// ("What the vendors actually measured").  Its decode reads 3.6x the bytes of the 2-bit
// format, so this kernel is built to stream pages at HBM rate with little work per byte.
//
// CTA = 4 warps = one (lane, KV head, split of F8_SPLIT tokens).  A page's K and V blocks of
// this layer and head (16 KB each, adjacent in the page) are copied by all 128 threads with
// 16 B cp.async into a F8_STAGES-deep shared-memory ring whose rows are padded from 256 to
// 272 B: with the fragment ownership below, every 16 B shared-memory read of a warp then hits
// eight different bank groups (unpadded rows 256 B apart put K reads 2-way and V reads 4-way
// in conflict).  Completion is an mbarrier of 128 cp.async arrivals; every wait is bounded.
// Warp w takes tokens 16w .. 16w + 15 of every page and runs its own online softmax over them:
//   S = K^ . q^T on mma.sync m16n8k16 (fp16 in, fp32 accumulate): A = K bytes turned into fp16
//     pairs by one cvt.e4m3x2 each (E4M3 -> fp16 is exact), B = q (fp16) of the group's heads
//     (padded to 8).  The contraction order over the 256 dims is permuted so that a thread's A
//     bytes of a k-step are one 32-bit word of its token row (thread column cq reads 16 B chunks
//     2cq + 8(c4 & 1) + (c4 >> 1), c4 = 0..3); a dot product does not depend on its order.  The
//     K scale multiplies the fp32 score.
//   O^T += V^ . P^T on the same MMA: A = V bytes of two tokens per fp16 pair (one byte permute,
//     two cvt), B = P (fp16, P <= 2^0.5 under the lazy rescale) moved from the S accumulator
//     layout to the B layout with movmatrix.trans.  Rows of O^T are dims: thread row g owns
//     dims 128 hh + 16 g + 0..15 (hh = 0, 1), 16 contiguous bytes of a token row per hh.
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
constexpr int F8_ROW = D + 16;                                // a padded 256 B page row
constexpr int F8_STAGE_BYTES = 2 * P * F8_ROW;                // K rows then V rows: 34,816 B
constexpr int F8_Q_OFF = F8_STAGES * F8_STAGE_BYTES;          // q as B fragments: [8][32 lanes] uint4
constexpr int F8_BAR_OFF = F8_Q_OFF + MAX_GROUP * D * 2;      // full[S]
constexpr int F8_SMEM = F8_BAR_OFF + F8_STAGES * 8;
constexpr float F8_LAZY = 0.5f;   // lazy rescale: a head's max moves only past +0.5 (log2), P <= 2^0.5

// 16 B chunk of thread column cq for k-step group c4 (conflict-free K reads, see above)
__device__ __forceinline__ int f8_kchunk(int cq, int c4) { return 2 * cq + 8 * (c4 & 1) + (c4 >> 1); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}

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
  if (const int e = lane_len_error(a, len)) {
    if (threadIdx.x == 0 && s == 0 && h == 0) flag(c.status, e);
    return;
  }
  const int t0 = s * a.split_tokens;
  if (t0 >= len) return;                      // the combine reads no record of this split
  const int t1 = min(t0 + a.split_tokens, len);
  const int p0 = t0 / P, np = (t1 - t0 + P - 1) / P;

  uint8_t* stage = smem;
  uint4* qf = reinterpret_cast<uint4*>(smem + F8_Q_OFF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + F8_BAR_OFF);
  auto FULL = [&](int i) { return smem_u32(&bars[i]); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < F8_STAGES; i++) mbar_init(FULL(i), F8_WARPS * 32);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  // q of head g of the group (zero past G) as this lane's fp16 B fragments: dims
  // 16 f8_kchunk(cq, k / 2) + 8 (k & 1) .. + 7 in qf[k * 32 + lane], k = 0..7, so the loop's reads
  // are lane-contiguous (no bank conflicts)
  if (warp == 0) {
#pragma unroll
    for (int k = 0; k < 8; k++) {
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (g < G)
        w = reinterpret_cast<const uint4*>(a.q + ((int64_t)b * Hq + h * G + g) * D)[2 * f8_kchunk(cq, k >> 1) + (k & 1)];
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; j++) o[j] = pack_h2(bf16_lo(u[j]), bf16_hi(u[j]));
      qf[k * 32 + lane] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
  __syncthreads();

  // page j of the split into stage j % F8_STAGES, by every thread: 16 B chunk q = thread + 128 i of
  // the page's 2,048 (K block then V block) to row q / 16, column q % 16 of the padded ring
  uint32_t valid = 0;   // bit per stage: the page is in the pool (same in every thread)
  auto issue = [&](int j) {
    const int st = j % F8_STAGES;
    const int32_t phys = c.page_table[(int64_t)b * c.max_pages + p0 + j];
    const bool ok = phys >= 0 && phys < c.pool_pages;
    valid = ok ? (valid | (1u << st)) : (valid & ~(1u << st));
    if (ok) {
      const uint8_t* src = c.pool + (int64_t)phys * c.page_bytes + block_offset(KVQ_FMT_FP8, H, c.layer, h, 0);
      const uint32_t dst = smem_u32(stage + st * F8_STAGE_BYTES);
#pragma unroll 4
      for (int i = 0; i < 2 * FP8_BLOCK / 16 / (F8_WARPS * 32); i++) {
        const int q = threadIdx.x + F8_WARPS * 32 * i;
        cp_async16(dst + (q >> 4) * F8_ROW + 16 * (q & 15), src + 16 * q);
      }
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(FULL(st)) : "memory");
    } else {
      if (threadIdx.x == 0) flag(c.status, KVQ_STATUS_PAGE_OOB);
      asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];\n" ::"r"(FULL(st)) : "memory");
    }
  };
  __syncthreads();   // barrier initialisation visible to every thread
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
    if (__syncthreads_or(!mbar_wait(FULL(st), par))) {   // every thread leaves together
      timed_out = true;
      break;
    }
    if (valid & (1u << st)) {
      const uint8_t* kb = stage + st * F8_STAGE_BYTES;
      const uint8_t* vb = kb + P * F8_ROW;
      // ---- S = K^ . q^T for tokens 16 warp + g (+8); k-step 4 c4 + i of thread column cq covers
      // dims 16 f + 4i + {0,1} (A regs 0/1) and {2,3} (regs 2/3), f = f8_kchunk(cq, c4)
      const uint8_t* krA = kb + (16 * warp + g) * F8_ROW;
      const uint8_t* krB = krA + 8 * F8_ROW;
      float S[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c4 = 0; c4 < 4; c4++) {
        const int f = f8_kchunk(cq, c4);
        const uint4 ka = *reinterpret_cast<const uint4*>(krA + 16 * f);
        const uint4 kbw = *reinterpret_cast<const uint4*>(krB + 16 * f);
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
      // ---- O^T += V^ . P^T; thread row g owns dims 128 hh + 16g + 0..15, tokens 2cq, 2cq+1,
      // 2cq+8, 2cq+9
      const uint8_t* vr = vb + (16 * warp + 2 * cq) * F8_ROW + 16 * g;
#pragma unroll
      for (int hh = 0; hh < 2; hh++) {
        const uint4 r0 = *reinterpret_cast<const uint4*>(vr + 128 * hh);
        const uint4 r1 = *reinterpret_cast<const uint4*>(vr + F8_ROW + 128 * hh);
        const uint4 r2 = *reinterpret_cast<const uint4*>(vr + 8 * F8_ROW + 128 * hh);
        const uint4 r3 = *reinterpret_cast<const uint4*>(vr + 9 * F8_ROW + 128 * hh);
        const uint32_t w0[4] = {r0.x, r0.y, r0.z, r0.w}, w1[4] = {r1.x, r1.y, r1.z, r1.w};
        const uint32_t w2[4] = {r2.x, r2.y, r2.z, r2.w}, w3[4] = {r3.x, r3.y, r3.z, r3.w};
#pragma unroll
        for (int dj = 0; dj < 8; dj++) {      // dims 128hh + 16g + 2dj, +1
          const uint32_t sel = (dj & 1) ? 0x7362u : 0x5140u;
          const uint32_t lo = __byte_perm(w0[dj >> 1], w1[dj >> 1], sel);   // tokens 2cq, 2cq+1
          const uint32_t hi = __byte_perm(w2[dj >> 1], w3[dj >> 1], sel);   // tokens 2cq+8, 2cq+9
          mma16816(O[8 * hh + dj], e4m3x2_to_h2(lo), e4m3x2_to_h2(lo >> 16), e4m3x2_to_h2(hi), e4m3x2_to_h2(hi >> 16),
                   b0, b1);
        }
      }
    }
    // every warp is done with this stage: refill it with page j + F8_STAGES
    __syncthreads();
    if (j + F8_STAGES < np) issue(j + F8_STAGES);
  }
  if (timed_out && threadIdx.x == 0) flag(c.status, KVQ_STATUS_TIMEOUT);
  // this thread's copies still in flight land before the stages are reused or the CTA exits
  asm volatile("cp.async.wait_all;\n" ::: "memory");
  __syncthreads();
  if (timed_out) return;   // (uniform) the status word reports it; no partial is written

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
      const int head = 2 * cq + (e & 1), dim = 128 * (i >> 3) + 16 * g + 2 * (i & 7) + (e >> 1);
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
    cudaFuncSetAttribute(decode_fp8_split, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
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

// decode_bf16.cu -- split-K decode attention over BF16 pages on the tensor cores.
//
// The BF16 format keeps every K and V value as it came, 512 B per head per token each: the
// exact reference the 2-bit format is measured against ("KV at 9 KB a token", "How it works";
// the decode price of the compressed cache against BF16 is quoted in "The numbers").  Its
// decode reads 7.1x the bytes of the 2-bit format and little arithmetic per byte, so this kernel
// only has to stream pages at HBM rate.
//
// CTA = 2 warps = one (lane, KV head, split of DECODE_SPLIT_BF16 tokens), two CTAs per SM, so
// one CTA's first copies overlap the other's steady stream.  A half page -- the K and V rows of
// 32 tokens of this layer and head -- is one stage: copied by the 64 threads with 16 B cp.async
// into a B16_STAGES-deep ring whose rows are padded from 512 to 528 B; completion is an mbarrier
// of 64 cp.async arrivals, every wait bounded.  Warp w takes tokens 16w .. 16w + 15 of every
// half page and runs its own online softmax:
//   S = K . q^T on mma.sync m16n8k16 with bf16 operands as they are stored: A = K rows, B = q of
//     the group's heads (padded to 8).  Thread column cq reads 16 contiguous bytes (the dims of
//     two k-steps) of its key rows, so the contraction order over the 256 dims is permuted; a dot
//     product does not depend on it.
//   O^T += V^T . P^T on the same MMA: A = V of two tokens per bf16 pair (one byte permute),
//     B = P as bf16 in two parts, P = P_hi + P_lo (P_lo = bf16(P - P_hi)), two MMAs with the same
//     A: together ~16 significant bits of every weight, so bf16 operands cost no accuracy
//     against the FP32 oracle.  Thread row g owns 32 contiguous dims of every value row, read in
//     four 16 B chunks whose order rotates with g so that a warp's reads spread over all banks.
// At the end the 2 warps' (m, l, O) merge in FP32 in shared memory into one partial record of
// the split; attn_combine merges the splits -- the two-level accumulation of "Half the Cache,
// Twice the Context", "The cliff is in the accumulator".
#include "kvq_internal.cuh"
#include "attn_args.cuh"
#include "mma_tma.cuh"

namespace kvq {

constexpr int B16_WARPS = 2;
constexpr int B16_STAGES = 3;                                 // half pages in the ring
constexpr int B16_T = 16 * B16_WARPS;                         // tokens a stage: 32
constexpr int B16_ROW = 2 * D + 16;                           // a padded 512 B row: 528 B
constexpr int B16_STAGE_BYTES = 2 * B16_T * B16_ROW;          // K rows then V rows: 33,792 B
constexpr int B16_Q_OFF = B16_STAGES * B16_STAGE_BYTES;       // q as B fragments: [8][32 lanes] uint4
constexpr int B16_BAR_OFF = B16_Q_OFF + 8 * 32 * 16;          // full[S]
constexpr int B16_SMEM = B16_BAR_OFF + B16_STAGES * 8;
constexpr float B16_LAZY = 0.5f;   // lazy rescale: a head's max moves only past +0.5 (log2), P <= 2^0.5

__device__ __forceinline__ void mma16816_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void b16_cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&r);
}

// the 16 B chunk of thread row g's j-th read in a value row (its 32 dims are chunks 4g .. 4g+3)
__device__ __forceinline__ int b16_vchunk(int g, int j) { return 4 * g + ((j + (g >> 1)) & 3); }

// grid (lanes * H, splits); 64 threads
__global__ void __launch_bounds__(B16_WARPS * 32, 2) decode_bf16_split(AttnArgs a) {
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
  // stages: half pages of the split (a split starts on a page boundary)
  const int p0 = t0 / P, np = (t1 - t0 + B16_T - 1) / B16_T;

  uint8_t* stage = smem;
  uint4* qf = reinterpret_cast<uint4*>(smem + B16_Q_OFF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + B16_BAR_OFF);
  auto FULL = [&](int i) { return smem_u32(&bars[i]); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < B16_STAGES; i++) mbar_init(FULL(i), B16_WARPS * 32);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  // q of head g of the group (zero past G) as this lane's bf16 B fragments: dims 32p + 8cq .. +7
  // in qf[p * 32 + lane], p = 0..7 (k-steps 2p, 2p+1), lane-contiguous reads in the loop
  if (warp == 0) {
#pragma unroll
    for (int p = 0; p < 8; p++) {
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (g < G) w = reinterpret_cast<const uint4*>(a.q + ((int64_t)b * Hq + h * G + g) * D)[4 * p + cq];
      qf[p * 32 + lane] = w;
    }
  }
  __syncthreads();

  // half page j of the split (tokens 32 (j % 2) .. + 31 of page p0 + j / 2) into stage
  // j % B16_STAGES, by every thread: 16 B chunk q = thread + 64 i of its 2,048 (K rows then V
  // rows) to row q / 32, column q % 32 of the padded ring
  uint32_t valid = 0;   // bit per stage: the page is in the pool (same in every thread)
  auto issue = [&](int j) {
    const int st = j % B16_STAGES;
    const int32_t phys = c.page_table[(int64_t)b * c.max_pages + p0 + j / 2];
    const bool ok = phys >= 0 && phys < c.pool_pages;
    valid = ok ? (valid | (1u << st)) : (valid & ~(1u << st));
    if (ok) {
      const uint8_t* kbl = c.pool + (int64_t)phys * c.page_bytes + block_offset(KVQ_FMT_BF16, H, c.layer, h, 0) +
                           (j & 1) * (B16_T * 2 * D);
      const uint32_t dst = smem_u32(stage + st * B16_STAGE_BYTES);
#pragma unroll 8
      for (int i = 0; i < 2 * B16_T * 2 * D / 16 / (B16_WARPS * 32); i++) {
        const int q = threadIdx.x + B16_WARPS * 32 * i;
        const int row = q >> 5;   // 0 .. 63: K rows then V rows of the half page
        const uint8_t* src = kbl + (row >= B16_T ? BF16_BLOCK - B16_T * 2 * D : 0) + 16 * q;
        b16_cp_async16(dst + row * B16_ROW + 16 * (q & 31), src);
      }
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(FULL(st)) : "memory");
    } else {
      if (threadIdx.x == 0) flag(c.status, KVQ_STATUS_PAGE_OOB);
      asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];\n" ::"r"(FULL(st)) : "memory");
    }
  };
  __syncthreads();   // barrier initialisation visible to every thread
  for (int j = 0; j < B16_STAGES && j < np; j++) issue(j);

  const float kscale = a.scale_log2;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // heads 2cq, 2cq+1
  float O[16][4];
#pragma unroll
  for (int i = 0; i < 16; i++)
#pragma unroll
    for (int e = 0; e < 4; e++) O[i][e] = 0.f;
  bool timed_out = false;
  for (int j = 0; j < np; j++) {
    const int st = j % B16_STAGES;
    const uint32_t par = (j / B16_STAGES) & 1;
    if (__syncthreads_or(!mbar_wait(FULL(st), par))) {   // every thread leaves together
      timed_out = true;
      break;
    }
    if (valid & (1u << st)) {
      const uint8_t* kb = stage + st * B16_STAGE_BYTES;
      const uint8_t* vb = kb + B16_T * B16_ROW;
      // ---- S = K . q^T for tokens 16 warp + g (+8); k-steps 2p, 2p+1 of thread column cq
      // cover dims 32p + 8cq .. +3 and +4 .. +7 (A regs 0/2: row g, 1/3: row g + 8)
      const uint8_t* krA = kb + (16 * warp + g) * B16_ROW + 16 * cq;
      const uint8_t* krB = krA + 8 * B16_ROW;
      float S[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int p = 0; p < 8; p++) {
        const uint4 ka = *reinterpret_cast<const uint4*>(krA + 64 * p);
        const uint4 kbw = *reinterpret_cast<const uint4*>(krB + 64 * p);
        const uint4 qw = qf[p * 32 + lane];
        mma16816_bf16(S, ka.x, kbw.x, ka.y, kbw.y, qw.x, qw.y);
        mma16816_bf16(S, ka.z, kbw.z, ka.w, kbw.w, qw.z, qw.w);
      }
      // scores (log2 domain), keys past the lane's length masked
      const int tok = p0 * P + j * B16_T + 16 * warp + g;
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
      if (mx0 > m0 + B16_LAZY) {
        if (m0 != -INFINITY) al0 = ex2(m0 - mx0);
        m0 = mx0;
      }
      if (mx1 > m1 + B16_LAZY) {
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
      // P = P_hi + P_lo in bf16, each moved from the accumulator layout to the B layout
      const uint32_t h01 = pack_bf2(pa, pb), h23 = pack_bf2(pc, pd);
      const uint32_t l01 = pack_bf2(pa - bf16_lo(h01), pb - bf16_hi(h01));
      const uint32_t l23 = pack_bf2(pc - bf16_lo(h23), pd - bf16_hi(h23));
      const uint32_t bh0 = movmatrix_t(h01), bh1 = movmatrix_t(h23);
      const uint32_t bl0 = movmatrix_t(l01), bl1 = movmatrix_t(l23);
      // ---- O^T += V^T . P^T; thread row g owns dims 32g .. 32g + 31 in four 16 B chunks (tokens
      // 2cq, 2cq+1, 2cq+8, 2cq+9 of the warp's 16); O[4 jc + i] holds dims
      // 8 b16_vchunk(g, jc) + 2i (rows g) and + 1 (rows g + 8)
      const uint8_t* vr = vb + (16 * warp + 2 * cq) * B16_ROW;
#pragma unroll
      for (int jc = 0; jc < 4; jc++) {
        const int off = 16 * b16_vchunk(g, jc);
        const uint4 r0 = *reinterpret_cast<const uint4*>(vr + off);
        const uint4 r1 = *reinterpret_cast<const uint4*>(vr + B16_ROW + off);
        const uint4 r2 = *reinterpret_cast<const uint4*>(vr + 8 * B16_ROW + off);
        const uint4 r3 = *reinterpret_cast<const uint4*>(vr + 9 * B16_ROW + off);
        const uint32_t w0[4] = {r0.x, r0.y, r0.z, r0.w}, w1[4] = {r1.x, r1.y, r1.z, r1.w};
        const uint32_t w2[4] = {r2.x, r2.y, r2.z, r2.w}, w3[4] = {r3.x, r3.y, r3.z, r3.w};
#pragma unroll
        for (int i = 0; i < 4; i++) {
          const uint32_t a0 = __byte_perm(w0[i], w1[i], 0x5410u), a1 = __byte_perm(w0[i], w1[i], 0x7632u);
          const uint32_t a2 = __byte_perm(w2[i], w3[i], 0x5410u), a3 = __byte_perm(w2[i], w3[i], 0x7632u);
          mma16816_bf16(O[4 * jc + i], a0, a1, a2, a3, bh0, bh1);
          mma16816_bf16(O[4 * jc + i], a0, a1, a2, a3, bl0, bl1);
        }
      }
    }
    // every warp is done with this stage: refill it with page j + B16_STAGES
    __syncthreads();
    if (j + B16_STAGES < np) issue(j + B16_STAGES);
  }
  if (timed_out && threadIdx.x == 0) flag(c.status, KVQ_STATUS_TIMEOUT);
  // this thread's copies still in flight land before the stages are reused or the CTA exits
  asm volatile("cp.async.wait_all;\n" ::: "memory");
  __syncthreads();
  if (timed_out) return;   // (uniform) the status word reports it; no partial is written

  // ---- merge the warps: per head the largest m, weights 2^(m_w - m), O and l summed in FP32
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, o);
    l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, o);
  }
  float* sm_m = reinterpret_cast<float*>(smem);                 // [warps][8]
  float* sm_l = sm_m + B16_WARPS * MAX_GROUP;                   // [warps][8]
  float* sm_o = sm_l + B16_WARPS * MAX_GROUP;                   // [warps][8 heads][256 dims]
  if (g == 0) {
    sm_m[warp * MAX_GROUP + 2 * cq] = m0;
    sm_m[warp * MAX_GROUP + 2 * cq + 1] = m1;
    sm_l[warp * MAX_GROUP + 2 * cq] = l0;
    sm_l[warp * MAX_GROUP + 2 * cq + 1] = l1;
  }
  __syncthreads();
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int w = 0; w < B16_WARPS; w++) {
    mx[0] = fmaxf(mx[0], sm_m[w * MAX_GROUP + 2 * cq]);
    mx[1] = fmaxf(mx[1], sm_m[w * MAX_GROUP + 2 * cq + 1]);
  }
  const float own[2] = {m0, m1};
  float wt[2];
#pragma unroll
  for (int e = 0; e < 2; e++) wt[e] = own[e] == -INFINITY ? 0.f : ex2(own[e] - mx[e]);
#pragma unroll
  for (int jc = 0; jc < 4; jc++)
#pragma unroll
    for (int i = 0; i < 4; i++)
#pragma unroll
      for (int e = 0; e < 4; e++) {
        const int head = 2 * cq + (e & 1), dim = 8 * b16_vchunk(g, jc) + 2 * i + (e >> 1);
        sm_o[(warp * MAX_GROUP + head) * D + dim] = O[4 * jc + i][e] * wt[e & 1];
      }
  __syncthreads();
  const int64_t base = ((int64_t)b * Hq + h * G) * a.max_splits + s;
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int head = i / D, dim = i % D;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < B16_WARPS; w++) v += sm_o[(w * MAX_GROUP + head) * D + dim];
    a.ws_o[(base + (int64_t)head * a.max_splits) * D + dim] = v;
  }
  if (threadIdx.x < G) {
    const int head = threadIdx.x;
    float m = -INFINITY, l = 0.f;
    for (int w = 0; w < B16_WARPS; w++) m = fmaxf(m, sm_m[w * MAX_GROUP + head]);
    for (int w = 0; w < B16_WARPS; w++) {
      const float mw = sm_m[w * MAX_GROUP + head];
      if (mw != -INFINITY) l += sm_l[w * MAX_GROUP + head] * ex2(mw - m);
    }
    reinterpret_cast<float2*>(a.ws_ml)[base + (int64_t)head * a.max_splits] = make_float2(m, l);
  }
}

int launch_attn_combine(const AttnArgs& a, int decode, cudaStream_t stream);

int launch_decode_bf16(const AttnArgs& a, cudaStream_t stream) {
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!attr_set[dev]) {
    cudaFuncSetAttribute(decode_bf16_split, cudaFuncAttributeMaxDynamicSharedMemorySize, B16_SMEM);
    cudaFuncSetAttribute(decode_bf16_split, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    attr_set[dev] = true;
  }
  const int splits = (int)((a.max_seq_len + a.split_tokens - 1) / a.split_tokens);
  if (splits > 0) {
    dim3 grid(a.lanes * a.c.num_kv_heads, splits);
    decode_bf16_split<<<grid, B16_WARPS * 32, B16_SMEM, stream>>>(a);
  }
  if (cudaGetLastError() != cudaSuccess) return KVQ_ERR_CUDA;
  return launch_attn_combine(a, 1, stream);
}

}  // namespace kvq

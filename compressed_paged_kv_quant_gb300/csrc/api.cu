// api.cu -- the C ABI of libkvq (declared in include/kvq.h): argument validation, sizing
// helpers, and the launches.  Every check here runs on the host before any kernel is
// enqueued, so a rejected call moves no byte; there is no CPU fallback for anything.
#include <stdio.h>

#include "kvq_internal.cuh"

namespace kvq {
int launch_append(int fmt, const CacheView& c, uint8_t* pool, __nv_bfloat16* ring, const int32_t* start_pos,
                  const int32_t* n_new, const int32_t* tok_offset, int max_new, int n_rows, int lanes,
                  const __nv_bfloat16* k, const __nv_bfloat16* v, cudaStream_t stream);
struct AttnArgs;
int launch_attn_generic(int fmt, const AttnArgs& a, int decode, cudaStream_t stream);
int launch_decode_hq2b(const AttnArgs& a, cudaStream_t stream);
int launch_append_last(const CacheView& c, uint8_t* pool, __nv_bfloat16* ring, const int32_t* start_pos,
                       const int32_t* n_new, const int32_t* tok_offset, int n_rows, int lanes,
                       const __nv_bfloat16* k, const __nv_bfloat16* v, cudaStream_t stream);
int launch_decode_fp8(const AttnArgs& a, cudaStream_t stream);
int launch_decode_bf16(const AttnArgs& a, cudaStream_t stream);
int decode_split_tokens(int fmt);
int prefill_split_tokens(int fmt);
int decode_hq2b_slots(int max_seq_len);
int launch_prefill_tc(int fmt, const AttnArgs& a, cudaStream_t stream);
int launch_attn_combine(const AttnArgs& a, int decode, cudaStream_t stream);
int launch_page_move(uint8_t* pool, uint8_t* arena, const int32_t* page_ids, int n_pages, int64_t page_bytes,
                     int64_t pool_pages, int gather, int32_t* status, cudaStream_t stream);
}  // namespace kvq

#include "attn_args.cuh"

using namespace kvq;

namespace {

constexpr float LOG2E = 1.4426950408889634f;

int check_geom(const kvq_geom* g) {
  if (!g) return KVQ_ERR_INVALID_ARG;
  if (g->format != KVQ_FMT_HQ2B && g->format != KVQ_FMT_BF16 && g->format != KVQ_FMT_HQ2B_HAD &&
      g->format != KVQ_FMT_HQ2B_TOK && g->format != KVQ_FMT_FP8)
    return KVQ_ERR_UNSUPPORTED;
  if (g->format == KVQ_FMT_FP8 && (!(g->k_scale >= 0.0f && g->k_scale <= 3.0e38f) ||
                                   !(g->v_scale >= 0.0f && g->v_scale <= 3.0e38f)))
    return KVQ_ERR_INVALID_ARG;
  if (g->head_dim != D || g->page_tokens != P) return KVQ_ERR_UNSUPPORTED;
  if (g->num_layers <= 0 || g->num_kv_heads <= 0 || g->num_q_heads <= 0) return KVQ_ERR_INVALID_ARG;
  if (g->num_layers > 4096 || g->num_kv_heads > 1024) return KVQ_ERR_UNSUPPORTED;
  if (g->num_q_heads % g->num_kv_heads != 0) return KVQ_ERR_INVALID_ARG;
  if (g->num_q_heads / g->num_kv_heads > MAX_GROUP) return KVQ_ERR_UNSUPPORTED;
  return KVQ_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// the byte layout a format uses: the rotated and per-token-K variants keep HQ2B's
int layout_fmt(int f) { return f == KVQ_FMT_HQ2B_HAD || f == KVQ_FMT_HQ2B_TOK ? KVQ_FMT_HQ2B : f; }
bool two_bit(int f) { return layout_fmt(f) == KVQ_FMT_HQ2B; }

size_t page_bytes_of(const kvq_geom* g) {
  return (size_t)g->num_layers * g->num_kv_heads * 2 * (size_t)block_bytes(g->format);
}

size_t partial_bytes(int64_t rows, int hq, int64_t splits) {
  const int64_t n = rows * hq * splits;
  size_t bytes = (size_t)n * D * sizeof(float) + (size_t)n * 2 * sizeof(float);
  return (bytes + 255) & ~(size_t)255;
}

int64_t splits_for(int64_t max_len, int split) { return max_len <= 0 ? 1 : (max_len + split - 1) / split; }

// partial records per (lane, query head) the decode kernels may write
int64_t decode_slots(int fmt, int max_seq_len) {
  fmt = layout_fmt(fmt);
  return fmt == KVQ_FMT_HQ2B ? decode_hq2b_slots(max_seq_len) : splits_for(max_seq_len, decode_split_tokens(fmt));
}

CacheView make_view(const kvq_geom* g, int layer, const void* pool, size_t pool_bytes, const void* ring,
                    const int32_t* page_table, int max_pages, int window, int32_t* status) {
  CacheView c;
  c.pool = static_cast<const uint8_t*>(pool);
  c.page_bytes = (int64_t)page_bytes_of(g);
  c.pool_pages = (int64_t)(pool_bytes / (size_t)c.page_bytes);
  c.ring = static_cast<const __nv_bfloat16*>(ring);
  c.page_table = page_table;
  c.max_pages = max_pages;
  c.num_layers = g->num_layers;
  c.num_kv_heads = g->num_kv_heads;
  c.num_q_heads = g->num_q_heads;
  c.group = g->num_q_heads / g->num_kv_heads;
  c.layer = layer;
  c.window = window;
  c.status = status;
  c.rotated = g->format == KVQ_FMT_HQ2B_HAD;
  c.ktok = g->format == KVQ_FMT_HQ2B_TOK;
  c.k_scale = g->format == KVQ_FMT_FP8 && g->k_scale != 0.0f ? g->k_scale : 1.0f;
  c.v_scale = g->format == KVQ_FMT_FP8 && g->v_scale != 0.0f ? g->v_scale : 1.0f;
  return c;
}

}  // namespace

namespace kvq {
// Checks shared by the attention entry points (the workspace pointer too unless
// need_workspace is false: the no-allocation decode supplies its own).
int check_attn_common(const kvq_geom* g, int layer, const void* pool, size_t pool_bytes, const void* ring,
                      int window, const int32_t* page_table, int max_pages, int lanes, const int32_t* seq_len,
                      int max_seq_len, const void* q, void* workspace, float* out, int32_t* d_status,
                      bool need_workspace) {
  int rc = check_geom(g);
  if (rc) return rc;
  if (layer < 0 || layer >= g->num_layers || lanes < 0 || max_pages < 0 || max_seq_len < 0) return KVQ_ERR_INVALID_ARG;
  if (window < 0 || window > P) return KVQ_ERR_INVALID_ARG;
  if ((int64_t)max_seq_len > (int64_t)max_pages * P) return KVQ_ERR_INVALID_ARG;
  if ((int64_t)max_pages * P > (int64_t)INT32_MAX) return KVQ_ERR_INVALID_ARG;
  if (lanes == 0) return KVQ_OK;
  if (!pool || !page_table || !seq_len || !q || (need_workspace && !workspace) || !out || !d_status)
    return KVQ_ERR_INVALID_ARG;
  if (two_bit(g->format) && !ring) return KVQ_ERR_INVALID_ARG;
  if (pool_bytes < page_bytes_of(g)) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(pool) || !aligned16(ring) || !aligned16(q) || !aligned16(workspace) || !aligned16(out))
    return KVQ_ERR_ALIGNMENT;
  return KVQ_OK;
}
}  // namespace kvq

namespace {

AttnArgs decode_args(const kvq_geom* g, int layer, const void* pool, size_t pool_bytes, const void* ring, int window,
                     const int32_t* page_table, int max_pages, int lanes, const int32_t* seq_len, int max_seq_len,
                     const void* q, float sm_scale, void* workspace, float* out, int32_t* d_status) {
  AttnArgs a{};
  a.c = make_view(g, layer, pool, pool_bytes, ring, page_table, max_pages, window, d_status);
  a.q_pos0 = a.n_q = a.q_offset = nullptr;
  a.seq_len = seq_len;
  a.lanes = lanes;
  a.max_n_q = 1;
  a.n_q_rows = lanes;
  a.split_tokens = decode_split_tokens(g->format);
  a.max_splits = (int)decode_slots(g->format, max_seq_len);
  a.grid_warps = 0;
  a.min_wp = 0;
  a.max_seq_len = max_seq_len;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.scale_log2 = sm_scale * LOG2E;
  a.ws_o = static_cast<float*>(workspace);
  a.ws_ml = a.ws_o + (int64_t)lanes * g->num_q_heads * a.max_splits * D;
  a.out = out;
  return a;
}

}  // namespace

extern "C" {

size_t kvq_page_bytes(const kvq_geom* g) { return check_geom(g) ? 0 : page_bytes_of(g); }

size_t kvq_token_bytes(const kvq_geom* g) { return check_geom(g) ? 0 : page_bytes_of(g) / P; }

size_t kvq_ring_bytes(const kvq_geom* g, int lanes) {
  if (check_geom(g) || lanes < 0 || !two_bit(g->format)) return 0;
  return (size_t)lanes * g->num_layers * g->num_kv_heads * P * D * 2;
}

int64_t kvq_pool_pages(const kvq_geom* g, size_t pool_bytes) {
  if (check_geom(g)) return -1;
  return (int64_t)(pool_bytes / page_bytes_of(g));
}

size_t kvq_decode_workspace_bytes(const kvq_geom* g, int lanes, int max_seq_len) {
  if (check_geom(g) || lanes < 0 || max_seq_len < 0) return 0;
  size_t bytes = partial_bytes(lanes, g->num_q_heads, decode_slots(g->format, max_seq_len));
  if (g->format == KVQ_FMT_HQ2B_HAD) bytes += (size_t)lanes * g->num_q_heads * D * 2;   // rotated q (fp16)
  return bytes;
}

size_t kvq_prefill_workspace_bytes(const kvq_geom* g, int n_q_rows, int max_seq_len) {
  if (check_geom(g) || n_q_rows < 0 || max_seq_len < 0) return 0;
  return partial_bytes(n_q_rows, g->num_q_heads, splits_for(max_seq_len, prefill_split_tokens(g->format)));
}

const char* kvq_strerror(int code) {
  switch (code) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported format or geometry (head_dim 256, page 64, group <= 8)";
    case KVQ_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case KVQ_ERR_CUDA: return "CUDA launch error";
    case KVQ_ERR_ALIGNMENT: return "a device pointer is not 16-byte aligned";
    case KVQ_ERR_SCRATCH_LIMIT: return "request exceeds the static scratch of paged_decode_attn_noalloc";
    default: return "unknown error";
  }
}

int kvq_build_arch(void) { return KVQ_SM; }

// host checks of kv_quant_append; 1 = valid but nothing to do
static int check_append(const kvq_geom* g, int layer, const void* pool, size_t pool_bytes, const void* ring,
                        const int32_t* page_table, int max_pages, int lanes, const int32_t* start_pos,
                        const int32_t* n_new, const int32_t* tok_offset, int max_new, int n_rows, const void* k,
                        const void* v, const int32_t* d_status) {
  int rc = check_geom(g);
  if (rc) return rc;
  if (layer < 0 || layer >= g->num_layers || lanes < 0 || max_new < 0 || n_rows < 0 || max_pages < 0)
    return KVQ_ERR_INVALID_ARG;
  if ((int64_t)max_pages * P > (int64_t)INT32_MAX) return KVQ_ERR_INVALID_ARG;
  if (lanes == 0 || max_new == 0) return 1;
  if (!pool || !page_table || !start_pos || !n_new || !tok_offset || !k || !v || !d_status)
    return KVQ_ERR_INVALID_ARG;
  if (two_bit(g->format) && !ring) return KVQ_ERR_INVALID_ARG;
  if (pool_bytes < page_bytes_of(g)) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(pool) || !aligned16(ring) || !aligned16(k) || !aligned16(v)) return KVQ_ERR_ALIGNMENT;
  return KVQ_OK;
}

int kv_quant_append(const kvq_geom* g, int layer, void* pool, size_t pool_bytes, void* ring,
                    const int32_t* page_table, int max_pages, int lanes, const int32_t* start_pos,
                    const int32_t* n_new, const int32_t* tok_offset, int max_new, int n_rows, const void* k,
                    const void* v, int32_t* d_status, kvq_stream_t stream) {
  const int rc = check_append(g, layer, pool, pool_bytes, ring, page_table, max_pages, lanes, start_pos, n_new,
                              tok_offset, max_new, n_rows, k, v, d_status);
  if (rc) return rc == 1 ? KVQ_OK : rc;
  CacheView c = make_view(g, layer, pool, pool_bytes, ring, page_table, max_pages, 0, d_status);
  return launch_append(layout_fmt(g->format), c, static_cast<uint8_t*>(pool), static_cast<__nv_bfloat16*>(ring), start_pos,
                       n_new, tok_offset, max_new, n_rows, lanes, static_cast<const __nv_bfloat16*>(k),
                       static_cast<const __nv_bfloat16*>(v), (cudaStream_t)stream);
}

int paged_decode_attn(const kvq_geom* g, int layer, const void* pool, size_t pool_bytes, const void* ring,
                      int window, const int32_t* page_table, int max_pages, int lanes, const int32_t* seq_len,
                      int max_seq_len, const void* q, float sm_scale, void* workspace, size_t ws_bytes,
                      float* out, int32_t* d_status, kvq_stream_t stream) {
  int rc = check_attn_common(g, layer, pool, pool_bytes, ring, window, page_table, max_pages, lanes, seq_len,
                             max_seq_len, q, workspace, out, d_status, true);
  if (rc || lanes == 0) return rc;
  if (ws_bytes < kvq_decode_workspace_bytes(g, lanes, max_seq_len)) return KVQ_ERR_WORKSPACE_TOO_SMALL;
  AttnArgs a = decode_args(g, layer, pool, pool_bytes, ring, window, page_table, max_pages, lanes, seq_len,
                           max_seq_len, q, sm_scale, workspace, out, d_status);
  if (g->format == KVQ_FMT_HQ2B_HAD) {
    if (lanes > 8192) return KVQ_ERR_UNSUPPORTED;
    // the rotated query sits after the partials
    a.q_rot = reinterpret_cast<__half*>(static_cast<uint8_t*>(workspace) +
                                        partial_bytes(lanes, g->num_q_heads, a.max_splits));
  }
  if (two_bit(g->format)) return launch_decode_hq2b(a, (cudaStream_t)stream);
  if (g->format == KVQ_FMT_FP8) return launch_decode_fp8(a, (cudaStream_t)stream);
  return launch_decode_bf16(a, (cudaStream_t)stream);
}

int paged_prefill_attn(const kvq_geom* g, int layer, const void* pool, size_t pool_bytes, const void* ring,
                       int window, const int32_t* page_table, int max_pages, int lanes, const int32_t* q_pos0,
                       const int32_t* n_q, const int32_t* q_offset, int max_n_q, int n_q_rows,
                       const int32_t* seq_len, int max_seq_len, const void* q, float sm_scale, void* workspace,
                       size_t ws_bytes, float* out, int32_t* d_status, kvq_stream_t stream) {
  int rc = check_attn_common(g, layer, pool, pool_bytes, ring, window, page_table, max_pages, lanes, seq_len,
                             max_seq_len, q, workspace, out, d_status, true);
  if (rc) return rc;
  if (max_n_q < 0 || n_q_rows < 0) return KVQ_ERR_INVALID_ARG;
  if (lanes == 0 || max_n_q == 0) return KVQ_OK;
  if (!q_pos0 || !n_q || !q_offset) return KVQ_ERR_INVALID_ARG;
  if (ws_bytes < kvq_prefill_workspace_bytes(g, n_q_rows, max_seq_len)) return KVQ_ERR_WORKSPACE_TOO_SMALL;
  AttnArgs a{};
  a.c = make_view(g, layer, pool, pool_bytes, ring, page_table, max_pages, window, d_status);
  a.q_pos0 = q_pos0;
  a.n_q = n_q;
  a.q_offset = q_offset;
  a.seq_len = seq_len;
  a.lanes = lanes;
  a.max_n_q = max_n_q;
  a.n_q_rows = n_q_rows;
  a.split_tokens = prefill_split_tokens(g->format);
  a.max_splits = (int)splits_for(max_seq_len, a.split_tokens);
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.scale_log2 = sm_scale * LOG2E;
  a.ws_o = static_cast<float*>(workspace);
  a.ws_ml = a.ws_o + (int64_t)n_q_rows * g->num_q_heads * a.max_splits * D;
  a.out = out;
  a.grid_warps = 0;
  a.min_wp = 0;
  a.max_seq_len = max_seq_len;
  if (g->format == KVQ_FMT_BF16)   // the exact reference pages: the CUDA-core split kernel
    return launch_attn_generic(KVQ_FMT_BF16, a, 0, (cudaStream_t)stream);
  // (the rotated format's prefill turns its page rows back to the original basis itself: q and
  // the output need no rotation)
  rc = launch_prefill_tc(g->format, a, (cudaStream_t)stream);
  return rc ? rc : launch_attn_combine(a, 0, (cudaStream_t)stream);
}

int kvq_decode_step(const kvq_geom* g, int layer, void* pool, size_t pool_bytes, void* ring, int window,
                    const int32_t* page_table, int max_pages, int lanes, const int32_t* start_pos,
                    const int32_t* n_new, const int32_t* tok_offset, int n_rows, const void* k, const void* v,
                    const int32_t* seq_len, int max_seq_len, const void* q, float sm_scale, void* workspace,
                    size_t ws_bytes, float* out, int32_t* d_status, kvq_stream_t stream) {
  int rc = check_attn_common(g, layer, pool, pool_bytes, ring, window, page_table, max_pages, lanes, seq_len,
                             max_seq_len, q, workspace, out, d_status, true);
  if (rc) return rc;
  if (n_rows < 0) return KVQ_ERR_INVALID_ARG;
  if (lanes == 0) return KVQ_OK;
  if (!start_pos || !n_new || !tok_offset || !k || !v) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v)) return KVQ_ERR_ALIGNMENT;
  if (ws_bytes < kvq_decode_workspace_bytes(g, lanes, max_seq_len)) return KVQ_ERR_WORKSPACE_TOO_SMALL;
  rc = check_append(g, layer, pool, pool_bytes, ring, page_table, max_pages, lanes, start_pos, n_new, tok_offset, 1,
                    n_rows, k, v, d_status);
  if (rc < 0) return rc;
  const bool fused = g->format == KVQ_FMT_HQ2B && lanes <= 8192;
  // With a window of a whole page nothing this step's attention reads is written by its append:
  // the main pages end before the window, the tail takes its keys from the ring slots the append
  // leaves alone and the step's own token from `k` / `v`.  The append then runs last, overlapping
  // the combine.  Otherwise it runs first (a one-launch decode append, at most one token a lane).
  const bool append_last = fused && window == P;
  if (!append_last) {
    rc = kv_quant_append(g, layer, pool, pool_bytes, ring, page_table, max_pages, lanes, start_pos, n_new,
                         tok_offset, 1, n_rows, k, v, d_status, stream);
    if (rc) return rc;
  }
  if (!fused)   // BF16, FP8, per-token-K or rotated pages, very many lanes: plain decode
    return paged_decode_attn(g, layer, pool, pool_bytes, ring, window, page_table, max_pages, lanes, seq_len,
                             max_seq_len, q, sm_scale, workspace, ws_bytes, out, d_status, stream);
  AttnArgs a = decode_args(g, layer, pool, pool_bytes, ring, window, page_table, max_pages, lanes, seq_len,
                           max_seq_len, q, sm_scale, workspace, out, d_status);
  a.step.start_pos = start_pos;
  a.step.n_new = n_new;
  a.step.tok_offset = tok_offset;
  a.step.n_rows = n_rows;
  a.step.k = static_cast<const __nv_bfloat16*>(k);
  a.step.v = static_cast<const __nv_bfloat16*>(v);
  a.step.active = 1;
  a.step.append_last = append_last ? 1 : 0;
  rc = launch_decode_hq2b(a, (cudaStream_t)stream);
  if (rc || !append_last) return rc;
  return launch_append_last(a.c, static_cast<uint8_t*>(pool), static_cast<__nv_bfloat16*>(ring), start_pos, n_new,
                            tok_offset, n_rows, lanes, static_cast<const __nv_bfloat16*>(k),
                            static_cast<const __nv_bfloat16*>(v), (cudaStream_t)stream);
}

static int page_move(const kvq_geom* g, void* pool, size_t pool_bytes, const int32_t* page_ids, int n_pages,
                     void* arena, int gather, int32_t* d_status, kvq_stream_t stream) {
  int rc = check_geom(g);
  if (rc) return rc;
  if (n_pages < 0) return KVQ_ERR_INVALID_ARG;
  if (n_pages == 0) return KVQ_OK;
  if (!pool || !page_ids || !arena || !d_status) return KVQ_ERR_INVALID_ARG;
  if (pool_bytes < page_bytes_of(g)) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(pool) || !aligned16(arena)) return KVQ_ERR_ALIGNMENT;
  const int64_t pb = (int64_t)page_bytes_of(g);
  return launch_page_move(static_cast<uint8_t*>(pool), static_cast<uint8_t*>(arena), page_ids, n_pages, pb,
                          (int64_t)(pool_bytes / pb), gather, d_status, (cudaStream_t)stream);
}

int kvq_pages_gather(const kvq_geom* g, const void* pool, size_t pool_bytes, const int32_t* page_ids, int n_pages,
                     void* arena, int32_t* d_status, kvq_stream_t stream) {
  return page_move(g, const_cast<void*>(pool), pool_bytes, page_ids, n_pages, arena, 1, d_status, stream);
}

int kvq_pages_scatter(const kvq_geom* g, void* pool, size_t pool_bytes, const int32_t* page_ids, int n_pages,
                      const void* arena, int32_t* d_status, kvq_stream_t stream) {
  return page_move(g, pool, pool_bytes, page_ids, n_pages, const_cast<void*>(arena), 0, d_status, stream);
}

}  // extern "C"

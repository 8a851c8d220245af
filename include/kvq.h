/*
 * kvq.h -- C ABI of libkvq: GQA attention over a paged KV cache kept in a 2-bit,
 * 72 B/head/token format (or in BF16 for comparison), hand-written CUDA for sm_103a.
 *
 * Sources (web pages; the library follows what they fix and documents what it chose where
 * they are silent):
 *   [KV9]  "KV at 9 KB a token" -- sections "How it works" (format table, 64-token pages,
 *          byte-sized pool) and "The numbers".
 *   [REUSE] "The KV cache and prompt reuse" -- section "What a sequence is made of" (pages of
 *          64 tokens shared by all lanes; the window of exact recent keys the compressed
 *          format keeps) and "Why reuse needs more than the KV pages" (prefix pages shared in
 *          place, reference counted).
 *   [HALF] "Half the Cache, Twice the Context" -- table "Two losses with one name" (K scaled
 *          per channel, V per token) and section "The cliff is in the accumulator, not the
 *          storage" (two-level accumulation into a real FP32 register).
 *
 * Conventions (every entry point):
 *   - Every pointer argument except `geom` is a DEVICE pointer owned by the caller.  The
 *     library allocates nothing, never synchronises, and enqueues its kernels on `stream`
 *     in order (stream-ordered like a cudaMemcpyAsync).
 *   - Host-detected problems return a negative KVQ_ERR_* code and launch nothing (a format or
 *     geometry the kernels do not support is refused before any byte moves; there is no CPU
 *     fallback).  0 means the kernels were enqueued.
 *   - Device-detected problems (a page id outside the pool, a length past the page table,
 *     a non-finite or out-of-range input) are OR-ed as KVQ_STATUS_* bits into *d_status
 *     (device int32; the caller zeroes it and reads it after the stream completes).  The
 *     unit that met the problem is skipped; the rest of the call proceeds.
 *   - Alignment: pool, ring, q, k, v, out and workspace must be 16-byte aligned.
 *   - geom->head_dim must be 256, geom->page_tokens 64, num_q_heads a multiple of
 *     num_kv_heads with group size G = num_q_heads / num_kv_heads <= 8.
 *   - Query head j reads KV head j / G (contiguous GQA groups).
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* kvq_stream_t; /* same handle as cudaStream_t; NULL = legacy stream */

/* KVQ_FMT_HQ2B_HAD: the HQ2B byte layout over K and V rows rotated by the normalized 256-point
 * Walsh-Hadamard transform H (H = H^T = H^-1) before quantization -- the rotation that "Half the
 * Cache, Twice the Context" ("What the vendors actually measured") credits with the accuracy
 * change of a low-bit cache.  The quantizer's input is the fast transform in float (stages
 * h = 1, 2, ..., 128, pairs (a + b, a - b), then x 1/16), so codes are reproducible bit for bit.
 * The ring keeps keys as they came.  Decode rotates the query (q.k = Hq.Hk) and turns the output
 * back (sum p Hv = H sum p v), so results approximate the same attention as HQ2B.
 * Every call takes it.  Its decode workspace is larger by lanes * num_q_heads * 512 B (the
 * rotated query); kvq_decode_workspace_bytes counts it.  Its prefill turns the page rows back to
 * the original basis before the tensor-core products, so q and the output are never rotated. */
/* KVQ_FMT_HQ2B_TOK: the HQ2B byte layout with each K row coded when it is appended, per token
 * and per 128-dim half, by the V rule (z = fp16(min), s = fp16((max - min)/3), k^ = z + c s):
 * the K block holds 64 code rows + 64 meta rows like a V block, and there is no page close.
 * This is the per-token axis that "Half the Cache, Twice the Context" ("What the cache loses
 * when you round it") weighs against per-channel K.  The ring still keeps the last 64 keys
 * exact; a key is read from it only inside the window (t >= seq_len - window), so with window 0
 * every key, the open page's included, comes from its codes.  All calls take it. */
/* KVQ_FMT_FP8: K and V rows as OCP FP8 E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa
 * bits, largest finite 448, no infinity), one byte per value: a (layer, head, K or V) block of a
 * page is 64 rows x 256 B = 16,384 B, half of BF16 -- the FP8 cache of the vLLM study quoted in
 * "Half the Cache, Twice the Context" ("What the vendors actually measured").  Append stores
 * E4M3(x / scale) with x / scale in fp32, rounded to nearest even and saturated at +-448; reads
 * decode the byte and multiply by the scale (kvq_geom.k_scale / v_scale, 0 meaning 1).  No
 * ring (ring may be NULL, ring bytes are 0) and no window: every key comes from its page. */
typedef enum { KVQ_FMT_HQ2B = 0, KVQ_FMT_BF16 = 1, KVQ_FMT_HQ2B_HAD = 2, KVQ_FMT_HQ2B_TOK = 3,
               KVQ_FMT_FP8 = 4 } kvq_format;

typedef struct {
  int32_t format;       /* kvq_format */
  int32_t num_layers;   /* layers that keep a KV cache (16 for the 27B geometry) */
  int32_t num_kv_heads; /* 4 for the 27B geometry */
  int32_t num_q_heads;  /* multiple of num_kv_heads, group <= 8 */
  int32_t head_dim;     /* must be 256 */
  int32_t page_tokens;  /* must be 64 */
  float k_scale;        /* KVQ_FMT_FP8: per-tensor scale of K (0 means 1; else finite, > 0) */
  float v_scale;        /* KVQ_FMT_FP8: per-tensor scale of V; other formats ignore both */
} kvq_geom;

/* host-side return codes */
#define KVQ_OK 0
#define KVQ_ERR_INVALID_ARG (-1)
#define KVQ_ERR_UNSUPPORTED (-2)
#define KVQ_ERR_WORKSPACE_TOO_SMALL (-3)
#define KVQ_ERR_CUDA (-4)
#define KVQ_ERR_ALIGNMENT (-5)
#define KVQ_ERR_SCRATCH_LIMIT (-6) /* paged_decode_attn_noalloc: request exceeds its static scratch */

/* device status bits OR-ed into *d_status */
#define KVQ_STATUS_PAGE_OOB 1      /* a page-table entry the call needed is outside [0, pool pages) */
#define KVQ_STATUS_LEN_GT_TABLE 2  /* a position lies past max_pages * 64 */
#define KVQ_STATUS_BAD_INPUT 4     /* a K/V input is NaN, Inf or |x| > 65504 (not quantized) */
#define KVQ_STATUS_BAD_LEN 8       /* a negative count, n_new > max_new, rows past n_rows, a
                                      seq_len[b] above max_seq_len (that lane is skipped), or a
                                      prefill query position >= seq_len */
#define KVQ_STATUS_TIMEOUT 16      /* a bounded wait on a shared-memory barrier gave up */

/*
 * Pool layout (the format; [KV9] "How it works"):
 *   The pool is `pool_bytes` of device memory cut into pages of kvq_page_bytes(geom) bytes;
 *   physical page p starts at byte p * page_bytes.  A page holds 64 tokens of every layer
 *   and KV head, in blocks ordered [layer][kv_head][K, V].
 *   KVQ_FMT_HQ2B, block = 4,608 B = 64 tokens x 72 B:
 *     K block: codes[64 slots][64 B] then scales[256] fp16 (one per channel, written when the
 *              page closes, i.e. when its slot 63 is appended);
 *     V block: codes[64 slots][64 B] then meta[64 slots][s0, z0, s1, z1] fp16.
 *     Code byte b of a 64 B row packs dims 4b..4b+3, dim 4b+j at bits 2j..2j+1.
 *     V (per token, per 128-dim half h): z = fp16(min), s = fp16((max - min) / 3),
 *       c = clamp(rint((x - z) / s), 0, 3), c = 0 if s == 0; v^ = z + c s.
 *     K (per channel d over the 64 keys of a closed page): s_d = fp16(max|x| / 3),
 *       c = clamp(rint((x / s_d + 3) / 2), 0, 3), c = 2 if s_d == 0; k^ = s_d (2c - 3).
 *     All steps are IEEE fp32 round-to-nearest-even; rint is half-even.
 *   KVQ_FMT_BF16, block = 32,768 B: rows[64 slots][256] bf16 for K and for V.
 *
 * Ring ([REUSE] "What a sequence is made of": the window of exact recent keys):
 *   bf16 [lanes][num_layers][num_kv_heads][64 slots][256]; position t of a lane lives in slot
 *   t % 64.  HQ2B only: keys of the page that is still open exist only here, and attention
 *   reads key t from the ring iff t >= min(seq_len - window, 64 * floor(seq_len / 64)).
 *
 * Page table: int32 [lanes][max_pages] (row stride max_pages); entry i of lane b is the
 *   physical page of the lane's tokens 64i .. 64i+63.  Several lanes may name the same page
 *   (a shared prefix, read in place); appending into a shared page is a caller error.
 */

/* Bytes of one page: num_layers * num_kv_heads * 2 * 64 * (72 | 512).  0 on a bad geom. */
size_t kvq_page_bytes(const kvq_geom* geom);
/* Bytes one token costs across all layers and heads, K and V (9,216 / 65,536 at 16 x 4). */
size_t kvq_token_bytes(const kvq_geom* geom);
/* Bytes of the exact-key ring for `lanes` lanes (HQ2B; 0 for BF16). */
size_t kvq_ring_bytes(const kvq_geom* geom, int lanes);
/* Whole pages a pool of pool_bytes holds; -1 on a bad geom. */
int64_t kvq_pool_pages(const kvq_geom* geom, size_t pool_bytes);
/* Workspace paged_decode_attn needs for `lanes` lanes of at most max_seq_len tokens. */
size_t kvq_decode_workspace_bytes(const kvq_geom* geom, int lanes, int max_seq_len);
/* Workspace paged_prefill_attn needs for n_q_rows query rows over at most max_seq_len keys. */
size_t kvq_prefill_workspace_bytes(const kvq_geom* geom, int n_q_rows, int max_seq_len);
/* Static text for a return code. */
const char* kvq_strerror(int code);
/* The SM target the kernels of this build were compiled for (103 for sm_103a). */
int kvq_build_arch(void);

/*
 * kv_quant_append -- quantize and append new tokens of one layer ([KV9] "How it works";
 * [HALF] "Two losses with one name" for the axes).
 *   For every lane b, rows tok_offset[b] .. tok_offset[b] + n_new[b] - 1 of k and v
 *   (bf16 [n_rows][num_kv_heads][256]) become positions start_pos[b] .. start_pos[b] +
 *   n_new[b] - 1 of the lane, placed through page_table.
 *   HQ2B: each V row is quantized into its page slot; each K row is stored in ring slot
 *   pos % 64, and every page whose slot 63 is appended by this call is closed: its K block
 *   is quantized per channel from the page's 64 keys (ring entries for keys appended by
 *   earlier calls, k rows for the rest).  The resulting bytes do not depend on how a
 *   sequence is split into calls.  BF16: both rows are stored as they are (ring unused).
 *   Arguments: layer in [0, num_layers); max_new >= every n_new[b] (host bound that sizes the
 *   grid); n_rows = rows of k and v; ring may be NULL only for BF16.
 *   Errors: KVQ_ERR_INVALID_ARG / UNSUPPORTED / ALIGNMENT / CUDA; device bits PAGE_OOB,
 *   LEN_GT_TABLE, BAD_INPUT (that token/head or page is not written), BAD_LEN.
 */
int kv_quant_append(const kvq_geom* geom, int layer, void* pool, size_t pool_bytes, void* ring,
                    const int32_t* page_table, int max_pages, int lanes, const int32_t* start_pos,
                    const int32_t* n_new, const int32_t* tok_offset, int max_new, int n_rows,
                    const void* k, const void* v, int32_t* d_status, kvq_stream_t stream);

/*
 * paged_decode_attn -- one query token per lane attends all of the lane's cached tokens
 * ([KV9] "How it works": attention reads the compressed pages directly, no decompressed
 * copy; [HALF] "The cliff is in the accumulator": FP32 partials merged once at the end).
 *   q: bf16 [lanes][num_q_heads][256]; out: fp32 [lanes][num_q_heads][256];
 *   out[b][j] = sum_t softmax_t(sm_scale * q[b][j] . k^_t) v^_t over t < seq_len[b]
 *   (seq_len counts the tokens after the step's append).  seq_len[b] == 0 gives zeros.
 *   window in [0, 64]: the last `window` keys are read exact from the ring (HQ2B).
 *   max_seq_len (host) >= every seq_len[b] sizes the split-K grid; it must not exceed
 *   max_pages * 64.  workspace: >= kvq_decode_workspace_bytes(geom, lanes, max_seq_len)
 *   bytes; its contents on entry are irrelevant (every byte read is first written by the
 *   same call).
 *   Errors: KVQ_ERR_*; device bits PAGE_OOB, LEN_GT_TABLE, BAD_LEN, TIMEOUT.
 */
int paged_decode_attn(const kvq_geom* geom, int layer, const void* pool, size_t pool_bytes,
                      const void* ring, int window, const int32_t* page_table, int max_pages,
                      int lanes, const int32_t* seq_len, int max_seq_len, const void* q,
                      float sm_scale, void* workspace, size_t ws_bytes, float* out,
                      int32_t* d_status, kvq_stream_t stream);

/*
 * paged_prefill_attn -- a chunk of query tokens attends causally over the cache
 * ([KV9] "How it works": since 0.7.3 prefill attention reads the compressed cache directly;
 * [KV9] "One cleanup came free": the workspace needs no zeroing).
 *   The chunk's own K/V must already be appended (kv_quant_append).  For lane b, query rows
 *   q_offset[b] .. q_offset[b] + n_q[b] - 1 of q (bf16 [n_q_rows][num_q_heads][256]) sit at
 *   positions q_pos0[b] + i and attend keys 0 .. q_pos0[b] + i (inclusive); out is fp32
 *   [n_q_rows][num_q_heads][256].  Keys are read from the cache state of seq_len[b] tokens
 *   (same window rule as decode).  max_n_q (host) >= every n_q[b]; max_seq_len (host) >=
 *   every seq_len[b]; workspace >= kvq_prefill_workspace_bytes(geom, n_q_rows, max_seq_len),
 *   contents on entry irrelevant.
 *   Errors: KVQ_ERR_*; device bits PAGE_OOB, LEN_GT_TABLE, BAD_LEN, TIMEOUT.
 */
int paged_prefill_attn(const kvq_geom* geom, int layer, const void* pool, size_t pool_bytes,
                       const void* ring, int window, const int32_t* page_table, int max_pages,
                       int lanes, const int32_t* q_pos0, const int32_t* n_q,
                       const int32_t* q_offset, int max_n_q, int n_q_rows,
                       const int32_t* seq_len, int max_seq_len, const void* q, float sm_scale,
                       void* workspace, size_t ws_bytes, float* out, int32_t* d_status,
                       kvq_stream_t stream);

/*
 * kvq_decode_step -- one decode step of one layer: kv_quant_append of at most one new token
 * per lane followed by paged_decode_attn over the cache that includes it ([KV9] "How it
 * works": tokens are quantized as they are appended and attention reads the compressed pages).
 *   Arguments are those of the two calls, with max_new = 1: n_new[b] in {0, 1}, the new token
 *   at position start_pos[b] == seq_len[b] - n_new[b]; k, v: bf16 [n_rows][num_kv_heads][256].
 *   Results: the pool and ring bytes and `out` equal those of kv_quant_append then
 *   paged_decode_attn on the same stream.  With HQ2B pages the decode kernels overlap the
 *   append kernel: the main kernel reads no page the append writes until it has waited for it
 *   (only a page the new token closes, and only with window 0, is such a page), and the tail
 *   takes the new token's key and value from k and v.  BF16 pages: the two calls in sequence.
 *   Errors: those of both calls; device bit BAD_LEN when start_pos[b] + n_new[b] != seq_len[b]
 *   (that lane's new token is then neither appended nor attended).
 */
int kvq_decode_step(const kvq_geom* geom, int layer, void* pool, size_t pool_bytes, void* ring,
                    int window, const int32_t* page_table, int max_pages, int lanes,
                    const int32_t* start_pos, const int32_t* n_new, const int32_t* tok_offset,
                    int n_rows, const void* k, const void* v, const int32_t* seq_len,
                    int max_seq_len, const void* q, float sm_scale, void* workspace,
                    size_t ws_bytes, float* out, int32_t* d_status, kvq_stream_t stream);

/*
 * kvq_pages_gather / kvq_pages_scatter -- bit-exact page moves between the pool and an arena
 * ([REUSE] "What a sequence is made of": pages are the unit a cache evicts to a slower tier
 * and brings back).
 *   gather:  arena slot i (page_bytes each, slot i at arena + i * kvq_page_bytes(geom)) <-
 *            pool page page_ids[i], for i < n_pages.
 *   scatter: pool page page_ids[i] <- arena slot i.
 *   A page is moved as opaque bytes -- every layer and head, codes, scales and metadata -- so
 *   scattering gathered pages to other page ids and pointing the page table at them leaves
 *   every attention result bit for bit the same.  The exact-key ring is per lane, not per
 *   page, and is not moved.  arena: device memory or pinned host memory the GPU can address
 *   (on a Grace host the kernel reads and writes it directly over NVLink-C2C); 16-byte
 *   aligned.  page_ids: device int32 [n_pages]; ids repeated in one scatter race.
 *   Errors: KVQ_ERR_INVALID_ARG / UNSUPPORTED / ALIGNMENT / CUDA; device bit PAGE_OOB (that
 *   page is not moved).
 */
int kvq_pages_gather(const kvq_geom* geom, const void* pool, size_t pool_bytes, const int32_t* page_ids,
                     int n_pages, void* arena, int32_t* d_status, kvq_stream_t stream);
int kvq_pages_scatter(const kvq_geom* geom, void* pool, size_t pool_bytes, const int32_t* page_ids,
                      int n_pages, const void* arena, int32_t* d_status, kvq_stream_t stream);

/*
 * kvq_selftest_wait_timeout -- the library's failure path, run on purpose.  Not an operation
 * of the method: it exists so that a caller can check, on a healthy GPU, what every kernel of
 * the library does when a shared-memory barrier wait runs out.  One warp waits, with the same
 * bounded wait the attention and append kernels use (2^16 tries of mbarrier.try_wait with a
 * ~1 us suspend hint each, so tens of milliseconds), on a barrier that nothing ever arrives
 * at; the wait gives up, the kernel ORs KVQ_STATUS_TIMEOUT into *d_status and returns.
 * Nothing faults or traps and the context stays usable.
 *   d_status: device int32, not cleared by the call.  Errors: KVQ_ERR_INVALID_ARG (null
 *   d_status) / KVQ_ERR_CUDA (launch failed).
 */
int kvq_selftest_wait_timeout(int32_t* d_status, kvq_stream_t stream);

/*
 * paged_decode_attn_noalloc -- paged_decode_attn without a caller workspace.  The pages have
 * no counterpart of this call: it exists for callers that cannot allocate device memory --
 * plugins of a serving engine whose allocator owns all of the GPU's memory and hands out no
 * scratch, hosts that forbid allocation after start-up, latency-critical loops where an
 * allocation (which may synchronise the device) is not allowed.
 *   Same arguments, results and errors as paged_decode_attn, minus `workspace`/`ws_bytes`:
 *   the split partials live in one static device array of KVQ_NOALLOC_SCRATCH_BYTES
 *   (32 MiB) inside the library, which every GPU that loads the library keeps until the
 *   process exits.  The call allocates nothing and calls no allocating routine.
 *   Limit: kvq_decode_workspace_bytes(geom, lanes, max_seq_len) must not exceed
 *   KVQ_NOALLOC_SCRATCH_BYTES, else KVQ_ERR_SCRATCH_LIMIT and nothing is launched (at the
 *   27B geometry that is room for 8 lanes x 40,960 tokens, 30.6 MiB of partials).  Every other
 *   argument is checked first, with the codes paged_decode_attn returns.
 *   The first call on a device looks up the array's device address (once per device, with
 *   that device current); make that first call before any stream capture.
 *   Every call shares the array: calls whose kernels may overlap on the GPU (different
 *   streams without ordering) race on it.  Nothing in it needs clearing -- each call writes
 *   every partial it reads.
 */
#define KVQ_NOALLOC_SCRATCH_BYTES (32u << 20)
int paged_decode_attn_noalloc(const kvq_geom* geom, int layer, const void* pool, size_t pool_bytes,
                              const void* ring, int window, const int32_t* page_table, int max_pages,
                              int lanes, const int32_t* seq_len, int max_seq_len, const void* q,
                              float sm_scale, float* out, int32_t* d_status, kvq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */

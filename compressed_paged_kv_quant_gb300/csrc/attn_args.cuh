// attn_args.cuh -- arguments of the attention kernels (decode and prefill share them).
#pragma once
#include "kvq_internal.cuh"

namespace kvq {

// The append of a fused decode step (kvq_decode_step), which the decode kernels overlap: at
// most one new token per lane, at position start_pos[b] == seq_len[b] - 1.
struct StepAppend {
  const int32_t* start_pos;
  const int32_t* n_new;
  const int32_t* tok_offset;
  int n_rows;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  int active;
  // 1: nothing this step reads is written by its append (window == 64), so the append runs last,
  // as the programmatic dependent of the combine kernel, instead of first
  int append_last;
};

struct AttnArgs {
  CacheView c;
  const int32_t* q_pos0;    // prefill only
  const int32_t* n_q;       // prefill only
  const int32_t* q_offset;  // prefill only
  const int32_t* seq_len;
  int lanes, max_n_q, n_q_rows, max_splits, split_tokens;
  const __nv_bfloat16* q;
  float scale_log2;  // sm_scale * log2(e)
  float* ws_o;       // [rows][Hq][max_splits][256]
  float* ws_ml;      // [rows][Hq][max_splits][2]
  float* out;        // [rows][Hq][256]
  int grid_warps;    // fast 2-bit decode: warps of the persistent grid
  int min_wp;        // fast 2-bit decode: least pages per warp (bounds the partials per lane/head)
  int max_seq_len;   // host bound on every seq_len[b]
  StepAppend step;   // fused decode step only (active == 0 otherwise)
  __half* q_rot;     // rotated format: H q per (lane, query head) in fp16 (workspace), else null
};

// Status bits for a lane length no kernel may use (0 when it is usable): past the page table
// (LEN_GT_TABLE), or negative or above the host bound max_seq_len that sized the grid and the
// split records of the workspace (BAD_LEN).  A lane that fails is skipped by every kernel of the
// call, so no kernel indexes a split record beyond the lane's share of the workspace.
__device__ __forceinline__ int lane_len_error(const AttnArgs& a, int len) {
  if (len < 0) return KVQ_STATUS_BAD_LEN;
  if (len > a.c.max_pages * P) return KVQ_STATUS_LEN_GT_TABLE;
  if (len > a.max_seq_len) return KVQ_STATUS_BAD_LEN;
  return 0;
}

// Resolve query i of lane b: its row, position, and key count.  Returns false (after
// flagging) when the lane's arguments are invalid or i is past the lane's queries.
__device__ __forceinline__ bool resolve_query(const AttnArgs& a, bool decode, int b, int i, int& row, int& n_keys,
                                              int& len, bool flag_errors) {
  const CacheView& c = a.c;
  len = a.seq_len[b];
  if (const int e = lane_len_error(a, len)) {
    if (flag_errors) flag(c.status, e);
    return false;
  }
  if (decode) {
    if (i > 0) return false;
    row = b;
    n_keys = len;
    return true;
  }
  const int nq = a.n_q[b], off = a.q_offset[b], pos0 = a.q_pos0[b];
  if (nq < 0 || nq > a.max_n_q || off < 0 || (int64_t)off + nq > a.n_q_rows || pos0 < 0) {
    if (flag_errors) flag(c.status, KVQ_STATUS_BAD_LEN);
    return false;
  }
  if (i >= nq) return false;
  const int pos = pos0 + i;
  if (pos >= len) {
    if (flag_errors) flag(c.status, KVQ_STATUS_BAD_LEN);
    return false;
  }
  row = off + i;
  n_keys = pos + 1;
  return true;
}

}  // namespace kvq

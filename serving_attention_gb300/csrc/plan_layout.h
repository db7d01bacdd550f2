// plan_layout.h -- layout of the int workspace written by the planner and
// read by the persistent kernel.  All fields are int32.
//
//   header[32]   FI_H_* below (the variant of the plan's config included:
//                  window_left, sink_tokens, soft-cap as float bits, RoPE;
//                  the partial rows and query tokens the plan uses, which the
//                  kernel compares with the buffers it was launched with;
//                  the cascade fields, 0 in a one-level plan)
//   cta_indptr   num_ctas + 1 entries: CTA c runs items [cta_indptr[c], cta_indptr[c+1])
//   items        FI_ITEM_INTS each: {b, hk, row0, row1, kv0, kv1, part, merge,
//                  qo_start, qo_len, page_start, kv_len, heads, 0, 0, 0}
//                  rows are packed rows of request b (row = token * G + g),
//                  heads = 0 for one KV head hk; heads = FI_MH_ROWS / G for
//                  a multi-head decode unit, which takes KV heads
//                  hk .. hk + heads - 1 of a one-token request of the plan's
//                  own page-1 cache at once (row = head offset * G + g; see
//                  fi_mh_heads),
//                  [kv0, kv1) the KV token range of this chunk,
//                  part = first fp32 partial-state row or -1 (unsplit),
//                  merge = merge unit or -1; then a copy of request b's
//                  entry of the request table, so that a work item arrives
//                  with one load instead of two dependent ones
//   merge units  FI_MERGE_INTS each: {b, hk, row0, row1, n_chunks, part_base, late, 0};
//                  chunk i of the unit wrote partial rows part_base + i * (row1 - row0) ...
//                  late = 1 (units of prefill-class tiles): merged after the run by
//                  a row-parallel merge launch; late = 0: merged inside the run by
//                  the CTA that finishes the unit's last chunk
//   counters     one per merge unit, zero between runs (the merging CTA resets it;
//                  late units merged after the run never touch theirs; when the run
//                  is not followed by the late merge, as when a graph was captured
//                  from a plan without late units, it merges them itself)
//   requests     FI_REQ_INTS each: {qo_start, qo_len, page_start, kv_len}
//                  (a cascade plan numbers its shared blocks first: requests
//                  b < num_shared read the shared KV cache and see every one
//                  of their keys; the others read the ordinary cache)
//   cascade      FI_CASCADE_INTS each (cascade plans only):
//                  {b, hk, row0, row1, n0, base0, stride0, n1, base1, stride1, 0, 0}:
//                  packed rows [row0, row1) (at most FI_CASCADE_ROWS of them)
//                  of ordinary request b; row r takes
//                  the partial rows base0 + c * stride0 + (r - row0), c < n0
//                  (its shared block's chunks) and base1 + c * stride1 +
//                  (r - row0), c < n1 (its own chunks), merged in that order
//                  by the cascade merge launched after the run
//   ...          (the rest of the plan capacity)
//   rope table   with RoPE: float2 (cos, sin) [rope_max_positions][64] at
//                  fi_rope_table_offset(capacity) bytes, filled by
//                  fi_rope_init, never part of a plan's copy
// Every section starts on a multiple of 4 ints (16 bytes).
//
// Float workspace: partial LSE (natural log) at [0, max_partial_rows), partial
// O (already divided by its own softmax sum) at
// fi_partial_o_offset(max_partial_rows), head_dim floats per row.
#pragma once
#include <stdint.h>

#define FI_PLAN_MAGIC 0x46495031
#define FI_HEADER_INTS 32
#define FI_ITEM_INTS 16
#define FI_MERGE_INTS 8
#define FI_REQ_INTS 4
#define FI_CASCADE_INTS 12
#define FI_CASCADE_ROWS 16  // packed rows per cascade merge entry, at most
#define FI_MERGE_LATE 6  // index of the late flag in a merge unit

#define FI_TILE_DECODE 16
#define FI_TILE_PREFILL 256  // two 128-row M tiles sharing each K/V tile
#define FI_GRANULE_DECODE 64
#define FI_GRANULE_PREFILL 128
#define FI_ITEM_COST_TOKENS 256  // fixed cost of a work item in the deal, in KV tokens of its class
#define FI_MH_ROWS 32            // packed query rows of a multi-head decode unit (heads * G)
#define FI_ITEM_HEADS 12         // item field: KV heads of a multi-head unit, else 0

enum {
  FI_H_MAGIC = 0,
  FI_H_NUM_ITEMS = 1,
  FI_H_NUM_MERGE = 2,
  FI_H_NUM_CTAS = 3,
  FI_H_BATCH = 4,
  FI_H_CAUSAL = 5,
  FI_H_OFF_CTA = 6,
  FI_H_OFF_ITEMS = 7,
  FI_H_OFF_MERGE = 8,
  FI_H_OFF_COUNTERS = 9,
  FI_H_OFF_REQUESTS = 10,
  FI_H_STATUS = 11,
  FI_H_NUM_QO_HEADS = 12,
  FI_H_NUM_KV_HEADS = 13,
  FI_H_PAGE_SIZE = 14,
  FI_H_TOTAL_INTS = 15,
  FI_H_WINDOW_LEFT = 16,
  FI_H_SINK_TOKENS = 17,
  FI_H_SOFT_CAP_BITS = 18,
  FI_H_ROPE_MAX_POS = 19,     // 0: no RoPE
  FI_H_ROPE_THETA_BITS = 20,
  FI_H_ROPE_SCALE_BITS = 21,
  FI_H_ROPE_TABLE_OFF = 22,   // ints from the workspace start to the cos/sin table
  FI_H_NUM_LATE_MERGE = 23,   // merge units flagged late
  FI_H_PARTIAL_ROWS = 24,     // fp32 partial-state rows the items write (0: no split unit)
  FI_H_TOTAL_QO = 25,         // query tokens of the batch (qo_indptr[batch])
  FI_H_NUM_SHARED = 26,       // cascade: shared blocks (requests 0 .. num_shared - 1); 0 otherwise
  FI_H_OFF_CASCADE = 27,      // cascade: offset of the cascade merge entries
  FI_H_NUM_CASCADE = 28,      // cascade: merge entries
  FI_H_SHARED_PAGE_SIZE = 29, // cascade: page size of the shared KV cache
  FI_H_NUM_DECODE_ITEMS = 30, // items of 16-row tiles (the CUDA-core path)
  FI_H_CASCADE_ROWS_MAX = 31  // cascade: the most packed rows of one merge entry; 0 otherwise
};

#define FI_ROPE_PAIRS 64  // dims i and i + 64 of head_dim 128 form a rotated pair

// Rows of the RoPE table: every position below rope_max_positions, and at
// least 16 (the kernels read the rows of their walk strides, 4 and 12).
static inline int64_t fi_rope_table_rows(int32_t rope_max_positions) {
  return rope_max_positions > 16 ? rope_max_positions : 16;
}

// Byte offset of the RoPE table in an int workspace whose plan region holds
// `plan_ints` int32 (256-byte aligned).
static inline int64_t fi_rope_table_offset(int64_t plan_ints) { return (plan_ints * 4 + 255) / 256 * 256; }

static inline int64_t fi_partial_o_offset(int64_t max_partial_rows) { return (max_partial_rows + 63) / 64 * 64; }

// KV heads of a multi-head decode unit for GQA group G and Hkv KV heads, or 1
// when such units cannot be formed: the unit's FI_MH_ROWS packed rows are
// eight groups of four rows, each group inside one KV head (G a multiple of
// 4), and the heads tile [0, Hkv).
static inline int32_t fi_mh_heads(int32_t group, int32_t num_kv_heads) {
  if (group < 4 || group > FI_MH_ROWS / 2 || group % 4) return 1;
  const int32_t h = FI_MH_ROWS / group;
  return num_kv_heads % h == 0 ? h : 1;
}

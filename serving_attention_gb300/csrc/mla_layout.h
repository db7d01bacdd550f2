// mla_layout.h -- layout of the int workspace of the absorbed-MLA decode
// path, written by the MLA planner and read by its two kernels.  All int32.
//
//   header[16]    FI_MLA_H_* below; the status word sits at the same index as
//                 in the GQA plan, so fi_get_device_status reads either
//   pair_indptr   num_pairs + 1 entries: pair p runs units [pair_indptr[p], pair_indptr[p+1])
//   units         FI_MLA_UNIT_INTS each: {b, kv0, kv1, part}
//                   [kv0, kv1) the KV tokens of request b in this chunk (kv0 a
//                   multiple of 64); part = partial-state slot, or -1 when the
//                   chunk is the whole request and writes the output itself
//   requests      FI_MLA_REQ_INTS each: {page_start (index into kv_indices), kv_len}
//   merge         FI_MLA_MERGE_INTS each: {b, part0, n_parts, 0} for every
//                   request with no chunk (n_parts 0: o = 0, lse = -inf) or
//                   with several (slots part0 .. part0 + n_parts - 1)
// Every section starts on a multiple of 4 ints.
//
// Float workspace: partial LSE (natural log) [max_parts][128] at 0, then the
// partial O (already divided by its own softmax sum) [max_parts][128][512]
// at fi_mla_partial_o_offset(max_parts) floats.
#pragma once
#include <stdint.h>

#include "plan_layout.h"

#define FI_MLA_MAGIC 0x464D4C31
#define FI_MLA_HEADER_INTS 16
#define FI_MLA_UNIT_INTS 4
#define FI_MLA_REQ_INTS 2
#define FI_MLA_MERGE_INTS 4
#define FI_MLA_BLOCK 64              // KV tokens per block of the decode kernel
#define FI_MLA_ROWS 128              // query heads per tile (the MMA's M)
#define FI_MLA_UNIT_COST_TOKENS 448  // fixed cost of a piece in the split, in KV tokens (measured)

enum {
  FI_MLA_H_MAGIC = 0,
  FI_MLA_H_NUM_UNITS = 1,
  FI_MLA_H_NUM_PAIRS = 2,
  FI_MLA_H_BATCH = 3,
  FI_MLA_H_NUM_HEADS = 4,
  FI_MLA_H_PAGE_SIZE = 5,
  FI_MLA_H_OFF_PAIR = 6,
  FI_MLA_H_OFF_UNITS = 7,
  FI_MLA_H_OFF_REQ = 8,
  FI_MLA_H_OFF_MERGE = 9,
  FI_MLA_H_NUM_MERGE = 10,
  FI_MLA_H_STATUS = FI_H_STATUS,
  FI_MLA_H_CHUNK = 12,
  FI_MLA_H_TOTAL_INTS = 13,
  FI_MLA_H_NUM_PARTS = 14
};
static_assert(FI_MLA_H_STATUS == 11, "status word shared with the GQA plan");

static inline int64_t fi_mla_round4(int64_t n) { return (n + 3) / 4 * 4; }

static inline int64_t fi_mla_partial_o_offset(int64_t max_parts) {
  return (max_parts * FI_MLA_ROWS + 63) / 64 * 64;
}

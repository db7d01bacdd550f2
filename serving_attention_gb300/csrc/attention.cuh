// attention.cuh -- parameters and shared-memory layout of the persistent
// paged-attention kernel (CUDA-core path).
#pragma once
#include <stdint.h>

#include "plan_layout.h"
#include "ptx.cuh"

namespace fi {

constexpr int kHeadDim = 128;
constexpr int kStageTokens = 64;       // KV tokens per pipeline stage
constexpr int kStages = 4;             // depth of the K/V ring
constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (1 + kConsumerWarps);  // warp 0 = producer
constexpr int kRowsPerGroup = 4;       // query rows a half-warp carries in registers
constexpr int kGroupsPerPass = 8;
constexpr int kRowsPerPass = kRowsPerGroup * kGroupsPerPass;
constexpr int kHalfWarps = 2 * kConsumerWarps;
constexpr int kTokBlock = 4;           // tokens a half-warp scores before one softmax update
constexpr float kLazyRescale = 8.0f;   // log2 units: keep a stale max until it is 2^8 off

struct RunParams {
  const uint16_t* q;
  int64_t q_stride_tok, q_stride_head;
  const uint16_t* k;
  int64_t k_stride_page, k_stride_slot, k_stride_head;
  const uint16_t* v;
  int64_t v_stride_page, v_stride_slot, v_stride_head;
  const int32_t* kv_indices;
  uint16_t* o;
  int64_t o_stride_tok, o_stride_head;
  float* lse;
  int32_t* iws;
  float* fws;
  int64_t partial_o_offset;  // floats
  float scale_log2;          // sm_scale * log2(e)
  int32_t num_qo_heads, num_kv_heads, group, page_size, log2_page;
};

struct alignas(128) RunSmem {
  uint16_t k[kStages][kStageTokens][kHeadDim];
  uint16_t v[kStages][kStageTokens][kHeadDim];
  float comb_o[kHalfWarps][kRowsPerGroup][kHeadDim];
  float comb_m[kHalfWarps][kRowsPerGroup];
  float comb_l[kHalfWarps][kRowsPerGroup];
  float4 xch[kHalfWarps][kTokBlock + 1];  // per half-warp: p of each token (4 rows), then alpha
  int32_t pidx[kStages][kStageTokens];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  volatile int abort;  // set by the role whose bounded wait ran out
  int merge_last;
};

struct Item {
  int32_t b, hk, row0, row1, kv0, kv1, part, merge;
};

struct Request {
  int32_t qo_start, qo_len, page_start, kv_len;
};

__device__ __forceinline__ Item load_item(const int32_t* iws, int32_t off_items, int32_t i) {
  const int4* p = reinterpret_cast<const int4*>(iws + off_items + FI_ITEM_INTS * i);
  int4 a = __ldg(p), c = __ldg(p + 1);
  return Item{a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
}

__device__ __forceinline__ Request load_request(const int32_t* iws, int32_t off_req, int32_t b) {
  int4 a = __ldg(reinterpret_cast<const int4*>(iws + off_req + FI_REQ_INTS * b));
  return Request{a.x, a.y, a.z, a.w};
}

}  // namespace fi

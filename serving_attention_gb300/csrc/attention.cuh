// attention.cuh -- parameters and shared-memory layout of the persistent
// paged-attention kernel.
#pragma once
#include <cuda.h>
#include <stdint.h>

#include "plan_layout.h"
#include "ptx.cuh"

namespace fi {

constexpr int kHeadDim = 128;

// CUDA-core path (16-row decode tiles; prefill-class items too when pages are < 8 tokens)
constexpr int kLog2StageTokens = 7;
constexpr int kStageTokens = 1 << kLog2StageTokens;  // KV rows per pipeline stage (tokens of one head)
constexpr int kStages = 3;             // depth of the K/V ring
constexpr int kBoxLanes = kStageTokens / 32;  // page boxes a producer lane issues per stage at page size 1
constexpr int kConsumerWarps = 8;
constexpr int kFirstConsumerWarp = 4;  // warps 4..11 consume (warp 0 produces)
constexpr int kThreads = 32 * 12;
constexpr int kRowsPerGroup = 4;       // query rows a half-warp carries in registers
constexpr int kGroupsPerPass = 8;
constexpr int kRowsPerPass = kRowsPerGroup * kGroupsPerPass;
constexpr int kHalfWarps = 2 * kConsumerWarps;
constexpr int kTokBlock = 8;           // tokens a half-warp scores before one softmax update
constexpr float kLazyRescale = 8.0f;   // log2 units: keep a stale max until it is 2^8 off

// Tensor-core path (prefill-class items of up to two 128-row M tiles):
// 128 x 128 S and O tiles in tensor memory.
constexpr int kTileM = 128;            // packed query rows per M tile
constexpr int kTileN = 128;            // KV tokens per tile
constexpr int kTmemCols = 512;         // S of M tiles A, B (128 cols each), then O of A, B
constexpr int kTmemO = 256;            // first column of O of M tile A
constexpr int kMinTmaPage = 8;         // pages of >= 8 tokens keep every TMA box 1024-byte aligned
constexpr int kSoftmaxWarp0 = 4;       // warps 4..7 own the rows of M tile A, warps 8..11 those of M tile B
constexpr int kSoftmaxThreads = 256;
// Register budgets of the tensor-core phase, per thread: warps 0..3 (loaders,
// MMA) drop to kRegsLoader, the two softmax warpgroups rise to kRegsSoftmax
// (a full 128-column S row per thread), and all return to kRegsLaunch before
// the CUDA-core phase.  kRegsLoader * 128 + kRegsSoftmax * 256 must not
// exceed the registers the CTA was launched with; the host launches only a
// build whose register count is at least kRegsLaunch (an increase that
// cannot be met would wait forever).
constexpr int kPhaseBarrier = 3;       // named barrier ending the tensor-core phase (1: decode, 2: merge)
constexpr int kEpilogueBarrier0 = 4;   // named barriers 4, 5: one per softmax warpgroup (output staging)
constexpr int kRegsLaunch = 168;
constexpr int kRegsLoader = 104;
constexpr int kRegsSoftmax = 192;
static_assert(kRegsLoader * 128 + kRegsSoftmax * 256 <= kRegsLaunch * kThreads, "register split exceeds the launch");
constexpr int kMmaWarp = 1;
constexpr int kVWarp = 2;              // loads V tiles; warp 0 loads Q and K tiles

// One KV cache as the kernel reads it: K and V [pages, P, Hkv, d], each
// through its own tensor maps (its own strides), and the page ids of its
// requests.
struct KvCache {
  CUtensorMap tm_k;   // boxes of (64 dims, 1 head, P slots, 1 page), 128-byte swizzle (tensor-core path)
  CUtensorMap tm_v;
  CUtensorMap tm_kd;  // boxes of (128 dims, 1 head, min(P, 128) slots, 1 page), no swizzle (CUDA-core path)
  CUtensorMap tm_vd;
  CUtensorMap tm_kg;  // page size 1: [pages * rows_per_page, d], rows of 128 dims gathered four at a time
  CUtensorMap tm_vg;
  CUtensorMap tm_kh;  // page size 1, multi-head units: boxes of (128 dims, mh_heads heads, 1 slot, 1 page)
  CUtensorMap tm_vh;
  const int32_t* kv_indices;
  int32_t page_size, log2_page, num_pages;
  int32_t tc;             // prefill-class items of this cache run on the tensor cores (tm_k, tm_v built)
  int32_t gather_rows;    // page size 1: decode stages by 4-row gathers of rows page * rows_k/v + head
  int32_t gather_rows_k;  // page stride / head stride of K (>= Hkv)
  int32_t gather_rows_v;  // the same for V
  int32_t mh_heads;       // KV heads of a multi-head unit's box (tm_kh, tm_vh built), else 0
};

struct RunParams {
  CUtensorMap tm_q;  // [q tokens, Hq, d] boxes of (64 dims, G heads, 128/G tokens), 128-byte swizzle
  CUtensorMap tm_o;  // O as [q tokens, Hq, d] with the boxes of tm_q: stores of whole 128-row output tiles
  // kv[0]: the cache of the plan's own requests; kv[1]: the shared blocks'
  // cache of a cascade plan (requests b < num_shared of the plan read it).
  KvCache kv[2];
  const uint16_t* q;
  int64_t q_stride_tok, q_stride_head;
  uint16_t* o;
  int64_t o_stride_tok, o_stride_head;
  float* lse;
  int32_t* iws;
  float* fws;
  int64_t partial_o_offset;  // floats
  int64_t max_partial_rows;  // partial-state rows the float workspace holds
  int32_t q_num_tokens;      // rows of Q and O
  float scale_log2;          // sm_scale * log2(e)
  int32_t num_qo_heads, num_kv_heads, group;
  int32_t has_shared;        // kv[1] was given (a cascade run)
  int32_t qk_prerotated;     // RoPE: tm_q and kv[0].tm_k read queries and keys of prefill-class requests
                             // already rotated (fp16) by a pass before the run
  int32_t late_merge;        // the late merge launch follows this run (else late units merge in the run)
};

// The cache request b reads (num_shared: the plan's shared blocks, 0 in a
// one-level plan).
__device__ __forceinline__ const KvCache& cache_of(const RunParams& p, int32_t b, int32_t num_shared) {
  return p.kv[b < num_shared ? 1 : 0];
}

struct DecodeBufs {
  uint16_t k[kStages][kStageTokens][kHeadDim];
  uint16_t v[kStages][kStageTokens][kHeadDim];
  union {  // xch while the stages stream, comb_o in the combine after them
    float comb_o[kHalfWarps][kRowsPerGroup][kHeadDim];
    float4 xch[kHalfWarps][kTokBlock + 1];  // per half-warp: p of each token (4 rows), then alpha
  };
  float comb_m[kHalfWarps][kRowsPerGroup];
  float comb_l[kHalfWarps][kRowsPerGroup];
};

// Every [128][64] block is one 16 KB operand half: 128 rows of 64 elements
// (128 bytes), 128-byte swizzled as TMA writes it and tcgen05 reads it.
struct PrefillBufs {
  uint16_t q[2][2][kTileM][64];     // [M tile][d half][row][dim]
  uint16_t k[2][2][kTileN][64];     // [stage][d half][token][dim]
  uint16_t v[2][2][kTileN][64];
  uint16_t ostage[2][kTileM][64];   // [M tile][row][dim]: one d half of an output tile on its way to a TMA store
};

struct alignas(1024) RunSmem {
  union {
    DecodeBufs dec;
    PrefillBufs pf;
  };
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t q_full, q_empty, drain;
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];   // [ring stage]
  uint64_t s_full[2], o_ready[2], o_free[2];  // [M tile of the item]
  uint64_t p_full[2][2];                      // [M tile][P of KV tokens 0..63, 64..127]
  uint64_t rot[kStages];                      // RoPE, decode: stage rotated (after full[])
  uint64_t q_rot, k_rot[2];                   // RoPE, prefill: Q tiles / K ring stage rotated
  uint32_t tmem_base;
  volatile int abort;  // set by the role whose bounded wait ran out
  int merge_last;
  int merge_last_pf;
};

constexpr size_t kSmemBytes = sizeof(RunSmem);
static_assert(kSmemBytes <= 227 * 1024, "shared memory of the run kernel exceeds one CTA's limit");

// Mask and logit variant of a plan (written into the workspace header by the
// planner): key j of a query at q_pos is visible only if j >= q_pos -
// window_left (window_left >= 0) or j < sink; with a soft-cap the logit is
// cap * tanh(scale * q.k / cap).  In the log2 domain the kernels work in,
// with u = scale * log2(e) * q.k, that is cap_a * tanh-form below with
// cap_a = cap * log2(e) and cap_b = 2 / cap.
struct Variant {
  int32_t window_left, sink;
  float cap_a, cap_b;
  const float2* rope_table;  // RoPE: (cos, sin)[position][64 pairs], or null
};

// Soft-capped log2-domain logit from the plain one, by the identity
// tanh y = 1 - 2 / (e^(2y) + 1): with t = 2^(u * cap_b) = e^(2y),
// cap_a * tanh y = cap_a - 2 cap_a / (t + 1).  t = +inf gives cap_a and
// t = 0 gives -cap_a, so the bound holds at both ends.
__device__ __forceinline__ float soft_cap_log2(float u, float cap_a, float cap_b) {
  const float t = ex2(u * cap_b);
  return cap_a - __fdividef(2.f * cap_a, t + 1.f);
}

// The hardware tanh (one MUFU operation; measured on GB300 against a double
// tanh over [-12, 12]: relative error below 1e-5, exactly +-1 past the
// saturation point).  The tensor-core softmax takes its soft-cap through it:
// that path is bound by instruction issue, and tanh(y), scaled by cap_a in
// the exponent's existing FMA, costs 1.5 instructions per logit (half a
// packed multiply and the tanh) against 3.5 for the exponential form above.
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Lowest visible key of a query at q_pos under the window (a bound below 0
// when there is no window).
__device__ __forceinline__ int window_low(const Variant& v, int q_pos) {
  return v.window_left >= 0 ? q_pos - v.window_left : -1;
}

struct Request {
  int32_t qo_start, qo_len, page_start, kv_len;
};

// A work item with its request's table entry (the plan writes both).
// heads: the KV heads hk .. hk + heads - 1 the item takes (1, or H of a
// multi-head unit, whose packed row r is head hk + r / G, query token 0).
struct Item {
  int32_t b, hk, row0, row1, kv0, kv1, part, merge;
  Request rq;
  int32_t heads;
};

__device__ __forceinline__ Item load_item(const int32_t* iws, int32_t off_items, int32_t i) {
  const int4* p = reinterpret_cast<const int4*>(iws + off_items + FI_ITEM_INTS * i);
  const int4 a = __ldg(p), c = __ldg(p + 1), r = __ldg(p + 2);
  const int32_t h = __ldg(reinterpret_cast<const int32_t*>(p + 3));
  return Item{a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w, Request{r.x, r.y, r.z, r.w}, h > 1 ? h : 1};
}

// Query token of packed row r of an item: r / G, and 0 in a multi-head item
// (one query token; its row r < heads * G is query head hk * G + r).  The
// query head is hk * G + r - t * G.
__device__ __forceinline__ int row_token(const Item& it, int r, int G) { return r / (it.heads * G); }

__device__ __forceinline__ Request load_request(const int32_t* iws, int32_t off_req, int32_t b) {
  int4 a = __ldg(reinterpret_cast<const int4*>(iws + off_req + FI_REQ_INTS * b));
  return Request{a.x, a.y, a.z, a.w};
}

}  // namespace fi

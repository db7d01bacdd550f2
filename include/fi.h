/*
 * fi.h -- C ABI of the GB300 (sm_103a) paged, block-sparse batched attention
 * library.  Plain C types only: device pointers are `void*`/typed pointers to
 * device memory, host pointers are marked HOST, a stream is a `cudaStream_t`
 * passed as `void*` (NULL = legacy default stream).
 *
 * The split of the work into a host "plan" and a device "run" follows the
 * FlashInfer paper summary, section "연구 방법론 / 3. 동적 부하 분산 스케줄링":
 * the work plan is built on the CPU from each request's runtime length so that
 * every SM gets an even share, it is then cached on the GPU, and the kernel
 * launch itself never changes, so it can be captured once in a CUDA graph.
 * The call shape (plan, then run(float workspace, int workspace, plan info,
 * q, kv cache, out, lse)) and the K/V stride comparison inside run follow the
 * BatchAttention PR page, section "코드 분석 §2".
 *
 * Ownership: the caller owns every buffer (device memory, the pinned host
 * staging buffer, the stream).  The library keeps no global allocations and
 * no handles.  Workspaces must outlive any CUDA graph that captured a run.
 *
 * Errors: every entry point returns an fi_status.  Argument and shape errors
 * are detected on the host before anything is enqueued, and then no device
 * memory is touched.  Kernel-side failures (a bounded wait that ran out) are
 * recorded in a status word inside the int workspace; read it with
 * fi_get_device_status().
 */
#ifndef FI_H_
#define FI_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FI_OK = 0,
    FI_ERR_INVALID_ARG = 1,  /* malformed indptr, lengths out of range, null pointer, ... */
    FI_ERR_UNSUPPORTED = 2,  /* head_dim, page_size, dtype or head ratio outside the supported set */
    FI_ERR_CAPACITY = 3,     /* plan does not fit the workspace capacities of the config */
    FI_ERR_ALIGNMENT = 4,    /* pointer or stride not 16-byte aligned */
    FI_ERR_CUDA = 5,         /* a CUDA runtime call failed */
    FI_ERR_DEVICE_CHECK = 6, /* the kernel recorded a failed device-side check */
    FI_ERR_TIMEOUT = 7       /* the kernel recorded a bounded wait that ran out */
} fi_status;

typedef enum { FI_FP16 = 0, FI_BF16 = 1, FI_FP32 = 2 } fi_dtype;

/* Fixed at workspace creation.  Every plan made with one config fits the same
 * workspaces and launches the same grid, which is what lets one captured
 * graph serve any plan. */
typedef struct {
    int32_t num_ctas;            /* persistent CTAs of run (grid size); <= SMs x resident CTAs per SM */
    int32_t max_batch;           /* requests per plan */
    int32_t max_items;           /* work items per plan */
    int32_t max_merge_units;     /* split units per plan */
    int64_t max_partial_rows;    /* rows of fp32 partial state (head_dim floats + 1 LSE each) */
    int32_t decode_min_chunk;    /* smallest KV chunk of a 16-row tile, tokens (default 256) */
    int32_t prefill_min_chunk;   /* smallest KV chunk of a 256-row tile, tokens (default 1024) */
    int32_t decode_cost_weight;  /* cost of one KV token in a 16-row tile (default 8) */
    int32_t prefill_cost_weight; /* cost of one KV token in a 256-row tile (default 9) */
    int32_t split_factor;        /* target chunks per CTA per tile class (default 1) */
    /* Mask and logit variant, constant for a model (FlashInfer 0.6 wiki page,
     * "Blackwell (SM100/SM103) 전용 경로 / CuTe-DSL GQA Decode 커널": sliding
     * window and attention sink; FlashInfer paper summary, "2. 유연한 어텐션
     * 변형 지원": logits transforms).  Query token t of a request with Lq
     * queries and Lkv keys sits at q_pos = Lkv - Lq + t.
     *   window_left >= 0: key j is visible only if j >= q_pos - window_left
     *     (-1, the default: no window); the plan skips KV chunks that no row
     *     of a tile can see;
     *   sink_tokens: keys j < sink_tokens stay visible whatever the window
     *     says (the causal bound still applies; default 0);
     *   logits_soft_cap > 0: the softmax logit is
     *     cap * tanh(sm_scale * q.k / cap) (0, the default: sm_scale * q.k);
     *     run then launches the capped kernel (fi_plan_info.variant bit 0).
     * Negative sink_tokens, window_left < -1 or a negative or non-finite cap
     * are FI_ERR_INVALID_ARG. */
    int32_t window_left;
    int32_t sink_tokens;
    float logits_soft_cap;
    /* RoPE fused into the attention loaders (FlashInfer paper summary,
     * "주요 성능 테스트 결과 / 2. 커널 수준 성능": a custom kernel fusing RoPE with attention).  The
     * cache holds keys WITHOUT rotation; the kernel rotates q and k on the
     * fly, Llama style: dims i and i + 64 form a pair rotated by the angle
     * (pos / rope_scale) * rope_theta^(-2i/128), i < 64, with key j at
     * position j and query token t of a request at position Lkv - Lq + t
     * (the bottom-right alignment of the causal mask).
     *   rope_max_positions > 0 turns it on: positions must stay below it (a
     *     plan with a longer request, or with Lq > Lkv, is
     *     FI_ERR_INVALID_ARG), and the int workspace then also holds a
     *     cos/sin table for these positions, filled by fi_rope_init;
     *   rope_theta > 0 (10000 for Llama 2, 500000 for Llama 3);
     *   rope_scale > 0 divides the positions (1 = no scaling).
     * Rotated keys (and the tensor-core path's rotated queries) are fp16
     * whatever the cache type; a rotated value past the fp16 range (|x| >
     * 65504, reachable from bf16 inputs) records FI_ERR_DEVICE_CHECK in the
     * status word, and the outputs of that run are undefined. */
    int32_t rope_max_positions;
    float rope_theta;
    float rope_scale;
    int32_t reserved;
} fi_plan_config;

/* Plain data returned by fi_plan; passed to run by value semantics. */
typedef struct {
    int32_t num_ctas;
    int32_t num_items;
    int32_t num_merge_units;
    int32_t batch;
    int64_t num_partial_rows;
    int32_t num_qo_heads, num_kv_heads, head_dim, page_size, causal;
    int32_t chunk_decode;        /* KV tokens per chunk chosen for 16-row tiles */
    int32_t chunk_prefill;       /* KV tokens per chunk chosen for 256-row tiles */
    int32_t num_decode_items, num_prefill_items;
    int32_t variant;             /* bit 0: logits soft-cap; bit 1: sliding window (and sink) mask; bit 2: RoPE */
    int64_t int_ws_bytes_used;   /* bytes of the int workspace written (and copied) by the plan */
    int64_t max_partial_rows;    /* capacity of the float workspace, from the config */
    int32_t num_late_merge_units; /* split units of prefill-class tiles: merged by a second launch */
    int32_t num_shared;          /* cascade plan: shared blocks (0 for a one-level plan) */
    int32_t num_cascade_merges;  /* cascade plan: entries of the cascade merge (a second launch) */
    int32_t prefill_caches;      /* caches read by prefill-class units: bit 0 the ordinary one, bit 1 the shared one */
} fi_plan_info;

/* Defaults, with num_ctas derived from the device's SM count and the run
 * kernel's occupancy (cudaOccupancyMaxActiveBlocksPerMultiprocessor), so a
 * plan never asks for more CTAs than can be resident at once. */
fi_status fi_default_plan_config(int device, fi_plan_config* out);

/* Workspace sizes for a config (bytes).  The int workspace holds the plan,
 * the merge counters and the device status word (and, with RoPE, the cos/sin
 * table after them); the float workspace holds fp32 partial states of split
 * work.  Both are device memory. */
size_t fi_int_workspace_bytes(const fi_plan_config* cfg);
size_t fi_float_workspace_bytes(const fi_plan_config* cfg, int32_t head_dim);

/*
 * fi_rope_init -- fill the RoPE cos/sin table of an int workspace made for
 * `cfg` (rope_max_positions > 0): cos and sin of (pos / rope_scale) *
 * rope_theta^(-2i/128) for pos < max(rope_max_positions, 16) and i < 64, computed in
 * fp64 and stored as fp32.  Once per workspace (and again if the config's
 * RoPE fields change); plans never overwrite the table.  Asynchronous on
 * `stream`.  FI_ERR_INVALID_ARG when the config has no RoPE or a theta or
 * scale <= 0.
 */
fi_status fi_rope_init(const fi_plan_config* cfg, void* int_workspace_dev, void* stream);

/*
 * fi_rope_apply_k -- the unfused form: rotate, outside attention, every key
 * of the plan's requests (key j at position j, the rotation the fused
 * kernel applies; paper summary, "주요 성능 테스트 결과 / 2. 커널 수준 성능",
 * compares the two forms) from k_in into k_out, both [num_pages, page_size,
 * num_kv_heads, 128] with their own strides (elements, multiples of 16
 * bytes) and the plan's page ids; k_out may be k_in.  Output in the cache's
 * own type.  Uses the plan in int_workspace_dev (request table and RoPE
 * table): FI_ERR_INVALID_ARG for a plan made without RoPE or a cascade plan.
 * One kernel, flat over the plan's key slots, its counts read from the
 * workspace (a captured graph serves later plans).  An fp16 cache whose
 * rotated value leaves the fp16 range records FI_ERR_DEVICE_CHECK in the
 * status word.  Asynchronous on `stream`.
 */
fi_status fi_rope_apply_k(const fi_plan_info* info, void* int_workspace_dev, const void* k_in,
                          const int64_t k_in_strides[3], void* k_out, const int64_t k_out_strides[3],
                          const int32_t* kv_indices_dev, fi_dtype dtype, void* stream);

/*
 * fi_rope_apply_q -- the unfused form for queries: rotate every query row of
 * the plan's requests (token t of a request at position kv_len - qo_len + t)
 * from q_in [tokens, num_qo_heads, 128] (strides q_in_stride_tok,
 * q_in_stride_head, 1) into q_out (its own strides; q_out may be q_in), in
 * the input's own type.  Arguments, checks, status and stream behaviour as
 * fi_rope_apply_k.
 */
fi_status fi_rope_apply_q(const fi_plan_info* info, void* int_workspace_dev, const void* q_in,
                          int64_t q_in_stride_tok, int64_t q_in_stride_head, void* q_out, int64_t q_out_stride_tok,
                          int64_t q_out_stride_head, fi_dtype dtype, void* stream);

/*
 * fi_plan -- build the load-balanced split-KV work list on the host and copy
 * it into int_workspace_dev with one cudaMemcpyAsync on `stream`.
 *
 * Paged KV as a block-sparse matrix (paper summary, "1. 통합된 KV 캐시 추상화";
 * wiki, "FlashInfer 아키텍처 / 1) 블록-스파스 KV 포맷"): request b owns query
 * tokens [qo_indptr[b], qo_indptr[b+1]) and pages
 * kv_indices[kv_indptr[b] .. kv_indptr[b+1]); its KV length is
 * (pages-1)*page_size + last_page_len[b] (0 when it has no page).
 *
 * All four arrays are HOST memory, int32: qo_indptr and kv_indptr have
 * batch+1 entries, start at 0 and never decrease; last_page_len has batch
 * entries in [1, page_size] for requests with pages; kv_indices has
 * kv_indptr[batch] entries (read only for validation against num_pages when
 * num_pages > 0).
 *
 * Supported: head_dim == 128; page_size a power of two in [1, 128];
 * num_qo_heads % num_kv_heads == 0 with group size <= 16.
 *
 * Work units are (request, KV head, tile of packed query rows), split into
 * KV chunks.  With page_size 1, no RoPE and a group size G in {4, 8, 16}
 * whose 32 / G divides num_kv_heads, a one-token request's units take 32 / G
 * KV heads at once (32 packed rows): such a unit pays the per-item cost once
 * for all its heads and each token of its KV arrives in one copy.
 *
 * pinned_staging_host: caller-owned pinned host buffer of at least
 * fi_int_workspace_bytes(cfg) bytes; the plan is written there and copied
 * from there asynchronously, so it must not be reused until the copy on
 * `stream` has completed.  The plan rule is deterministic: equal inputs give
 * byte-identical workspaces.
 */
fi_status fi_plan(const fi_plan_config* cfg, const int32_t* qo_indptr, const int32_t* kv_indptr,
                  const int32_t* kv_indices, const int32_t* last_page_len, int32_t batch,
                  int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                  int32_t causal, int32_t num_pages, void* int_workspace_dev, void* pinned_staging_host,
                  size_t staging_bytes, void* stream, fi_plan_info* info_out);

/*
 * fi_plan_host -- the same rule as fi_plan, writing the workspace image into
 * a HOST buffer only (no CUDA call).  Used to inspect a plan.
 */
fi_status fi_plan_host(const fi_plan_config* cfg, const int32_t* qo_indptr, const int32_t* kv_indptr,
                       const int32_t* kv_indices, const int32_t* last_page_len, int32_t batch,
                       int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                       int32_t causal, int32_t num_pages, void* workspace_host, size_t workspace_bytes,
                       fi_plan_info* info_out);

/*
 * fi_plan_cascade -- plan one launch over a two-level KV layout: every query
 * row attends to the keys of its shared block (level 0, read from a shared
 * cache; e.g. a prompt prefix common to several requests, stored once as a
 * dense block) and to its own request's pages (level 1), and the two partial
 * results are merged by their log-sum-exp (paper summary, "1. 통합된 KV 캐시
 * 추상화": composable formats -- a shared prefix as one dense block, the
 * request-specific suffixes as a sparse format, computed apart and merged;
 * and "주요 성능 테스트 결과 / 1. 엔드투엔드 성능", parallel generation).  One
 * run then computes both levels in a single persistent launch (the shared
 * blocks' units on the tensor cores when they have more than 16 packed rows)
 * and a second, small launch merges them.
 *
 * Level 1 is an ordinary batch (qo_indptr, kv_indptr, kv_indices,
 * last_page_len: HOST arrays as for fi_plan, pages of page_size in the
 * requests' own cache), covering query rows [0, qo_indptr[batch]).  Level 0:
 * num_shared >= 1 blocks (HOST arrays, num_shared + 1 / num_shared + 1 /
 * shared_kv_indptr[num_shared] / num_shared entries); block s owns query rows
 * [shared_qo_indptr[s], shared_qo_indptr[s+1]) -- the blocks start at 0, cover
 * every row, and no request straddles two -- and the pages
 * shared_kv_indices[shared_kv_indptr[s] .. shared_kv_indptr[s+1]) of the
 * shared cache (pages of shared_page_size, its last page holding
 * shared_last_page_len[s] slots).  A block with no page adds nothing.
 *
 * Visibility: every key of a row's block is visible to the row (the block
 * precedes all of its queries); the row's own keys follow `causal`, aligned
 * to the bottom right of the request's own keys, and a causal request must
 * hold at least as many keys as queries (its queries are among its keys).
 * That is attention over the concatenation block ++ own pages with the
 * bottom-right causal mask.  The logits soft-cap applies; a sliding window,
 * sink tokens or RoPE in `cfg` are FI_ERR_UNSUPPORTED here (their positions
 * would have to span two caches).
 *
 * The plan numbers the blocks first in its request table; every unit writes
 * fp32 partial states (float workspace) and fi_plan_info.num_cascade_merges
 * > 0 tells the run to follow with the cascade merge.  Other rules, errors,
 * staging and copy as for fi_plan; FI_ERR_CAPACITY also when the merge
 * entries (runs of up to 16 packed rows of one unit) exceed
 * cfg->max_merge_units or the requests and blocks together exceed
 * cfg->max_batch.
 */
fi_status fi_plan_cascade(const fi_plan_config* cfg, const int32_t* shared_qo_indptr,
                          const int32_t* shared_kv_indptr, const int32_t* shared_kv_indices,
                          const int32_t* shared_last_page_len, int32_t num_shared, int32_t shared_page_size,
                          int32_t shared_num_pages, const int32_t* qo_indptr, const int32_t* kv_indptr,
                          const int32_t* kv_indices, const int32_t* last_page_len, int32_t batch,
                          int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                          int32_t causal, int32_t num_pages, void* int_workspace_dev, void* pinned_staging_host,
                          size_t staging_bytes, void* stream, fi_plan_info* info_out);

/* fi_plan_cascade_host -- the same rule, writing the workspace image into a
 * HOST buffer only (no CUDA call). */
fi_status fi_plan_cascade_host(const fi_plan_config* cfg, const int32_t* shared_qo_indptr,
                               const int32_t* shared_kv_indptr, const int32_t* shared_kv_indices,
                               const int32_t* shared_last_page_len, int32_t num_shared, int32_t shared_page_size,
                               int32_t shared_num_pages, const int32_t* qo_indptr, const int32_t* kv_indptr,
                               const int32_t* kv_indices, const int32_t* last_page_len, int32_t batch,
                               int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                               int32_t causal, int32_t num_pages, void* workspace_host, size_t workspace_bytes,
                               fi_plan_info* info_out);

/*
 * fi_batch_paged_attention_run -- one persistent kernel over the planned
 * work list: O = softmax(scale * Q K^T + mask) V per query row and head, and
 * LSE = log sum exp(scale * q.k) (natural log) over the visible keys.
 *
 * Layouts (all element strides; the last dimension is contiguous):
 *   q  [q_num_tokens, num_qo_heads, head_dim]      strides (q_stride_tok, q_stride_head, 1)
 *   k  [num_pages, page_size, num_kv_heads, d]     strides k_strides[0..2], 1
 *   v  [num_pages, page_size, num_kv_heads, d]     strides v_strides[0..2], 1
 *   o  [q_num_tokens, num_qo_heads, head_dim]      strides (o_stride_tok, o_stride_head, 1)
 *   lse[q_num_tokens, num_qo_heads] fp32, contiguous; may be NULL.
 * q, k, v and o share `dtype` (FI_FP16 or FI_BF16).  Every base pointer and
 * every stride in bytes must be a multiple of 16.  K and V strides may differ
 * (the equal-stride case is detected here, BatchAttention PR page, "코드 분석
 * §2").  kv_indices_dev is the device copy of the page table given to the
 * plan.  q_num_tokens and num_pages are the extents of the buffers (they may
 * exceed what the plan uses, so a graph can be captured once at capacity).
 * Query head h reads KV head h / (num_qo_heads / num_kv_heads); a query row
 * with no visible key gets O = 0 and LSE = -inf.  Causal masks are aligned to
 * the bottom right: query token t of a request sees key j iff
 * j <= kv_len - qo_len + t.
 *
 * Asynchronous on `stream`; never allocates, synchronizes or copies from the
 * host, so it can be captured in a CUDA graph.  The kernel reads the counts
 * of the current plan from the int workspace, and before any work checks that
 * plan against this launch: its CTA count (the grid), its partial-state rows
 * (info->max_partial_rows, the float workspace's capacity), its query tokens
 * (q_num_tokens), its head counts and its page size.  A mismatch -- a
 * workspace re-planned after `info` was taken, or `info` of another config --
 * records FI_ERR_DEVICE_CHECK in the status word and nothing is written.  When info->num_late_merge_units
 * > 0 (split units of prefill-class tiles) a second kernel follows on the
 * same stream and merges those units row-parallel, reading its counts from
 * the workspace too; it merges nothing when the run has set the status word.
 * With info->num_late_merge_units == 0 (as in a graph captured from a plan
 * without late units) the run merges any late units of the current plan
 * itself, one CTA per unit: correct either way, faster with the second
 * kernel, so capture from a plan with late units when later plans may have
 * them.
 */
fi_status fi_batch_paged_attention_run(const fi_plan_info* info, const void* q, int64_t q_stride_tok,
                                       int64_t q_stride_head, int32_t q_num_tokens, const void* k_cache,
                                       const int64_t k_strides[3], const void* v_cache,
                                       const int64_t v_strides[3], int32_t num_pages,
                                       const int32_t* kv_indices_dev, void* o, int64_t o_stride_tok,
                                       int64_t o_stride_head, float* lse, fi_dtype dtype, float sm_scale,
                                       void* int_workspace_dev, void* float_workspace_dev, void* stream);

/*
 * fi_batch_paged_attention_run_rope_prerotated -- fi_batch_paged_attention_run
 * for a plan made with RoPE (fi_plan_config.rope_max_positions > 0), with the
 * queries and keys of prefill-class requests (more than 16 packed query rows)
 * rotated once before the kernel instead of inside it (paper summary, "주요
 * 성능 테스트 결과 / 2. 커널 수준 성능": RoPE fused with attention).
 * Decode-class requests read each key once, and the kernel keeps rotating
 * their queries and keys as it loads them.  A prefill-class request's keys
 * are read by every 256-row work item of the request (tens of times for a
 * long causal prefill), and the tensor-core phase has only two warps free to
 * rotate them, so they are rotated by one pass over the request's keys into
 * k_rot -- its queries into q_rot -- and the tensor cores read both from
 * there.  The arguments are those of fi_batch_paged_attention_run plus two
 * caller-owned device buffers in **fp16** (rotated values are fp16 whatever
 * the cache type, as on the fused path: q and k meet only each other in
 * S = q.k):
 *   q_rot [q_num_tokens, num_qo_heads, 128], strides (q_rot_stride_tok,
 *         q_rot_stride_head, 1), rows of prefill-class requests written;
 *   k_rot [num_pages, page_size, num_kv_heads, 128], strides k_rot_strides,
 *         written at the pages of prefill-class requests (same page ids as
 *         the cache); the rest of both buffers is left alone.
 * Strides are elements, multiples of 16 bytes.  FI_ERR_INVALID_ARG for a plan
 * without RoPE or a cascade plan.  With pages under 8 tokens (no tensor-core
 * path), or when `info` has no prefill-class item, the call is the fully
 * fused run and the buffers are not touched.  Otherwise two kernels on
 * `stream`: the rotation pass (its counts read from the workspace, so a
 * captured graph serves later plans), then the run -- on the kernel without
 * RoPE when `info` has no decode-class item.  That kernel refuses a
 * workspace re-planned since with decode-class items (FI_ERR_DEVICE_CHECK,
 * nothing written): capture such graphs from a plan with decode-class items.
 * A rotated value past the fp16 range (|x| > 65504, reachable from bf16
 * inputs) records FI_ERR_DEVICE_CHECK; the outputs of that run are then
 * undefined.  The fully fused run reports the same.  Asynchronous.
 */
fi_status fi_batch_paged_attention_run_rope_prerotated(
    const fi_plan_info* info, const void* q, int64_t q_stride_tok, int64_t q_stride_head, int32_t q_num_tokens,
    const void* k_cache, const int64_t k_strides[3], const void* v_cache, const int64_t v_strides[3],
    int32_t num_pages, const int32_t* kv_indices_dev, void* q_rot, int64_t q_rot_stride_tok,
    int64_t q_rot_stride_head, void* k_rot, const int64_t k_rot_strides[3], void* o, int64_t o_stride_tok,
    int64_t o_stride_head, float* lse, fi_dtype dtype, float sm_scale, void* int_workspace_dev,
    void* float_workspace_dev, void* stream);

/*
 * fi_batch_paged_attention_run_cascade -- the run of a plan made by
 * fi_plan_cascade: the arguments of fi_batch_paged_attention_run for the
 * requests' own cache (k_cache, v_cache, their strides, num_pages,
 * kv_indices_dev), plus the shared blocks' cache: shared_k_cache and
 * shared_v_cache [shared_num_pages, shared_page_size, num_kv_heads, d] with
 * their own strides (elements, multiples of 16 bytes) and the device copy of
 * shared_kv_indices.  The two caches may be views of one allocation (a dense
 * prefix viewed as pages of 16 inside a pool of pages of 1, say).  One
 * persistent launch computes every unit of both levels into the float
 * workspace, then a second launch merges each row's shared and own states in
 * that order and writes O (storage type) and LSE (natural log).  A row whose
 * block and own pages are both empty gets O = 0, LSE = -inf.  Asynchronous,
 * capture-safe and checked on the device as fi_batch_paged_attention_run
 * (the plan's shared page size must equal shared_page_size).
 * fi_batch_paged_attention_run given a cascade plan returns
 * FI_ERR_INVALID_ARG (it has no shared cache).
 */
fi_status fi_batch_paged_attention_run_cascade(
    const fi_plan_info* info, const void* q, int64_t q_stride_tok, int64_t q_stride_head, int32_t q_num_tokens,
    const void* k_cache, const int64_t k_strides[3], const void* v_cache, const int64_t v_strides[3],
    int32_t num_pages, const int32_t* kv_indices_dev, const void* shared_k_cache, const int64_t shared_k_strides[3],
    const void* shared_v_cache, const int64_t shared_v_strides[3], int32_t shared_num_pages,
    const int32_t* shared_kv_indices_dev, int32_t shared_page_size, void* o, int64_t o_stride_tok,
    int64_t o_stride_head, float* lse, fi_dtype dtype, float sm_scale, void* int_workspace_dev,
    void* float_workspace_dev, void* stream);

/*
 * fi_batch_paged_attention_run_static_scratch -- fi_batch_paged_attention_run
 * for callers that cannot allocate device memory.  The paper has no
 * counterpart; it exists for this library's users.
 *
 * Who needs it: code that has no device allocator at hand or must not call
 * one at this point -- a plugin that its host runtime gives only fixed input
 * and output buffers, a server that reserved all device memory up front, or
 * code for which an allocation would synchronise the device.  Such a caller
 * cannot provide the float workspace, so here the split-KV partial states
 * live in one fixed device array inside the library, sized for at most 32768
 * partial rows (about 17 MB; every GPU that loads the library holds it until
 * the process exits).  The call itself allocates nothing.
 *
 * Arguments are those of fi_batch_paged_attention_run without
 * float_workspace_dev; the caller still passes the inputs, the outputs and
 * the int workspace filled by fi_plan.  Returns FI_ERR_CAPACITY, before
 * anything is enqueued, when info->num_partial_rows exceeds 32768 (plan with
 * fewer CTAs, a larger split chunk or a smaller batch).  The kernel repeats
 * that check on the plan it finds in the int workspace: a workspace
 * re-planned beyond 32768 partial rows after `info` was taken is refused on
 * the device (FI_ERR_DEVICE_CHECK in the status word, nothing written, the
 * array never written past its end).
 *
 * The first call on a device looks up the array's device address on that
 * device (the current one).
 * All calls share the one array and it keeps the last call's contents;
 * nothing in it has to start at zero (every partial row is written before it
 * is read; the merge counters live in the int workspace).  Calls whose
 * kernels overlap on the GPU (other streams, other threads) race on the
 * array: serialise them.
 */
fi_status fi_batch_paged_attention_run_static_scratch(const fi_plan_info* info, const void* q, int64_t q_stride_tok,
                                                      int64_t q_stride_head, int32_t q_num_tokens, const void* k_cache,
                                                      const int64_t k_strides[3], const void* v_cache,
                                                      const int64_t v_strides[3], int32_t num_pages,
                                                      const int32_t* kv_indices_dev, void* o, int64_t o_stride_tok,
                                                      int64_t o_stride_head, float* lse, fi_dtype dtype,
                                                      float sm_scale, void* int_workspace_dev, void* stream);

/*
 * fi_merge_states -- merge two attention states row by row (paper summary,
 * "1. 통합된 KV 캐시 추상화": a shared dense prefix and per-request sparse
 * suffixes are computed separately and combined):
 *   s = log(exp(s_a) + exp(s_b)),  v = exp(s_a - s) v_a + exp(s_b - s) v_b.
 * (v, -inf) is the identity; two -inf states give (0, -inf).
 *   v_a, v_b, v_out [rows, heads, head_dim] contiguous, element type dtype
 *   (FI_FP16, FI_BF16 or FI_FP32); s_a, s_b, s_out [rows, heads] fp32.
 * v_out may alias v_a or v_b, s_out may alias s_a or s_b.  Asynchronous.
 */
fi_status fi_merge_states(const void* v_a, const float* s_a, const void* v_b, const float* s_b, void* v_out,
                          float* s_out, int32_t rows, int32_t heads, int32_t head_dim, fi_dtype dtype,
                          void* stream);

/* Reads the device status word of an int workspace (synchronizes `stream`).
 * *status_out is FI_OK, FI_ERR_TIMEOUT or FI_ERR_DEVICE_CHECK. */
fi_status fi_get_device_status(const void* int_workspace_dev, void* stream, int32_t* status_out);

/*
 * fi_selftest_bounded_wait -- check the failure path without a fault: one
 * warp waits, with the kernels' own bounded wait (about 0.5 s of SM clocks),
 * on a barrier that nothing completes; when the wait gives up it records
 * FI_ERR_TIMEOUT in the status word of int_workspace_dev (the next plan
 * copied into that workspace clears it).  Asynchronous on `stream`; read the
 * result with fi_get_device_status.  The context stays usable.
 */
fi_status fi_selftest_bounded_wait(void* int_workspace_dev, void* stream);

const char* fi_status_string(fi_status s);

#ifdef __cplusplus
}
#endif

#endif /* FI_H_ */

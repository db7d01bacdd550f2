/*
 * fi_mla.h -- C ABI of the absorbed-MLA decode path of the GB300 (sm_103a)
 * attention library.  Same conventions as fi.h (plain C types, HOST marks
 * host pointers, a stream is a cudaStream_t passed as void*, every entry
 * returns an fi_status, the caller owns every buffer).
 *
 * What it computes (FlashInfer 0.6 wiki page, section "MLA(Multi-head Latent
 * Attention) 커널": the cache keeps one latent vector per token and the
 * up-projections are folded into the attention, which then runs on the
 * latents directly).  DeepSeek-V3 shapes: latent 512, RoPE key 64.  For
 * request b with L cached tokens and query head h < num_heads:
 *
 *   s_j   = sm_scale * (q_nope[b,h,:] . ckv[j,:] + q_pe[b,h,:] . kpe[j,:])
 *   o     = sum_j softmax_j(s) ckv[j,:]                 (512 dims)
 *   lse   = log sum_j exp(s_j)                          (natural log)
 *
 * q_nope is the query already multiplied by the absorbed key up-projection;
 * the value up-projection of o is left to the caller.  A request with no
 * cached token gets o = 0 and lse = -inf.  One query token per request.
 *
 * Work split (the wiki's section "Blackwell (SM100/SM103) 전용 경로 / SM103
 * (B300) MLA 디코드" names a cluster-aware split-KV MLA decode on B300): the
 * plan cuts each request's KV into chunks and deals them to CTA pairs; the
 * two CTAs of a pair (a thread-block cluster) each own half of the 512
 * output dims and exchange their halves of the logits through distributed
 * shared memory.  Chunks of one request are merged by a second kernel.
 */
#ifndef FI_MLA_H_
#define FI_MLA_H_

#include <stddef.h>
#include <stdint.h>

#include "fi.h"

#ifdef __cplusplus
extern "C" {
#endif

#define FI_MLA_LATENT_DIM 512
#define FI_MLA_ROPE_DIM 64
#define FI_MLA_MAX_HEADS 128

/* Fixed at workspace creation; plans made with one config fit the same
 * workspaces and launch the same grids (so one captured graph serves all). */
typedef struct {
    int32_t num_pairs;      /* CTA pairs of the decode kernel (grid = 2 x num_pairs) */
    int32_t max_batch;      /* requests per plan */
    int32_t max_units;      /* KV chunks per plan */
    int32_t max_parts;      /* chunks of split requests per plan (fp32 partial states) */
    int32_t min_chunk;      /* shortest piece cut off a request (a request's last piece may be
                               shorter), tokens, a multiple of 64 (default 256) */
    int32_t reserved[3];
} fi_mla_config;

typedef struct {
    int32_t num_pairs;
    int32_t num_units;
    int32_t num_parts;
    int32_t num_merge;      /* requests with 0 or >= 2 chunks (finished by the merge kernel) */
    int32_t batch;
    int32_t num_heads;
    int32_t page_size;
    int32_t chunk;          /* the first pair's budget, token-equivalents (tokens + 192 per piece) */
    int64_t int_ws_bytes_used;
    int32_t max_parts;
    int32_t reserved;
} fi_mla_plan_info;

/* Defaults; num_pairs = the device's cudaOccupancyMaxActiveClusters for the
 * decode kernel with clusters of 2 (every pair resident at once). */
fi_status fi_mla_default_config(int device, fi_mla_config* out);

/* Workspace sizes (bytes, device memory).  The int workspace holds the plan
 * and the device status word (read with fi_get_device_status); the float
 * workspace the fp32 partial states: max_parts x 128 rows of 512 floats plus
 * one LSE each. */
size_t fi_mla_int_workspace_bytes(const fi_mla_config* cfg);
size_t fi_mla_float_workspace_bytes(const fi_mla_config* cfg);

/*
 * fi_mla_plan -- build the work list on the host and copy it into
 * int_workspace_dev with one cudaMemcpyAsync on `stream` from the caller's
 * pinned staging buffer (>= fi_mla_int_workspace_bytes bytes; not reused
 * until the copy has completed).
 *
 * kv_indptr (batch + 1 entries), kv_indices (kv_indptr[batch]) and
 * last_page_len (batch) are HOST int32 arrays with the meaning of fi_plan's;
 * kv_indices is read only to validate ids against num_pages when
 * num_pages > 0.  page_size is 8, 16, 32 or 64; 1 <= num_heads <= 128.
 * Deterministic: equal inputs give byte-identical workspaces.
 */
fi_status fi_mla_plan(const fi_mla_config* cfg, const int32_t* kv_indptr, const int32_t* kv_indices,
                      const int32_t* last_page_len, int32_t batch, int32_t num_heads, int32_t page_size,
                      int32_t num_pages, void* int_workspace_dev, void* pinned_staging_host, size_t staging_bytes,
                      void* stream, fi_mla_plan_info* info_out);

/* The same rule, writing the workspace image into a HOST buffer only. */
fi_status fi_mla_plan_host(const fi_mla_config* cfg, const int32_t* kv_indptr, const int32_t* kv_indices,
                           const int32_t* last_page_len, int32_t batch, int32_t num_heads, int32_t page_size,
                           int32_t num_pages, void* workspace_host, size_t workspace_bytes,
                           fi_mla_plan_info* info_out);

/*
 * fi_mla_decode_run -- the decode kernel over the plan, then the merge
 * kernel; two launches with fixed grids, no allocation, no host copy
 * (capturable in a CUDA graph).
 *
 * Layouts (bf16; element strides; the last dimension contiguous):
 *   q_nope [q_rows, num_heads, 512]  strides (q_nope_stride_tok, q_nope_stride_head, 1)
 *   q_pe   [q_rows, num_heads, 64]   strides (q_pe_stride_tok, q_pe_stride_head, 1)
 *   ckv    [num_pages, page_size, 512]  strides (ckv_stride_page, ckv_stride_slot, 1)
 *   kpe    [num_pages, page_size, 64]   strides (kpe_stride_page, kpe_stride_slot, 1)
 *   o      [q_rows, num_heads, 512]  bf16, contiguous
 *   lse    [q_rows, num_heads]       fp32, contiguous (may be NULL)
 * Row b of q and o belongs to request b (q_rows >= the plan's batch).
 * Every base pointer and every stride in bytes is a multiple of 16.
 * kv_indices_dev is the device copy of the plan's page table.
 */
fi_status fi_mla_decode_run(const fi_mla_plan_info* info, const void* q_nope, int64_t q_nope_stride_tok,
                            int64_t q_nope_stride_head, const void* q_pe, int64_t q_pe_stride_tok,
                            int64_t q_pe_stride_head, int32_t q_rows, const void* ckv, int64_t ckv_stride_page,
                            int64_t ckv_stride_slot, const void* kpe, int64_t kpe_stride_page,
                            int64_t kpe_stride_slot, int32_t num_pages, const int32_t* kv_indices_dev, void* o,
                            float* lse, float sm_scale, void* int_workspace_dev, void* float_workspace_dev,
                            void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FI_MLA_H_ */

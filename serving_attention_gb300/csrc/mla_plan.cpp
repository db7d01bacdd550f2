// mla_plan.cpp -- host planner of the absorbed-MLA decode kernel.
//
// The same idea as the GQA planner (FlashInfer paper summary, section "연구
// 방법론 / 3. 동적 부하 분산 스케줄링": the CPU turns the requests' lengths
// into an even per-SM work list once per step, and the launch never
// changes), with the split-KV of the wiki's "SM103 (B300) MLA 디코드"
// section.  Rule (this library's reading; the pages give no cost model):
//  * the requests with tokens form one stream in index order, and the pairs
//    are filled one after another with consecutive pieces of it;
//  * a piece costs its tokens + FI_MLA_UNIT_COST_TOKENS; pair c's budget is
//    max(ceil(R / (P - c)), FI_MLA_UNIT_COST_TOKENS + min_chunk), where R =
//    the tokens left + FI_MLA_UNIT_COST_TOKENS x (requests with tokens left +
//    pairs left - 1): each pair boundary still to come splits one request;
//  * a pair takes the next piece of at most its remaining budget minus the
//    piece cost, rounded down to the 64-token block (the whole rest of the
//    request when that fits); it stops when that would cut a piece shorter
//    than min_chunk off a request, or when less than one block fits; the
//    last pair takes everything left, whatever its budget;
//  * a request cut into several pieces gets one fp32 partial-state slot per
//    piece and a merge entry; a request with no tokens gets a merge entry
//    that writes (0, -inf).
// The budget counts what is still to be split, so every pair but the last
// stays within its budget and the loads differ by little more than a piece
// cost, where dealing fixed-size chunks longest-first left the busiest pair
// of the decode length mix 24 % above the mean.  The piece cost (448 tokens:
// Q into tensor memory, pipeline refill, epilogue) is measured: charging
// 192 / 320 / 448 / 640 gave 181.4 / 171.1 / 167.0 / 167.0 us on that mix.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <vector>

#include "../../include/fi_mla.h"
#include "mla_layout.h"

namespace {

int64_t capacity_ints(const fi_mla_config* c) {
  return FI_MLA_HEADER_INTS + fi_mla_round4(int64_t(c->num_pairs) + 1) + int64_t(FI_MLA_UNIT_INTS) * c->max_units +
         fi_mla_round4(int64_t(FI_MLA_REQ_INTS) * c->max_batch) + int64_t(FI_MLA_MERGE_INTS) * c->max_batch;
}

bool config_ok(const fi_mla_config* c) {
  return c && c->num_pairs >= 1 && c->max_batch >= 1 && c->max_units >= 1 && c->max_parts >= 0 &&
         c->min_chunk >= FI_MLA_BLOCK && c->min_chunk % FI_MLA_BLOCK == 0;
}

struct Unit {
  int32_t b, kv0, kv1, part;
};

}  // namespace

extern "C" size_t fi_mla_int_workspace_bytes(const fi_mla_config* cfg) {
  if (!config_ok(cfg)) return 0;
  return size_t(capacity_ints(cfg)) * 4;
}

extern "C" size_t fi_mla_float_workspace_bytes(const fi_mla_config* cfg) {
  if (!config_ok(cfg)) return 0;
  const int64_t parts = std::max<int64_t>(cfg->max_parts, 1);
  return size_t(fi_mla_partial_o_offset(parts) + parts * FI_MLA_ROWS * FI_MLA_LATENT_DIM) * 4;
}

extern "C" fi_status fi_mla_plan_host(const fi_mla_config* cfg, const int32_t* kv_indptr, const int32_t* kv_indices,
                                      const int32_t* last_page_len, int32_t batch, int32_t num_heads,
                                      int32_t page_size, int32_t num_pages, void* workspace_host,
                                      size_t workspace_bytes, fi_mla_plan_info* info_out) {
  if (!config_ok(cfg) || !workspace_host || !info_out || batch < 0 || !kv_indptr) return FI_ERR_INVALID_ARG;
  if (batch > 0 && !last_page_len) return FI_ERR_INVALID_ARG;
  if (num_heads < 1 || num_heads > FI_MLA_MAX_HEADS) return FI_ERR_UNSUPPORTED;
  if (page_size != 8 && page_size != 16 && page_size != 32 && page_size != 64) return FI_ERR_UNSUPPORTED;
  if (batch > cfg->max_batch) return FI_ERR_CAPACITY;
  if (kv_indptr[0] != 0) return FI_ERR_INVALID_ARG;
  std::vector<int32_t> kv_len(batch);
  for (int32_t b = 0; b < batch; ++b) {
    const int64_t n = int64_t(kv_indptr[b + 1]) - kv_indptr[b];
    if (n < 0) return FI_ERR_INVALID_ARG;
    if (n == 0) {
      kv_len[b] = 0;
      continue;
    }
    const int32_t lp = last_page_len[b];
    if (lp < 1 || lp > page_size) return FI_ERR_INVALID_ARG;
    const int64_t len = (n - 1) * page_size + lp;
    if (len > (int64_t(1) << 30)) return FI_ERR_INVALID_ARG;
    kv_len[b] = int32_t(len);
  }
  if (num_pages > 0) {
    if (!kv_indices && kv_indptr[batch] > 0) return FI_ERR_INVALID_ARG;
    for (int32_t i = 0; i < kv_indptr[batch]; ++i)
      if (kv_indices[i] < 0 || kv_indices[i] >= num_pages) return FI_ERR_INVALID_ARG;
  }

  const int64_t P = cfg->num_pairs, CU = FI_MLA_UNIT_COST_TOKENS, MC = cfg->min_chunk;
  int64_t tokens_left = 0, reqs_left = 0;
  for (int32_t b = 0; b < batch; ++b) {
    tokens_left += kv_len[b];
    reqs_left += kv_len[b] > 0;
  }

  // the walk: pieces in stream order, each tagged with its pair
  std::vector<Unit> units;
  std::vector<std::vector<int32_t>> per_pair(P);
  int64_t first_budget = 0;
  int32_t b = 0;
  int64_t k = 0;  // tokens of request b already placed
  while (b < batch && kv_len[b] == 0) ++b;
  for (int64_t c = 0; c < P && b < batch; ++c) {
    const int64_t pairs_left = P - c;
    const int64_t want = tokens_left + CU * (reqs_left + pairs_left - 1);
    const int64_t budget = std::max((want + pairs_left - 1) / pairs_left, CU + MC);
    if (c == 0) first_budget = budget;
    int64_t r = budget;
    while (b < batch) {
      const int64_t left = kv_len[b] - k;
      int64_t take = left;
      if (c < P - 1) {
        take = std::min(left, std::max<int64_t>(0, (r - CU) / FI_MLA_BLOCK * FI_MLA_BLOCK));
        if (take < left && take < MC) break;
      }
      per_pair[c].push_back(int32_t(units.size()));
      units.push_back(Unit{b, int32_t(k), int32_t(k + take), -1});
      r -= take + CU;
      tokens_left -= take;
      k += take;
      if (k == kv_len[b]) {
        --reqs_left;
        k = 0;
        ++b;
        while (b < batch && kv_len[b] == 0) ++b;
      }
      if (c < P - 1 && r - CU < FI_MLA_BLOCK) break;
    }
  }

  // partial slots (consecutive per request, in stream order) and merge entries
  std::vector<int32_t> merge;
  int32_t parts = 0;
  std::vector<int32_t> first_unit(batch, -1), n_units_of(batch, 0);
  for (size_t u = 0; u < units.size(); ++u) {
    if (first_unit[units[u].b] < 0) first_unit[units[u].b] = int32_t(u);
    ++n_units_of[units[u].b];
  }
  for (int32_t q = 0; q < batch; ++q) {
    if (kv_len[q] == 0) {
      merge.insert(merge.end(), {q, 0, 0, 0});
    } else if (n_units_of[q] > 1) {
      for (int32_t i = 0; i < n_units_of[q]; ++i) units[first_unit[q] + i].part = parts + i;
      merge.insert(merge.end(), {q, parts, n_units_of[q], 0});
      parts += n_units_of[q];
    }
  }
  const int64_t n_units = int64_t(units.size()), n_merge = int64_t(merge.size() / FI_MLA_MERGE_INTS);
  if (n_units > cfg->max_units || parts > cfg->max_parts) return FI_ERR_CAPACITY;
  const int64_t chunk = first_budget;

  const int64_t off_pair = FI_MLA_HEADER_INTS;
  const int64_t off_units = off_pair + fi_mla_round4(P + 1);
  const int64_t off_req = off_units + FI_MLA_UNIT_INTS * n_units;
  const int64_t off_merge = off_req + fi_mla_round4(int64_t(FI_MLA_REQ_INTS) * batch);
  const int64_t total_ints = off_merge + FI_MLA_MERGE_INTS * n_merge;
  if (total_ints > capacity_ints(cfg) || size_t(total_ints) * 4 > workspace_bytes) return FI_ERR_CAPACITY;

  int32_t* ws = static_cast<int32_t*>(workspace_host);
  std::memset(ws, 0, size_t(total_ints) * 4);
  int32_t at = 0;
  for (int32_t p = 0; p < P; ++p) {
    ws[off_pair + p] = at;
    for (int32_t u : per_pair[p]) {
      int32_t* f = ws + off_units + int64_t(FI_MLA_UNIT_INTS) * at++;
      f[0] = units[u].b;
      f[1] = units[u].kv0;
      f[2] = units[u].kv1;
      f[3] = units[u].part;
    }
  }
  ws[off_pair + P] = at;
  for (int32_t b = 0; b < batch; ++b) {
    ws[off_req + 2 * b] = kv_indptr[b];
    ws[off_req + 2 * b + 1] = kv_len[b];
  }
  if (n_merge) std::memcpy(ws + off_merge, merge.data(), merge.size() * 4);
  const int32_t header[FI_MLA_HEADER_INTS] = {FI_MLA_MAGIC,       int32_t(n_units),   int32_t(P),
                                              batch,              num_heads,          page_size,
                                              int32_t(off_pair),  int32_t(off_units), int32_t(off_req),
                                              int32_t(off_merge), int32_t(n_merge),   0,
                                              int32_t(chunk),     int32_t(total_ints), parts,
                                              0};
  std::memcpy(ws, header, sizeof header);

  fi_mla_plan_info info;
  std::memset(&info, 0, sizeof info);
  info.num_pairs = int32_t(P);
  info.num_units = int32_t(n_units);
  info.num_parts = parts;
  info.num_merge = int32_t(n_merge);
  info.batch = batch;
  info.num_heads = num_heads;
  info.page_size = page_size;
  info.chunk = int32_t(chunk);
  info.int_ws_bytes_used = total_ints * 4;
  info.max_parts = cfg->max_parts;
  *info_out = info;
  return FI_OK;
}

extern "C" fi_status fi_mla_plan(const fi_mla_config* cfg, const int32_t* kv_indptr, const int32_t* kv_indices,
                                 const int32_t* last_page_len, int32_t batch, int32_t num_heads, int32_t page_size,
                                 int32_t num_pages, void* int_workspace_dev, void* pinned_staging_host,
                                 size_t staging_bytes, void* stream, fi_mla_plan_info* info_out) {
  if (!int_workspace_dev || !pinned_staging_host) return FI_ERR_INVALID_ARG;
  fi_status st = fi_mla_plan_host(cfg, kv_indptr, kv_indices, last_page_len, batch, num_heads, page_size,
                                  num_pages, pinned_staging_host, staging_bytes, info_out);
  if (st != FI_OK) return st;
  cudaError_t e = cudaMemcpyAsync(int_workspace_dev, pinned_staging_host, size_t(info_out->int_ws_bytes_used),
                                  cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FI_OK : FI_ERR_CUDA;
}

// plan.cpp -- host planner of the persistent paged-attention kernel.
//
// FlashInfer paper summary, section "연구 방법론 / 3. 동적 부하 분산
// 스케줄링": tile sizes are fixed when the kernel is compiled; at run time the
// scheduler takes every request's sequence length and builds, on the CPU, a
// plan that gives all SMs an even share of the work.  The plan is copied to
// the GPU once per step and the kernel launch never changes, so one CUDA graph
// replays any plan.  The two tile classes follow the CTA_TILE_Q_1 = 128 /
// CTA_TILE_Q_2 = 16 pair of the BatchAttention PR page, section "코드 분석 §1":
// 16 rows for decode work, and for prefill work two 128-row halves that share
// every K/V tile (256 rows).
//
// Rule (this library's reading of that goal; the pages give no cost model):
//  * request b -> R = qo_len * G packed rows (row t*G+g = token t, head hk*G+g);
//    tile T = 16 when R <= 16, else 256;
//  * unit (b, hk, q-tile) with its visible KV ranges: [0, hi) with hi the
//    bottom-right causal end; with a sliding window W and S sink tokens, the
//    window range starts at the first token's q_pos - W rounded down to the
//    class granule, and the sink range [0, min(S, hi)) comes first unless
//    the two touch (then one range [0, hi));
//  * per tile class, a KV chunk length = max(min_chunk, total / (CTAs * split))
//    rounded up to the class granule, where the decode class counts only the
//    CTAs left free by the prefill-class items when those take at most half
//    of them; units longer than a chunk are split into chunks whose fp32
//    partial states are merged by the kernel;
//  * chunks are dealt out longest-first to the least-loaded CTA (LPT); an
//    item's cost is its KV length plus a fixed FI_ITEM_COST_TOKENS (the
//    per-item latency of the kernel), times the class weight, so that many
//    short items do not pile up on one CTA.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <utility>
#include <vector>

#include "../../include/fi.h"
#include "plan_layout.h"
#include "workspace.h"

namespace {

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round4(int64_t n) { return (n + 3) & ~int64_t(3); }

struct Unit {
  int32_t b, hk, qt, tile, row0, row1;
  int32_t heads;                 // KV heads hk .. hk + heads - 1 (more than one: a multi-head decode unit)
  int64_t r_begin[2], r_end[2];  // visible KV ranges, in KV order
  int32_t n_ranges;
  int64_t kv_eff;                // summed length of the ranges
};

struct Chunk {
  int64_t cost;
  int32_t tile, b, hk, qt, idx;
  int32_t fields[FI_ITEM_INTS];
};

// The deal's sort key of a chunk (the chunk itself stays where it is).
struct DealKey {
  int64_t cost;
  int32_t tile, b, hk, qt, idx, pos;
};

// Order of the longest-processing-time deal: cost descending, then the
// prefill class first, then (b, hk, q-tile, chunk) ascending.  Keys are unique.
bool deal_before(const DealKey& x, const DealKey& y) {
  if (x.cost != y.cost) return x.cost > y.cost;
  if (x.tile != y.tile) return x.tile > y.tile;
  if (x.b != y.b) return x.b < y.b;
  if (x.hk != y.hk) return x.hk < y.hk;
  if (x.qt != y.qt) return x.qt < y.qt;
  return x.idx < y.idx;
}

// Min-heap of (load, CTA), ties to the lower CTA: the least-loaded CTA is at
// the top, and giving it an item is one sift-down from the top.
struct CtaHeap {
  std::vector<std::pair<int64_t, int32_t>> h;
  explicit CtaHeap(int32_t n) : h(size_t(n)) {
    for (int32_t c = 0; c < n; ++c) h[size_t(c)] = {0, c};  // already a heap: equal loads, rising CTAs
  }
  int32_t top() const { return h[0].second; }
  void add_to_top(int64_t cost) {
    auto x = h[0];
    x.first += cost;
    const size_t n = h.size();
    size_t i = 0;
    while (true) {
      size_t c = 2 * i + 1;
      if (c >= n) break;
      if (c + 1 < n && h[c + 1] < h[c]) ++c;
      if (!(h[c] < x)) break;
      h[i] = h[c];
      i = c;
    }
    h[i] = x;
  }
};

}  // namespace

int64_t fi::plan_capacity_ints(const fi_plan_config* cfg) {
  return FI_HEADER_INTS + round4(int64_t(cfg->num_ctas) + 1) + int64_t(FI_ITEM_INTS) * cfg->max_items +
         int64_t(FI_MERGE_INTS) * cfg->max_merge_units + round4(cfg->max_merge_units) +
         int64_t(FI_REQ_INTS) * cfg->max_batch + int64_t(FI_CASCADE_INTS) * cfg->max_merge_units;
}

extern "C" size_t fi_int_workspace_bytes(const fi_plan_config* cfg) {
  if (!cfg) return 0;
  const int64_t plan_ints = fi::plan_capacity_ints(cfg);
  if (cfg->rope_max_positions <= 0) return size_t(plan_ints) * 4;
  return size_t(fi_rope_table_offset(plan_ints) + fi_rope_table_rows(cfg->rope_max_positions) * FI_ROPE_PAIRS * 8);
}

extern "C" size_t fi_float_workspace_bytes(const fi_plan_config* cfg, int32_t head_dim) {
  if (!cfg || head_dim <= 0) return 0;
  return size_t(fi_partial_o_offset(cfg->max_partial_rows) + cfg->max_partial_rows * int64_t(head_dim)) * 4;
}

namespace {

// One request of the plan's request table: its query tokens, its pages and
// its KV length.  A cascade plan lists its shared blocks first.
struct Req {
  int32_t qo_start, qo_len, page_start, kv_len;
};

// Checks one level's host arrays and appends its requests.
fi_status read_level(const int32_t* qo_indptr, const int32_t* kv_indptr, const int32_t* kv_indices,
                     const int32_t* last_page_len, int32_t batch, int32_t page_size, int32_t num_pages,
                     int32_t rope_max, std::vector<Req>* out) {
  if (batch > 0 && (!qo_indptr || !kv_indptr || !last_page_len)) return FI_ERR_INVALID_ARG;
  const int32_t* qo = qo_indptr;
  const int32_t* kvp = kv_indptr;
  if (batch > 0 && (qo[0] != 0 || kvp[0] != 0)) return FI_ERR_INVALID_ARG;
  for (int32_t b = 0; b < batch; ++b) {
    if (qo[b + 1] < qo[b] || kvp[b + 1] < kvp[b]) return FI_ERR_INVALID_ARG;
    const int32_t pages = kvp[b + 1] - kvp[b];
    if (pages > 0 && (last_page_len[b] < 1 || last_page_len[b] > page_size)) return FI_ERR_INVALID_ARG;
    const int64_t len = pages == 0 ? 0 : int64_t(pages - 1) * page_size + last_page_len[b];
    if (len > INT32_MAX) return FI_ERR_UNSUPPORTED;
    const int32_t lq = qo[b + 1] - qo[b];
    // RoPE positions: keys 0 .. Lkv-1 and queries Lkv-Lq .. Lkv-1 inside the table
    if (rope_max > 0 && (len > rope_max || lq > len)) return FI_ERR_INVALID_ARG;
    out->push_back(Req{qo[b], lq, kvp[b], int32_t(len)});
  }
  if (num_pages > 0 && batch > 0) {
    if (!kv_indices && kvp[batch] > 0) return FI_ERR_INVALID_ARG;
    // one pass without early exit (it vectorises): every id in [0, num_pages),
    // negative ids read as unsigned values past num_pages
    uint32_t bad = 0;
    const uint32_t* ids = reinterpret_cast<const uint32_t*>(kv_indices);
    const uint32_t np = uint32_t(num_pages);
    for (int32_t i = 0; i < kvp[batch]; ++i) bad |= uint32_t(ids[i] >= np);
    if (bad) return FI_ERR_INVALID_ARG;
  }
  return FI_OK;
}

fi_status check_config(const fi_plan_config* cfg, int32_t head_dim, int32_t num_qo_heads, int32_t num_kv_heads,
                       int32_t page_size, int32_t causal) {
  if (head_dim != 128) return FI_ERR_UNSUPPORTED;
  if (page_size < 1 || page_size > 128 || (page_size & (page_size - 1))) return FI_ERR_UNSUPPORTED;
  if (num_qo_heads < 1 || num_kv_heads < 1 || num_qo_heads % num_kv_heads) return FI_ERR_UNSUPPORTED;
  if (num_qo_heads / num_kv_heads > 16) return FI_ERR_UNSUPPORTED;
  if ((causal != 0 && causal != 1) || cfg->num_ctas < 1 || cfg->split_factor < 1) return FI_ERR_INVALID_ARG;
  if (cfg->decode_min_chunk < 1 || cfg->prefill_min_chunk < 1) return FI_ERR_INVALID_ARG;
  const float cap = cfg->logits_soft_cap;
  if (cfg->window_left < -1 || cfg->sink_tokens < 0 || !(cap >= 0.f) || cap == HUGE_VALF) return FI_ERR_INVALID_ARG;
  const int32_t rope_max = cfg->rope_max_positions;
  if (rope_max < 0 || (rope_max > 0 && !(cfg->rope_theta > 0.f && cfg->rope_theta < HUGE_VALF &&
                                         cfg->rope_scale > 0.f && cfg->rope_scale < HUGE_VALF)))
    return FI_ERR_INVALID_ARG;
  return FI_OK;
}

// The plan rule over a request table.  Requests b < num_shared are the
// shared blocks of a cascade plan: all their keys are visible, every unit of
// the plan writes fp32 partial states, and the cascade merge entries say
// which partial rows make up each output row.
fi_status plan_requests(const fi_plan_config* cfg, const std::vector<Req>& reqs, int32_t num_shared,
                        int32_t shared_page_size, const std::vector<int32_t>& block_of, int32_t total_qo,
                        int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                        int32_t causal, void* workspace_host, fi_plan_info* info_out) {
  const int32_t batch = int32_t(reqs.size());
  const int32_t group = num_qo_heads / num_kv_heads;
  const bool cascade = num_shared > 0;
  const int32_t window = cfg->window_left, sink = cfg->sink_tokens;
  const float cap = cfg->logits_soft_cap;
  const int32_t rope_max = cfg->rope_max_positions;
  // Chunk boundaries fall on pages of every cache the plan reads.
  const int32_t max_page = std::max(page_size, cascade ? shared_page_size : page_size);

  // Units, in (b, hk, q-tile) order, and per-class visible-KV totals.
  std::vector<Unit> units;
  units.reserve(size_t(batch) * num_kv_heads);
  std::vector<int32_t> first_unit(batch, -1);  // index of unit (b, 0, 0)
  int64_t total_dec = 0, total_pre = 0;
  for (int32_t b = 0; b < batch; ++b) {
    const Req& rq = reqs[b];
    const int64_t rows = int64_t(rq.qo_len) * group;
    if (rows == 0) continue;
    first_unit[b] = int32_t(units.size());
    const bool causal_b = causal && b >= num_shared;  // a shared block's keys precede all its queries
    const int32_t tile = rows <= FI_TILE_DECODE ? FI_TILE_DECODE : FI_TILE_PREFILL;
    const int32_t tiles = int32_t(ceil_div(rows, tile));
    // One query token of the plan's own page-1 cache: fi_mh_heads() KV heads
    // per unit (FI_MH_ROWS packed rows), so that short requests pay the
    // per-item cost once per unit, not once per head, and every TMA box brings
    // one token of all the unit's heads.
    const int32_t cache_page = b < num_shared ? shared_page_size : page_size;
    const int32_t heads = (tile == FI_TILE_DECODE && rq.qo_len == 1 && cache_page == 1 && rope_max == 0 &&
                           b >= num_shared)
                              ? fi_mh_heads(group, num_kv_heads)
                              : 1;
    for (int32_t hk = 0; hk < num_kv_heads; hk += heads) {
      for (int32_t qt = 0; qt < tiles; ++qt) {
        Unit u;
        u.b = b;
        u.hk = hk;
        u.qt = qt;
        u.tile = tile;
        u.heads = heads;
        u.row0 = qt * tile;
        u.row1 = heads > 1 ? int32_t(rows * heads) : int32_t(std::min<int64_t>(rows, int64_t(qt + 1) * tile));
        // query tokens of the unit's first and last rows (a multi-head unit: token 0)
        const int64_t t_first = heads > 1 ? 0 : u.row0 / group, t_last = heads > 1 ? 0 : (u.row1 - 1) / group;
        const int64_t q_first = int64_t(rq.kv_len) - rq.qo_len + t_first;
        const int64_t q_last = int64_t(rq.kv_len) - rq.qo_len + t_last;
        int64_t hi = causal_b ? std::min<int64_t>(rq.kv_len, q_last + 1) : int64_t(rq.kv_len);
        if (hi < 0) hi = 0;
        u.n_ranges = 1;
        u.r_begin[0] = 0;
        u.r_end[0] = hi;
        if (window >= 0) {
          const int64_t gran = tile == FI_TILE_DECODE ? std::max(max_page, FI_GRANULE_DECODE)
                                                      : std::max(max_page, FI_GRANULE_PREFILL);
          const int64_t lo = std::max<int64_t>(0, q_first - window) / gran * gran;
          const int64_t sink_end = std::min<int64_t>(sink, hi);
          if (lo > sink_end) {
            u.n_ranges = 0;
            if (sink_end > 0) {
              u.r_begin[0] = 0;
              u.r_end[0] = sink_end;
              u.n_ranges = 1;
            }
            u.r_begin[u.n_ranges] = lo;
            u.r_end[u.n_ranges] = hi;
            ++u.n_ranges;
          }
        }
        u.kv_eff = 0;
        for (int r = 0; r < u.n_ranges; ++r) u.kv_eff += u.r_end[r] - u.r_begin[r];
        (tile == FI_TILE_DECODE ? total_dec : total_pre) += u.kv_eff * heads;
        units.push_back(u);
      }
    }
  }

  auto pick_chunk = [&](int64_t total, int64_t min_chunk, int64_t granule, int64_t slots) {
    int64_t c = std::max<int64_t>(min_chunk, ceil_div(total, slots));
    return ceil_div(c, granule) * granule;
  };
  const int64_t gran_dec = std::max(max_page, FI_GRANULE_DECODE);
  const int64_t chunk_pre = pick_chunk(total_pre, cfg->prefill_min_chunk, std::max(max_page, FI_GRANULE_PREFILL),
                                       int64_t(cfg->num_ctas) * cfg->split_factor);
  // Prefill-class items are long; when they take at most half the CTAs, the
  // decode work is spread over the CTAs they leave free (finer decode chunks
  // would only add per-item costs beside them).
  int64_t n_pre = 0;
  for (const Unit& u : units) {
    if (u.tile != FI_TILE_PREFILL) continue;
    int64_t n = 0;
    for (int r = 0; r < u.n_ranges; ++r) n += ceil_div(u.r_end[r] - u.r_begin[r], chunk_pre);
    n_pre += std::max<int64_t>(n, 1);
  }
  const int64_t dec_ctas = (n_pre > 0 && 2 * n_pre <= cfg->num_ctas) ? cfg->num_ctas - n_pre : cfg->num_ctas;
  const int64_t chunk_dec = pick_chunk(total_dec, cfg->decode_min_chunk, gran_dec, dec_ctas * cfg->split_factor);
  // a multi-head unit's chunk: the K/V bytes of a one-head chunk, rounded up
  const int32_t mh = fi_mh_heads(group, num_kv_heads);
  const int64_t chunk_mh = std::max(gran_dec, ceil_div(ceil_div(chunk_dec, mh), gran_dec) * gran_dec);

  // Chunks of every unit; split units become merge units in unit order.  In
  // a cascade plan every unit writes partial states and none is merged in
  // the run: the cascade merge combines them across the two levels.
  std::vector<Chunk> chunks;
  chunks.reserve(units.size() * 2);
  std::vector<int32_t> merge_rows;  // FI_MERGE_INTS per merge unit
  std::vector<int64_t> unit_base(units.size(), -1), unit_n(units.size(), 0);
  int64_t partial_rows = 0;
  int32_t n_late = 0;  // merge units of prefill-class tiles, merged after the run
  int32_t prefill_caches = 0;
  for (size_t ui = 0; ui < units.size(); ++ui) {
    const Unit& u = units[ui];
    const int64_t chunk = u.tile == FI_TILE_DECODE ? (u.heads > 1 ? chunk_mh : chunk_dec) : chunk_pre;
    const int64_t weight = u.tile == FI_TILE_DECODE ? cfg->decode_cost_weight : cfg->prefill_cost_weight;
    if (u.tile == FI_TILE_PREFILL) prefill_caches |= u.b < num_shared ? 2 : 1;
    int64_t n = 0;
    for (int r = 0; r < u.n_ranges; ++r) n += ceil_div(u.r_end[r] - u.r_begin[r], chunk);
    const bool empty = n == 0;
    if (empty) n = 1;
    int32_t merge_id = -1;
    int64_t base = -1;
    const int32_t nrows = u.row1 - u.row0;
    if (n > 1 || cascade) {
      base = partial_rows;
      partial_rows += n * nrows;
    }
    if (n > 1 && !cascade) {
      merge_id = int32_t(merge_rows.size() / FI_MERGE_INTS);
      const int32_t late = u.tile == FI_TILE_DECODE ? 0 : 1;
      const int32_t m[FI_MERGE_INTS] = {u.b, u.hk, u.row0, u.row1, int32_t(n), int32_t(base), late, 0};
      merge_rows.insert(merge_rows.end(), m, m + FI_MERGE_INTS);
      n_late += late;
    }
    unit_base[ui] = base;
    unit_n[ui] = n;
    // chunk i of the unit: ranges in KV order, chunk numbers running across them
    int64_t i = 0;
    auto emit = [&](int64_t k0, int64_t k1) {
      Chunk c;
      c.cost = ((k1 - k0) * u.heads + FI_ITEM_COST_TOKENS) * weight;
      c.tile = u.tile;
      c.b = u.b;
      c.hk = u.hk;
      c.qt = u.qt;
      c.idx = int32_t(i);
      const Req& rq = reqs[u.b];
      const int32_t f[FI_ITEM_INTS] = {u.b,         u.hk,        u.row0,
                                       u.row1,      int32_t(k0), int32_t(k1),
                                       base >= 0 ? int32_t(base + i * nrows) : -1, merge_id,
                                       rq.qo_start, rq.qo_len,   rq.page_start,
                                       rq.kv_len,   u.heads > 1 ? u.heads : 0, 0,
                                       0,           0};
      std::memcpy(c.fields, f, sizeof f);
      chunks.push_back(c);
      ++i;
    };
    if (empty) {
      emit(0, 0);
    } else {
      for (int r = 0; r < u.n_ranges; ++r)
        for (int64_t k0 = u.r_begin[r]; k0 < u.r_end[r]; k0 += chunk) emit(k0, std::min(u.r_end[r], k0 + chunk));
    }
  }
  // Cascade merge entries, in ordinary-unit order: the rows of each unit in
  // runs of at most FI_CASCADE_ROWS from the unit's first row, also cut
  // where they cross from one shared unit (q-tile of their block) into the
  // next.
  std::vector<int32_t> cascade_rows;  // FI_CASCADE_INTS per entry
  if (cascade) {
    for (size_t ui = 0; ui < units.size(); ++ui) {
      const Unit& u = units[ui];
      if (u.b < num_shared) continue;
      const int32_t s = block_of[u.b];
      const Req& blk = reqs[s];
      const int64_t srows = int64_t(blk.qo_len) * group;
      const int32_t stile = srows <= FI_TILE_DECODE ? FI_TILE_DECODE : FI_TILE_PREFILL;
      const int32_t stiles = int32_t(ceil_div(srows, stile));
      const int64_t shift = int64_t(reqs[u.b].qo_start - blk.qo_start) * group;  // row r -> block row r + shift
      // A multi-head unit's entries are per KV head, in one-head row numbering;
      // head h's rows sit at offset h * G of the unit's partial rows.
      for (int32_t h = 0; h < u.heads; ++h) {
        const int32_t hk = u.hk + h;
        const int32_t row0 = u.heads > 1 ? 0 : u.row0, row1 = u.heads > 1 ? group : u.row1;
        const int64_t own0 = unit_base[ui] + (u.heads > 1 ? int64_t(h) * group : 0);  // partial row of row0
        for (int32_t ra = row0; ra < row1;) {
          const int64_t rs = ra + shift;
          const int32_t qt0 = int32_t(rs / stile);
          const size_t si = size_t(first_unit[s]) + size_t(hk) * stiles + qt0;
          const Unit& su = units[si];
          const int32_t run_end = row0 + ((ra - row0) / FI_CASCADE_ROWS + 1) * FI_CASCADE_ROWS;
          const int32_t rb = int32_t(std::min<int64_t>(std::min(row1, run_end), ra + (su.row1 - rs)));
          const int32_t e[FI_CASCADE_INTS] = {u.b, hk, ra, rb,
                                              int32_t(unit_n[si]), int32_t(unit_base[si] + (rs - su.row0)),
                                              su.row1 - su.row0, int32_t(unit_n[ui]),
                                              int32_t(own0 + (ra - row0)), u.row1 - u.row0, 0, 0};
          cascade_rows.insert(cascade_rows.end(), e, e + FI_CASCADE_INTS);
          ra = rb;
        }
      }
    }
  }
  const int64_t n_items = int64_t(chunks.size());
  const int64_t n_merge = int64_t(merge_rows.size() / FI_MERGE_INTS);
  const int64_t n_cascade = int64_t(cascade_rows.size() / FI_CASCADE_INTS);
  int32_t cascade_rows_max = 0;  // the merge launch gives each entry this many row tasks
  for (int64_t e = 0; e < n_cascade; ++e)
    cascade_rows_max = std::max(cascade_rows_max, cascade_rows[size_t(e) * FI_CASCADE_INTS + 3] -
                                                      cascade_rows[size_t(e) * FI_CASCADE_INTS + 2]);
  if (n_items > cfg->max_items || n_merge > cfg->max_merge_units || n_cascade > cfg->max_merge_units ||
      partial_rows > cfg->max_partial_rows || partial_rows > INT32_MAX)
    return FI_ERR_CAPACITY;

  // Longest processing time first onto the least-loaded CTA (ties: lower CTA).
  std::vector<DealKey> order(chunks.size());
  for (size_t i = 0; i < chunks.size(); ++i) {
    const Chunk& c = chunks[i];
    order[i] = DealKey{c.cost, c.tile, c.b, c.hk, c.qt, c.idx, int32_t(i)};
  }
  std::sort(order.begin(), order.end(), deal_before);
  const int32_t C = cfg->num_ctas;
  CtaHeap least(C);
  std::vector<int32_t> owner(chunks.size());  // by position in `order`
  std::vector<int32_t> per_cta(C, 0);
  for (size_t i = 0; i < order.size(); ++i) {
    const int32_t c = least.top();
    owner[i] = c;
    per_cta[c] += 1;
    least.add_to_top(order[i].cost);
  }

  const int64_t off_cta = FI_HEADER_INTS;
  const int64_t off_items = off_cta + round4(C + 1);
  const int64_t off_merge = off_items + FI_ITEM_INTS * n_items;
  const int64_t off_cnt = off_merge + FI_MERGE_INTS * n_merge;
  const int64_t off_req = off_cnt + round4(n_merge);
  const int64_t off_cascade = off_req + int64_t(FI_REQ_INTS) * batch;
  const int64_t total_ints = off_cascade + int64_t(FI_CASCADE_INTS) * n_cascade;
  if (total_ints > fi::plan_capacity_ints(cfg)) return FI_ERR_CAPACITY;

  int32_t* ws = static_cast<int32_t*>(workspace_host);
  std::memset(ws, 0, size_t(total_ints) * 4);
  // CTA c's items occupy [start[c], start[c+1]): its prefill-class items first,
  // then its 16-row items, each kept in the order the deal handed them out
  // (one switch between the kernel's two tile paths per CTA at most).
  std::vector<int32_t> start(C + 1, 0);
  for (int32_t c = 0; c < C; ++c) start[c + 1] = start[c] + per_cta[c];
  for (int32_t c = 0; c <= C; ++c) ws[off_cta + c] = start[c];
  std::vector<int32_t> fill(start.begin(), start.end() - 1);
  int64_t n_decode = 0;
  for (int pass = 0; pass < 2; ++pass) {
    const int32_t tile = pass == 0 ? FI_TILE_PREFILL : FI_TILE_DECODE;
    for (size_t i = 0; i < order.size(); ++i) {
      if (order[i].tile != tile) continue;
      const int32_t slot = fill[owner[i]]++;
      const Chunk& c = chunks[size_t(order[i].pos)];
      std::memcpy(ws + off_items + int64_t(FI_ITEM_INTS) * slot, c.fields, sizeof c.fields);
      if (tile == FI_TILE_DECODE) ++n_decode;
    }
  }
  if (n_merge) std::memcpy(ws + off_merge, merge_rows.data(), merge_rows.size() * 4);
  for (int32_t b = 0; b < batch; ++b) {
    int32_t* r = ws + off_req + int64_t(FI_REQ_INTS) * b;
    r[0] = reqs[b].qo_start;
    r[1] = reqs[b].qo_len;
    r[2] = reqs[b].page_start;
    r[3] = reqs[b].kv_len;
  }
  if (n_cascade) std::memcpy(ws + off_cascade, cascade_rows.data(), cascade_rows.size() * 4);
  int32_t cap_bits, theta_bits = 0, scale_bits = 0;
  std::memcpy(&cap_bits, &cap, 4);
  if (rope_max > 0) {
    std::memcpy(&theta_bits, &cfg->rope_theta, 4);
    std::memcpy(&scale_bits, &cfg->rope_scale, 4);
  }
  const int32_t rope_off = rope_max > 0 ? int32_t(fi_rope_table_offset(fi::plan_capacity_ints(cfg)) / 4) : 0;
  const int32_t header[FI_HEADER_INTS] = {
      FI_PLAN_MAGIC,        int32_t(n_items),   int32_t(n_merge),   C,
      batch,                causal,             int32_t(off_cta),   int32_t(off_items),
      int32_t(off_merge),   int32_t(off_cnt),   int32_t(off_req),   0,
      num_qo_heads,         num_kv_heads,       page_size,          int32_t(total_ints),
      window,               sink,               cap_bits,           rope_max,
      theta_bits,           scale_bits,         rope_off,           n_late,
      int32_t(partial_rows), total_qo,          num_shared,         cascade ? int32_t(off_cascade) : 0,
      int32_t(n_cascade),   cascade ? shared_page_size : 0, int32_t(n_decode), cascade_rows_max};
  std::memcpy(ws, header, sizeof header);

  fi_plan_info info;
  std::memset(&info, 0, sizeof info);
  info.num_ctas = C;
  info.num_items = int32_t(n_items);
  info.num_merge_units = int32_t(n_merge);
  info.num_late_merge_units = n_late;
  info.batch = batch;
  info.num_partial_rows = partial_rows;
  info.num_qo_heads = num_qo_heads;
  info.num_kv_heads = num_kv_heads;
  info.head_dim = head_dim;
  info.page_size = page_size;
  info.causal = causal;
  info.chunk_decode = int32_t(chunk_dec);
  info.chunk_prefill = int32_t(chunk_pre);
  info.num_decode_items = int32_t(n_decode);
  info.num_prefill_items = int32_t(n_items - n_decode);
  info.int_ws_bytes_used = total_ints * 4;
  info.max_partial_rows = cfg->max_partial_rows;
  info.variant = (cap > 0.f ? 1 : 0) | (window >= 0 ? 2 : 0) | (rope_max > 0 ? 4 : 0);
  info.num_shared = num_shared;
  info.num_cascade_merges = int32_t(n_cascade);
  info.prefill_caches = prefill_caches;
  *info_out = info;
  return FI_OK;
}

}  // namespace

extern "C" fi_status fi_plan_host(const fi_plan_config* cfg, const int32_t* qo_indptr, const int32_t* kv_indptr,
                                  const int32_t* kv_indices, const int32_t* last_page_len, int32_t batch,
                                  int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t page_size, int32_t causal, int32_t num_pages, void* workspace_host,
                                  size_t workspace_bytes, fi_plan_info* info_out) {
  if (!cfg || !info_out || !workspace_host || batch < 0) return FI_ERR_INVALID_ARG;
  fi_status st = check_config(cfg, head_dim, num_qo_heads, num_kv_heads, page_size, causal);
  if (st != FI_OK) return st;
  if (batch > cfg->max_batch) return FI_ERR_CAPACITY;
  if (workspace_bytes < size_t(fi::plan_capacity_ints(cfg)) * 4) return FI_ERR_CAPACITY;
  std::vector<Req> reqs;
  reqs.reserve(batch);
  st = read_level(qo_indptr, kv_indptr, kv_indices, last_page_len, batch, page_size, num_pages,
                  cfg->rope_max_positions, &reqs);
  if (st != FI_OK) return st;
  return plan_requests(cfg, reqs, 0, page_size, {}, batch > 0 ? qo_indptr[batch] : 0, num_qo_heads, num_kv_heads,
                       head_dim, page_size, causal, workspace_host, info_out);
}

extern "C" fi_status fi_plan_cascade_host(
    const fi_plan_config* cfg, const int32_t* shared_qo_indptr, const int32_t* shared_kv_indptr,
    const int32_t* shared_kv_indices, const int32_t* shared_last_page_len, int32_t num_shared,
    int32_t shared_page_size, int32_t shared_num_pages, const int32_t* qo_indptr, const int32_t* kv_indptr,
    const int32_t* kv_indices, const int32_t* last_page_len, int32_t batch, int32_t num_qo_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t page_size, int32_t causal, int32_t num_pages,
    void* workspace_host, size_t workspace_bytes, fi_plan_info* info_out) {
  if (!cfg || !info_out || !workspace_host || batch < 0 || num_shared < 1) return FI_ERR_INVALID_ARG;
  fi_status st = check_config(cfg, head_dim, num_qo_heads, num_kv_heads, page_size, causal);
  if (st != FI_OK) return st;
  if (shared_page_size < 1 || shared_page_size > 128 || (shared_page_size & (shared_page_size - 1)))
    return FI_ERR_UNSUPPORTED;
  // Positions of the two levels are not tied to one sequence here: the
  // position-dependent variants (sliding window, sink, RoPE) are not offered.
  if (cfg->window_left >= 0 || cfg->rope_max_positions > 0) return FI_ERR_UNSUPPORTED;
  if (int64_t(batch) + num_shared > cfg->max_batch) return FI_ERR_CAPACITY;
  if (workspace_bytes < size_t(fi::plan_capacity_ints(cfg)) * 4) return FI_ERR_CAPACITY;
  std::vector<Req> reqs;
  reqs.reserve(size_t(num_shared) + batch);
  st = read_level(shared_qo_indptr, shared_kv_indptr, shared_kv_indices, shared_last_page_len, num_shared,
                  shared_page_size, shared_num_pages, 0, &reqs);
  if (st != FI_OK) return st;
  st = read_level(qo_indptr, kv_indptr, kv_indices, last_page_len, batch, page_size, num_pages, 0, &reqs);
  if (st != FI_OK) return st;
  // The blocks cover the query rows exactly and no request straddles two of
  // them; a causal request's queries are among its own keys.
  const int32_t total_qo = batch > 0 ? qo_indptr[batch] : 0;
  if (shared_qo_indptr[num_shared] != total_qo) return FI_ERR_INVALID_ARG;
  std::vector<int32_t> block_of(size_t(num_shared) + batch, -1);
  int32_t s = 0;
  for (int32_t b = 0; b < batch; ++b) {
    const Req& rq = reqs[size_t(num_shared) + b];
    if (causal && rq.kv_len < rq.qo_len) return FI_ERR_INVALID_ARG;
    if (rq.qo_len == 0) continue;  // no rows, no units
    while (s < num_shared && shared_qo_indptr[s + 1] <= rq.qo_start) ++s;
    if (s == num_shared || rq.qo_start + rq.qo_len > shared_qo_indptr[s + 1]) return FI_ERR_INVALID_ARG;
    block_of[size_t(num_shared) + b] = s;
  }
  return plan_requests(cfg, reqs, num_shared, shared_page_size, block_of, total_qo, num_qo_heads, num_kv_heads,
                       head_dim, page_size, causal, workspace_host, info_out);
}

extern "C" fi_status fi_plan(const fi_plan_config* cfg, const int32_t* qo_indptr, const int32_t* kv_indptr,
                             const int32_t* kv_indices, const int32_t* last_page_len, int32_t batch,
                             int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                             int32_t causal, int32_t num_pages, void* int_workspace_dev, void* pinned_staging_host,
                             size_t staging_bytes, void* stream, fi_plan_info* info_out) {
  if (!int_workspace_dev || !pinned_staging_host) return FI_ERR_INVALID_ARG;
  fi_status st = fi_plan_host(cfg, qo_indptr, kv_indptr, kv_indices, last_page_len, batch, num_qo_heads,
                              num_kv_heads, head_dim, page_size, causal, num_pages, pinned_staging_host,
                              staging_bytes, info_out);
  if (st != FI_OK) return st;
  cudaError_t e = cudaMemcpyAsync(int_workspace_dev, pinned_staging_host, size_t(info_out->int_ws_bytes_used),
                                  cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FI_OK : FI_ERR_CUDA;
}

extern "C" fi_status fi_plan_cascade(
    const fi_plan_config* cfg, const int32_t* shared_qo_indptr, const int32_t* shared_kv_indptr,
    const int32_t* shared_kv_indices, const int32_t* shared_last_page_len, int32_t num_shared,
    int32_t shared_page_size, int32_t shared_num_pages, const int32_t* qo_indptr, const int32_t* kv_indptr,
    const int32_t* kv_indices, const int32_t* last_page_len, int32_t batch, int32_t num_qo_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t page_size, int32_t causal, int32_t num_pages,
    void* int_workspace_dev, void* pinned_staging_host, size_t staging_bytes, void* stream,
    fi_plan_info* info_out) {
  if (!int_workspace_dev || !pinned_staging_host) return FI_ERR_INVALID_ARG;
  fi_status st = fi_plan_cascade_host(cfg, shared_qo_indptr, shared_kv_indptr, shared_kv_indices,
                                      shared_last_page_len, num_shared, shared_page_size, shared_num_pages,
                                      qo_indptr, kv_indptr, kv_indices, last_page_len, batch, num_qo_heads,
                                      num_kv_heads, head_dim, page_size, causal, num_pages, pinned_staging_host,
                                      staging_bytes, info_out);
  if (st != FI_OK) return st;
  cudaError_t e = cudaMemcpyAsync(int_workspace_dev, pinned_staging_host, size_t(info_out->int_ws_bytes_used),
                                  cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FI_OK : FI_ERR_CUDA;
}

extern "C" const char* fi_status_string(fi_status s) {
  switch (s) {
    case FI_OK: return "ok";
    case FI_ERR_INVALID_ARG: return "invalid argument";
    case FI_ERR_UNSUPPORTED: return "unsupported shape, page size or dtype";
    case FI_ERR_CAPACITY: return "plan exceeds workspace capacity";
    case FI_ERR_ALIGNMENT: return "pointer or stride not 16-byte aligned";
    case FI_ERR_CUDA: return "CUDA runtime error";
    case FI_ERR_DEVICE_CHECK: return "device-side check failed";
    case FI_ERR_TIMEOUT: return "device-side bounded wait ran out";
  }
  return "unknown status";
}

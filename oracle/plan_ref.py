"""Independent re-derivation of the work plan.  TEST INFRASTRUCTURE ONLY.

The pages fix only the goal of the planner (FlashInfer paper summary, section
"연구 방법론 / 3. 동적 부하 분산 스케줄링"): from each request's runtime
sequence length, build on the CPU a plan that spreads the work evenly over all
cores, with the tile size fixed at compile time; the plan is cached on the GPU
and run by a fixed kernel launch.  The two tile classes follow the pair of
CTA tile heights on the BatchAttention PR page, section "코드 분석 §1"
(CTA_TILE_Q_1 = 128, CTA_TILE_Q_2 = 16): 16-row decode tiles, and prefill
tiles of two 128-row halves that share every K/V tile (256 rows).  The rule
below is this library's own
reading of that goal; this module restates it in plain Python, without sharing
code with the C++ planner, so the two can be compared byte for byte.

Rule:
 1. Request b has Lq query tokens, Lkv keys, R = Lq * G packed rows (packed row
    r = t * G + g is query token t, head hk * G + g).  Tile height T = 16 if
    R <= 16 (decode class) else 256 (prefill class).
 2. Units (b, hk, qt) for qt < ceil(R / T); rows [qt*T, min(R, (qt+1)*T)),
    tokens t_first = row0 // G .. t_last = (row_end - 1) // G, at KV positions
    q_pos(t) = Lkv - Lq + t (bottom-right alignment).  Visible end hi = Lkv,
    or with the causal mask min(Lkv, q_pos(t_last) + 1), floored at 0.
    Visible KV ranges: [0, hi) without a sliding window.  With window W >= 0
    and S sink tokens: lo = max(0, q_pos(t_first) - W) rounded down to the
    class granule (below); if lo <= min(S, hi) one range [0, hi), else the
    sink range [0, min(S, hi)) (when not empty) followed by [lo, hi).
    kv_eff = the summed length of the ranges.
    Multi-head units: when Lq = 1, the request reads the plan's own cache,
    the page size is 1, there is no RoPE, G is a multiple of 4 with G <= 16
    and H = 32 / G divides Hkv, the decode-class units are (b, hk) for hk a
    multiple of H, each taking KV heads hk .. hk + H - 1 at once: 32 rows,
    row = h * G + g for head hk + h, all of query token 0.
 3. Per class, total = sum of kv_eff (times H for a multi-head unit); chunk = max(min_chunk,
    ceil(total / (ctas * split_factor))) rounded up to a multiple of the
    class granule max(page_size, 64) (decode) or max(page_size, 128) (prefill).
    ctas = num_ctas, except for the decode class when the prefill-class
    items (n_pre of them: per 256-row unit, its ranges' chunk counts, at
    least 1) are at least one and at most num_ctas / 2: then num_ctas - n_pre.
    A multi-head unit's chunk is max(granule, ceil(ceil(chunk / H) / granule)
    * granule) keys (the K/V bytes of a one-head chunk).
 4. A unit with kv_eff = 0 gives one empty item.  Otherwise each range
    [s, e) splits into ceil((e - s) / chunk) items [s + i*chunk,
    min(e, s + (i+1)*chunk)), ranges in order, chunk numbers running across
    them.  When a unit has n > 1 items it becomes a merge unit (numbered in
    unit order) and its items get consecutive fp32 partial-state rows,
    n * rows in all.  A merge unit of a 256-row (prefill-class) unit carries
    the flag 1 in its seventh field ("late": merged after the run by a
    launch of its own), a 16-row unit 0 (merged inside the run); a header
    field counts the late units.
 5. cost = (kv length of the item * H + 256) * class weight (H = 1 for a
    one-head unit), the 256 standing for
    the fixed per-item latency of the kernel.  Items are sorted by
    (-cost, -T, b, hk, qt, chunk) and each goes to the CTA with the smallest
    load, ties to the smaller CTA index (longest processing time first).
 6. Output: header (with the variant: window, sink, soft-cap bits, and for
    RoPE its position capacity, theta and scale bits and the table offset;
    then the count of late units, the partial rows used, the batch's query
    tokens, the cascade fields, the count of 16-row items and the most rows of
    a cascade merge entry (0 without cascade)), per-CTA
    CSR offsets, items in CTA order (an item: its 8 fields, its request's
    table entry, H for a multi-head unit or 0, three zeros; within a CTA the 256-row items first,
    then the 16-row items, each in the order dealt), merge units, zeroed merge
    counters, request table.
"""
from __future__ import annotations

import heapq

import numpy as np

MAGIC = 0x46495031
TILE_DECODE, TILE_PREFILL = 16, 256
HEADER_INTS = 32
ROPE_PAIRS = 64
ITEM_INTS = 16
MERGE_INTS = 8
REQ_INTS = 4
CASCADE_INTS = 12
CASCADE_ROWS = 16
ITEM_COST_TOKENS = 256
MH_ROWS = 32  # packed query rows of a multi-head decode unit (its KV heads x G)

# fi_status values
OK, INVALID_ARG, UNSUPPORTED, CAPACITY = 0, 1, 2, 3


def _align4(n: int) -> int:
    return (n + 3) // 4 * 4


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def int_workspace_ints(cfg: dict) -> int:
    return (HEADER_INTS + _align4(cfg["num_ctas"] + 1) + ITEM_INTS * cfg["max_items"]
            + MERGE_INTS * cfg["max_merge_units"] + _align4(cfg["max_merge_units"])
            + REQ_INTS * cfg["max_batch"] + CASCADE_INTS * cfg["max_merge_units"])


def _pow2_page(page_size: int) -> bool:
    return 1 <= page_size <= 128 and page_size & (page_size - 1) == 0


def _config_status(cfg, head_dim, num_qo_heads, num_kv_heads, page_size, causal):
    """Status of the config and shapes (0 when they are acceptable)."""
    if head_dim != 128 or not _pow2_page(page_size):
        return UNSUPPORTED
    if num_qo_heads < 1 or num_kv_heads < 1 or num_qo_heads % num_kv_heads:
        return UNSUPPORTED
    if num_qo_heads // num_kv_heads > 16:
        return UNSUPPORTED
    if causal not in (0, 1) or cfg["num_ctas"] < 1 or cfg["split_factor"] < 1:
        return INVALID_ARG
    window, sink = cfg.get("window_left", -1), cfg.get("sink_tokens", 0)
    cap = float(np.float32(cfg.get("logits_soft_cap", 0.0)))
    if window < -1 or sink < 0 or not (cap >= 0.0) or cap == float("inf"):
        return INVALID_ARG
    rope_max = cfg.get("rope_max_positions", 0)
    theta = float(np.float32(cfg.get("rope_theta", 10000.0)))
    rscale = float(np.float32(cfg.get("rope_scale", 1.0)))
    if rope_max < 0 or (rope_max > 0 and not (0 < theta < float("inf") and 0 < rscale < float("inf"))):
        return INVALID_ARG
    return OK


def _requests_of(qo_indptr, kv_indptr, kv_indices, last_page_len, page_size, num_pages, rope_max):
    """One level's requests as [qo_start, qo_len, page_start, kv_len] lists
    (status, list): the indptr arrays start at 0 and never decrease, a
    request with pages fills its last page with 1..page_size slots, page ids
    lie in [0, num_pages) when num_pages > 0, and with RoPE every position
    lies in the table."""
    qo = [int(x) for x in qo_indptr]
    kvp = [int(x) for x in kv_indptr]
    lpl = [int(x) for x in last_page_len]
    batch = len(qo) - 1
    if batch < 0 or len(kvp) != batch + 1 or len(lpl) < batch:
        return INVALID_ARG, None
    if batch > 0 and (qo[0] != 0 or kvp[0] != 0):
        return INVALID_ARG, None
    reqs = []
    for b in range(batch):
        if qo[b + 1] < qo[b] or kvp[b + 1] < kvp[b]:
            return INVALID_ARG, None
        n_pg = kvp[b + 1] - kvp[b]
        if n_pg > 0 and not (1 <= lpl[b] <= page_size):
            return INVALID_ARG, None
        lkv_b = 0 if n_pg == 0 else (n_pg - 1) * page_size + lpl[b]
        lq_b = qo[b + 1] - qo[b]
        if rope_max > 0 and (lkv_b > rope_max or lq_b > lkv_b):
            return INVALID_ARG, None
        reqs.append([qo[b], lq_b, kvp[b], lkv_b])
    if num_pages > 0 and batch > 0:
        idx = np.asarray(kv_indices[:kvp[batch]], dtype=np.int64)
        if idx.size and (idx.min() < 0 or idx.max() >= num_pages):
            return INVALID_ARG, None
    return OK, reqs


def make_plan(cfg: dict, qo_indptr, kv_indptr, kv_indices, last_page_len, num_qo_heads: int,
              num_kv_heads: int, head_dim: int, page_size: int, causal: int, num_pages: int):
    """Returns (status, workspace int32 array or None, info dict or None)."""
    st = _config_status(cfg, head_dim, num_qo_heads, num_kv_heads, page_size, causal)
    if st:
        return st, None, None
    if len(qo_indptr) - 1 > cfg["max_batch"]:
        return CAPACITY, None, None
    st, reqs = _requests_of(qo_indptr, kv_indptr, kv_indices, last_page_len, page_size, num_pages,
                            cfg.get("rope_max_positions", 0))
    if st:
        return st, None, None
    total_qo = int(qo_indptr[-1]) if len(reqs) else 0
    return _plan(cfg, reqs, 0, page_size, [], total_qo, num_qo_heads, num_kv_heads, head_dim, page_size, causal)


def make_cascade_plan(cfg: dict, shared_qo_indptr, shared_kv_indptr, shared_kv_indices, shared_last_page_len,
                      shared_page_size: int, shared_num_pages: int, qo_indptr, kv_indptr, kv_indices,
                      last_page_len, num_qo_heads: int, num_kv_heads: int, head_dim: int, page_size: int,
                      causal: int, num_pages: int):
    """The two-level (cascade) plan: shared blocks, then the ordinary
    requests, in one request table.  Block s covers query rows
    [shared_qo_indptr[s], shared_qo_indptr[s+1]) -- the blocks cover every
    row and no request straddles two -- and its keys (a shared cache, pages
    of shared_page_size) are all visible to those rows; each ordinary
    request's own keys follow the causal flag, and a causal request has at
    least as many keys as queries.  Every unit writes partial states; the
    cascade merge entries name, per run of output rows, the partial rows of
    the block's chunks and of the request's chunks.  Windows, sinks and RoPE
    are not offered with two levels."""
    num_shared = len(shared_qo_indptr) - 1
    if num_shared < 1:
        return INVALID_ARG, None, None
    st = _config_status(cfg, head_dim, num_qo_heads, num_kv_heads, page_size, causal)
    if st:
        return st, None, None
    if not _pow2_page(shared_page_size):
        return UNSUPPORTED, None, None
    if cfg.get("window_left", -1) >= 0 or cfg.get("rope_max_positions", 0) > 0:
        return UNSUPPORTED, None, None
    batch = len(qo_indptr) - 1
    if batch + num_shared > cfg["max_batch"]:
        return CAPACITY, None, None
    st, shared = _requests_of(shared_qo_indptr, shared_kv_indptr, shared_kv_indices, shared_last_page_len,
                              shared_page_size, shared_num_pages, 0)
    if st:
        return st, None, None
    st, own = _requests_of(qo_indptr, kv_indptr, kv_indices, last_page_len, page_size, num_pages, 0)
    if st:
        return st, None, None
    total_qo = int(qo_indptr[-1]) if batch > 0 else 0
    bounds = [int(x) for x in shared_qo_indptr]
    if bounds[-1] != total_qo:
        return INVALID_ARG, None, None
    block_of = [-1] * num_shared
    for q0, lq, _, lkv in own:
        if causal and lkv < lq:
            return INVALID_ARG, None, None
        if lq == 0:
            block_of.append(-1)
            continue
        # the block whose row range holds this request's first row
        s = next((i for i in range(num_shared) if bounds[i] <= q0 < bounds[i + 1]), None)
        if s is None or q0 + lq > bounds[s + 1]:
            return INVALID_ARG, None, None
        block_of.append(s)
    return _plan(cfg, shared + own, num_shared, shared_page_size, block_of, total_qo, num_qo_heads,
                 num_kv_heads, head_dim, page_size, causal)


def _plan(cfg, reqs, num_shared, shared_page_size, block_of, total_qo, num_qo_heads, num_kv_heads, head_dim,
          page_size, causal):
    group = num_qo_heads // num_kv_heads
    cascade = num_shared > 0
    window, sink = cfg.get("window_left", -1), cfg.get("sink_tokens", 0)
    cap = float(np.float32(cfg.get("logits_soft_cap", 0.0)))
    rope_max = cfg.get("rope_max_positions", 0)
    theta = float(np.float32(cfg.get("rope_theta", 10000.0)))
    rscale = float(np.float32(cfg.get("rope_scale", 1.0)))
    batch = len(reqs)
    C = cfg["num_ctas"]
    lq = [r[1] for r in reqs]
    lkv = [r[3] for r in reqs]
    # chunk ends fall on the pages of every cache the plan reads
    page_gran = max(page_size, shared_page_size if cascade else page_size)
    granule = {TILE_DECODE: max(page_gran, 64), TILE_PREFILL: max(page_gran, 128)}

    def ranges_of(b, T, r0, r1, heads=1):
        # query tokens of the first and last rows (a multi-head unit: token 0)
        q_first = lkv[b] - lq[b] + (0 if heads > 1 else r0 // group)
        q_last = lkv[b] - lq[b] + (0 if heads > 1 else (r1 - 1) // group)
        causal_b = causal and b >= num_shared
        hi = max(0, min(lkv[b], q_last + 1) if causal_b else lkv[b])
        if window < 0:
            return [(0, hi)]
        lo = max(0, q_first - window) // granule[T] * granule[T]
        sink_end = min(sink, hi)
        if lo <= sink_end:
            return [(0, hi)]
        return ([(0, sink_end)] if sink_end > 0 else []) + [(lo, hi)]

    def tile_of(b):
        return TILE_DECODE if lq[b] * group <= TILE_DECODE else TILE_PREFILL

    # units in (b, hk, qt) order: (b, hk, qt, T, row0, row1, ranges, heads).  A
    # one-token request of the plan's own page-1 cache takes MH_ROWS / G KV
    # heads at once (rows = head offset * G + g) when G is a multiple of 4 and
    # those heads tile [0, Hkv): a short request then pays the per-item cost
    # once per unit instead of once per head.
    mh = MH_ROWS // group if (group % 4 == 0 and group <= MH_ROWS // 2
                              and num_kv_heads % (MH_ROWS // group) == 0) else 1
    units = []
    unit_at = {}
    total = {TILE_DECODE: 0, TILE_PREFILL: 0}
    for b in range(batch):
        R = lq[b] * group
        if R == 0:
            continue
        T = tile_of(b)
        cache_page = shared_page_size if b < num_shared else page_size
        heads = mh if (T == TILE_DECODE and lq[b] == 1 and cache_page == 1 and rope_max == 0
                       and b >= num_shared) else 1
        for hk in range(0, num_kv_heads, heads):
            for qt in range(_ceil_div(R, T)):
                r0, r1 = (0, R * heads) if heads > 1 else (qt * T, min(R, (qt + 1) * T))
                rng = ranges_of(b, T, r0, r1, heads)
                unit_at[(b, hk, qt)] = len(units)
                units.append((b, hk, qt, T, r0, r1, rng, heads))
                total[T] += sum(e - s for s, e in rng) * heads

    def pick(T, min_chunk, ctas):
        want = max(min_chunk, _ceil_div(total[T], ctas * cfg["split_factor"]))
        return _ceil_div(want, granule[T]) * granule[T]

    chunk = {TILE_PREFILL: pick(TILE_PREFILL, cfg["prefill_min_chunk"], C)}
    # prefill-class items; the decode class counts the CTAs they leave free when they take at most half
    n_pre = sum(max(1, sum(_ceil_div(e - s, chunk[TILE_PREFILL]) for s, e in u[6]))
                for u in units if u[3] == TILE_PREFILL)
    chunk[TILE_DECODE] = pick(TILE_DECODE, cfg["decode_min_chunk"], C - n_pre if 0 < 2 * n_pre <= C else C)
    weight = {TILE_DECODE: cfg["decode_cost_weight"], TILE_PREFILL: cfg["prefill_cost_weight"]}
    # a multi-head unit's chunk holds the K/V bytes of a one-head chunk, rounded up to the granule
    g = granule[TILE_DECODE]
    chunk_mh = max(g, _ceil_div(_ceil_div(chunk[TILE_DECODE], mh), g) * g)

    items = []   # (sort key, fields)
    merges = []
    part_rows = 0
    unit_parts = []  # per unit: (first partial row or -1, number of chunks)
    prefill_caches = 0
    for (b, hk, qt, T, r0, r1, rng, heads) in units:
        if T == TILE_PREFILL:
            prefill_caches |= 2 if b < num_shared else 1
        ck = chunk_mh if heads > 1 else chunk[T]
        pieces = [(s_ + i * ck, min(e_, s_ + (i + 1) * ck))
                  for s_, e_ in rng for i in range(_ceil_div(e_ - s_, ck))]
        n = max(1, len(pieces))
        nrows = r1 - r0
        base, m = -1, -1
        if n > 1 or cascade:
            base = part_rows
            part_rows += n * nrows
        if n > 1 and not cascade:
            m = len(merges)
            merges.append((b, hk, r0, r1, n, base, 0 if T == TILE_DECODE else 1, 0))
        unit_parts.append((base, n))
        for i, (k0, k1) in enumerate(pieces or [(0, 0)]):
            cost = ((k1 - k0) * heads + ITEM_COST_TOKENS) * weight[T]
            part = base + i * nrows if base >= 0 else -1
            # the request's table entry rides along with the item
            items.append(((-cost, -T, b, hk, qt, i),
                          (b, hk, r0, r1, k0, k1, part, m, *reqs[b], heads if heads > 1 else 0, 0, 0, 0)))

    # cascade merge entries, per ordinary unit: runs of at most CASCADE_ROWS
    # rows counted from the unit's first row, cut again at the block's q-tile bounds
    entries = []
    for u, (b, hk_u, qt, T, r0_u, r1_u, _, heads) in enumerate(units):
        if not cascade or b < num_shared:
            continue
        s = block_of[b]
        TS = tile_of(s)
        shift = (reqs[b][0] - reqs[s][0]) * group
        # a multi-head unit: entries per KV head, rows numbered as for one
        # head, head h's partial rows at offset h * G of the unit's
        for h in range(heads):
            hk = hk_u + h
            r0, r1 = (0, group) if heads > 1 else (r0_u, r1_u)
            b1, n1 = unit_parts[u]
            own0 = b1 + (h * group if heads > 1 else 0)
            r = r0
            while r < r1:
                sr = r + shift
                su = unit_at[(s, hk, sr // TS)]
                s_r0, s_r1 = units[su][4], units[su][5]
                r_end = min(r1, r0 + ((r - r0) // CASCADE_ROWS + 1) * CASCADE_ROWS, r + (s_r1 - sr))
                b0, n0 = unit_parts[su]
                entries.append((b, hk, r, r_end, n0, b0 + sr - s_r0, s_r1 - s_r0, n1, own0 + r - r0, r1_u - r0_u, 0, 0))
                r = r_end

    if len(items) > cfg["max_items"] or len(merges) > cfg["max_merge_units"] \
            or len(entries) > cfg["max_merge_units"] or part_rows > cfg["max_partial_rows"]:
        return CAPACITY, None, None

    items.sort(key=lambda it: it[0])
    heap = [(0, c) for c in range(C)]
    per_cta = [[] for _ in range(C)]
    for key, fields in items:
        load, c = heapq.heappop(heap)
        per_cta[c].append(fields)
        heapq.heappush(heap, (load - key[0], c))

    n_items, n_merge = len(items), len(merges)
    off_cta = HEADER_INTS
    off_items = off_cta + _align4(C + 1)
    off_merge = off_items + ITEM_INTS * n_items
    off_cnt = off_merge + MERGE_INTS * n_merge
    off_req = off_cnt + _align4(n_merge)
    off_cascade = off_req + REQ_INTS * batch
    total_ints = off_cascade + CASCADE_INTS * len(entries)
    if total_ints > int_workspace_ints(cfg):
        return CAPACITY, None, None

    ws = np.zeros(total_ints, dtype=np.int32)
    def bits(x):
        return int(np.array([x], dtype=np.float32).view(np.int32)[0])

    rope_off = (int_workspace_ints(cfg) * 4 + 255) // 256 * 256 // 4 if rope_max > 0 else 0
    n_dec = sum(1 for _, f in items if lq[f[0]] * group <= 16)
    ws[:HEADER_INTS] = [MAGIC, n_items, n_merge, C, batch, causal, off_cta, off_items, off_merge,
                        off_cnt, off_req, 0, num_qo_heads, num_kv_heads, page_size, total_ints,
                        window, sink, bits(cap), rope_max,
                        bits(theta) if rope_max > 0 else 0, bits(rscale) if rope_max > 0 else 0, rope_off,
                        sum(1 for m in merges if m[6]), part_rows, total_qo, num_shared,
                        off_cascade if cascade else 0, len(entries), shared_page_size if cascade else 0, n_dec,
                        max((e[3] - e[2] for e in entries), default=0)]
    pos = 0
    for c in range(C):
        ws[off_cta + c] = pos
        # prefill-class tiles first, then 16-row tiles, each in the order dealt
        mine = [f for f in per_cta[c] if lq[f[0]] * group > 16] + [f for f in per_cta[c] if lq[f[0]] * group <= 16]
        for fields in mine:
            ws[off_items + ITEM_INTS * pos: off_items + ITEM_INTS * (pos + 1)] = fields
            pos += 1
    ws[off_cta + C] = pos
    for m, fields in enumerate(merges):
        ws[off_merge + MERGE_INTS * m: off_merge + MERGE_INTS * (m + 1)] = fields
    for b in range(batch):
        ws[off_req + REQ_INTS * b: off_req + REQ_INTS * (b + 1)] = reqs[b]
    for e, fields in enumerate(entries):
        ws[off_cascade + CASCADE_INTS * e: off_cascade + CASCADE_INTS * (e + 1)] = fields

    info = dict(num_ctas=C, num_items=n_items, num_merge_units=n_merge,
                num_late_merge_units=sum(1 for m in merges if m[6]), batch=batch,
                num_partial_rows=part_rows, num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads,
                head_dim=head_dim, page_size=page_size, causal=causal, chunk_decode=chunk[16],
                chunk_prefill=chunk[TILE_PREFILL], num_decode_items=n_dec, num_prefill_items=n_items - n_dec,
                int_ws_bytes_used=4 * total_ints, max_partial_rows=cfg["max_partial_rows"],
                variant=(1 if cap > 0 else 0) | (2 if window >= 0 else 0) | (4 if rope_max > 0 else 0),
                num_shared=num_shared, num_cascade_merges=len(entries), prefill_caches=prefill_caches)
    return OK, ws, info


# ---------------------------------------------------------------- MLA decode plan

MLA_MAGIC = 0x464D4C31
MLA_HEADER_INTS = 16
MLA_BLOCK = 64
MLA_UNIT_COST_TOKENS = 448


def mla_make_plan(kv_indptr, last_page_len, page_size: int, num_heads: int, num_pairs: int,
                  min_chunk: int) -> np.ndarray:
    """The absorbed-MLA decode plan, restated.  Rule:
     1. L_b = (pages_b - 1) * page_size + last_page_len[b] (0 without pages).
     2. The requests with L_b > 0, in index order, are one stream of tokens;
        the pairs take consecutive pieces of it, pair 0 first.
     3. A piece costs its tokens + 448.  When pair c starts, with T tokens
        and n requests (started or not) still unplaced and q = pairs - c
        pairs left, its budget is max(ceil((T + 448 * (n + q - 1)) / q),
        448 + min_chunk).
     4. Pair c repeatedly takes the next piece of the current request: the
        rest of the request if that fits in (budget left - 448) rounded down
        to a multiple of 64, else that rounded amount; it takes nothing and
        stops if the piece would be shorter than both the rest and
        min_chunk.  After each piece it stops when the budget left minus 448
        is under 64.  The last pair takes all that is left, whatever its
        budget.
     5. A request in several pieces gets consecutive partial slots in stream
        order and a merge entry (b, first slot, count); a request with no
        tokens a merge entry (b, 0, 0); merge entries in request order.
     6. Image: header[16] (its chunk field = pair 0's budget), pair offsets
        (pairs + 1, padded to 4), units {b, kv0, kv1, slot or -1} pair by
        pair in the order taken, requests {kv_indptr[b], L_b} (padded to 4),
        merge entries {b, slot0, count, 0}."""
    kv_indptr = [int(x) for x in kv_indptr]
    B = len(kv_indptr) - 1
    L = []
    for b in range(B):
        n = kv_indptr[b + 1] - kv_indptr[b]
        L.append(0 if n == 0 else (n - 1) * page_size + int(last_page_len[b]))
    cost = MLA_UNIT_COST_TOKENS
    stream = [b for b in range(B) if L[b] > 0]
    owned = [[] for _ in range(num_pairs)]   # pieces [b, kv0, kv1, slot] per pair
    pos, done = 0, 0                         # stream position, tokens of stream[pos] placed
    first_budget = 0
    for c in range(num_pairs):
        if pos == len(stream):
            break
        q = num_pairs - c
        unplaced = sum(L[b] for b in stream[pos:]) - done
        budget = max(-(-(unplaced + cost * (len(stream) - pos + q - 1)) // q), cost + min_chunk)
        if c == 0:
            first_budget = budget
        left_budget = budget
        while pos < len(stream):
            b = stream[pos]
            rest = L[b] - done
            if c == num_pairs - 1:
                piece = rest
            else:
                fits = max(0, (left_budget - cost) // MLA_BLOCK * MLA_BLOCK)
                piece = min(rest, fits)
                if piece < rest and piece < min_chunk:
                    break
            owned[c].append([b, done, done + piece, -1])
            left_budget -= piece + cost
            done += piece
            if done == L[b]:
                pos, done = pos + 1, 0
            if c < num_pairs - 1 and left_budget - cost < MLA_BLOCK:
                break
    pieces_of = {}
    for c in range(num_pairs):
        for piece in owned[c]:
            pieces_of.setdefault(piece[0], []).append(piece)
    merge, slots = [], 0
    for b in range(B):
        if L[b] == 0:
            merge.append((b, 0, 0, 0))
        elif len(pieces_of[b]) > 1:
            for i, piece in enumerate(pieces_of[b]):
                piece[3] = slots + i
            merge.append((b, slots, len(pieces_of[b]), 0))
            slots += len(pieces_of[b])
    n_pieces = sum(len(o) for o in owned)
    chunk = first_budget

    def r4(n):
        return (n + 3) // 4 * 4

    off_pair = MLA_HEADER_INTS
    off_units = off_pair + r4(num_pairs + 1)
    off_req = off_units + 4 * n_pieces
    off_merge = off_req + r4(2 * B)
    total_ints = off_merge + 4 * len(merge)
    img = np.zeros(total_ints, dtype=np.int32)
    img[:MLA_HEADER_INTS] = [MLA_MAGIC, n_pieces, num_pairs, B, num_heads, page_size, off_pair, off_units,
                             off_req, off_merge, len(merge), 0, chunk, total_ints, slots, 0]
    at = 0
    for p in range(num_pairs):
        img[off_pair + p] = at
        for piece in owned[p]:
            img[off_units + 4 * at:off_units + 4 * at + 4] = piece
            at += 1
    img[off_pair + num_pairs] = at
    for b in range(B):
        img[off_req + 2 * b] = kv_indptr[b]
        img[off_req + 2 * b + 1] = L[b]
    for k, m in enumerate(merge):
        img[off_merge + 4 * k:off_merge + 4 * k + 4] = m
    return img

"""CUDA path (through the C ABI) against the fp64 oracle.

Small cases compare every output element; the full-size workloads compare
sampled (row, head) outputs that the oracle computes one by one.  Bar:
O max-abs <= 8e-3 and LSE abs <= 1e-3 against the fp64 values; rows without a
visible key must be exactly (0, -inf)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import serving_attention_gb300 as fi
import workloads
from helpers import LSE_TOL, O_TOL, compare, gpu_run, oracle_problem

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _full_check(b, cfg=None):
    o, lse, info, ws = gpu_run(b, cfg=cfg)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0
    o_ref, l_ref = oracle.attention(oracle_problem(b))
    n = b.total_qo
    err_o, err_l = compare(o[:n], lse[:n], o_ref, l_ref)
    assert err_o <= O_TOL and err_l <= LSE_TOL, (err_o, err_l)
    return info


def _sample_rows(b, per_request=3):
    rows = []
    for r in range(b.batch):
        q0, q1 = int(b.qo_indptr[r]), int(b.qo_indptr[r + 1])
        if q1 > q0:
            rows += sorted({q0, (q0 + q1 - 1) // 2, q1 - 1})[:per_request]
    return np.array(rows, np.int64)


def _sampled_check(b, o, lse, heads=None, rows=None):
    rows = _sample_rows(b) if rows is None else rows
    heads = np.arange(b.num_qo_heads) if heads is None else np.asarray(heads)
    rr = np.repeat(rows, len(heads))
    hh = np.tile(heads, len(rows))
    o_ref, l_ref = oracle.attention_select(oracle_problem(b), rr, hh)
    og = o[torch.as_tensor(rr), torch.as_tensor(hh)]
    lg = lse[torch.as_tensor(rr), torch.as_tensor(hh)]
    err_o, err_l = compare(og, lg, o_ref, l_ref)
    assert err_o <= O_TOL and err_l <= LSE_TOL, (err_o, err_l)
    return err_o, err_l


def test_tiny_decode_full():
    info = _full_check(workloads.tiny_decode(device=DEV))
    assert info.num_items > 0


@pytest.mark.parametrize("qo,kv,causal,dtype", [
    ([32], [128], 0, "bf16"),          # one 128-row M tile against one 128-token KV tile
    ([32], [128], 1, "bf16"),          # the same with the causal diagonal
    ([32], [77], 0, "fp16"),           # ragged KV tail inside the tile
    ([40], [300], 1, "bf16"),          # two row tiles (128 + 32 rows), three KV tiles
    ([64, 33], [1000, 40], 1, "bf16"), # two requests, long and short
    ([100], [600], 1, "bf16"),         # 400 rows: a 256-row item and a 144-row item
])
def test_tensor_core_tiles(qo, kv, causal, dtype):
    """Prefill-class items (one or two 128-row M tiles) on the tensor cores, page 16, G 4."""
    b = workloads.make_batch("tc", dtype, qo, kv, 8, 2, 16, causal, 300 + len(qo) + kv[0], DEV,
                             pool_pages=sum((k + 15) // 16 for k in kv) + 2)
    info = _full_check(b)
    assert info.num_prefill_items > 0


@pytest.mark.parametrize("scale,dtype", [(1.5, "bf16"), (2.0, "bf16"), (4.0, "bf16"), (4.0, "fp16"), (8.0, "fp16")])
@pytest.mark.parametrize("prefill_min_chunk", [1024, 512])
def test_peaked_softmax_tensor_cores(scale, dtype, prefill_min_chunk):
    """Queries scaled up so a few keys dominate each row, whole (1024-token
    chunks) and split in two (512, merged by the late merge).  P enters the
    P V MMA rounded to 16 bits; O is divided by the sum of those rounded P,
    so a key that dominates its row passes its value through unchanged, and
    LSE comes from the sum of the fp32 P.  The bar is the flat 8e-3 wherever
    the stored outputs stay below 4 in magnitude.  At bf16 x4 single keys
    push |o| past 4, where half an ulp of the stored bf16 value is 2^-6 by
    itself, more than the whole bar; there the bar adds that storage
    rounding (2^-8 |o_ref|)."""
    b = workloads.make_batch("peak", dtype, [64, 33], [1000, 40], 8, 2, 16, 1, 777, DEV, pool_pages=70)
    b.q.mul_(scale)
    cfg = fi.default_plan_config(0, prefill_min_chunk=prefill_min_chunk)
    o, lse, info, ws = gpu_run(b, cfg=cfg)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0 and info.num_prefill_items > 0
    assert (info.num_late_merge_units > 0) == (prefill_min_chunk == 512)
    o_ref, l_ref = oracle.attention(oracle_problem(b))
    n = b.total_qo
    err_o, err_l = compare(o[:n], lse[:n], o_ref, l_ref)
    assert err_l <= LSE_TOL, err_l
    if dtype == "bf16" and scale > 2.0:
        assert np.abs(o_ref).max() > 4.0  # the storage rounding alone can exceed the flat bar
        excess = np.abs(o[:n].float().cpu().numpy() - o_ref) - (O_TOL + 2.0 ** -8 * np.abs(o_ref))
        assert excess.max() <= 0, float(excess.max())
    else:
        assert err_o <= O_TOL, err_o


@pytest.mark.parametrize("seed,page,group,causal,dtype,qo_max,kv_max", [
    (101, 16, 4, 0, "bf16", 1, 700), (102, 1, 4, 0, "bf16", 1, 300), (103, 4, 1, 1, "fp16", 3, 500),
    (104, 16, 8, 1, "bf16", 2, 900), (105, 64, 4, 1, "bf16", 40, 400), (106, 16, 4, 1, "fp16", 70, 300),
    (107, 2, 2, 0, "bf16", 9, 260), (108, 128, 16, 1, "bf16", 12, 700), (109, 32, 4, 1, "bf16", 5, 2000),
])
def test_random_small_full(seed, page, group, causal, dtype, qo_max, kv_max):
    """Several tiles, ragged tails, splits (small chunks on few CTAs), empty requests."""
    hkv = 2
    b = workloads.random_batch(seed, batch=6, qo_max=qo_max, kv_max=kv_max, num_qo_heads=hkv * group,
                               num_kv_heads=hkv, page_size=page, causal=causal, dtype=dtype, device=DEV)
    cfg = fi.default_plan_config(0, num_ctas=5, decode_min_chunk=64, prefill_min_chunk=128, split_factor=3)
    info = _full_check(b, cfg=cfg)
    assert info.num_items >= 6


def test_late_merge_of_prefill_split_units():
    """Prefill-class split units are merged after the run by the row-parallel
    merge launch: 3 to 19 chunks per unit (past the merge's 4-wide load
    groups, with ragged tails), row counts that are not multiples of the
    8-row blocks, causal rows that see few keys."""
    b = workloads.random_batch(221, batch=5, qo_max=130, kv_max=2600, num_qo_heads=8, num_kv_heads=2,
                               page_size=16, causal=1, device=DEV, qo_min=37, kv_min=200)
    cfg = fi.default_plan_config(0, num_ctas=40, prefill_min_chunk=128, split_factor=6)
    info = _full_check(b, cfg=cfg)
    assert info.num_late_merge_units == info.num_merge_units == 16  # 3 to 19 chunks per unit


def test_graph_templates_with_and_without_late_units():
    """A graph captured from a plan without late units replays a plan with
    them (the run merges them itself); a graph captured from a plan with late
    units replays one without (the late merge finds nothing) and one with
    them again.  Both merges give the same bits, and every replay matches the
    oracle."""
    cfg = fi.default_plan_config(0, num_ctas=40, prefill_min_chunk=128, decode_min_chunk=64, split_factor=6)
    bB = workloads.make_batch("graph_pf", "bf16", [80, 45, 61, 90], [1900, 1200, 1500, 1000], 8, 2, 16, 1, 231,
                              DEV, poison=False)
    rng = np.random.default_rng(232)
    kvA = rng.integers(1, 600, size=6)
    kvpA, lplA = workloads._pages_for(kvA, 16)
    kviA = rng.permutation(bB.num_pages)[:kvpA[-1]].astype(np.int32)
    bA = workloads.PagedBatch("graph_dec", "bf16", np.arange(7, dtype=np.int32), kvpA, kviA, lplA, 8, 2, 16, 0,
                              bB.sm_scale, bB.q, bB.k, bB.v, bB.k_base, bB.v_base)
    kvi_buf = torch.zeros(bB.num_pages, dtype=torch.int32, device=DEV)
    refs = {}

    def replan(ws, b):
        info = fi.plan(ws, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, 8, 2, 128, 16, b.causal,
                       b.num_pages)
        kvi_buf[:b.kv_indices.size].copy_(torch.as_tensor(b.kv_indices, device=DEV))
        return info

    def check(b, o, lse):
        if b.name not in refs:
            refs[b.name] = oracle.attention(oracle_problem(b))
        n = b.total_qo
        err_o, err_l = compare(o[:n], lse[:n], *refs[b.name])
        assert err_o <= O_TOL and err_l <= LSE_TOL, (b.name, err_o, err_l)

    outs = {}
    for first, later in ((bA, [bB]), (bB, [bA, bB])):
        ws = fi.Workspace(cfg, device=DEV)
        o = torch.full_like(bB.q, float("nan"))
        lse = torch.full(bB.q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
        info = replan(ws, first)
        assert (info.num_late_merge_units > 0) == (first is bB)
        fi.run(ws, info, bB.q, bB.k, bB.v, kvi_buf, o, lse, bB.sm_scale)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fi.run(ws, info, bB.q, bB.k, bB.v, kvi_buf, o, lse, bB.sm_scale)
        for b in [first] + later:
            info_b = replan(ws, b)
            assert info_b.num_ctas == info.num_ctas
            o.fill_(float("nan"))
            lse.fill_(float("nan"))
            graph.replay()
            torch.cuda.synchronize()
            assert fi.device_status(ws) == 0
            check(b, o, lse)
            if b is bB:
                outs[first.name] = (o[:b.total_qo].clone(), lse[:b.total_qo].clone())
        del graph
    # bB merged in the run (template bA) and by the late merge (template bB)
    assert torch.equal(outs["graph_dec"][0], outs["graph_pf"][0])
    assert torch.equal(outs["graph_dec"][1], outs["graph_pf"][1])


def test_empty_and_blind_rows():
    b = workloads.make_batch("edge", "bf16", [2, 1, 4, 3], [0, 5, 2, 40], 8, 2, 4, 1, 77, DEV, pool_pages=20)
    _full_check(b)


def test_equal_and_unequal_strides_agree():
    b = workloads.random_batch(201, batch=5, qo_max=3, kv_max=800, num_qo_heads=8, num_kv_heads=2, page_size=16,
                               causal=1, device=DEV, v_pad_heads=1)
    o1, l1, _, _ = gpu_run(b)
    v_eq = b.v.contiguous()
    b2 = workloads.PagedBatch(b.name, b.dtype, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len,
                              b.num_qo_heads, b.num_kv_heads, b.page_size, b.causal, b.sm_scale, b.q, b.k, v_eq,
                              b.k_base, v_eq)
    o2, l2, _, _ = gpu_run(b2)
    torch.cuda.synchronize()
    n = b.total_qo
    assert torch.equal(o1[:n], o2[:n]) and torch.equal(l1[:n], l2[:n])


def _pad_pages(t: torch.Tensor, pad: int):
    """The same values in a cache whose pages are `pad` elements longer (page
    stride no longer a whole number of head strides)."""
    pool, P, H, D = t.shape
    buf = torch.zeros((pool, P * H * D + pad), dtype=t.dtype, device=t.device)
    view = buf.as_strided((pool, P, H, D), (P * H * D + pad, H * D, D, 1))
    view.copy_(t)
    return buf, view


def test_page1_gather_and_box_fetches_agree():
    """Page size 1.  K contiguous (2 rows per page) and V with a padding head
    (3 rows per page) are fetched by four-row gathers; padded pages (page
    stride 264 elements, not a multiple of the 128-element head stride) by one
    box per token.  Both match the oracle, and both fetches land the same
    bytes in shared memory, so the outputs are identical."""
    b = workloads.random_batch(211, batch=7, qo_max=1, kv_max=700, num_qo_heads=8, num_kv_heads=2, page_size=1,
                               causal=0, device=DEV, kv_min=0, v_pad_heads=1)
    cfg = fi.default_plan_config(0, num_ctas=6, decode_min_chunk=64, split_factor=3)
    _full_check(b, cfg=cfg)
    o1, l1, _, _ = gpu_run(b, cfg=cfg)
    kb, kp = _pad_pages(b.k, 8)
    vb, vp = _pad_pages(b.v, 8)
    b2 = workloads.PagedBatch(b.name, b.dtype, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len,
                              b.num_qo_heads, b.num_kv_heads, b.page_size, b.causal, b.sm_scale, b.q, kp, vp, kb, vb)
    _full_check(b2, cfg=cfg)
    o2, l2, _, _ = gpu_run(b2, cfg=cfg)
    torch.cuda.synchronize()
    n = b.total_qo
    assert torch.equal(o1[:n], o2[:n]) and torch.equal(l1[:n], l2[:n])


def test_llama8b_decode_sampled():
    b = workloads.llama8b_decode(device=DEV)
    o, lse, info, ws = gpu_run(b)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0
    assert info.num_merge_units > 0, "the long requests must be split"
    _sampled_check(b, o, lse)
    del b, o, lse
    torch.cuda.empty_cache()


def test_ragged_prefill_sampled():
    b = workloads.ragged_prefill(device=DEV)
    o, lse, info, ws = gpu_run(b)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0
    rows = _sample_rows(b)
    _sampled_check(b, o, lse, heads=[0, 3, 4, 17, 31], rows=rows)
    del b, o, lse
    torch.cuda.empty_cache()


def test_shared_prefix_composable():
    d = workloads.shared_prefix(device=DEV)
    pre, suf, flat = d["prefix"], d["suffix"], d["flat"]
    o_p, l_p, _, _ = gpu_run(pre)
    o_s, l_s, _, _ = gpu_run(suf)
    o_m = torch.empty_like(o_p)
    l_m = torch.empty_like(l_p)
    fi.merge_states(o_p, l_p, o_s, l_s, o_m, l_m)
    o_f, l_f, _, _ = gpu_run(flat)
    torch.cuda.synchronize()
    rows = np.arange(flat.total_qo)
    _sampled_check(flat, o_m, l_m, heads=[0, 9, 31], rows=rows)
    # composable result agrees with the flat layout run
    assert float((o_m.float() - o_f.float()).abs().max()) <= 2 * O_TOL
    assert float((l_m - l_f).abs().max()) <= 2 * LSE_TOL


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_merge_states_kernel(dtype):
    g = torch.Generator(device=DEV).manual_seed(5)
    rows, heads = 37, 5
    va = torch.randn(rows, heads, 128, generator=g, device=DEV).to(dtype)
    vb = torch.randn(rows, heads, 128, generator=g, device=DEV).to(dtype)
    sa = torch.randn(rows, heads, generator=g, device=DEV) * 4
    sb = torch.randn(rows, heads, generator=g, device=DEV) * 4
    sa[0, 0] = float("-inf")
    sb[1, 1] = float("-inf")
    sa[2, 2] = sb[2, 2] = float("-inf")
    vo = torch.empty_like(va)
    so = torch.empty_like(sa)
    fi.merge_states(va, sa, vb, sb, vo, so)
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.merge_states(va.double().cpu().numpy(), sa.double().cpu().numpy(),
                                       vb.double().cpu().numpy(), sb.double().cpu().numpy())
    err_o, err_l = compare(vo.reshape(-1, 128), so.reshape(-1), o_ref.reshape(-1, 128), s_ref.reshape(-1))
    assert err_o <= O_TOL and err_l <= LSE_TOL
    # in place: the output may alias an input
    fi.merge_states(va, sa, vb, sb, va, sa)
    torch.cuda.synchronize()
    assert torch.equal(va, vo) and torch.equal(sa, so)


def test_continuous_batch_graph_replans():
    """One captured graph serves 10 seeded re-plans of the mix (unequal K/V
    strides); graph output is bit-identical to an eager run of the same plan
    and matches the oracle on sampled rows."""
    pages, tokens = workloads.continuous_batch_capacity(10)
    cfg = fi.default_plan_config(0)
    ws = fi.Workspace(cfg, device=DEV)
    b0 = workloads.continuous_batch(device=DEV, replan=0, pool_pages=pages, q_tokens=tokens)
    q_buf = b0.q
    k_buf, v_base = b0.k_base, b0.v_base
    v_buf = b0.v
    kvi_buf = torch.zeros(pages, dtype=torch.int32, device=DEV)
    o = torch.zeros_like(q_buf)
    lse = torch.zeros(q_buf.shape[:2], dtype=torch.float32, device=DEV)
    info = fi.plan(ws, b0.qo_indptr, b0.kv_indptr, b0.kv_indices, b0.last_page_len, 32, 8, 128, 16, 1, pages)
    kvi_buf[:b0.kv_indices.size].copy_(torch.as_tensor(b0.kv_indices, device=DEV))
    fi.run(ws, info, q_buf, k_buf, v_buf, kvi_buf, o, lse, b0.sm_scale)  # warm-up outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fi.run(ws, info, q_buf, k_buf, v_buf, kvi_buf, o, lse, b0.sm_scale)
    for r in range(10):
        if r > 0:
            b = workloads.continuous_batch(device=DEV, replan=r, pool_pages=pages, q_tokens=tokens)
            q_buf.copy_(b.q)
            k_buf.copy_(b.k_base)
            v_base.copy_(b.v_base)
        else:
            b = b0
        info_r = fi.plan(ws, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, 32, 8, 128, 16, 1, pages)
        kvi_buf[:b.kv_indices.size].copy_(torch.as_tensor(b.kv_indices, device=DEV))
        assert info_r.num_ctas == info.num_ctas
        graph.replay()
        torch.cuda.synchronize()
        assert fi.device_status(ws) == 0
        n = int(b.qo_indptr[-1])
        o_g, l_g = o[:n].clone(), lse[:n].clone()
        fi.run(ws, info_r, q_buf, k_buf, v_buf, kvi_buf, o, lse, b.sm_scale)
        torch.cuda.synchronize()
        assert torch.equal(o_g, o[:n]) and torch.equal(l_g, lse[:n]), f"graph != eager at replan {r}"
        if r in (0, 3, 9):
            view = workloads.PagedBatch(b.name, b.dtype, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len,
                                        32, 8, 16, 1, b.sm_scale, q_buf, k_buf, v_buf, k_buf, v_base)
            heads = [0, 13, 31]
            _sampled_check(view, o, lse, heads=heads)
    del graph
    torch.cuda.empty_cache()

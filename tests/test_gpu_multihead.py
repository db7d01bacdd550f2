"""Multi-head decode units on the CUDA path, through the C ABI, against the
fp64 oracle (every element).

A one-token request on a cache of one-token pages, with a GQA group G that is
a multiple of 4, is planned as units of 32 / G KV heads: one work item scores
all of them, and one TMA box per token brings that token's rows of every head
of the unit.  The cases cover the three unit widths (8, 4 and 2 heads), split
units (merged inside the run) and whole ones, one-head units of multi-token
requests in the same plan, empty and one-token requests, stages cut short by
the chunk, a padded V cache (its own strides), the mask and soft-cap
variants with a sink longer than a chunk, and the shared-prefix layout of two
levels.  Bar: O max-abs <= 8e-3 and LSE abs <= 1e-3."""
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


def _heads_of_items(ws):
    """Per work item of the plan in a device workspace: its KV-head count."""
    iws = ws.int_ws.cpu().numpy()
    n, off = int(iws[1]), int(iws[7])
    return iws[off:off + 16 * n].reshape(-1, 16)[:, 12]


def _lengths(seed, n=9):
    rng = np.random.default_rng(seed)
    kv = rng.integers(2, 700, size=n)
    kv[0], kv[1], kv[2], kv[3] = 0, 1, 17, 64  # empty, one key, one stage and one key, one granule
    qo = np.ones(n, np.int64)
    qo[5] = 3                                  # a three-token request: one-head units beside the others
    return qo, kv


@pytest.mark.parametrize("seed,group,hkv,dtype,causal,split,v_pad", [
    (1101, 4, 8, "bf16", 0, False, 0),
    (1102, 4, 8, "fp16", 1, True, 0),
    (1103, 8, 4, "bf16", 1, True, 0),
    (1104, 16, 2, "bf16", 0, True, 0),
    (1105, 16, 4, "fp16", 1, False, 0),
    (1106, 4, 8, "bf16", 1, True, 3),   # V pages padded by 3 heads: V's page stride differs from K's
])
def test_multi_head_decode_matches_oracle(seed, group, hkv, dtype, causal, split, v_pad):
    qo, kv = _lengths(seed)
    b = workloads.make_batch("mh", dtype, qo, kv, hkv * group, hkv, 1, causal, seed, DEV, v_pad_heads=v_pad)
    cfg = (fi.default_plan_config(0, num_ctas=5, decode_min_chunk=64, split_factor=3) if split
           else fi.default_plan_config(0))
    o, lse, info, ws = gpu_run(b, cfg=cfg)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0
    heads = _heads_of_items(ws)
    assert (heads == 32 // group).any() and (heads == 0).any()
    if split:
        assert info.num_merge_units > 0
    o_ref, l_ref = oracle.attention(oracle_problem(b))
    n = b.total_qo
    err_o, err_l = compare(o[:n], lse[:n], o_ref, l_ref)
    assert err_o <= O_TOL and err_l <= LSE_TOL, (err_o, err_l)


@pytest.mark.parametrize("window,sink,cap", [(100, 300, 0.0), (40, 3, 30.0), (-1, 0, 20.0), (250, 700, 0.0)])
def test_multi_head_decode_variants(window, sink, cap):
    """Window, sink (longer than the 64-token chunks in two cases) and soft-cap
    on multi-head units, split over small chunks."""
    qo, kv = _lengths(1110)
    kv[6] = 1500
    b = workloads.make_batch("mh_var", "bf16", qo, kv, 32, 8, 1, 1, 1110, DEV)
    cfg = fi.default_plan_config(0, num_ctas=7, decode_min_chunk=64, split_factor=3, window_left=window,
                                 sink_tokens=sink, logits_soft_cap=cap)
    o, lse, info, ws = gpu_run(b, cfg=cfg)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0 and (_heads_of_items(ws) == 8).any()
    o_ref, l_ref = oracle.attention(oracle_problem(b, window, sink, cap))
    n = b.total_qo
    err_o, err_l = compare(o[:n], lse[:n], o_ref, l_ref)
    assert err_o <= O_TOL and err_l <= LSE_TOL, (err_o, err_l)


@pytest.mark.parametrize("page,causal,sink", [(1, 1, 300), (4, 1, 200), (16, 0, 150)])
def test_sink_longer_than_a_chunk_and_the_causal_range(page, causal, sink):
    """Sink tokens past a chunk's end, or past a query's causal range, stay
    invisible to it: multi-token requests on the CUDA-core path with chunks of
    64 keys and a sink of 150 to 300 keys."""
    rng = np.random.default_rng(1120 + page)
    kv = rng.integers(200, 900, size=5)
    qo = np.array([1, 4, 9, 2, 1])
    b = workloads.make_batch("sink_long", "bf16", qo, kv, 8, 2, page, causal, 1120 + page, DEV)
    cfg = fi.default_plan_config(0, num_ctas=6, decode_min_chunk=64, split_factor=4, window_left=30,
                                 sink_tokens=sink)
    o, lse, info, ws = gpu_run(b, cfg=cfg)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0 and info.num_merge_units > 0
    o_ref, l_ref = oracle.attention(oracle_problem(b, 30, sink))
    n = b.total_qo
    err_o, err_l = compare(o[:n], lse[:n], o_ref, l_ref)
    assert err_o <= O_TOL and err_l <= LSE_TOL, (err_o, err_l)


@pytest.mark.parametrize("seed,group,hkv", [(1131, 4, 8), (1132, 8, 4)])
def test_multi_head_units_in_a_cascade(seed, group, hkv):
    """Two-level plans whose own requests are one-token branches at page 1:
    the branch units take 32 / G heads, the cascade merge combines each
    head's rows with its block's."""
    d = workloads.cascade_batch(seed, [3, 2, 4], 1, 600, 2500, hkv * group, hkv, 1, 16, 0, device=DEV, shared_min=0)
    sh, own = d["shared"], d["own"]
    cfg = fi.default_plan_config(0, num_ctas=23, decode_min_chunk=64, split_factor=3)
    ws = fi.Workspace(cfg, device=DEV)
    info = fi.plan_cascade(ws, sh.qo_indptr, sh.kv_indptr, sh.kv_indices, sh.last_page_len, sh.page_size,
                           own.qo_indptr, own.kv_indptr, own.kv_indices, own.last_page_len, own.num_qo_heads,
                           own.num_kv_heads, 128, own.page_size, own.causal, own.num_pages, sh.num_pages)
    assert (_heads_of_items(ws) == 32 // group).any()
    kvi = torch.as_tensor(own.kv_indices, device=DEV)
    skvi = torch.as_tensor(sh.kv_indices if sh.kv_indices.size else np.zeros(1, np.int32), device=DEV)
    o = torch.full_like(own.q, float("nan"))
    lse = torch.full(own.q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    fi.run_cascade(ws, info, own.q, own.k, own.v, kvi, sh.k, sh.v, skvi, o, lse, own.sm_scale)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0
    o_ref, l_ref = oracle.attention(oracle_problem(d["flat"]))
    n = own.total_qo
    err_o, err_l = compare(o[:n], lse[:n], o_ref, l_ref)
    assert err_o <= O_TOL and err_l <= LSE_TOL, (err_o, err_l)

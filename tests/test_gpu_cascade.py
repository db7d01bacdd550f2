"""Two-level (cascade) runs through the C ABI against the fp64 oracle.

A cascade batch -- shared blocks (one cache) and each request's own pages
(another cache) -- is planned by fi_plan_cascade and run as one persistent
launch plus the cascade merge; the oracle computes the same attention over
each request's block keys followed by its own keys as one page-1 batch.  Bar:
O max-abs <= 8e-3 and LSE abs <= 1e-3 against the fp64 values."""
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


def cascade_run(d, cfg=None, ws=None, o=None, lse=None):
    sh, own = d["shared"], d["own"]
    cfg = cfg if cfg is not None else fi.default_plan_config(0)
    ws = ws if ws is not None else fi.Workspace(cfg, device=DEV)
    info = fi.plan_cascade(ws, sh.qo_indptr, sh.kv_indptr, sh.kv_indices, sh.last_page_len, sh.page_size,
                           own.qo_indptr, own.kv_indptr, own.kv_indices, own.last_page_len, own.num_qo_heads,
                           own.num_kv_heads, 128, own.page_size, own.causal, own.num_pages, sh.num_pages)
    kvi = torch.as_tensor(own.kv_indices if own.kv_indices.size else np.zeros(1, np.int32), device=DEV)
    skvi = torch.as_tensor(sh.kv_indices if sh.kv_indices.size else np.zeros(1, np.int32), device=DEV)
    o = o if o is not None else torch.full_like(own.q, float("nan"))
    lse = lse if lse is not None else torch.full(own.q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    fi.run_cascade(ws, info, own.q, own.k, own.v, kvi, sh.k, sh.v, skvi, o, lse, own.sm_scale)
    return o, lse, info, ws


@pytest.mark.parametrize("seed,blocks,qo_max,page,spage,group,causal,dtype", [
    (301, [4, 1, 3], 1, 1, 16, 4, 0, "bf16"),     # decode branches at page 1 (gathers), blocks on tensor cores
    (302, [2, 3], 5, 16, 16, 4, 1, "bf16"),       # multi-token branches, causal own keys
    (303, [1, 2, 2], 70, 4, 8, 2, 1, "fp16"),     # prefill-class requests (own cache on CUDA cores, page 4)
    (304, [3, 3], 2, 1, 1, 8, 0, "bf16"),         # both caches at page 1: blocks on the CUDA-core path
    (305, [6], 40, 16, 64, 4, 1, "bf16"),         # one block, both levels on tensor cores
    (306, [2, 2, 1], 3, 2, 16, 1, 0, "fp16"),     # G 1
])
def test_cascade_matches_oracle(seed, blocks, qo_max, page, spage, group, causal, dtype):
    d = workloads.cascade_batch(seed, blocks, qo_max, 700, 2500, 2 * group, 2, page, spage, causal, dtype=dtype,
                                device=DEV, shared_min=0)
    cfg = fi.default_plan_config(0, num_ctas=37, decode_min_chunk=64, prefill_min_chunk=128, split_factor=3)
    o, lse, info, ws = cascade_run(d, cfg)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0 and info.num_cascade_merges > 0
    o_ref, l_ref = oracle.attention(oracle_problem(d["flat"]))
    n = d["own"].total_qo
    err_o, err_l = compare(o[:n], lse[:n], o_ref, l_ref)
    assert err_o <= O_TOL and err_l <= LSE_TOL, (err_o, err_l)


def test_cascade_with_empty_blocks_and_requests():
    """Blocks without keys, requests without keys, and a request whose block
    is empty too: its rows see no key at all and get (0, -inf)."""
    d = workloads.cascade_batch(315, [2, 2, 2], 2, 3, 3, 8, 2, 16, 16, 0, device=DEV)
    skv, okv = d["shared"].kv_lens(), d["own"].kv_lens()
    assert skv[1] == 0 and okv[2] == 0 and (skv == 0).sum() == 2
    o, lse, info, ws = cascade_run(d)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0
    o_ref, l_ref = oracle.attention(oracle_problem(d["flat"]))
    n = d["own"].total_qo
    assert np.isneginf(l_ref).any()
    err_o, err_l = compare(o[:n], lse[:n], o_ref, l_ref)  # also: the empty rows are exactly (0, -inf)
    assert err_o <= O_TOL and err_l <= LSE_TOL, (err_o, err_l)


def test_shared_prefix_in_one_launch():
    """The parallel-generation workload as a cascade: the 8192-token dense
    prefix (pages of 16, identity ids) is one block for all 64 branches, the
    page-1 suffixes are the requests' own keys.  Sampled rows against the
    oracle on the flat layout, and everything against the flat GPU run."""
    d = workloads.shared_prefix(device=DEV)
    pre, suf, flat = d["prefix"], d["suffix"], d["flat"]
    o, lse, info, ws = cascade_run({"shared": pre, "own": suf})
    o_f, l_f, _, _ = gpu_run(flat)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0 and info.num_shared == 1 and info.prefill_caches == 2
    rows = np.arange(flat.total_qo)
    heads = np.array([0, 9, 31])
    rr, hh = np.repeat(rows, len(heads)), np.tile(heads, len(rows))
    o_ref, l_ref = oracle.attention_select(oracle_problem(flat), rr, hh)
    err_o, err_l = compare(o[torch.as_tensor(rr), torch.as_tensor(hh)], lse[torch.as_tensor(rr), torch.as_tensor(hh)],
                           o_ref, l_ref)
    assert err_o <= O_TOL and err_l <= LSE_TOL, (err_o, err_l)
    assert float((o.float() - o_f.float()).abs().max()) <= 2 * O_TOL
    assert float((lse - l_f).abs().max()) <= 2 * LSE_TOL


def test_cascade_graph_replays_new_plans():
    """One graph captured from a cascade plan replays re-plans with other
    suffix lengths bit for bit like eager runs, and matches the oracle."""
    cfg = fi.default_plan_config(0)
    ws = fi.Workspace(cfg, device=DEV)
    # no poison: the re-plans pick their pages anywhere in the two pools
    d0 = workloads.cascade_batch(321, [3, 3], 1, 600, 3000, 32, 8, 1, 16, 0, device=DEV, poison=False)
    sh0, own0 = d0["shared"], d0["own"]
    # buffers at capacity: the same pools for every draw, page tables rewritten
    kvi = torch.zeros(own0.num_pages, dtype=torch.int32, device=DEV)
    skvi = torch.zeros(sh0.num_pages, dtype=torch.int32, device=DEV)
    o = torch.zeros_like(own0.q)
    lse = torch.zeros(own0.q.shape[:2], dtype=torch.float32, device=DEV)

    def plan(sh, own):
        info = fi.plan_cascade(ws, sh.qo_indptr, sh.kv_indptr, sh.kv_indices, sh.last_page_len, 16, own.qo_indptr,
                               own.kv_indptr, own.kv_indices, own.last_page_len, 32, 8, 128, 1, 0, own0.num_pages,
                               sh0.num_pages)
        kvi[:own.kv_indices.size].copy_(torch.as_tensor(own.kv_indices, device=DEV))
        skvi[:sh.kv_indices.size].copy_(torch.as_tensor(sh.kv_indices, device=DEV))
        return info

    info0 = plan(sh0, own0)
    run = lambda info: fi.run_cascade(ws, info, own0.q, own0.k, own0.v, kvi, sh0.k, sh0.v, skvi, o, lse,  # noqa: E731
                                      own0.sm_scale)
    run(info0)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run(info0)
    rng = np.random.default_rng(322)
    for r in range(4):
        # same pools and queries, new lengths and page choices inside them
        own_kv = rng.integers(1, own0.num_pages // 6 + 1, size=6)
        sh_kv = rng.integers(0, sh0.num_pages * 16 // 2 + 1, size=2)
        own_kvp, own_lpl = workloads._pages_for(own_kv, 1)
        sh_kvp, sh_lpl = workloads._pages_for(sh_kv, 16)
        own = workloads.PagedBatch("own", "bf16", own0.qo_indptr, own_kvp,
                                   rng.permutation(own0.num_pages)[:int(own_kvp[-1])].astype(np.int32), own_lpl,
                                   32, 8, 1, 0, own0.sm_scale, own0.q, own0.k, own0.v, own0.k_base, own0.v_base)
        sh = workloads.PagedBatch("shared", "bf16", sh0.qo_indptr, sh_kvp,
                                  rng.permutation(sh0.num_pages)[:int(sh_kvp[-1])].astype(np.int32), sh_lpl,
                                  32, 8, 16, 0, own0.sm_scale, own0.q, sh0.k, sh0.v, sh0.k_base, sh0.v_base)
        info = plan(sh, own)
        g.replay()
        torch.cuda.synchronize()
        assert fi.device_status(ws) == 0
        o_g, l_g = o.clone(), lse.clone()
        run(info)
        torch.cuda.synchronize()
        assert torch.equal(o_g, o) and torch.equal(l_g, lse), r
        # the oracle: the block's attention merged with the request's own
        # (the two-level reading, pinned against attention over the
        # concatenated keys in the oracle's tests)
        so, sl = oracle.attention(oracle_problem(sh))
        oo, ol = oracle.attention(oracle_problem(own))
        mo, ml = oracle.merge_states(so, sl, oo, ol)
        err_o, err_l = compare(o, lse, mo, ml)
        assert err_o <= O_TOL and err_l <= LSE_TOL, (r, err_o, err_l)


def test_one_level_run_refuses_a_cascade_plan():
    d = workloads.cascade_batch(331, [2], 1, 50, 60, 8, 2, 16, 16, 0, device=DEV)
    sh, own = d["shared"], d["own"]
    ws = fi.Workspace(fi.default_plan_config(0), device=DEV)
    info = fi.plan_cascade(ws, sh.qo_indptr, sh.kv_indptr, sh.kv_indices, sh.last_page_len, 16, own.qo_indptr,
                           own.kv_indptr, own.kv_indices, own.last_page_len, 8, 2, 128, 16, 0)
    with pytest.raises(fi.FIError) as e:
        fi.run(ws, info, own.q, own.k, own.v, torch.as_tensor(own.kv_indices, device=DEV), torch.empty_like(own.q),
               None, own.sm_scale)
    assert e.value.status == 1


@pytest.mark.parametrize("seed,kv_max,shared_min,shared_max", [
    (341, 3, 6000, 9000),   # long blocks on the tensor cores, one to three own keys per branch
    (342, 900, 0, 40),      # short blocks, long own keys
])
def test_cascade_long_blocks_or_long_suffixes(seed, kv_max, shared_min, shared_max):
    """Blocks of 20 to 28 packed rows (tensor-core units) with one-token
    branches at page 1 (multi-head units), either side the longer one; the
    merge launch behind the run waits for it, and two runs give the same
    bits."""
    d = workloads.cascade_batch(seed, [6, 7, 5], 1, kv_max, shared_max, 32, 8, 1, 16, 0, device=DEV,
                                shared_min=shared_min)
    o, lse, info, ws = cascade_run(d)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0 and info.num_cascade_merges > 0
    assert info.prefill_caches & 2  # the blocks' units run on the tensor cores
    o_ref, l_ref = oracle.attention(oracle_problem(d["flat"]))
    n = d["own"].total_qo
    err_o, err_l = compare(o[:n], lse[:n], o_ref, l_ref)
    assert err_o <= O_TOL and err_l <= LSE_TOL, (err_o, err_l)
    o2, lse2, _, _ = cascade_run(d, ws=ws, o=torch.full_like(o, float("nan")), lse=torch.full_like(lse, float("nan")))
    torch.cuda.synchronize()
    assert torch.equal(o2[:n], o[:n]) and torch.equal(lse2[:n], lse[:n])

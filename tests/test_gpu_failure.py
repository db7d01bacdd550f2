"""Failure detection on the GPU without a fault: a bounded wait that runs out
and a plan that does not match its launch both end in a status word the host
reads, and the context and the workspace stay usable afterwards."""
from __future__ import annotations

import pytest
import torch

from helpers import LSE_TOL, O_TOL, compare, gpu_run, oracle_problem
import oracle
import serving_attention_gb300 as fi
from serving_attention_gb300 import mla
import workloads

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
FI_ERR_DEVICE_CHECK, FI_ERR_TIMEOUT = 6, 7


def _tiny():
    return workloads.random_batch(901, batch=4, qo_max=1, kv_max=600, num_qo_heads=8, num_kv_heads=2, page_size=16,
                                  causal=0, device=DEV, kv_min=1)


def _check_parity(b, o, lse):
    o_ref, l_ref = oracle.attention(oracle_problem(b))
    n = b.total_qo
    err_o, err_l = compare(o[:n], lse[:n], o_ref, l_ref)
    assert err_o <= O_TOL and err_l <= LSE_TOL, (err_o, err_l)


def test_bounded_wait_runs_out_and_the_context_survives():
    b = _tiny()
    cfg = fi.default_plan_config(0)
    ws = fi.Workspace(cfg, device=DEV)
    fi.selftest_bounded_wait(ws)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == FI_ERR_TIMEOUT
    # a new plan clears the status word; the same workspace then runs normally
    o, lse, _, _ = gpu_run(b, cfg=cfg, ws=ws)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0
    _check_parity(b, o, lse)


def test_plan_that_does_not_match_the_launch_is_reported():
    b = _tiny()
    cfg = fi.default_plan_config(0)
    ws = fi.Workspace(cfg, device=DEV)
    info = fi.plan(ws, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, 8, 2, 128, 16, 0, b.num_pages)
    bad = fi.PlanInfo.from_buffer_copy(info)
    bad.num_ctas = info.num_ctas - 2  # grid no longer matches the plan's header
    kvi = torch.as_tensor(b.kv_indices, device=DEV)
    o = torch.full_like(b.q, float("nan"))
    lse = torch.full(b.q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    fi.run(ws, bad, b.q, b.k, b.v, kvi, o, lse, b.sm_scale)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == FI_ERR_DEVICE_CHECK
    assert torch.isnan(o).all()  # no CTA did any work
    o, lse, _, _ = gpu_run(b, cfg=cfg, ws=ws)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0
    _check_parity(b, o, lse)


def test_late_merge_skips_a_failed_run():
    """With split prefill units the run is followed by the late merge launch;
    when the run reports an error the merge writes nothing either."""
    b = workloads.random_batch(903, batch=3, qo_max=60, kv_max=1500, num_qo_heads=8, num_kv_heads=2,
                               page_size=16, causal=1, device=DEV, qo_min=20, kv_min=600)
    cfg = fi.default_plan_config(0, num_ctas=6, prefill_min_chunk=128, split_factor=4)
    ws = fi.Workspace(cfg, device=DEV)
    info = fi.plan(ws, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, 8, 2, 128, 16, 1, b.num_pages)
    assert info.num_late_merge_units > 0
    bad = fi.PlanInfo.from_buffer_copy(info)
    bad.num_ctas = info.num_ctas - 1
    kvi = torch.as_tensor(b.kv_indices, device=DEV)
    o = torch.full_like(b.q, float("nan"))
    lse = torch.full(b.q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    fi.run(ws, bad, b.q, b.k, b.v, kvi, o, lse, b.sm_scale)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == FI_ERR_DEVICE_CHECK
    assert torch.isnan(o).all() and torch.isnan(lse).all()
    o, lse, _, _ = gpu_run(b, cfg=cfg, ws=ws)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0
    _check_parity(b, o, lse)


def test_mla_plan_that_does_not_match_the_launch_is_reported():
    b = workloads.make_mla_batch("mla_bad", [300, 64], 128, 64, 902, device=DEV, pool_pages=8)
    cfg = mla.default_config(0)
    ws = mla.MlaWorkspace(cfg, device=DEV)
    info = mla.plan(ws, b.kv_indptr, b.kv_indices, b.last_page_len, b.num_heads, b.page_size, b.num_pages)
    bad = mla.MlaPlanInfo.from_buffer_copy(info)
    bad.num_pairs = info.num_pairs - 1
    kvi = torch.as_tensor(b.kv_indices, device=DEV)
    o = torch.empty(b.q_nope.shape, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(b.q_nope.shape[:2], dtype=torch.float32, device=DEV)
    mla.decode_run(ws, bad, b.q_nope, b.q_pe, b.ckv, b.kpe, kvi, o, lse, b.sm_scale)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == FI_ERR_DEVICE_CHECK
    # re-planned, the same workspace runs normally
    info = mla.plan(ws, b.kv_indptr, b.kv_indices, b.last_page_len, b.num_heads, b.page_size, b.num_pages)
    mla.decode_run(ws, info, b.q_nope, b.q_pe, b.ckv, b.kpe, kvi, o, lse, b.sm_scale)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0
    assert torch.isfinite(o.float()).all()


def _replanned_split_batch(num_qo_heads, num_kv_heads, seed):
    """One prefill request whose 16 query tokens meet 20,000 keys in 128-token
    chunks: each unit splits into 157 chunks of 16 * G partial rows."""
    return workloads.make_batch("many_partials", "bf16", [16], [20000], num_qo_heads, num_kv_heads, 16, 1, seed, DEV,
                                pool_pages=1260)


def test_workspace_replanned_past_the_float_workspace_is_refused():
    """The kernel compares the plan it finds in the int workspace with the
    float workspace it was launched with: a plan info taken from a small
    plan, used after the workspace was re-planned with more partial rows
    than the float workspace holds, ends in FI_ERR_DEVICE_CHECK before any
    write, and the workspace then runs normally once re-planned."""
    small = fi.default_plan_config(0, max_partial_rows=4096)
    big = fi.default_plan_config(0, prefill_min_chunk=128, split_factor=64)
    assert fi.int_workspace_bytes(small) == fi.int_workspace_bytes(big)
    ws = fi.Workspace(small, device=DEV)  # float workspace for 4096 partial rows
    b = _replanned_split_batch(32, 8, 911)
    a = workloads.llama8b_decode(device=DEV, batch=16)
    info_a = fi.plan(ws, a.qo_indptr, a.kv_indptr, a.kv_indices, a.last_page_len, 32, 8, 128, 16, 0, a.num_pages)
    assert info_a.num_partial_rows <= 4096
    ws.cfg = big
    info_b = fi.plan(ws, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, 32, 8, 128, 16, 1, b.num_pages)
    assert info_b.num_partial_rows > 4096 and info_b.num_ctas == info_a.num_ctas
    kvi = torch.as_tensor(b.kv_indices, device=DEV)
    o = torch.full_like(b.q, float("nan"))
    lse = torch.full(b.q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    stale = fi.PlanInfo.from_buffer_copy(info_a)
    stale.causal, stale.variant, stale.num_late_merge_units = info_b.causal, info_b.variant, info_b.num_late_merge_units
    fi.run(ws, stale, b.q, b.k, b.v, kvi, o, lse, b.sm_scale)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == FI_ERR_DEVICE_CHECK
    assert torch.isnan(o).all() and torch.isnan(lse).all()  # nothing written, the late merge skipped too
    ws.cfg = small
    o, lse, info, _ = gpu_run(a, cfg=small, ws=ws)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0
    _check_parity(a, o, lse)


def test_mla_workspace_replanned_past_the_float_workspace_is_refused():
    small = mla.default_config(0, max_parts=4)
    big = mla.default_config(0, min_chunk=64)
    assert mla.int_workspace_bytes(small) == mla.int_workspace_bytes(big)
    ws = mla.MlaWorkspace(small, device=DEV)
    a = workloads.make_mla_batch("mla_small", [300, 64], 128, 64, 912, device=DEV, pool_pages=8)
    info_a = mla.plan(ws, a.kv_indptr, a.kv_indices, a.last_page_len, a.num_heads, a.page_size, a.num_pages)
    assert info_a.num_parts <= 4
    b = workloads.make_mla_batch("mla_many_parts", [20000, 9000], 128, 64, 913, device=DEV, pool_pages=460)
    ws.cfg = big
    info_b = mla.plan(ws, b.kv_indptr, b.kv_indices, b.last_page_len, b.num_heads, b.page_size, b.num_pages)
    assert info_b.num_parts > 4 and info_b.num_pairs == info_a.num_pairs
    kvi = torch.as_tensor(b.kv_indices, device=DEV)
    o = torch.full(b.q_nope.shape, float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full(b.q_nope.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    mla.decode_run(ws, info_a, b.q_nope, b.q_pe, b.ckv, b.kpe, kvi, o, lse, b.sm_scale)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == FI_ERR_DEVICE_CHECK
    assert torch.isnan(o.float()).all() and torch.isnan(lse).all()  # the merge kernel skipped as well
    ws.cfg = small
    info_a = mla.plan(ws, a.kv_indptr, a.kv_indices, a.last_page_len, a.num_heads, a.page_size, a.num_pages)
    kva = torch.as_tensor(a.kv_indices, device=DEV)
    oa = torch.empty(a.q_nope.shape, dtype=torch.bfloat16, device=DEV)
    la = torch.empty(a.q_nope.shape[:2], dtype=torch.float32, device=DEV)
    mla.decode_run(ws, info_a, a.q_nope, a.q_pe, a.ckv, a.kpe, kva, oa, la, a.sm_scale)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0 and torch.isfinite(oa.float()).all()

"""fi_batch_paged_attention_run_static_scratch against fi_batch_paged_attention_run.

The static-scratch entry point serves callers that cannot allocate device
memory (no allocator reachable where they run, all memory reserved up front,
or an allocation would synchronise the device): it keeps the split-KV partial
states in a fixed array inside the library instead of a caller-provided float
workspace.  Its output must match the regular entry point's on the same plan,
call after call (the array keeps the previous call's contents), and a plan
that needs more partial rows than the array holds must be refused: by the
host before anything is enqueued, and by the kernel, before any write, when
the workspace was re-planned after the host looked at the plan info.  This
file is collected last on purpose."""
from __future__ import annotations

import ctypes

import pytest
import torch

import serving_attention_gb300 as fi
import workloads

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _outputs(b):
    o = torch.full_like(b.q, float("nan"))
    lse = torch.full(b.q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    return o, lse


@pytest.mark.parametrize("case", ["decode", "prefill"])
def test_static_scratch_matches_regular_run(case):
    if case == "decode":
        b = workloads.llama8b_decode(device=DEV, batch=16)
        cfg = fi.default_plan_config(0)
    else:  # prefill-class items split into 256-token chunks
        b = workloads.make_batch("split_prefill", "bf16", [64, 40], [1500, 700], 8, 2, 16, 1, 4242, DEV,
                                 pool_pages=160)
        cfg = fi.default_plan_config(0, prefill_min_chunk=256, split_factor=16)
    ws = fi.Workspace(cfg, device=DEV)
    info = fi.plan(ws, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, b.num_qo_heads, b.num_kv_heads,
                   128, b.page_size, b.causal, b.num_pages)
    assert 0 < info.num_partial_rows <= fi.STATIC_SCRATCH_PARTIAL_ROWS, "the case must use split-KV partial states"
    kvi = torch.as_tensor(b.kv_indices, device=DEV)
    n = b.total_qo
    o_ref, lse_ref = _outputs(b)
    fi.run(ws, info, b.q, b.k, b.v, kvi, o_ref, lse_ref, b.sm_scale)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0
    for call in range(2):
        o, lse = _outputs(b)
        fi.run_static_scratch(ws, info, b.q, b.k, b.v, kvi, o, lse, b.sm_scale)
        torch.cuda.synchronize()
        assert fi.device_status(ws) == 0, f"device status after call {call}"
        # the same kernel on the same plan, only the partial states elsewhere:
        # the same bits
        assert torch.equal(o[:n], o_ref[:n]) and torch.equal(lse[:n], lse_ref[:n]), call


def test_static_scratch_refuses_oversized_plan():
    lib = fi.load()
    info = fi.PlanInfo(num_ctas=1, head_dim=128, page_size=16, num_qo_heads=8, num_kv_heads=2,
                       num_partial_rows=fi.STATIC_SCRATCH_PARTIAL_ROWS + 1)
    ks = (ctypes.c_int64 * 3)(4096, 256, 128)
    st = lib.fi_batch_paged_attention_run_static_scratch(ctypes.byref(info), 16, 1024, 128, 4, 32, ks, 64, ks, 10, 48,
                                                         80, 1024, 128, None, fi.BF16, 0.1, 96, None)
    assert st == 3  # FI_ERR_CAPACITY, returned before anything is enqueued


def test_static_scratch_refuses_a_workspace_replanned_past_the_array():
    """The host checks the plan info it is given; a workspace re-planned
    afterwards with more partial rows than the array holds is refused by the
    kernel itself (FI_ERR_DEVICE_CHECK, nothing written), and the workspace
    runs normally once re-planned."""
    cfg = fi.default_plan_config(0, prefill_min_chunk=128, split_factor=64)
    ws = fi.Workspace(cfg, device=DEV)
    a = workloads.llama8b_decode(device=DEV, batch=16)
    info_a = fi.plan(ws, a.qo_indptr, a.kv_indptr, a.kv_indices, a.last_page_len, 32, 8, 128, 16, 0, a.num_pages)
    assert info_a.num_partial_rows <= fi.STATIC_SCRATCH_PARTIAL_ROWS
    # 8 units of 64 packed rows, each split into 157 chunks: 80,384 partial rows
    b = workloads.make_batch("many_partials", "bf16", [16], [20000], 32, 8, 16, 1, 4243, DEV, pool_pages=1260)
    info_b = fi.plan(ws, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, 32, 8, 128, 16, 1, b.num_pages)
    assert info_b.num_partial_rows > fi.STATIC_SCRATCH_PARTIAL_ROWS
    stale = fi.PlanInfo.from_buffer_copy(info_a)
    stale.causal, stale.variant, stale.num_late_merge_units = info_b.causal, info_b.variant, info_b.num_late_merge_units
    o, lse = _outputs(b)
    fi.run_static_scratch(ws, stale, b.q, b.k, b.v, torch.as_tensor(b.kv_indices, device=DEV), o, lse, b.sm_scale)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 6  # FI_ERR_DEVICE_CHECK
    assert torch.isnan(o).all() and torch.isnan(lse).all()
    info_a = fi.plan(ws, a.qo_indptr, a.kv_indptr, a.kv_indices, a.last_page_len, 32, 8, 128, 16, 0, a.num_pages)
    kva = torch.as_tensor(a.kv_indices, device=DEV)
    o_ref, lse_ref = _outputs(a)
    fi.run(ws, info_a, a.q, a.k, a.v, kva, o_ref, lse_ref, a.sm_scale)
    o, lse = _outputs(a)
    fi.run_static_scratch(ws, info_a, a.q, a.k, a.v, kva, o, lse, a.sm_scale)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0
    n = a.total_qo
    assert torch.equal(o[:n], o_ref[:n]) and torch.equal(lse[:n], lse_ref[:n])

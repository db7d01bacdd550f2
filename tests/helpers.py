"""Shared test helpers: PagedBatch -> oracle problem, GPU runs through the C ABI."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads

ORACLE_DTYPE = {"fp16": oracle.FP16, "bf16": oracle.BF16}

# Tolerances stated for the GPU path against the fp64 oracle.
O_TOL = 8e-3
LSE_TOL = 1e-3


def oracle_problem(b: workloads.PagedBatch, window_left: int = -1, sink_tokens: int = 0,
                   logits_soft_cap: float = 0.0, rope: int = 0, rope_theta: float = 10000.0,
                   rope_scale: float = 1.0) -> oracle.Problem:
    q, k, v = workloads.host_views(b)
    return oracle.Problem(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, b.num_qo_heads,
                          b.num_kv_heads, b.page_size, b.causal, b.sm_scale, ORACLE_DTYPE[b.dtype], q, k, v,
                          window_left=window_left, sink_tokens=sink_tokens, logits_soft_cap=logits_soft_cap,
                          rope=rope, rope_theta=rope_theta, rope_scale=rope_scale)


def gpu_run(b: workloads.PagedBatch, cfg=None, ws=None, stream=None, o=None, lse=None):
    """Plan + run one batch on the GPU; returns (o, lse, info, ws)."""
    import serving_attention_gb300 as fi

    dev = b.q.device
    if cfg is None:
        cfg = fi.default_plan_config(dev.index or 0)
    if ws is None:
        ws = fi.Workspace(cfg, device=dev)
    info = fi.plan(ws, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, b.num_qo_heads, b.num_kv_heads,
                   128, b.page_size, b.causal, b.num_pages, stream=stream)
    kvi = torch.as_tensor(b.kv_indices if b.kv_indices.size else np.zeros(1, np.int32), device=dev)
    if o is None:
        o = torch.full_like(b.q, float("nan"))
    if lse is None:
        lse = torch.full(b.q.shape[:2], float("nan"), dtype=torch.float32, device=dev)
    fi.run(ws, info, b.q, b.k, b.v, kvi, o, lse, b.sm_scale, stream=stream)
    return o, lse, info, ws


def compare(o_gpu: torch.Tensor, lse_gpu: torch.Tensor, o_ref: np.ndarray, lse_ref: np.ndarray):
    """Max-abs errors of O and LSE; -inf LSE must match exactly (and O there must be 0)."""
    og = o_gpu.float().cpu().numpy().astype(np.float64)
    lg = lse_gpu.cpu().numpy().astype(np.float64)
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lg), empty), "rows without visible keys disagree"
    assert np.all(np.isfinite(og)), "non-finite values in O"
    err_o = float(np.abs(og - o_ref).max()) if og.size else 0.0
    fin = ~empty
    err_l = float(np.abs(lg[fin] - lse_ref[fin]).max()) if fin.any() else 0.0
    if empty.any():
        assert np.all(og[empty] == 0.0)
    return err_o, err_l

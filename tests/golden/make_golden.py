"""Writes the regression fixtures of this folder from the oracle alone.

The pages print no worked example (no input with its attention output), so
these files are not the pages' values: they freeze what the oracle computes on
a few small seeded inputs, so that a later change to the oracle's arithmetic
shows up as a failing test and has to name the passage that justifies it.
Inputs are regenerated from their seeds by workloads.py; the fixtures store
the seeds, the shapes, and the expected outputs rounded to 12 significant
digits (far below any GPU tolerance, far above fp64 summation-order noise);
O keeps every 8th dim of each row and head (DIM_STRIDE), every LSE is kept.

    python tests/golden/make_golden.py
"""
from __future__ import annotations

import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from oracle import mla  # noqa: E402
import workloads  # noqa: E402

CASES_GQA = [
    # name, make_batch arguments (name, dtype, qo, kv, Hq, Hkv, page, causal, seed), variant kwargs
    ("decode_fp16", ("g1", "fp16", [1, 1, 1], [7, 33, 64], 4, 2, 4, 0, 11), {}),
    ("prefill_bf16_causal", ("g2", "bf16", [3, 5], [9, 5], 4, 2, 4, 1, 12), {}),
    ("window_sink_cap", ("g3", "bf16", [2, 1], [40, 17], 4, 1, 8, 1, 13),
     dict(window_left=5, sink_tokens=2, logits_soft_cap=2.0)),
    ("rope", ("g4", "bf16", [2, 1], [30, 9], 2, 2, 4, 1, 14), dict(rope=1, rope_theta=10000.0, rope_scale=1.0)),
]
CASES_MLA = [("mla_small", dict(kv_lens=[1, 70, 5], num_heads=2, page_size=8, seed=15))]
DIM_STRIDE = 8


def gqa_case(args, kw):
    b = workloads.make_batch(*args, pool_pages=None, poison=True)
    q, k, v = workloads.host_views(b)
    dt = oracle.FP16 if b.dtype == "fp16" else oracle.BF16
    p = oracle.Problem(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, b.num_qo_heads, b.num_kv_heads,
                       b.page_size, b.causal, b.sm_scale, dt, q, k, v, **kw)
    return oracle.attention(p)


def mla_case(c):
    b = workloads.make_mla_batch("golden", c["kv_lens"], c["num_heads"], c["page_size"], c["seed"],
                                 pool_pages=None)
    f = lambda t: t.double().numpy()  # noqa: E731
    return mla.mla_decode(b.kv_indptr, b.kv_indices, b.last_page_len, b.page_size, b.sm_scale, f(b.q_nope),
                          f(b.q_pe), f(b.ckv), f(b.kpe))


def _r(a):
    return [float(f"{x:.12g}") if np.isfinite(x) else str(x) for x in np.asarray(a, dtype=np.float64).ravel()]


def main():
    for name, args, kw in CASES_GQA:
        o, lse = gqa_case(args, kw)
        with open(os.path.join(HERE, f"oracle_{name}.json"), "w") as fh:
            json.dump({"kind": "gqa", "make_batch": list(args), "variant": kw, "o_shape": list(o.shape),
                       "dim_stride": DIM_STRIDE, "o": _r(o[..., ::DIM_STRIDE]), "lse": _r(lse)}, fh)
    for name, c in CASES_MLA:
        o, lse = mla_case(c)
        with open(os.path.join(HERE, f"oracle_{name}.json"), "w") as fh:
            json.dump({"kind": "mla", "case": c, "o_shape": list(o.shape), "dim_stride": DIM_STRIDE,
                       "o": _r(o[..., ::DIM_STRIDE]), "lse": _r(lse)}, fh)


if __name__ == "__main__":
    main()

"""The oracle against the regression fixtures in tests/golden (written by
tests/golden/make_golden.py from the oracle alone; the pages print no worked
example).  A change to the oracle's arithmetic fails here and has to say which
passage, or which reading of one, justifies it."""
from __future__ import annotations

import json
import os
import sys

import numpy as np
import pytest

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
sys.path.insert(0, HERE)
import make_golden  # noqa: E402

FILES = sorted(f for f in os.listdir(HERE) if f.endswith(".json"))


def _vals(lst):
    return np.array([float(x) for x in lst], dtype=np.float64)


def test_every_case_has_a_fixture():
    names = {f"oracle_{n}.json" for n, _, _ in make_golden.CASES_GQA} | {f"oracle_{n}.json" for n, _ in
                                                                          make_golden.CASES_MLA}
    assert names == set(FILES)


@pytest.mark.parametrize("fname", FILES)
def test_oracle_matches_fixture(fname):
    with open(os.path.join(HERE, fname)) as fh:
        g = json.load(fh)
    if g["kind"] == "gqa":
        o, lse = make_golden.gqa_case(tuple(g["make_batch"]), g["variant"])
    else:
        o, lse = make_golden.mla_case(g["case"])
    assert list(o.shape) == g["o_shape"]
    o_ref, l_ref = _vals(g["o"]), _vals(g["lse"])
    got_o, got_l = o[..., ::g["dim_stride"]].ravel(), lse.ravel()
    assert np.array_equal(np.isneginf(got_l), np.isneginf(l_ref))
    fin = np.isfinite(l_ref)
    np.testing.assert_allclose(got_l[fin], l_ref[fin], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(got_o, o_ref, rtol=1e-11, atol=1e-12)

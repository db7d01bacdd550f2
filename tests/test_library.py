"""The C-ABI library loads on a machine without a GPU, exports every symbol its
header declares, and rejects bad arguments on the host before touching CUDA."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import serving_attention_gb300 as fi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            names |= set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(fi_[a-z_0-9]+)\s*\(", text, re.M))
    return names


def test_exports_every_declared_symbol():
    lib = fi.load()
    names = _declared()
    assert {"fi_plan", "fi_batch_paged_attention_run", "fi_merge_states"} <= names
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert set(fi.EXPORTS) <= names


def test_status_strings():
    lib = fi.load()
    for s in range(8):
        assert lib.fi_status_string(s)


def test_run_rejects_bad_arguments_before_cuda():
    lib = fi.load()
    info = fi.PlanInfo(num_ctas=1, head_dim=128, page_size=16, num_qo_heads=8, num_kv_heads=2)
    ks = (ctypes.c_int64 * 3)(4096, 256, 128)
    args = [ctypes.byref(info), 16, 1024, 128, 4, 32, ks, 64, ks, 10, 48, 80, 1024, 128, None, fi.BF16, 0.1, 96,
            112, None]
    # the pointers are fake: only argument checks that return before any CUDA call are exercised
    bad = list(args)
    bad[0] = None
    assert lib.fi_batch_paged_attention_run(*bad) == 1
    bad = list(args)
    bad[1] = 18  # misaligned q
    assert lib.fi_batch_paged_attention_run(*bad) == 4
    bad = list(args)
    bad[15] = fi.FP32
    assert lib.fi_batch_paged_attention_run(*bad) == 2
    bad = list(args)
    bad[6] = (ctypes.c_int64 * 3)(4096, 250, 128)  # stride not a multiple of 16 bytes
    assert lib.fi_batch_paged_attention_run(*bad) == 4


def test_merge_rejects_bad_arguments_before_cuda():
    lib = fi.load()
    assert lib.fi_merge_states(None, 16, 32, 48, 64, 80, 4, 2, 128, fi.BF16, None) == 1
    assert lib.fi_merge_states(16, 16, 32, 48, 64, 80, 4, 2, 64, fi.BF16, None) == 2
    assert lib.fi_merge_states(18, 16, 32, 48, 64, 80, 4, 2, 128, fi.BF16, None) == 4
    assert lib.fi_merge_states(16, 16, 32, 48, 64, 80, 0, 2, 128, fi.BF16, None) == 0  # nothing to do


def test_workspace_sizes():
    cfg = fi.make_plan_config(152)
    assert fi.int_workspace_bytes(cfg) % 16 == 0
    assert fi.float_workspace_bytes(cfg, 128) >= cfg.max_partial_rows * 129 * 4


def test_mla_run_rejects_bad_arguments_before_cuda():
    from serving_attention_gb300 import mla

    lib = mla.load()
    info = mla.MlaPlanInfo(num_pairs=2, batch=2, num_heads=128, page_size=64, max_parts=4)
    # fake, 16-byte aligned pointers: only checks that return before any CUDA call run
    args = [ctypes.byref(info), 16, 65536, 512, 32, 8192, 64, 2, 48, 32768, 512, 64, 4096, 64, 10, 80, 96, 112,
            0.07, 128, 144, None]
    bad = list(args)
    bad[0] = None
    assert lib.fi_mla_decode_run(*bad) == 1                     # no plan info
    bad = list(args)
    bad[7] = 1
    assert lib.fi_mla_decode_run(*bad) == 1                     # fewer query rows than the plan's batch
    bad = list(args)
    bad[1] = 24
    assert lib.fi_mla_decode_run(*bad) == 4                     # misaligned q_nope
    bad = list(args)
    bad[10] = 500
    assert lib.fi_mla_decode_run(*bad) == 4                     # slot stride not a multiple of 16 bytes
    info_bad = mla.MlaPlanInfo(num_pairs=2, batch=2, num_heads=128, page_size=4, max_parts=4)
    bad = list(args)
    bad[0] = ctypes.byref(info_bad)
    assert lib.fi_mla_decode_run(*bad) == 2                     # page size 4
    info_bad = mla.MlaPlanInfo(num_pairs=2, batch=2, num_heads=129, page_size=64, max_parts=4)
    bad[0] = ctypes.byref(info_bad)
    assert lib.fi_mla_decode_run(*bad) == 2                     # more than 128 heads
    info_split = mla.MlaPlanInfo(num_pairs=2, batch=2, num_heads=128, page_size=64, max_parts=4, num_parts=3)
    bad = list(args)
    bad[0] = ctypes.byref(info_split)
    bad[20] = None
    assert lib.fi_mla_decode_run(*bad) == 1                     # split chunks need the float workspace


def test_rope_utilities_reject_bad_arguments_before_cuda():
    """The rotation passes refuse, before any CUDA call: a plan without RoPE,
    a cascade plan (two caches), misaligned buffers and unsupported types."""
    lib = fi.load()
    rope = fi.PlanInfo(num_ctas=1, batch=1, head_dim=128, page_size=16, num_qo_heads=8, num_kv_heads=2, variant=4)
    plain = fi.PlanInfo(num_ctas=1, batch=1, head_dim=128, page_size=16, num_qo_heads=8, num_kv_heads=2, variant=0)
    cascade = fi.PlanInfo(num_ctas=1, batch=2, head_dim=128, page_size=16, num_qo_heads=8, num_kv_heads=2,
                          variant=4, num_shared=1)
    ks = (ctypes.c_int64 * 3)(4096, 256, 128)
    # fake pointers: every case returns before touching memory
    assert lib.fi_rope_apply_k(ctypes.byref(plain), 16, 32, ks, 48, ks, 64, fi.BF16, None) == 1
    assert lib.fi_rope_apply_k(ctypes.byref(cascade), 16, 32, ks, 48, ks, 64, fi.BF16, None) == 1
    assert lib.fi_rope_apply_k(ctypes.byref(rope), 16, 34, ks, 48, ks, 64, fi.BF16, None) == 4
    assert lib.fi_rope_apply_k(ctypes.byref(rope), 16, 32, ks, 48, ks, 64, fi.FP32, None) == 2
    assert lib.fi_rope_apply_q(ctypes.byref(plain), 16, 32, 1024, 128, 48, 1024, 128, fi.BF16, None) == 1
    assert lib.fi_rope_apply_q(ctypes.byref(cascade), 16, 32, 1024, 128, 48, 1024, 128, fi.BF16, None) == 1
    assert lib.fi_rope_apply_q(ctypes.byref(rope), 16, 32, 1020, 128, 48, 1024, 128, fi.BF16, None) == 4
    assert lib.fi_rope_apply_q(ctypes.byref(rope), None, 32, 1024, 128, 48, 1024, 128, fi.BF16, None) == 1


def test_prerotated_run_rejects_bad_arguments_before_cuda():
    """The pre-rotated run needs a RoPE plan and both rotation buffers, and
    refuses a cascade plan (it reads one cache)."""
    lib = fi.load()
    ks = (ctypes.c_int64 * 3)(4096, 256, 128)

    def call(info, q_rot=208, k_rot=224):
        return lib.fi_batch_paged_attention_run_rope_prerotated(
            ctypes.byref(info), 16, 1024, 128, 4, 32, ks, 64, ks, 10, 48, q_rot, 1024, 128, k_rot, ks, 80, 1024, 128,
            None, fi.BF16, 0.1, 96, 112, None)

    rope = fi.PlanInfo(num_ctas=1, batch=1, head_dim=128, page_size=16, num_qo_heads=8, num_kv_heads=2, variant=4)
    plain = fi.PlanInfo(num_ctas=1, batch=1, head_dim=128, page_size=16, num_qo_heads=8, num_kv_heads=2, variant=0)
    cascade = fi.PlanInfo(num_ctas=1, batch=2, head_dim=128, page_size=16, num_qo_heads=8, num_kv_heads=2,
                          variant=4, num_shared=1)
    assert call(rope, q_rot=None) == 1
    assert call(rope, k_rot=None) == 1
    assert call(cascade) == 1
    # (a plan without RoPE and misaligned rotation buffers are refused after
    # the tensor maps are built, which needs the CUDA driver: GPU tests)
    del plain

"""The oracle: plain, slow, fp64 CPU reference of paged batched attention.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's CPU
baseline leg may import this package.  It shares no code with the CUDA library
(`serving_attention_gb300`) and never imports it.

* `attention` / `attention_select` -- attn_oracle.c: the definition of the
  result, walking the page table (see that file's header for the passages).
* `merge_states` -- attn_oracle.c: the LSE-weighted merge of two states.
* `plan_ref.make_plan` -- the plan rule restated in Python.
* `mla.mla_decode` -- absorbed-MLA decode (latent cache), numpy fp64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liborc.so")
_lock = threading.Lock()
_lib = None

FP16, BF16, FP32 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile attn_oracle.c with gcc (-O2, OpenMP) into oracle/_build/liborc.so."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Problem(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("qo_indptr", ctypes.c_void_p),
        ("kv_indptr", ctypes.c_void_p),
        ("kv_indices", ctypes.c_void_p),
        ("last_page_len", ctypes.c_void_p),
        ("num_qo_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("causal", ctypes.c_int32),
        ("sm_scale", ctypes.c_double),
        ("dtype", ctypes.c_int32),
        ("q", ctypes.c_void_p),
        ("q_stride_tok", ctypes.c_int64),
        ("q_stride_head", ctypes.c_int64),
        ("k", ctypes.c_void_p),
        ("k_stride_page", ctypes.c_int64),
        ("k_stride_slot", ctypes.c_int64),
        ("k_stride_head", ctypes.c_int64),
        ("v", ctypes.c_void_p),
        ("v_stride_page", ctypes.c_int64),
        ("v_stride_slot", ctypes.c_int64),
        ("v_stride_head", ctypes.c_int64),
        ("window_left", ctypes.c_int32),
        ("sink_tokens", ctypes.c_int32),
        ("logits_soft_cap", ctypes.c_double),
        ("rope", ctypes.c_int32),
        ("rope_theta", ctypes.c_double),
        ("rope_scale", ctypes.c_double),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.POINTER(_Problem)
            vp = ctypes.c_void_p
            lib.orc_attention_all.argtypes = [P, vp, vp]
            lib.orc_attention_all.restype = ctypes.c_int
            lib.orc_attention_select.argtypes = [P, ctypes.c_int64, vp, vp, vp, vp]
            lib.orc_attention_select.restype = ctypes.c_int
            lib.orc_merge_states.argtypes = [ctypes.c_int64, ctypes.c_int32, vp, vp, vp, vp, vp, vp]
            lib.orc_merge_states.restype = None
            lib.orc_decode_fp16.argtypes = [ctypes.c_uint16]
            lib.orc_decode_fp16.restype = ctypes.c_double
            lib.orc_decode_bf16.argtypes = [ctypes.c_uint16]
            lib.orc_decode_bf16.restype = ctypes.c_double
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _elem_strides(a: np.ndarray):
    st = [s // a.itemsize for s in a.strides]
    if any(s * a.itemsize != b for s, b in zip(st, a.strides)) or st[-1] != 1:
        raise ValueError("oracle needs element-aligned strides and a contiguous last dimension")
    return st


def _check_storage(a: np.ndarray, dtype: int):
    want = np.float32 if dtype == FP32 else np.uint16
    if a.dtype != want:
        raise TypeError(f"dtype code {dtype} needs {np.dtype(want)} storage, got {a.dtype}")


class Problem:
    """One batch: host int32 index arrays, q/k/v storage (uint16 bit patterns
    for fp16/bf16, float32 for fp32) with arbitrary element strides."""

    def __init__(self, qo_indptr, kv_indptr, kv_indices, last_page_len, num_qo_heads, num_kv_heads,
                 page_size, causal, sm_scale, dtype, q, k, v, window_left=-1, sink_tokens=0, logits_soft_cap=0.0,
                 rope=0, rope_theta=10000.0, rope_scale=1.0):
        self.qo_indptr = np.ascontiguousarray(qo_indptr, dtype=np.int32)
        self.kv_indptr = np.ascontiguousarray(kv_indptr, dtype=np.int32)
        self.kv_indices = np.ascontiguousarray(kv_indices, dtype=np.int32)
        self.last_page_len = np.ascontiguousarray(last_page_len, dtype=np.int32)
        for a in (q, k, v):
            _check_storage(a, dtype)
        if q.ndim != 3 or k.ndim != 4 or v.ndim != 4:
            raise ValueError("q is [tokens, Hq, d]; k and v are [pages, page_size, Hkv, d]")
        self.q, self.k, self.v = q, k, v
        qs, ks, vs = _elem_strides(q), _elem_strides(k), _elem_strides(v)
        batch = len(self.qo_indptr) - 1
        if len(self.kv_indptr) != batch + 1 or len(self.last_page_len) < batch:
            raise ValueError("index array lengths disagree")
        if k.shape[1] != page_size or v.shape[1] != page_size:
            raise ValueError("page_size disagrees with the cache shape")
        self.num_qo_heads = num_qo_heads
        self.head_dim = q.shape[2]
        self._c = _Problem(batch, _ptr(self.qo_indptr), _ptr(self.kv_indptr),
                           _ptr(self.kv_indices) if self.kv_indices.size else 0, _ptr(self.last_page_len),
                           num_qo_heads, num_kv_heads, q.shape[2], page_size, int(causal), float(sm_scale),
                           dtype, _ptr(q), qs[0], qs[1], _ptr(k), ks[0], ks[1], ks[2], _ptr(v), vs[0], vs[1],
                           vs[2], int(window_left), int(sink_tokens), float(logits_soft_cap), int(rope),
                           float(rope_theta), float(rope_scale))
        if rope and q.shape[2] > 512:
            raise ValueError("the oracle's RoPE path holds at most 512 dims")

    @property
    def num_rows(self) -> int:
        return int(self.qo_indptr[-1])


def attention(p: Problem):
    """All rows: returns (o [rows, Hq, d] fp64, lse [rows, Hq] fp64)."""
    lib = _load()
    o = np.zeros((p.num_rows, p.num_qo_heads, p.head_dim), dtype=np.float64)
    lse = np.zeros((p.num_rows, p.num_qo_heads), dtype=np.float64)
    if p.num_rows:
        if lib.orc_attention_all(ctypes.byref(p._c), _ptr(o), _ptr(lse)) != 0:
            raise MemoryError("oracle scratch allocation failed")
    return o, lse


def attention_select(p: Problem, rows, heads):
    """Selected (row, head) pairs: returns (o [n, d] fp64, lse [n] fp64)."""
    lib = _load()
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    heads = np.ascontiguousarray(heads, dtype=np.int32)
    n = rows.size
    o = np.zeros((n, p.head_dim), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    if n:
        rc = lib.orc_attention_select(ctypes.byref(p._c), n, _ptr(rows), _ptr(heads), _ptr(o), _ptr(lse))
        if rc != 0:
            raise ValueError(f"oracle select failed ({rc})")
    return o, lse


def merge_states(o_a, s_a, o_b, s_b):
    """Merge two fp64 states row by row: o [..., d], s [...]."""
    lib = _load()
    o_a = np.ascontiguousarray(o_a, dtype=np.float64)
    o_b = np.ascontiguousarray(o_b, dtype=np.float64)
    s_a = np.ascontiguousarray(s_a, dtype=np.float64)
    s_b = np.ascontiguousarray(s_b, dtype=np.float64)
    d = o_a.shape[-1]
    n = s_a.size
    o = np.empty_like(o_a)
    s = np.empty_like(s_a)
    lib.orc_merge_states(n, d, _ptr(o_a), _ptr(s_a), _ptr(o_b), _ptr(s_b), _ptr(o), _ptr(s))
    return o, s


def decode_fp16(bits: int) -> float:
    return _load().orc_decode_fp16(bits)


def decode_bf16(bits: int) -> float:
    return _load().orc_decode_bf16(bits)

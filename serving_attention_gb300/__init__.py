"""Python binding of libfi_gb300 (paged, block-sparse batched attention on sm_103a).

Argument marshalling only: torch supplies device memory, pinned host memory and
streams; every step of the hot path runs in the library's CUDA kernels (the
planner runs on the host, as the plan/run split prescribes).  There is no CPU
fallback: if the shared library is missing or fails to load, every call
raises.

    cfg = default_plan_config(0)
    ws = Workspace(cfg)
    info = plan(ws, qo_indptr, kv_indptr, kv_indices, last_page_len, 32, 8, 128, 16, causal=0)
    run(ws, info, q, k_cache, v_cache, kv_indices_dev, o, lse, sm_scale)
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import _build

FP16, BF16, FP32 = 0, 1, 2
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "capacity", 4: "alignment", 5: "cuda error",
          6: "device check failed", 7: "device timeout"}
_DTYPE = {torch.float16: FP16, torch.bfloat16: BF16, torch.float32: FP32}


class FIError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS.get(status, status)} ({status})")
        self.status = status


class PlanConfig(ctypes.Structure):
    _fields_ = [("num_ctas", ctypes.c_int32), ("max_batch", ctypes.c_int32), ("max_items", ctypes.c_int32),
                ("max_merge_units", ctypes.c_int32), ("max_partial_rows", ctypes.c_int64),
                ("decode_min_chunk", ctypes.c_int32), ("prefill_min_chunk", ctypes.c_int32),
                ("decode_cost_weight", ctypes.c_int32), ("prefill_cost_weight", ctypes.c_int32),
                ("split_factor", ctypes.c_int32), ("window_left", ctypes.c_int32), ("sink_tokens", ctypes.c_int32),
                ("logits_soft_cap", ctypes.c_float), ("rope_max_positions", ctypes.c_int32),
                ("rope_theta", ctypes.c_float), ("rope_scale", ctypes.c_float), ("reserved", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {f: getattr(self, f) for f, _ in self._fields_ if f != "reserved"}


class PlanInfo(ctypes.Structure):
    _fields_ = [("num_ctas", ctypes.c_int32), ("num_items", ctypes.c_int32), ("num_merge_units", ctypes.c_int32),
                ("batch", ctypes.c_int32), ("num_partial_rows", ctypes.c_int64), ("num_qo_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("causal", ctypes.c_int32), ("chunk_decode", ctypes.c_int32), ("chunk_prefill", ctypes.c_int32),
                ("num_decode_items", ctypes.c_int32), ("num_prefill_items", ctypes.c_int32),
                ("variant", ctypes.c_int32), ("int_ws_bytes_used", ctypes.c_int64),
                ("max_partial_rows", ctypes.c_int64), ("num_late_merge_units", ctypes.c_int32),
                ("num_shared", ctypes.c_int32), ("num_cascade_merges", ctypes.c_int32),
                ("prefill_caches", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {f: getattr(self, f) for f, _ in self._fields_}


EXPORTS = ["fi_default_plan_config", "fi_int_workspace_bytes", "fi_float_workspace_bytes", "fi_plan",
           "fi_plan_host", "fi_plan_cascade", "fi_plan_cascade_host", "fi_batch_paged_attention_run",
           "fi_batch_paged_attention_run_cascade", "fi_batch_paged_attention_run_rope_prerotated",
           "fi_batch_paged_attention_run_static_scratch",
           "fi_merge_states", "fi_get_device_status", "fi_status_string", "fi_rope_init", "fi_rope_apply_k",
           "fi_rope_apply_q", "fi_selftest_bounded_wait"]

_lib = None


def load(build_if_stale: bool = True) -> ctypes.CDLL:
    """Load libfi_gb300.so (building it in-tree first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build() if build_if_stale else _build.LIB_PATH
    lib = ctypes.CDLL(path)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    cfgp, infop = ctypes.POINTER(PlanConfig), ctypes.POINTER(PlanInfo)
    lib.fi_default_plan_config.argtypes = [ctypes.c_int, cfgp]
    lib.fi_int_workspace_bytes.argtypes = [cfgp]
    lib.fi_int_workspace_bytes.restype = sz
    lib.fi_float_workspace_bytes.argtypes = [cfgp, i32]
    lib.fi_float_workspace_bytes.restype = sz
    lib.fi_plan.argtypes = [cfgp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp, sz, vp, infop]
    lib.fi_plan_host.argtypes = [cfgp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, sz, infop]
    lib.fi_plan_cascade_host.argtypes = [cfgp, vp, vp, vp, vp, i32, i32, i32, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                         i32, i32, vp, sz, infop]
    lib.fi_plan_cascade.argtypes = [cfgp, vp, vp, vp, vp, i32, i32, i32, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                    i32, vp, vp, sz, vp, infop]
    lib.fi_batch_paged_attention_run_rope_prerotated.argtypes = [infop, vp, i64, i64, i32, vp, vp, vp, vp, i32, vp, vp,
                                                                 i64, i64, vp, vp, vp, i64, i64, vp, ctypes.c_int,
                                                                 ctypes.c_float, vp, vp, vp]
    lib.fi_batch_paged_attention_run_cascade.argtypes = [infop, vp, i64, i64, i32, vp, vp, vp, vp, i32, vp, vp, vp,
                                                         vp, vp, i32, vp, i32, vp, i64, i64, vp, ctypes.c_int,
                                                         ctypes.c_float, vp, vp, vp]
    lib.fi_batch_paged_attention_run.argtypes = [infop, vp, i64, i64, i32, vp, vp, vp, vp, i32, vp, vp, i64, i64,
                                                 vp, ctypes.c_int, ctypes.c_float, vp, vp, vp]
    lib.fi_batch_paged_attention_run_static_scratch.argtypes = [infop, vp, i64, i64, i32, vp, vp, vp, vp, i32, vp, vp,
                                                                i64, i64, vp, ctypes.c_int, ctypes.c_float, vp, vp]
    lib.fi_batch_paged_attention_run_static_scratch.restype = ctypes.c_int
    lib.fi_merge_states.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, ctypes.c_int, vp]
    lib.fi_get_device_status.argtypes = [vp, vp, ctypes.POINTER(i32)]
    lib.fi_rope_init.argtypes = [cfgp, vp, vp]
    lib.fi_rope_apply_k.argtypes = [infop, vp, vp, vp, vp, vp, vp, ctypes.c_int, vp]
    lib.fi_rope_apply_q.argtypes = [infop, vp, vp, i64, i64, vp, i64, i64, ctypes.c_int, vp]
    lib.fi_selftest_bounded_wait.argtypes = [vp, vp]
    lib.fi_selftest_bounded_wait.restype = ctypes.c_int
    lib.fi_status_string.argtypes = [ctypes.c_int]
    lib.fi_status_string.restype = ctypes.c_char_p
    for name in ("fi_default_plan_config", "fi_plan", "fi_plan_host", "fi_plan_cascade", "fi_plan_cascade_host",
                 "fi_batch_paged_attention_run", "fi_batch_paged_attention_run_cascade",
                 "fi_batch_paged_attention_run_rope_prerotated", "fi_merge_states",
                 "fi_get_device_status", "fi_rope_init", "fi_rope_apply_k", "fi_rope_apply_q"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _check(status: int, where: str):
    if status != 0:
        raise FIError(status, where)


def _stream_ptr(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=np.int32)


def default_plan_config(device: int = 0, **overrides) -> PlanConfig:
    cfg = PlanConfig()
    _check(load().fi_default_plan_config(device, ctypes.byref(cfg)), "fi_default_plan_config")
    for k, v in overrides.items():
        setattr(cfg, k, v)
    return cfg


def make_plan_config(num_ctas: int, **overrides) -> PlanConfig:
    """A config without asking the device (host-side planning and tests)."""
    cfg = PlanConfig(num_ctas=num_ctas, max_batch=8192, max_items=1 << 17, max_merge_units=1 << 15,
                     max_partial_rows=1 << 19, decode_min_chunk=256, prefill_min_chunk=1024, decode_cost_weight=8,
                     prefill_cost_weight=9, split_factor=1, window_left=-1, sink_tokens=0, logits_soft_cap=0.0,
                     rope_max_positions=0, rope_theta=10000.0, rope_scale=1.0)
    for k, v in overrides.items():
        setattr(cfg, k, v)
    return cfg


def int_workspace_bytes(cfg: PlanConfig) -> int:
    return int(load().fi_int_workspace_bytes(ctypes.byref(cfg)))


def float_workspace_bytes(cfg: PlanConfig, head_dim: int = 128) -> int:
    return int(load().fi_float_workspace_bytes(ctypes.byref(cfg), head_dim))


class Workspace:
    """Device int/float workspaces plus two pinned staging buffers for plans."""

    def __init__(self, cfg: PlanConfig, head_dim: int = 128, device="cuda"):
        self.cfg = cfg
        self.device = torch.device(device)
        ib, fb = int_workspace_bytes(cfg), float_workspace_bytes(cfg, head_dim)
        self.int_ws = torch.zeros((ib + 15) // 16 * 4, dtype=torch.int32, device=self.device)
        self.float_ws = torch.zeros((fb + 15) // 16 * 4, dtype=torch.float32, device=self.device)
        self._staging = [torch.empty(ib, dtype=torch.uint8, pin_memory=True) for _ in range(2)]
        self._events = [None, None]
        self._next = 0
        if cfg.rope_max_positions > 0:  # the RoPE cos/sin table lives in the int workspace
            with torch.cuda.device(self.device):
                _check(load().fi_rope_init(ctypes.byref(cfg), self.int_ws.data_ptr(), _stream_ptr(None)),
                       "fi_rope_init")


def plan_host(cfg: PlanConfig, qo_indptr, kv_indptr, kv_indices, last_page_len, num_qo_heads: int,
              num_kv_heads: int, head_dim: int, page_size: int, causal: int, num_pages: int = 0):
    """Host-only planning: returns (status, int32 workspace image or None, PlanInfo)."""
    lib = load()
    qo, kvp, kvi, lpl = _i32(qo_indptr), _i32(kv_indptr), _i32(kv_indices), _i32(last_page_len)
    nbytes = int_workspace_bytes(cfg)
    buf = np.zeros(nbytes // 4, dtype=np.int32)
    info = PlanInfo()
    st = lib.fi_plan_host(ctypes.byref(cfg), qo.ctypes.data, kvp.ctypes.data, kvi.ctypes.data if kvi.size else None,
                          lpl.ctypes.data if lpl.size else None, len(qo) - 1, num_qo_heads, num_kv_heads, head_dim,
                          page_size, causal, num_pages, buf.ctypes.data, nbytes, ctypes.byref(info))
    if st != 0:
        return st, None, info
    return st, buf[:info.int_ws_bytes_used // 4].copy(), info


def plan(ws: Workspace, qo_indptr, kv_indptr, kv_indices, last_page_len, num_qo_heads: int, num_kv_heads: int,
         head_dim: int, page_size: int, causal: int, num_pages: int = 0, stream=None) -> PlanInfo:
    """Plan on the host and enqueue the copy of the work list into ws.int_ws."""
    lib = load()
    qo, kvp, kvi, lpl = _i32(qo_indptr), _i32(kv_indptr), _i32(kv_indices), _i32(last_page_len)
    i = ws._next
    ws._next ^= 1
    if ws._events[i] is not None:
        ws._events[i].synchronize()  # the staging buffer's previous copy has landed
    info = PlanInfo()
    staging = ws._staging[i]
    st = lib.fi_plan(ctypes.byref(ws.cfg), qo.ctypes.data, kvp.ctypes.data, kvi.ctypes.data if kvi.size else None,
                     lpl.ctypes.data if lpl.size else None, len(qo) - 1, num_qo_heads, num_kv_heads, head_dim,
                     page_size, causal, num_pages, ws.int_ws.data_ptr(), staging.data_ptr(), staging.numel(),
                     _stream_ptr(stream), ctypes.byref(info))
    _check(st, "fi_plan")
    ev = torch.cuda.Event()
    ev.record(stream if stream is not None else torch.cuda.current_stream())
    ws._events[i] = ev
    return info


def _ptr_or_none(a: np.ndarray):
    return a.ctypes.data if a.size else None


def _cascade_args(shared_qo_indptr, shared_kv_indptr, shared_kv_indices, shared_last_page_len, shared_page_size,
                  shared_num_pages, qo_indptr, kv_indptr, kv_indices, last_page_len):
    arrs = [_i32(a) for a in (shared_qo_indptr, shared_kv_indptr, shared_kv_indices, shared_last_page_len,
                              qo_indptr, kv_indptr, kv_indices, last_page_len)]
    sqo, skvp, skvi, slpl, qo, kvp, kvi, lpl = arrs
    head = [sqo.ctypes.data, skvp.ctypes.data, _ptr_or_none(skvi), _ptr_or_none(slpl), len(sqo) - 1,
            shared_page_size, shared_num_pages, qo.ctypes.data, kvp.ctypes.data, _ptr_or_none(kvi),
            _ptr_or_none(lpl), len(qo) - 1]
    return arrs, head


def plan_cascade_host(cfg: PlanConfig, shared_qo_indptr, shared_kv_indptr, shared_kv_indices, shared_last_page_len,
                      shared_page_size: int, qo_indptr, kv_indptr, kv_indices, last_page_len, num_qo_heads: int,
                      num_kv_heads: int, head_dim: int, page_size: int, causal: int, num_pages: int = 0,
                      shared_num_pages: int = 0):
    """Host-only two-level (cascade) planning: (status, int32 workspace image or None, PlanInfo)."""
    keep, head = _cascade_args(shared_qo_indptr, shared_kv_indptr, shared_kv_indices, shared_last_page_len,
                               shared_page_size, shared_num_pages, qo_indptr, kv_indptr, kv_indices, last_page_len)
    nbytes = int_workspace_bytes(cfg)
    buf = np.zeros(nbytes // 4, dtype=np.int32)
    info = PlanInfo()
    st = load().fi_plan_cascade_host(ctypes.byref(cfg), *head, num_qo_heads, num_kv_heads, head_dim, page_size,
                                     causal, num_pages, buf.ctypes.data, nbytes, ctypes.byref(info))
    del keep
    if st != 0:
        return st, None, info
    return st, buf[:info.int_ws_bytes_used // 4].copy(), info


def plan_cascade(ws: Workspace, shared_qo_indptr, shared_kv_indptr, shared_kv_indices, shared_last_page_len,
                 shared_page_size: int, qo_indptr, kv_indptr, kv_indices, last_page_len, num_qo_heads: int,
                 num_kv_heads: int, head_dim: int, page_size: int, causal: int, num_pages: int = 0,
                 shared_num_pages: int = 0, stream=None) -> PlanInfo:
    """Plan a two-level (cascade) batch and enqueue the copy of the work list into ws.int_ws."""
    keep, head = _cascade_args(shared_qo_indptr, shared_kv_indptr, shared_kv_indices, shared_last_page_len,
                               shared_page_size, shared_num_pages, qo_indptr, kv_indptr, kv_indices, last_page_len)
    i = ws._next
    ws._next ^= 1
    if ws._events[i] is not None:
        ws._events[i].synchronize()  # the staging buffer's previous copy has landed
    info = PlanInfo()
    staging = ws._staging[i]
    st = load().fi_plan_cascade(ctypes.byref(ws.cfg), *head, num_qo_heads, num_kv_heads, head_dim, page_size, causal,
                                num_pages, ws.int_ws.data_ptr(), staging.data_ptr(), staging.numel(),
                                _stream_ptr(stream), ctypes.byref(info))
    del keep
    _check(st, "fi_plan_cascade")
    ev = torch.cuda.Event()
    ev.record(stream if stream is not None else torch.cuda.current_stream())
    ws._events[i] = ev
    return info


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPE:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return _DTYPE[t.dtype]


def run(ws: Workspace, info: PlanInfo, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
        kv_indices_dev: torch.Tensor, o: torch.Tensor, lse: torch.Tensor | None, sm_scale: float, stream=None):
    """Enqueue the persistent attention kernel for the current plan of `ws`."""
    lib = load()
    if kv_indices_dev.dtype != torch.int32 or not kv_indices_dev.is_contiguous():
        raise TypeError("kv_indices must be a contiguous int32 device tensor")
    if lse is not None and (lse.dtype != torch.float32 or not lse.is_contiguous()):
        raise TypeError("lse must be contiguous fp32")
    if q.dtype != k_cache.dtype or q.dtype != v_cache.dtype or q.dtype != o.dtype:
        raise TypeError("q, k, v and o must share one dtype")
    ks = (ctypes.c_int64 * 3)(*k_cache.stride()[:3])
    vs = (ctypes.c_int64 * 3)(*v_cache.stride()[:3])
    st = lib.fi_batch_paged_attention_run(
        ctypes.byref(info), q.data_ptr(), q.stride(0), q.stride(1), q.shape[0], k_cache.data_ptr(), ks,
        v_cache.data_ptr(), vs, k_cache.shape[0], kv_indices_dev.data_ptr(), o.data_ptr(), o.stride(0), o.stride(1),
        lse.data_ptr() if lse is not None else None, _dtype_code(q), float(sm_scale), ws.int_ws.data_ptr(),
        ws.float_ws.data_ptr(), _stream_ptr(stream))
    _check(st, "fi_batch_paged_attention_run")


def run_rope_prerotated(ws: Workspace, info: PlanInfo, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                        kv_indices_dev: torch.Tensor, q_rot: torch.Tensor, k_rot: torch.Tensor, o: torch.Tensor,
                        lse: torch.Tensor | None, sm_scale: float, stream=None):
    """run() of a RoPE plan with the queries and keys of prefill-class
    requests rotated once into q_rot and k_rot (fp16, the shapes of q and the
    cache) before the kernel."""
    if kv_indices_dev.dtype != torch.int32 or not kv_indices_dev.is_contiguous():
        raise TypeError("kv_indices must be a contiguous int32 device tensor")
    if lse is not None and (lse.dtype != torch.float32 or not lse.is_contiguous()):
        raise TypeError("lse must be contiguous fp32")
    if q.dtype != k_cache.dtype or q.dtype != v_cache.dtype or q.dtype != o.dtype:
        raise TypeError("q, k, v and o share one dtype")
    if k_rot.dtype != torch.float16 or q_rot.dtype != torch.float16:
        raise TypeError("q_rot and k_rot are fp16")
    ks = (ctypes.c_int64 * 3)(*k_cache.stride()[:3])
    vs = (ctypes.c_int64 * 3)(*v_cache.stride()[:3])
    rs = (ctypes.c_int64 * 3)(*k_rot.stride()[:3])
    st = load().fi_batch_paged_attention_run_rope_prerotated(
        ctypes.byref(info), q.data_ptr(), q.stride(0), q.stride(1), q.shape[0], k_cache.data_ptr(), ks,
        v_cache.data_ptr(), vs, k_cache.shape[0], kv_indices_dev.data_ptr(), q_rot.data_ptr(), q_rot.stride(0),
        q_rot.stride(1), k_rot.data_ptr(), rs, o.data_ptr(),
        o.stride(0), o.stride(1), lse.data_ptr() if lse is not None else None, _dtype_code(q), float(sm_scale),
        ws.int_ws.data_ptr(), ws.float_ws.data_ptr(), _stream_ptr(stream))
    _check(st, "fi_batch_paged_attention_run_rope_prerotated")


def run_cascade(ws: Workspace, info: PlanInfo, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                kv_indices_dev: torch.Tensor, shared_k: torch.Tensor, shared_v: torch.Tensor,
                shared_kv_indices_dev: torch.Tensor, o: torch.Tensor, lse: torch.Tensor | None, sm_scale: float,
                stream=None):
    """Enqueue the run of a two-level (cascade) plan: the requests' own cache
    (k_cache, v_cache, kv_indices_dev) and the shared blocks' cache (shared_k,
    shared_v, shared_kv_indices_dev), then the cascade merge."""
    for t in (kv_indices_dev, shared_kv_indices_dev):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise TypeError("page tables must be contiguous int32 device tensors")
    if lse is not None and (lse.dtype != torch.float32 or not lse.is_contiguous()):
        raise TypeError("lse must be contiguous fp32")
    if any(t.dtype != q.dtype for t in (k_cache, v_cache, shared_k, shared_v, o)):
        raise TypeError("q, the caches and o must share one dtype")
    ks = (ctypes.c_int64 * 3)(*k_cache.stride()[:3])
    vs = (ctypes.c_int64 * 3)(*v_cache.stride()[:3])
    sks = (ctypes.c_int64 * 3)(*shared_k.stride()[:3])
    svs = (ctypes.c_int64 * 3)(*shared_v.stride()[:3])
    st = load().fi_batch_paged_attention_run_cascade(
        ctypes.byref(info), q.data_ptr(), q.stride(0), q.stride(1), q.shape[0], k_cache.data_ptr(), ks,
        v_cache.data_ptr(), vs, k_cache.shape[0], kv_indices_dev.data_ptr(), shared_k.data_ptr(), sks,
        shared_v.data_ptr(), svs, shared_k.shape[0], shared_kv_indices_dev.data_ptr(), shared_k.shape[1],
        o.data_ptr(), o.stride(0), o.stride(1), lse.data_ptr() if lse is not None else None, _dtype_code(q),
        float(sm_scale), ws.int_ws.data_ptr(), ws.float_ws.data_ptr(), _stream_ptr(stream))
    _check(st, "fi_batch_paged_attention_run_cascade")


STATIC_SCRATCH_PARTIAL_ROWS = 32768


def run_static_scratch(ws: Workspace, info: PlanInfo, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                       kv_indices_dev: torch.Tensor, o: torch.Tensor, lse: torch.Tensor | None, sm_scale: float,
                       stream=None):
    """run() for callers that cannot allocate: the split-KV partial states go
    to the library's fixed device array (at most 32768 partial rows) instead
    of ws.float_ws.  Calls that overlap on the GPU race on that array."""
    lib = load()
    if kv_indices_dev.dtype != torch.int32 or not kv_indices_dev.is_contiguous():
        raise TypeError("kv_indices must be a contiguous int32 device tensor")
    if q.dtype != k_cache.dtype or q.dtype != v_cache.dtype or q.dtype != o.dtype:
        raise TypeError("q, k, v and o must share one dtype")
    ks = (ctypes.c_int64 * 3)(*k_cache.stride()[:3])
    vs = (ctypes.c_int64 * 3)(*v_cache.stride()[:3])
    st = lib.fi_batch_paged_attention_run_static_scratch(
        ctypes.byref(info), q.data_ptr(), q.stride(0), q.stride(1), q.shape[0], k_cache.data_ptr(), ks,
        v_cache.data_ptr(), vs, k_cache.shape[0], kv_indices_dev.data_ptr(), o.data_ptr(), o.stride(0), o.stride(1),
        lse.data_ptr() if lse is not None else None, _dtype_code(q), float(sm_scale), ws.int_ws.data_ptr(),
        _stream_ptr(stream))
    _check(st, "fi_batch_paged_attention_run_static_scratch")


def merge_states(v_a, s_a, v_b, s_b, v_out, s_out, stream=None):
    """v_* [rows, heads, 128] (fp16/bf16/fp32, contiguous), s_* [rows, heads] fp32."""
    lib = load()
    for t in (v_a, v_b, v_out, s_a, s_b, s_out):
        if not t.is_contiguous():
            raise TypeError("merge_states needs contiguous tensors")
    rows, heads, d = v_a.shape
    st = lib.fi_merge_states(v_a.data_ptr(), s_a.data_ptr(), v_b.data_ptr(), s_b.data_ptr(), v_out.data_ptr(),
                             s_out.data_ptr(), rows, heads, d, _dtype_code(v_a), _stream_ptr(stream))
    _check(st, "fi_merge_states")


def rope_apply_k(ws: Workspace, info: PlanInfo, k_in, k_out, kv_indices, stream=None):
    """Unfused RoPE: rotate the keys of the plan's requests from k_in into k_out
    ([pages, page_size, Hkv, 128], same dtype; k_out may be k_in)."""
    ks_in = (ctypes.c_int64 * 3)(*k_in.stride()[:3])
    ks_out = (ctypes.c_int64 * 3)(*k_out.stride()[:3])
    _check(load().fi_rope_apply_k(ctypes.byref(info), ws.int_ws.data_ptr(), k_in.data_ptr(), ks_in, k_out.data_ptr(),
                                  ks_out, kv_indices.data_ptr(), _dtype_code(k_in), _stream_ptr(stream)),
           "fi_rope_apply_k")


def rope_apply_q(ws: Workspace, info: PlanInfo, q_in, q_out, stream=None):
    """Unfused RoPE: rotate the query rows of the plan's requests from q_in
    into q_out ([tokens, Hq, 128], same dtype; q_out may be q_in)."""
    _check(load().fi_rope_apply_q(ctypes.byref(info), ws.int_ws.data_ptr(), q_in.data_ptr(), q_in.stride(0),
                                  q_in.stride(1), q_out.data_ptr(), q_out.stride(0), q_out.stride(1),
                                  _dtype_code(q_in), _stream_ptr(stream)), "fi_rope_apply_q")


def selftest_bounded_wait(ws, stream=None):
    """Enqueue the bounded-wait self-test on ws's int workspace (see fi.h)."""
    _check(load().fi_selftest_bounded_wait(ws.int_ws.data_ptr(), _stream_ptr(stream)), "fi_selftest_bounded_wait")


def device_status(ws: Workspace, stream=None) -> int:
    """Status word of the last run on ws (0 = ok, 7 = a bounded wait ran out)."""
    out = ctypes.c_int32(0)
    _check(load().fi_get_device_status(ws.int_ws.data_ptr(), _stream_ptr(stream), ctypes.byref(out)),
           "fi_get_device_status")
    return out.value

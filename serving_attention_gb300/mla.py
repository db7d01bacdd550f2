"""Python binding of the absorbed-MLA decode entry points (include/fi_mla.h).

Argument marshalling only, like the package's GQA binding: the planner runs on
the host in the library, the decode and merge run in its CUDA kernels, and
there is no fallback.

    cfg = default_config(0)
    ws = MlaWorkspace(cfg)
    info = plan(ws, kv_indptr, kv_indices, last_page_len, num_heads=128, page_size=64)
    decode_run(ws, info, q_nope, q_pe, ckv, kpe, kv_indices_dev, o, lse, sm_scale)
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import _check, _i32, _stream_ptr, load as _load_lib

LATENT_DIM, ROPE_DIM, MAX_HEADS = 512, 64, 128
EXPORTS = ["fi_mla_default_config", "fi_mla_int_workspace_bytes", "fi_mla_float_workspace_bytes", "fi_mla_plan",
           "fi_mla_plan_host", "fi_mla_decode_run"]


class MlaConfig(ctypes.Structure):
    _fields_ = [("num_pairs", ctypes.c_int32), ("max_batch", ctypes.c_int32), ("max_units", ctypes.c_int32),
                ("max_parts", ctypes.c_int32), ("min_chunk", ctypes.c_int32), ("reserved", ctypes.c_int32 * 3)]

    def as_dict(self) -> dict:
        return {k: getattr(self, k) for k, _ in self._fields_ if k != "reserved"}


class MlaPlanInfo(ctypes.Structure):
    _fields_ = [("num_pairs", ctypes.c_int32), ("num_units", ctypes.c_int32), ("num_parts", ctypes.c_int32),
                ("num_merge", ctypes.c_int32), ("batch", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("chunk", ctypes.c_int32), ("int_ws_bytes_used", ctypes.c_int64),
                ("max_parts", ctypes.c_int32), ("reserved", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {k: getattr(self, k) for k, _ in self._fields_ if k != "reserved"}


_bound = False


def load() -> ctypes.CDLL:
    global _bound
    lib = _load_lib()
    if not _bound:
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        cfgp, infop = ctypes.POINTER(MlaConfig), ctypes.POINTER(MlaPlanInfo)
        lib.fi_mla_default_config.argtypes = [ctypes.c_int, cfgp]
        lib.fi_mla_int_workspace_bytes.argtypes = [cfgp]
        lib.fi_mla_int_workspace_bytes.restype = sz
        lib.fi_mla_float_workspace_bytes.argtypes = [cfgp]
        lib.fi_mla_float_workspace_bytes.restype = sz
        lib.fi_mla_plan.argtypes = [cfgp, vp, vp, vp, i32, i32, i32, i32, vp, vp, sz, vp, infop]
        lib.fi_mla_plan_host.argtypes = [cfgp, vp, vp, vp, i32, i32, i32, i32, vp, sz, infop]
        lib.fi_mla_decode_run.argtypes = [infop, vp, i64, i64, vp, i64, i64, i32, vp, i64, i64, vp, i64, i64, i32,
                                          vp, vp, vp, ctypes.c_float, vp, vp, vp]
        for name in ("fi_mla_default_config", "fi_mla_plan", "fi_mla_plan_host", "fi_mla_decode_run"):
            getattr(lib, name).restype = ctypes.c_int
        _bound = True
    return lib


def default_config(device: int = 0, **overrides) -> MlaConfig:
    cfg = MlaConfig()
    _check(load().fi_mla_default_config(device, ctypes.byref(cfg)), "fi_mla_default_config")
    for k, v in overrides.items():
        setattr(cfg, k, v)
    return cfg


def make_config(num_pairs: int, **overrides) -> MlaConfig:
    """A config without a device query (host planning, tests)."""
    cfg = MlaConfig(num_pairs=num_pairs, max_batch=4096, max_units=1 << 15, max_parts=512, min_chunk=256)
    for k, v in overrides.items():
        setattr(cfg, k, v)
    return cfg


def int_workspace_bytes(cfg: MlaConfig) -> int:
    return int(load().fi_mla_int_workspace_bytes(ctypes.byref(cfg)))


def float_workspace_bytes(cfg: MlaConfig) -> int:
    return int(load().fi_mla_float_workspace_bytes(ctypes.byref(cfg)))


class MlaWorkspace:
    """Device int/float workspaces plus two pinned staging buffers for plans."""

    def __init__(self, cfg: MlaConfig, device="cuda"):
        self.cfg = cfg
        self.device = torch.device(device)
        ib, fb = int_workspace_bytes(cfg), float_workspace_bytes(cfg)
        if ib == 0 or fb == 0:
            raise ValueError("invalid MLA config")
        self.int_ws = torch.zeros((ib + 15) // 16 * 4, dtype=torch.int32, device=self.device)
        self.float_ws = torch.zeros((fb + 15) // 16 * 4, dtype=torch.float32, device=self.device)
        self._staging = [torch.empty(ib, dtype=torch.uint8, pin_memory=True) for _ in range(2)]
        self._events = [None, None]
        self._next = 0


def plan_host(cfg: MlaConfig, kv_indptr, kv_indices, last_page_len, num_heads: int, page_size: int,
              num_pages: int = 0):
    """Host-only planning: returns (status, int32 workspace image or None, MlaPlanInfo)."""
    lib = load()
    kvp, kvi, lpl = _i32(kv_indptr), _i32(kv_indices), _i32(last_page_len)
    nbytes = int_workspace_bytes(cfg)
    buf = np.zeros(max(nbytes, 4) // 4, dtype=np.int32)
    info = MlaPlanInfo()
    st = lib.fi_mla_plan_host(ctypes.byref(cfg), kvp.ctypes.data, kvi.ctypes.data if kvi.size else None,
                              lpl.ctypes.data if lpl.size else None, len(kvp) - 1, num_heads, page_size, num_pages,
                              buf.ctypes.data, nbytes, ctypes.byref(info))
    if st != 0:
        return st, None, info
    return st, buf[:info.int_ws_bytes_used // 4].copy(), info


def plan(ws: MlaWorkspace, kv_indptr, kv_indices, last_page_len, num_heads: int, page_size: int,
         num_pages: int = 0, stream=None) -> MlaPlanInfo:
    """Plan on the host and enqueue the copy of the work list into ws.int_ws."""
    lib = load()
    kvp, kvi, lpl = _i32(kv_indptr), _i32(kv_indices), _i32(last_page_len)
    i = ws._next
    ws._next ^= 1
    if ws._events[i] is not None:
        ws._events[i].synchronize()  # the staging buffer's previous copy has landed
    info = MlaPlanInfo()
    staging = ws._staging[i]
    st = lib.fi_mla_plan(ctypes.byref(ws.cfg), kvp.ctypes.data, kvi.ctypes.data if kvi.size else None,
                         lpl.ctypes.data if lpl.size else None, len(kvp) - 1, num_heads, page_size, num_pages,
                         ws.int_ws.data_ptr(), staging.data_ptr(), staging.numel(), _stream_ptr(stream),
                         ctypes.byref(info))
    _check(st, "fi_mla_plan")
    ev = torch.cuda.Event()
    ev.record(stream if stream is not None else torch.cuda.current_stream())
    ws._events[i] = ev
    return info


def decode_run(ws: MlaWorkspace, info: MlaPlanInfo, q_nope: torch.Tensor, q_pe: torch.Tensor, ckv: torch.Tensor,
               kpe: torch.Tensor, kv_indices_dev: torch.Tensor, o: torch.Tensor, lse: torch.Tensor | None,
               sm_scale: float, stream=None):
    """Enqueue the MLA decode and merge kernels for the current plan of `ws`."""
    for t in (q_nope, q_pe, ckv, kpe, o):
        if t.dtype != torch.bfloat16:
            raise TypeError("q_nope, q_pe, ckv, kpe and o are bf16")
    if kv_indices_dev.dtype != torch.int32 or not kv_indices_dev.is_contiguous():
        raise TypeError("kv_indices must be a contiguous int32 device tensor")
    if not o.is_contiguous() or (lse is not None and (lse.dtype != torch.float32 or not lse.is_contiguous())):
        raise TypeError("o (bf16) and lse (fp32) must be contiguous")
    st = load().fi_mla_decode_run(
        ctypes.byref(info), q_nope.data_ptr(), q_nope.stride(0), q_nope.stride(1), q_pe.data_ptr(), q_pe.stride(0),
        q_pe.stride(1), q_nope.shape[0], ckv.data_ptr(), ckv.stride(0), ckv.stride(1), kpe.data_ptr(),
        kpe.stride(0), kpe.stride(1), ckv.shape[0], kv_indices_dev.data_ptr(), o.data_ptr(),
        lse.data_ptr() if lse is not None else None, float(sm_scale), ws.int_ws.data_ptr(), ws.float_ws.data_ptr(),
        _stream_ptr(stream))
    _check(st, "fi_mla_decode_run")

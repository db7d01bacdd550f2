"""Benchmark of the paged-attention hot path on GB300.

Headline (N=1): the Llama-3-8B-shaped decode batch -- 64 requests, one query
token each, KV lengths floor(exp U(ln 512, ln 32768)), 32 query / 8 KV heads,
head_dim 128, pages of 16 shuffled over a pool sized to the total, bf16.  One
step = fi_plan on the host (work list copied to the device) + one launch of
the persistent kernel through the C ABI.  The metric is algorithmic HBM bytes
(K and V of every visible token once per KV head, plus Q, O and LSE) per
second of device time; the KV cache (2 GB) is larger than L2, so no flush is
needed between steps.

The same JSON line also reports the ragged causal prefill batch (TFLOP/s,
tensor-core bound) and the continuous-batching mix replayed through one CUDA
graph across 10 re-plans (with its decode requests also timed on their own),
each against its own roof.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun (N > 1) every rank runs its own replica of the workload (the
path has no exchange step); rank 0 prints the line with the max over ranks.
`--impl reference` times the fp64 CPU oracle on bounded samples of the same
workload on the host cores.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged-KV attention: decode HBM GB/s, prefill TFLOPS (fraction of GB300 roof)"
WORKLOAD = ("llama8b_decode: 64 requests, qo_len 1, kv_len floor(exp U(ln 512, ln 32768)), 32 q / 8 kv heads, "
            "head_dim 128, page 16, shuffled pages, bf16, N(0,1)")
HOT_KERNEL = "paged_attention_kernel"


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def _kernel_hash() -> str:
    """Hash of the sources the paged-attention kernel is built from (the MLA
    files build other kernels and are left out)."""
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "serving_attention_gb300", "csrc", "*"))):
        if os.path.basename(f).startswith("mla") or not os.path.isfile(f):
            continue
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _traffic_per_launch(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        e = t.get(workload)
        if e and e.get("kernel_hash") == _kernel_hash():
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class NvmlClockSampler:
    """SM clock and clock-event reasons read through NVML (read-only queries)
    by a thread polling every millisecond while the timed region runs, so even
    a region of a few milliseconds gets samples."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int):
        import ctypes
        import threading

        self.ct = ctypes
        self.samples, self.reason_bits = [], 0
        self.stop = threading.Event()
        self.thread = None
        self.max_mhz = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            h = ctypes.c_void_p()
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            parts = [p for p in vis.split(",") if p.strip()]
            phys = int(parts[index]) if index < len(parts) and parts[index].strip().isdigit() else index
            if lib.nvmlDeviceGetHandleByIndex_v2(phys, ctypes.byref(h)) != 0:
                raise OSError("no NVML handle")
            self.lib, self.h = lib, h
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.reasons_fn = fn
        except Exception:
            self.lib = None

    def _poll(self):
        ct = self.ct
        clk, rs = ct.c_uint(), ct.c_ulonglong()
        while True:
            if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(clk)) == 0:
                self.samples.append(float(clk.value))
            if self.reasons_fn(self.h, ct.byref(rs)) == 0:
                self.reason_bits |= int(rs.value)
            if self.stop.wait(0.001):
                break

    def __enter__(self):
        import threading

        if self.lib is not None:
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
        return self

    def __exit__(self, *a):
        if self.thread is not None:
            self.stop.set()
            self.thread.join()

    def summary(self):
        if self.lib is None:
            return None
        reasons = sorted(n for b, n in self.REASONS.items() if self.reason_bits & b)
        return {"sm_mhz": float(np.median(self.samples)) if self.samples else None, "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(self.samples), "source": "nvml"}


class ClockSampler:
    """nvidia-smi samples (200 ms) while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"fi_clocks_{os.getpid()}_{index}.csv")

    def __enter__(self):
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.out,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.out.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")

        sm = np.array([num(r[1]) for r in rows])
        mx = np.array([num(r[2]) for r in rows])
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": float(np.nanmedian(sm)), "sm_max_mhz": float(np.nanmax(mx)), "reasons": reasons,
                "samples": len(rows)}


# ----------------------------------------------------------------- workload


def algorithmic(b):
    """Decode bytes (KV once per KV head + Q + O + LSE) and attention FLOPs of a batch.
    FLOPs: 'formula' = 4*qo*kv*d*Hq (halved when causal), 'exact' = 4*d*Hq*visible pairs."""
    kv = b.kv_lens().astype(np.float64)
    qo = b.qo_lens().astype(np.float64)
    d, hq, hkv = 128, b.num_qo_heads, b.num_kv_heads
    kv_bytes = float((kv * hkv * d * 2 * 2).sum())
    io_bytes = float(qo.sum() * hq * (d * 2 * 2 + 4))
    pairs = qo * (kv - qo) + qo * (qo + 1) / 2 if b.causal else qo * kv
    exact = float((4 * d * hq * pairs).sum())
    formula = float((4 * d * hq * qo * kv).sum() / (2 if b.causal else 1))
    return kv_bytes + io_bytes, formula, exact


def _device_setup(local_rank):
    import torch

    torch.cuda.set_device(local_rank)
    return torch.device("cuda", local_rank)


def bench_decode(dev, steps, warmup, clocks_index):
    import torch

    import serving_attention_gb300 as fi
    import workloads

    b = workloads.llama8b_decode(device=dev)
    cfg = fi.default_plan_config(dev.index)
    # Two workspaces, used by alternate steps: the plan of step i + 1 (host
    # planning and its copy to the device, on a side stream) overlaps the
    # kernel of step i, as in a serving loop; a workspace is re-planned only
    # once the kernel that read it has finished.
    wss = [fi.Workspace(cfg, device=dev), fi.Workspace(cfg, device=dev)]
    kvi = torch.as_tensor(b.kv_indices, device=dev)
    o = torch.empty_like(b.q)
    lse = torch.empty(b.q.shape[:2], dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream(device=dev)
    args = (b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, 32, 8, 128, 16, 0, b.num_pages)
    released = [None, None]  # per workspace: event after the last kernel that read it

    def plan_on_side(k, copies=()):
        with torch.cuda.stream(side):
            if released[k] is not None:
                side.wait_event(released[k])
            for dst, src in copies:
                dst.copy_(src, non_blocking=True)
            info = fi.plan(wss[k], *args, stream=side)
            ready = torch.cuda.Event()
            ready.record(side)
        stream.wait_event(ready)
        return info

    def step(i, ev=None):
        k = i & 1
        info = plan_on_side(k)
        if ev is not None:
            ev[0].record(stream)
        fi.run(wss[k], info, b.q, b.k, b.v, kvi, o, lse, b.sm_scale)
        if ev is not None:
            ev[1].record(stream)
        released[k] = torch.cuda.Event()
        released[k].record(stream)
        return info

    for i in range(warmup):
        info = step(i)
    torch.cuda.synchronize()
    assert all(fi.device_status(w) == 0 for w in wss), "device status not ok"
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier()
    torch.cuda.synchronize()
    nv = NvmlClockSampler(clocks_index)
    with (nv if nv.lib is not None else ClockSampler(clocks_index)) as cs:
        t0.record(stream)
        for i in range(steps):
            step(i, kev[i])
        t1.record(stream)
        torch.cuda.synchronize()
    total_ms = t0.elapsed_time(t1)
    kern_ms = [a.elapsed_time(c) for a, c in kev]
    assert all(fi.device_status(w) == 0 for w in wss), "device status not ok"
    nbytes, _, _ = algorithmic(b)

    # end to end through the public API from pinned host buffers: Q and the
    # page table in (plus the plan's work list), O and LSE out, every step.
    # The KV cache stays resident in HBM: it is the serving state that
    # persists across steps.  Inputs of step i + 1 go in on the side stream
    # while step i computes, outputs of step i come back on a third stream
    # while step i + 1 computes (double-buffered device copies).
    q_h = b.q.cpu().pin_memory()
    kvi_h = torch.as_tensor(b.kv_indices).pin_memory()
    o_h = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
    lse_h = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(2)]
    q_d = [torch.empty_like(b.q) for _ in range(2)]
    kvi_d = [torch.empty_like(kvi) for _ in range(2)]
    o_d = [torch.empty_like(o) for _ in range(2)]
    lse_d = [torch.empty_like(lse) for _ in range(2)]
    out = torch.cuda.Stream(device=dev)
    drained = [None, None]  # per buffer set: event after its outputs were copied back
    h2d = q_h.numel() * q_h.element_size() + kvi_h.numel() * 4
    d2h = o_h[0].numel() * o_h[0].element_size() + lse_h[0].numel() * 4

    def e2e_step(i):
        k = i & 1
        info = plan_on_side(k, ((q_d[k], q_h), (kvi_d[k], kvi_h)))
        if drained[k] is not None:
            stream.wait_event(drained[k])
        fi.run(wss[k], info, q_d[k], b.k, b.v, kvi_d[k], o_d[k], lse_d[k], b.sm_scale)
        released[k] = torch.cuda.Event()
        released[k].record(stream)
        with torch.cuda.stream(out):
            out.wait_event(released[k])
            o_h[k].copy_(o_d[k], non_blocking=True)
            lse_h[k].copy_(lse_d[k], non_blocking=True)
            drained[k] = torch.cuda.Event()
            drained[k].record(out)
        return info

    for i in range(warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        info_e = e2e_step(i)
    stream.wait_stream(out)  # the last step's outputs are on the host before the clock stops
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    # the pipelined copies moved the right data: same inputs, same (deterministic) kernel
    assert torch.equal(o_h[(steps - 1) & 1], o.cpu()), "end-to-end output differs from the device-timed run"
    plan_bytes = info_e.int_ws_bytes_used
    plan_us = []
    for _ in range(20):
        t = time.perf_counter()
        fi.plan_host(cfg, *args)
        plan_us.append((time.perf_counter() - t) * 1e6)
    return dict(batch=b, total_ms=total_ms, kern_ms=kern_ms, bytes=nbytes, clocks=cs.summary(), e2e_ms=e2e_ms,
                h2d=h2d + plan_bytes, d2h=d2h, info=info, plan_host_us=float(np.median(plan_us)))


def bench_secondary(dev, reps=5):
    """Prefill TFLOP/s and the continuous-batching mix, CUDA events, L2 flushed between reps."""
    import torch

    import serving_attention_gb300 as fi
    import workloads

    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    out = {}
    cfg = fi.default_plan_config(dev.index)
    ws = fi.Workspace(cfg, device=dev)
    for name, maker in (("ragged_prefill", workloads.ragged_prefill),):
        b = maker(device=dev)
        info = fi.plan(ws, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, b.num_qo_heads, b.num_kv_heads,
                       128, b.page_size, b.causal, b.num_pages)
        kvi = torch.as_tensor(b.kv_indices, device=dev)
        o = torch.empty_like(b.q)
        lse = torch.empty(b.q.shape[:2], dtype=torch.float32, device=dev)
        fi.run(ws, info, b.q, b.k, b.v, kvi, o, lse, b.sm_scale)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fi.run(ws, info, b.q, b.k, b.v, kvi, o, lse, b.sm_scale)
        ts = _replay_times(g, flush, 4 * reps)
        warm = _replay_times(g, None, 4 * reps)
        assert fi.device_status(ws) == 0
        ms = float(np.median(ts))
        nbytes, formula, exact = algorithmic(b)
        out[name] = dict(ms=ms, ms_p10_p90=_p10_p90(ts), warm_l2_ms=float(np.median(warm)),
                         tflops_formula=formula / ms / 1e9, tflops_exact=exact / ms / 1e9,
                         decode_gbs=nbytes / ms / 1e6, items=info.num_items)
        del b, o, lse, g
        torch.cuda.empty_cache()
    out["tiny_decode"] = bench_tiny(dev, flush, reps)
    out["continuous_batch"] = bench_mix(dev, flush, reps)
    out["shared_prefix"] = bench_shared_prefix(dev, flush, reps)
    out["kv_strides"] = bench_kv_strides(dev, flush, reps)
    out["variants"] = bench_variants(dev, flush, reps)
    out["mla"] = bench_mla(dev, flush, reps)
    return out


def bench_tiny(dev, flush, reps=5):
    """The tiny fp16 decode batch (4 requests, kv U{1..512}, 8 q / 2 kv heads):
    about 1 MB of KV, so the launch and one item's load chain set its time;
    graph replay, L2 flushed between replays."""
    import torch

    import serving_attention_gb300 as fi
    import workloads

    b = workloads.tiny_decode(device=dev)
    ws = fi.Workspace(fi.default_plan_config(dev.index), device=dev)
    info = fi.plan(ws, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, b.num_qo_heads, b.num_kv_heads, 128,
                   b.page_size, b.causal, b.num_pages)
    kvi = torch.as_tensor(b.kv_indices, device=dev)
    o = torch.empty_like(b.q)
    lse = torch.empty(b.q.shape[:2], dtype=torch.float32, device=dev)
    fi.run(ws, info, b.q, b.k, b.v, kvi, o, lse, b.sm_scale)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fi.run(ws, info, b.q, b.k, b.v, kvi, o, lse, b.sm_scale)
    ts = _replay_times(g, flush, 20 * reps)
    assert fi.device_status(ws) == 0
    ms = float(np.median(ts))
    nbytes, _, _ = algorithmic(b)
    return {"workload": "tiny_decode: 4 requests, kv U{1..512}, 8 q / 2 kv heads, page 16, fp16", "ms": ms,
            "ms_p10_p90": _p10_p90(ts), "gbs": nbytes / ms / 1e6, "algorithmic_bytes": nbytes, "items": info.num_items,
            "graded": False}


def _replay_times(g, flush, reps):
    """CUDA-event times (ms) of `reps` replays of graph g, each after an L2
    flush when `flush` is a buffer (else back to back, warm L2)."""
    import torch

    ts = []
    for _ in range(reps):
        if flush is not None:
            flush.zero_()
        a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        c.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(c))
    return ts


def _p10_p90(ts):
    return [float(np.percentile(ts, 10)), float(np.percentile(ts, 90))]


def tail_requests(b, first: int):
    """Requests first.. of a batch as a batch of their own: (qo_indptr,
    kv_indptr, kv_indices, last_page_len) re-based to start at 0, and the
    query row where they start in the original batch."""
    start = int(b.qo_indptr[first])
    k0, k1 = int(b.kv_indptr[first]), int(b.kv_indptr[-1])
    return (b.qo_indptr[first:] - start, b.kv_indptr[first:] - k0, b.kv_indices[k0:k1],
            b.last_page_len[first:len(b.qo_indptr) - 1], start)


def bench_mix(dev, flush, reps=5, replans=10):
    """The continuous-batching mix as a serving loop runs it: buffers at the
    capacity of the first `replans` seeded draws, one graph captured from
    draw 0, then per draw new contents, a re-plan (host, with its copy) and
    `reps` replays with L2 flushed.  Reports the median over draws of each
    draw's median, p10/p90 over all replays, and the decode part alone: the
    120 decode requests of every draw planned on their own and replayed
    through a second graph (their queries and outputs are the buffers' rows
    after the 8 x 512 prefill tokens)."""
    import torch

    import serving_attention_gb300 as fi
    import workloads

    pages, tokens = workloads.continuous_batch_capacity(replans)
    cfg = fi.default_plan_config(dev.index)
    b0 = workloads.continuous_batch(device=dev, replan=0, pool_pages=pages, q_tokens=tokens)
    n_pf = 8
    s0 = int(b0.qo_indptr[n_pf])  # decode rows start after the prefill tokens (the same for every draw)
    q_buf, k_buf, v_base, v_buf = b0.q, b0.k_base, b0.v_base, b0.v
    kvi_buf = torch.zeros(pages, dtype=torch.int32, device=dev)
    kvi_dec = torch.zeros(pages, dtype=torch.int32, device=dev)
    o = torch.zeros_like(q_buf)
    lse = torch.zeros(q_buf.shape[:2], dtype=torch.float32, device=dev)
    ws, ws_d = fi.Workspace(cfg, device=dev), fi.Workspace(cfg, device=dev)

    def decode_part(b):
        qo, kvp, kvi, lpl, start = tail_requests(b, n_pf)
        assert start == s0
        return workloads.PagedBatch("continuous_batch.decode", b.dtype, qo, kvp, kvi, lpl, 32, 8, 16, 1,
                                    b.sm_scale, q_buf[s0:], k_buf, v_buf, k_buf, v_base)

    def plan(wsx, b, kvi):
        info = fi.plan(wsx, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, 32, 8, 128, 16, 1, pages)
        kvi[:b.kv_indices.size].copy_(torch.as_tensor(b.kv_indices, device=dev))
        return info

    d0 = decode_part(b0)
    info = plan(ws, b0, kvi_buf)
    info_d = plan(ws_d, d0, kvi_dec)
    run_all = lambda: fi.run(ws, info, q_buf, k_buf, v_buf, kvi_buf, o, lse, b0.sm_scale)  # noqa: E731
    run_dec = lambda: fi.run(ws_d, info_d, q_buf[s0:], k_buf, v_buf, kvi_dec, o[s0:], lse[s0:],  # noqa: E731
                             b0.sm_scale)
    graphs = []
    for fn in (run_all, run_dec):
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        graphs.append(g)
    per, per_d, all_ts, gbs_d, plan_us, tf_exact, dec_gbs = [], [], [], [], [], [], []
    for r in range(replans):
        if r == 0:
            b = b0
        else:
            b = workloads.continuous_batch(device=dev, replan=r, pool_pages=pages, q_tokens=tokens)
            q_buf.copy_(b.q)
            k_buf.copy_(b.k_base)
            v_base.copy_(b.v_base)
            b.q, b.k, b.v, b.k_base, b.v_base = q_buf, k_buf, v_buf, k_buf, v_base  # frees the draw's own copies
        t = time.perf_counter()
        fi.plan_host(cfg, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, 32, 8, 128, 16, 1, pages)
        plan_us.append((time.perf_counter() - t) * 1e6)
        info_r = plan(ws, b, kvi_buf)
        assert info_r.num_ctas == info.num_ctas
        ts = _replay_times(graphs[0], flush, reps)
        assert fi.device_status(ws) == 0
        all_ts += ts
        ms = float(np.median(ts))
        per.append(ms)
        nbytes, _, exact = algorithmic(b)
        tf_exact.append(exact / ms / 1e9)
        dec_gbs.append(nbytes / ms / 1e6)
        d = decode_part(b)
        plan(ws_d, d, kvi_dec)
        ts_d = _replay_times(graphs[1], flush, reps)
        assert fi.device_status(ws_d) == 0
        ms_d = float(np.median(ts_d))
        per_d.append(ms_d)
        gbs_d.append(algorithmic(d)[0] / ms_d / 1e6)
    del graphs
    torch.cuda.synchronize()
    return dict(ms=float(np.median(per)), ms_per_replan=per, ms_p10_p90=_p10_p90(all_ts),
                tflops_exact=float(np.median(tf_exact)), decode_gbs=float(np.median(dec_gbs)),
                decode_part_ms=float(np.median(per_d)), decode_part_gbs=float(np.median(gbs_d)),
                decode_part_gbs_per_replan=gbs_d, plan_host_us=float(np.median(plan_us)), replans=replans,
                items=info.num_items)


def mla_algorithmic(b):
    """Bytes and flops of one absorbed-MLA decode: every cached latent (512)
    and RoPE key (64) once, the page ids, q (576) and o (512) per head, the
    LSE; flops 2 * H * (576 + 512) per cached token (Q K^T and P V)."""
    lens = b.kv_lens().astype(np.int64)
    tok = int(lens.sum())
    H, B = b.num_heads, b.batch
    pages = int(b.kv_indptr[-1])
    nbytes = tok * (512 + 64) * 2 + pages * 4 + B * H * ((576 + 512) * 2 + 4)
    flops = 2 * H * (576 + 512) * tok
    return nbytes, flops


def bench_mla(dev, flush, reps=5):
    """Absorbed-MLA decode (decode kernel + merge kernel, one C-ABI call) on
    the 64-request length-mix workload, graph-replayed, L2 flushed."""
    import torch

    from serving_attention_gb300 import mla
    import workloads

    b = workloads.mla_decode(device=dev)
    cfg = mla.default_config(dev.index)
    ws = mla.MlaWorkspace(cfg, device=dev)
    info = mla.plan(ws, b.kv_indptr, b.kv_indices, b.last_page_len, b.num_heads, b.page_size, b.num_pages)
    kvi = torch.as_tensor(b.kv_indices, device=dev)
    o = torch.empty(b.q_nope.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(b.q_nope.shape[:2], dtype=torch.float32, device=dev)
    ms = _graph_ms(lambda: mla.decode_run(ws, info, b.q_nope, b.q_pe, b.ckv, b.kpe, kvi, o, lse, b.sm_scale),
                   flush, reps)
    import serving_attention_gb300 as fi
    assert fi.device_status(ws) == 0
    nbytes, flops = mla_algorithmic(b)
    out = {"workload": "mla_decode: 64 requests, kv floor(exp U(ln 512, ln 32768)), 128 heads, latent 512 + RoPE 64,"
                       " page 64, bf16", "ms": ms, "gbs": nbytes / ms / 1e6, "tflops": flops / ms / 1e9,
           "algorithmic_bytes": nbytes, "flops": flops, "pairs": info.num_pairs, "chunks": info.num_units,
           "split_chunks": info.num_parts, "launches": 2}
    del b, o, lse, ws
    torch.cuda.empty_cache()
    return out


def _graph_ms(fn, flush, reps):
    import torch

    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    ts = []
    for _ in range(reps):
        flush.zero_()
        a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        c.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(c))
    del g
    return float(np.median(ts))


def bench_variants(dev, flush, reps=5):
    """Mask and logit variants: the decode workload with a 4096-token sliding
    window and 4 sink tokens (GB/s over the keys a query can see; the plan
    skips the rest), and the ragged prefill with a logits soft-cap of 30."""
    import torch

    import serving_attention_gb300 as fi
    import workloads

    out = {}
    b = workloads.llama8b_decode(device=dev)
    kvi = torch.as_tensor(b.kv_indices, device=dev)
    o = torch.empty_like(b.q)
    lse = torch.empty(b.q.shape[:2], dtype=torch.float32, device=dev)
    window, sink = 4096, 4
    times = {}
    for tag, kw in (("full", {}), ("window", dict(window_left=window, sink_tokens=sink))):
        cfg = fi.default_plan_config(dev.index, **kw)
        ws = fi.Workspace(cfg, device=dev)
        info = fi.plan(ws, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, b.num_qo_heads, b.num_kv_heads,
                       128, b.page_size, b.causal, b.num_pages)
        times[tag] = _graph_ms(lambda: fi.run(ws, info, b.q, b.k, b.v, kvi, o, lse, b.sm_scale), flush, reps)
        assert fi.device_status(ws) == 0
    kv = b.kv_lens().astype(np.int64)
    visible = np.minimum(kv, window + 1) + np.clip(kv - (window + 1), 0, sink)
    vis_bytes = float(visible.sum()) * b.num_kv_heads * 128 * 2 * 2 + b.batch * b.num_qo_heads * (128 * 2 * 2 + 4)
    out["window_decode"] = {"workload": "llama8b_decode with window_left 4096, sink_tokens 4",
                            "ms": times["window"], "full_ms": times["full"],
                            "gbs_visible": vis_bytes / times["window"] / 1e6,
                            "speedup_vs_full": times["full"] / times["window"]}
    del b, o, lse, kvi
    torch.cuda.empty_cache()
    b = workloads.ragged_prefill(device=dev)
    kvi = torch.as_tensor(b.kv_indices, device=dev)
    o = torch.empty_like(b.q)
    lse = torch.empty(b.q.shape[:2], dtype=torch.float32, device=dev)
    for tag, kw in (("plain", {}), ("capped", dict(logits_soft_cap=30.0))):
        cfg = fi.default_plan_config(dev.index, **kw)
        ws = fi.Workspace(cfg, device=dev)
        info = fi.plan(ws, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, b.num_qo_heads, b.num_kv_heads,
                       128, b.page_size, b.causal, b.num_pages)
        times[tag] = _graph_ms(lambda: fi.run(ws, info, b.q, b.k, b.v, kvi, o, lse, b.sm_scale), flush, reps)
        assert fi.device_status(ws) == 0
    _, _, exact = algorithmic(b)
    out["capped_prefill"] = {"workload": "ragged_prefill with logits_soft_cap 30", "ms": times["capped"],
                             "plain_ms": times["plain"], "tflops_exact": exact / times["capped"] / 1e9,
                             "cost_vs_plain": times["capped"] / times["plain"]}
    del b, o, lse, kvi
    torch.cuda.empty_cache()
    out["rope"] = bench_rope(dev, flush, reps)
    return out


def bench_rope(dev, flush, reps=5):
    """RoPE on unrotated queries and cached keys: fused into the attention
    loaders, against the unfused form -- the queries and every cached key
    rotated into copies by separate passes (fi_rope_apply_q, fi_rope_apply_k:
    read, rotate, write), then the plain kernel on the copies -- and against
    the plain kernel alone (no rotation at all).  The library's RoPE path for
    a batch is `rope_ms`: the fused run, except that with query and key
    buffers the queries and keys of prefill-class requests (keys read by
    every 256-row item of their request) are rotated once by a pass before
    the kernel (fi_batch_paged_attention_run_rope_prerotated,
    `prerotated_ms`); decode-class requests stay fully fused.
    fusion_speedup = unfused / rope_ms."""
    import torch

    import serving_attention_gb300 as fi
    import workloads

    res = {}
    for name, maker, theta, max_pos in (("llama8b_decode", workloads.llama8b_decode, 500000.0, 32768),
                                        ("ragged_prefill", workloads.ragged_prefill, 10000.0, 8192)):
        b = maker(device=dev)
        kvi = torch.as_tensor(b.kv_indices, device=dev)
        o = torch.empty_like(b.q)
        lse = torch.empty(b.q.shape[:2], dtype=torch.float32, device=dev)
        k_rot = torch.empty_like(b.k)
        q_rot = torch.empty_like(b.q)
        k_rot16 = torch.empty(b.k.shape, dtype=torch.float16, device=dev)
        q_rot16 = torch.empty(b.q.shape, dtype=torch.float16, device=dev)
        cfg_p = fi.default_plan_config(dev.index)
        cfg_r = fi.default_plan_config(dev.index, rope_max_positions=max_pos, rope_theta=theta)
        ws_p, ws_r = fi.Workspace(cfg_p, device=dev), fi.Workspace(cfg_r, device=dev)
        args = (b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, b.num_qo_heads, b.num_kv_heads, 128,
                b.page_size, b.causal, b.num_pages)
        info_p, info_r = fi.plan(ws_p, *args), fi.plan(ws_r, *args)

        def fused():
            fi.run(ws_r, info_r, b.q, b.k, b.v, kvi, o, lse, b.sm_scale)

        def unfused():
            fi.rope_apply_q(ws_r, info_r, b.q, q_rot)
            fi.rope_apply_k(ws_r, info_r, b.k, k_rot, kvi)
            fi.run(ws_p, info_p, q_rot, k_rot, b.v, kvi, o, lse, b.sm_scale)

        def plain():
            fi.run(ws_p, info_p, b.q, b.k, b.v, kvi, o, lse, b.sm_scale)

        def prerotated():
            fi.run_rope_prerotated(ws_r, info_r, b.q, b.k, b.v, kvi, q_rot16, k_rot16, o, lse, b.sm_scale)

        t = {k: _graph_ms(f, flush, reps) for k, f in (("fused", fused), ("unfused", unfused), ("plain", plain),
                                                         ("prerotated", prerotated))}
        assert fi.device_status(ws_r) == 0 and fi.device_status(ws_p) == 0
        rope_ms = t["prerotated"] if info_r.num_prefill_items > 0 else t["fused"]
        res[name] = {"fused_ms": t["fused"], "prerotated_ms": t["prerotated"], "rope_ms": rope_ms,
                     "unfused_ms": t["unfused"], "plain_ms": t["plain"], "fusion_speedup": t["unfused"] / rope_ms,
                     "fully_fused_speedup": t["unfused"] / t["fused"], "fused_cost_vs_plain": t["fused"] / t["plain"]}
        del b, o, lse, kvi, k_rot, q_rot, k_rot16, q_rot16, ws_p, ws_r
        torch.cuda.empty_cache()
    res["workload"] = ("queries and cached keys unrotated; llama8b_decode with theta 5e5, ragged_prefill with theta "
                       "1e4; unfused = fi_rope_apply_q and fi_rope_apply_k (every query and cached key), then the "
                       "plain kernel; rope_ms = the library's path: prerotated when the plan has prefill-class units, "
                       "else fully fused")
    return res


def bench_kv_strides(dev, flush, reps=5):
    """Equal against independent K/V strides on the same values: V either
    shares K's layout or sits in a pool with one padding head (its slot and
    page strides then differ from K's).  The BatchAttention PR page reports
    the equal-stride module 1.0456x faster on B200; here both layouts run
    the same kernel, the copy engine computing K and V addresses from their
    own tensor maps."""
    import torch

    import serving_attention_gb300 as fi
    import workloads

    cfg = fi.default_plan_config(dev.index)
    res = {}
    for name, maker in (("llama8b_decode", workloads.llama8b_decode), ("continuous_batch", workloads.continuous_batch)):
        b = maker(device=dev)
        ws = fi.Workspace(cfg, device=dev)
        info = fi.plan(ws, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, b.num_qo_heads, b.num_kv_heads,
                       128, b.page_size, b.causal, b.num_pages)
        kvi = torch.as_tensor(b.kv_indices, device=dev)
        o = torch.empty_like(b.q)
        lse = torch.empty(b.q.shape[:2], dtype=torch.float32, device=dev)
        shape = list(b.v.shape)
        v_equal = b.v.contiguous()
        v_pool = torch.empty(shape[:2] + [shape[2] + 1, shape[3]], dtype=b.v.dtype, device=dev)
        v_pool[:, :, :shape[2]].copy_(b.v)
        v_unequal = v_pool[:, :, :shape[2]]
        times = {}
        for tag, v in (("equal", v_equal), ("unequal", v_unequal)):
            fi.run(ws, info, b.q, b.k, v, kvi, o, lse, b.sm_scale)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fi.run(ws, info, b.q, b.k, v, kvi, o, lse, b.sm_scale)
            ts = []
            for _ in range(reps):
                flush.zero_()
                a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                g.replay()
                c.record()
                torch.cuda.synchronize()
                ts.append(a.elapsed_time(c))
            times[tag] = float(np.median(ts))
            del g
        assert fi.device_status(ws) == 0
        res[name] = {"equal_ms": times["equal"], "unequal_ms": times["unequal"],
                     "equal_speedup": times["unequal"] / times["equal"]}
        del b, o, lse, v_equal, v_pool, v_unequal
        torch.cuda.empty_cache()
    res["workload"] = "llama8b_decode and continuous_batch with V in K's layout or in a pool with a padding head"
    return res


def bench_shared_prefix(dev, flush, reps=5):
    """Composable format as one cascade plan: the dense prefix is the shared
    block of all 64 branch queries (tensor cores), the page-1 suffixes their
    own keys, in one persistent launch followed by the cascade merge; against
    the same step as separate calls (prefix run with its late merge, suffix
    run, fi_merge_states) and one run over the flat page-1 layout (prefix
    pages repeated in every branch's page list).  Each captured in a CUDA
    graph, L2 flushed between replays."""
    import torch

    cascade, separate, flat_run, nbytes, late = _shared_prefix_runs(dev)
    res, spread = {}, {}
    for name, fn in (("cascade", cascade), ("separate", separate), ("flat", flat_run)):
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        ts = _replay_times(g, flush, reps if name == "flat" else 20 * reps)
        res[name] = float(np.median(ts))
        spread[name] = _p10_p90(ts)
    assert cascade.check() == 0
    return {"workload": "shared_prefix: 8192-token dense prefix + 64 branches, suffix U[64,512] at page 1",
            "composable_ms": res["cascade"], "composable_ms_p10_p90": spread["cascade"],
            "composable_gbs": nbytes / res["cascade"] / 1e6, "launches": 2,
            "form": "one cascade plan: one persistent launch + the cascade merge",
            "separate_ms": res["separate"], "separate_launches": 3 + late, "flat_ms": res["flat"],
            "speedup_vs_flat": res["flat"] / res["cascade"], "speedup_vs_separate": res["separate"] / res["cascade"],
            "algorithmic_bytes": nbytes}


def _shared_prefix_runs(dev):
    """The shared-prefix workload planned three ways: returns the cascade step
    (one plan: prefix block + suffixes), the separate step (prefix run, suffix
    run, state merge), the flat run, the algorithmic bytes of the composable
    form and how many late-merge launches the separate step adds."""
    import torch

    import serving_attention_gb300 as fi
    import workloads

    d = workloads.shared_prefix(device=dev)
    pre, suf, flat = d["prefix"], d["suffix"], d["flat"]
    cfg = fi.default_plan_config(dev.index)

    def prepared(b):
        ws = fi.Workspace(cfg, device=dev)
        info = fi.plan(ws, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, b.num_qo_heads, b.num_kv_heads,
                       128, b.page_size, b.causal, b.num_pages)
        kvi = torch.as_tensor(b.kv_indices, device=dev)
        o = torch.empty_like(b.q)
        lse = torch.empty(b.q.shape[:2], dtype=torch.float32, device=dev)
        return ws, info, kvi, o, lse

    P, S, F = prepared(pre), prepared(suf), prepared(flat)
    o_m = torch.empty_like(pre.q)
    l_m = torch.empty(pre.q.shape[:2], dtype=torch.float32, device=dev)
    wsc = fi.Workspace(cfg, device=dev)
    info_c = fi.plan_cascade(wsc, pre.qo_indptr, pre.kv_indptr, pre.kv_indices, pre.last_page_len, pre.page_size,
                             suf.qo_indptr, suf.kv_indptr, suf.kv_indices, suf.last_page_len, 32, 8, 128, 1, 0,
                             suf.num_pages, pre.num_pages)
    o_c = torch.empty_like(suf.q)
    l_c = torch.empty(suf.q.shape[:2], dtype=torch.float32, device=dev)

    def cascade():
        fi.run_cascade(wsc, info_c, suf.q, suf.k, suf.v, S[2], pre.k, pre.v, P[2], o_c, l_c, suf.sm_scale)

    def composable():
        fi.run(P[0], P[1], pre.q, pre.k, pre.v, P[2], P[3], P[4], pre.sm_scale)
        fi.run(S[0], S[1], suf.q, suf.k, suf.v, S[2], S[3], S[4], suf.sm_scale)
        fi.merge_states(P[3], P[4], S[3], S[4], o_m, l_m)

    def flat_run():
        fi.run(F[0], F[1], flat.q, flat.k, flat.v, F[2], F[3], F[4], flat.sm_scale)

    # algorithmic bytes of the composable form: the prefix KV once, every suffix token once, Q in, O/LSE out
    suffix_tokens = int(suf.kv_lens().sum())
    nbytes = (pre.meta["prefix_len"] + suffix_tokens) * 8 * 128 * 2 * 2 + 64 * 32 * (128 * 2 * 2 + 4)
    late = (1 if P[1].num_late_merge_units else 0) + (1 if S[1].num_late_merge_units else 0)

    def check():
        return max(fi.device_status(x) for x in (P[0], S[0], F[0], wsc))

    cascade.check = composable.check = check
    return cascade, composable, flat_run, nbytes, late


PROFILE_CASES = {
    "llama8b_decode": lambda dev: __import__("workloads").llama8b_decode(device=dev),
    "llama8b_decode_16": lambda dev: __import__("workloads").llama8b_decode(device=dev, batch=16),
    "tiny_decode": lambda dev: __import__("workloads").tiny_decode(device=dev),
    "ragged_prefill": lambda dev: __import__("workloads").ragged_prefill(device=dev),
    "ragged_prefill_4": lambda dev: __import__("workloads").ragged_prefill(device=dev, batch=4),
    "continuous_batch": lambda dev: __import__("workloads").continuous_batch(device=dev),
    # the mix with 30 of its 120 decode requests: the same kernel on about a GB (counter captures)
    "continuous_batch_small": lambda dev: __import__("workloads").continuous_batch(device=dev, n_decode=30),
    "mla_decode": lambda dev: __import__("workloads").mla_decode(device=dev),
    "mla_decode_16": lambda dev: __import__("workloads").mla_decode(device=dev, batch=16),
    "shared_prefix": None,  # the cascade step: one persistent launch + the cascade merge
    "shared_prefix_separate": None,  # prefix run (+ late merge), suffix run, state merge
}


def profile_case(name: str, launches: int) -> int:
    """A few launches of the run kernel on one workload, untimed: the program
    that ncu captures (the first launch warms up; capture with -s 1)."""
    import torch

    import serving_attention_gb300 as fi

    dev = _device_setup(0)
    if name in ("shared_prefix", "shared_prefix_separate"):
        cascade, separate, _, nbytes, late = _shared_prefix_runs(dev)
        fn = cascade if name == "shared_prefix" else separate
        for _ in range(launches):
            fn()
        torch.cuda.synchronize()
        st = fn.check()
        print(json.dumps({"profile": name, "launches": launches,
                          "kernels_per_launch": 2 if name == "shared_prefix" else 3 + late, "status": st,
                          "algorithmic_bytes": nbytes}))
        return 0 if st == 0 else 3
    b = PROFILE_CASES[name](dev)
    if name.startswith("mla"):
        return _profile_mla(name, b, dev, launches)
    ws = fi.Workspace(fi.default_plan_config(0), device=dev)
    info = fi.plan(ws, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, b.num_qo_heads, b.num_kv_heads, 128,
                   b.page_size, b.causal, b.num_pages)
    kvi = torch.as_tensor(b.kv_indices, device=dev)
    o = torch.empty_like(b.q)
    lse = torch.empty(b.q.shape[:2], dtype=torch.float32, device=dev)
    for _ in range(launches):
        fi.run(ws, info, b.q, b.k, b.v, kvi, o, lse, b.sm_scale)
    torch.cuda.synchronize()
    st = fi.device_status(ws)
    nbytes, formula, exact = algorithmic(b)
    print(json.dumps({"profile": name, "launches": launches, "items": info.num_items, "status": st,
                      "algorithmic_bytes": nbytes, "flops_exact": exact, "flops_formula": formula}))
    return 0 if st == 0 else 3


def _profile_mla(name, b, dev, launches: int) -> int:
    import torch

    import serving_attention_gb300 as fi
    from serving_attention_gb300 import mla

    ws = mla.MlaWorkspace(mla.default_config(0), device=dev)
    info = mla.plan(ws, b.kv_indptr, b.kv_indices, b.last_page_len, b.num_heads, b.page_size, b.num_pages)
    kvi = torch.as_tensor(b.kv_indices, device=dev)
    o = torch.empty(b.q_nope.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(b.q_nope.shape[:2], dtype=torch.float32, device=dev)
    for _ in range(launches):
        mla.decode_run(ws, info, b.q_nope, b.q_pe, b.ckv, b.kpe, kvi, o, lse, b.sm_scale)
    torch.cuda.synchronize()
    st = fi.device_status(ws)
    nbytes, flops = mla_algorithmic(b)
    print(json.dumps({"profile": name, "launches": launches, "chunks": info.num_units, "status": st,
                      "algorithmic_bytes": nbytes, "flops": flops}))
    return 0 if st == 0 else 3


# ----------------------------------------------------------------- reference arm


def _oracle_problem(b):
    import oracle
    import workloads

    q, k, v = workloads.host_views(b)
    dt = oracle.BF16 if b.dtype == "bf16" else oracle.FP16
    return oracle.Problem(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, b.num_qo_heads, b.num_kv_heads,
                          b.page_size, b.causal, b.sm_scale, dt, q, k, v)


def _time_rows(prob, rows_list, budget_s, work_of):
    """Run the oracle on whole query rows (all heads each), one group of rows
    per call, cycling through rows_list until about budget_s of CPU time;
    returns (work done, seconds, calls)."""
    import oracle

    heads = np.arange(prob.num_qo_heads, dtype=np.int32)
    done, t_used, calls, i = 0.0, 0.0, 0, 0
    while t_used < budget_s:
        rows = rows_list[i % len(rows_list)]
        rr = np.repeat(np.asarray(rows, np.int32), heads.size)
        hh = np.tile(heads, len(rows))
        t0 = time.perf_counter()
        oracle.attention_select(prob, rr, hh)
        t_used += time.perf_counter() - t0
        done += work_of(rows)
        calls += 1
        i += 1
    return done, t_used, calls


def reference_sample(budget_s: float):
    """Time the fp64 oracle on whole requests of the decode workload (all heads)
    until about budget_s of CPU work; returns (GB/s of algorithmic bytes, sample text, cores, seconds)."""
    import workloads

    b = workloads.llama8b_decode(device="cpu")
    prob = _oracle_problem(b)
    kv = b.kv_lens()
    order = np.argsort(kv)  # short requests first so a small budget still spans several
    rows_list = [[int(b.qo_indptr[r])] for r in order]
    row_req = {int(b.qo_indptr[r]): int(r) for r in range(b.batch)}
    nbytes = lambda rows: sum(kv[row_req[x]] * 8 * 128 * 2 * 2 + 32 * (128 * 2 * 2 + 4) for x in rows)  # noqa: E731
    done, t_used, calls = _time_rows(prob, rows_list, budget_s, nbytes)
    sample = f"{calls} request decodes (all 32 heads each) of the 64-request batch, {done / 1e9:.2f} GB of KV"
    return done / t_used / 1e9, sample, _omp_threads(), t_used


def reference_sample_prefill(budget_s: float):
    """The oracle on query rows (all 32 heads) spread over the ragged prefill
    batch; returns (TFLOP/s over visible pairs, sample text, seconds)."""
    import workloads

    b = workloads.ragged_prefill(device="cpu")
    prob = _oracle_problem(b)
    qo, kv = b.qo_lens(), b.kv_lens()
    rng = np.random.default_rng(31)
    rows_list, vis = [], {}
    for r in range(b.batch):
        for t in rng.choice(int(qo[r]), size=4, replace=False):
            row = int(b.qo_indptr[r]) + int(t)
            vis[row] = int(kv[r]) - int(qo[r]) + int(t) + 1  # bottom-right causal: keys the row sees
            rows_list.append([row])
    rng.shuffle(rows_list)
    flops = lambda rows: sum(4.0 * 128 * 32 * vis[x] for x in rows)  # noqa: E731
    done, t_used, calls = _time_rows(prob, rows_list, budget_s, flops)
    sample = f"{calls} query rows (all 32 heads each) drawn over the 16 prefill requests, {done / 1e12:.3f} TFLOP"
    return done / t_used / 1e12, sample, t_used


def reference_sample_mix(budget_s: float):
    """The oracle on the continuous-batching mix (draw 0): its 8 prefill
    chunks and 16 of its 120 decode requests (a seeded choice) are built as
    one batch of the same lengths; rows of both parts are timed, and the
    step time is extrapolated from each part's rate (visible-pair FLOPs for
    the prefill chunks, KV bytes for the decode requests).  Returns
    (estimated ms per mix step, detail dict, seconds)."""
    import workloads

    rng = np.random.default_rng(1000 * 5)
    qo, kv = workloads.continuous_batch_lengths(rng)
    pick = np.sort(np.random.default_rng(32).choice(np.arange(8, 128), size=16, replace=False))
    idx = np.concatenate([np.arange(8), pick])
    b = workloads.make_batch("continuous_batch.sample", "bf16", qo[idx], kv[idx], 32, 8, 16, 1, 5032, "cpu")
    prob = _oracle_problem(b)
    rows_p, vis = [], {}
    for r in range(8):
        for t in np.random.default_rng(33 + r).choice(512, size=4, replace=False):
            row = int(b.qo_indptr[r]) + int(t)
            vis[row] = int(kv[idx[r]]) - 512 + int(t) + 1
            rows_p.append([row])
    rows_d = [[int(b.qo_indptr[r])] for r in range(8, 24)]
    dkv = {int(b.qo_indptr[r]): int(kv[idx[r]]) for r in range(8, 24)}
    fp, tp, cp = _time_rows(prob, rows_p, budget_s / 2, lambda rows: sum(4.0 * 128 * 32 * vis[x] for x in rows))
    by, td, cd = _time_rows(prob, rows_d, budget_s / 2, lambda rows: sum(dkv[x] * 8 * 128 * 4.0 for x in rows))
    full_flops = float(sum(4.0 * 128 * 32 * (kv[r] - 512 + t + 1) for r in range(8) for t in range(512)))
    full_bytes = float((kv[8:] * 8 * 128 * 4.0).sum())
    step_s = full_flops / (fp / tp) + full_bytes / (by / td)
    detail = {"prefill_tflops": fp / tp / 1e12, "decode_gbs": by / td / 1e9,
              "sample": f"{cp} prefill-chunk query rows and {cd} decode requests (all 32 heads each) of draw 0; "
                        "step time = its prefill FLOPs and decode KV bytes at the sampled rates"}
    return step_s * 1e3, detail, tp + td


def _omp_threads() -> int:
    v = os.environ.get("OMP_NUM_THREADS", "")
    return int(v) if v.isdigit() and int(v) > 0 else (os.cpu_count() or 1)


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform

    return platform.machine()


def cpu_leg(name: str, budget_s: float) -> dict:
    """One CPU-baseline leg, as a dict (also the body of --cpu-leg)."""
    if name == "decode":
        v, sample, cores, t = reference_sample(budget_s)
        return {"value": v, "unit": "GB/s", "cores": cores, "sample": sample, "seconds": t}
    if name == "prefill":
        v, sample, t = reference_sample_prefill(budget_s)
        return {"value": v, "unit": "TFLOP/s", "cores": _omp_threads(), "sample": sample, "seconds": t}
    ms, detail, t = reference_sample_mix(budget_s)
    return dict(detail, value=ms, unit="ms per step (estimated)", cores=_omp_threads(), seconds=t)


def cpu_leg_one_core(name: str, budget_s: float):
    """The same leg in a child process limited to one OpenMP thread."""
    env = dict(os.environ, OMP_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    try:
        out = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-leg", name, "--cpu-budget",
                              str(budget_s)], capture_output=True, text=True, env=env, timeout=600)
        return json.loads(out.stdout.strip().splitlines()[-1])
    except Exception as e:  # reported, not fatal: the all-core figure stands
        return {"error": f"{type(e).__name__}: {e}"[:200]}


def cpu_baselines(budget_s: float) -> dict:
    """The oracle on the host cores: decode (the headline's workload), ragged
    prefill and the continuous-batching mix on all cores, and decode and
    prefill on one core, with the CPU model."""
    dec = cpu_leg("decode", budget_s)
    out = {"value": dec["value"], "unit": "GB/s", "cores": dec["cores"], "kind": "oracle",
           "sample": dec["sample"] + f", {dec['seconds']:.1f} s", "cpu_model": cpu_model()}
    out["one_core"] = {"decode": cpu_leg_one_core("decode", budget_s / 3),
                       "prefill": cpu_leg_one_core("prefill", budget_s / 3)}
    out["prefill"] = cpu_leg("prefill", budget_s / 2)
    out["mix"] = cpu_leg("mix", budget_s / 2)
    return out


# ----------------------------------------------------------------- driver


def _dist():
    """torch.distributed from the torchrun environment: NCCL on GPUs, gloo on a
    machine without one (the multi-process tests)."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch
        import torch.distributed as dist

        if not dist.is_initialized():
            dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        return dist, int(os.environ.get("RANK", "0")), ws, int(os.environ.get("LOCAL_RANK", "0"))
    return None, 0, 1, 0


def whole_job_gbs(bytes_per_rank: float, world: int, max_total_ms: float, steps: int) -> float:
    """Whole-job GB/s: every rank processed bytes_per_rank per step; the job's
    time is the slowest rank's (max over ranks)."""
    return bytes_per_rank * world / (max_total_ms / steps) / 1e6


_DIST = None


def _barrier():
    if _DIST is not None:
        _DIST.barrier()


def _max_over_ranks(x: float, dev) -> float:
    if _DIST is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=dev)
    _DIST.all_reduce(t, op=_DIST.ReduceOp.MAX)
    return float(t.item())


def main():
    global _DIST
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--profile", choices=sorted(PROFILE_CASES), help="only launch the kernel on this workload")
    ap.add_argument("--launches", type=int, default=2)
    ap.add_argument("--cpu-leg", choices=["decode", "prefill", "mix"], help=argparse.SUPPRESS)
    a = ap.parse_args()
    if a.profile:
        sys.exit(profile_case(a.profile, a.launches))
    if a.cpu_leg:  # one CPU-baseline leg in this process (the one-core child of cpu_baselines)
        print(json.dumps(cpu_leg(a.cpu_leg, a.cpu_budget)))
        return
    dist, rank, world, local = _dist()
    _DIST = dist
    hbm, tf, tf_sus, peak_src = _peaks()

    if a.impl == "reference":
        if rank != 0:
            return
        steps = max(1, a.steps)
        per = max(0.5, min(a.cpu_budget, 150.0 / (steps + a.warmup)))
        for _ in range(a.warmup):
            reference_sample(per / 4)
        vals, used = [], 0.0
        for _ in range(steps):
            gbs, sample, cores, t = reference_sample(per)
            vals.append(gbs)
            used += t
        v = float(np.median(vals))
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world, "steps": steps,
                "warmup": a.warmup, "ms_per_step": used / steps * 1e3, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": WORKLOAD, "global_batch": 64, "kind": "fp64 CPU oracle"},
                "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
                "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch

    import serving_attention_gb300 as fi

    fi.load()
    dev = _device_setup(local)
    r = bench_decode(dev, a.steps, a.warmup, clocks_index=local)
    total_ms = _max_over_ranks(r["total_ms"], dev)
    value = whole_job_gbs(r["bytes"], world, total_ms, a.steps)
    kern_ms = float(np.mean(r["kern_ms"]))
    achieved = r["bytes"] / kern_ms / 1e6
    e2e_ms = _max_over_ranks(r["e2e_ms"], dev)
    e2e = whole_job_gbs(r["bytes"], world, e2e_ms, a.steps)
    traffic = _traffic_per_launch("llama8b_decode")
    sec = None if (a.no_secondary or rank != 0) else bench_secondary(dev)
    cpu = None
    if rank == 0 and world == 1:
        cpu = cpu_baselines(a.cpu_budget)
    if rank != 0:
        return
    info = r["info"]
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": total_ms / a.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": 64 * world, "per_gpu_batch": 64,
                   "parallelism": f"replicas{world}",
                   "l2": f"inputs larger than L2 ({r['bytes'] / 1e9:.2f} GB of KV per step)",
                   "step": "fi_plan (host, work list copied to device) + one persistent kernel launch",
                   "num_ctas": info.num_ctas, "items": info.num_items, "split_units": info.num_merge_units},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": traffic, "kernel": HOT_KERNEL, "peak_source": peak_src,
                     "algorithmic_bytes_per_launch": r["bytes"], "kernel_ms": kern_ms,
                     "kernel_ms_p10_p90": _p10_p90(r["kern_ms"])},
        "plan_host_us": r["plan_host_us"],
        "e2e": {"value": e2e, "unit": "GB/s", "h2d_bytes_per_step": int(r["h2d"]), "d2h_bytes_per_step": int(r["d2h"])},
        "gpu_launches": a.steps,
        "clocks": r["clocks"],
        "cpu_baseline": cpu,
    }
    if sec:
        p = sec["ragged_prefill"]
        m = sec["continuous_batch"]
        line["prefill"] = {"workload": "ragged_prefill: 16 requests, qo U[128,4096], prefix U[0,2048], causal",
                           "ms": p["ms"], "tflops_formula": p["tflops_formula"], "tflops_exact": p["tflops_exact"],
                           "peak_tflops": tf, "frac_formula": p["tflops_formula"] / tf, "bound": "tensor"}
        line["prefill"].update(ms_p10_p90=p["ms_p10_p90"], warm_l2_ms=p["warm_l2_ms"])
        line["mix"] = {"workload": "continuous_batch: 8 chunked prefill (512) + 120 zipf decode, unequal K/V strides, "
                                   f"{m['replans']} re-plans through one graph",
                       "ms": m["ms"], "ms_per_replan": m["ms_per_replan"], "ms_p10_p90": m["ms_p10_p90"],
                       "decode_gbs_over_kernel": m["decode_gbs"], "tflops_exact_over_kernel": m["tflops_exact"],
                       "decode_part": {"ms": m["decode_part_ms"], "gbs": m["decode_part_gbs"],
                                       "frac_of_hbm": m["decode_part_gbs"] / hbm,
                                       "gbs_per_replan": m["decode_part_gbs_per_replan"]},
                       "plan_host_us": m["plan_host_us"]}
        t1 = sec["tiny_decode"]
        line["tiny_decode"] = dict(t1, frac_of_hbm=t1["gbs"] / hbm)
        sp = sec["shared_prefix"]
        line["shared_prefix"] = dict(sp, frac_of_hbm=sp["composable_gbs"] / hbm)
        line["kv_strides"] = sec["kv_strides"]
        line["variants"] = sec["variants"]
        ml = sec["mla"]
        line["mla"] = dict(ml, frac_of_hbm=ml["gbs"] / hbm, frac_of_tensor=ml["tflops"] / tf)
    print(json.dumps(line))


if __name__ == "__main__":
    main()

"""RoPE fused into the loaders: CUDA path (through the C ABI) against the fp64
oracle (q and unrotated k rotated exactly, then attention), same bar as the
plain path."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import serving_attention_gb300 as fi
import workloads
from helpers import LSE_TOL, O_TOL, compare, gpu_run, oracle_problem

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _cfg(max_pos, theta=10000.0, scale=1.0, **kw):
    return fi.default_plan_config(0, rope_max_positions=max_pos, rope_theta=theta, rope_scale=scale, **kw)


def _full(b, max_pos, theta=10000.0, scale=1.0, window=-1, sink=0, cap=0.0, **kw):
    cfg = _cfg(max_pos, theta, scale, window_left=window, sink_tokens=sink, logits_soft_cap=cap, **kw)
    o, lse, info, ws = gpu_run(b, cfg=cfg)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0
    assert info.variant & 4
    o_ref, l_ref = oracle.attention(oracle_problem(b, window, sink, cap, rope=1, rope_theta=theta, rope_scale=scale))
    n = b.total_qo
    err_o, err_l = compare(o[:n], lse[:n], o_ref, l_ref)
    assert err_o <= O_TOL and err_l <= LSE_TOL, (err_o, err_l)
    return info


@pytest.mark.parametrize("seed,page,group,causal,qo_max,theta,scale", [
    (401, 16, 4, 0, 1, 10000.0, 1.0),     # decode
    (402, 16, 8, 1, 3, 500000.0, 1.0),    # decode, several tokens per 16-row tile, Llama-3 theta
    (403, 4, 2, 1, 9, 10000.0, 8.0),      # page 4: prefill-class rows on the CUDA cores, scaled positions
    (404, 32, 4, 1, 40, 10000.0, 1.0),    # prefill-class rows on the tensor cores
    (405, 1, 4, 0, 2, 500000.0, 2.0),     # page 1
])
def test_rope_small_full(seed, page, group, causal, qo_max, theta, scale):
    hkv = 2
    b = workloads.random_batch(seed, batch=6, qo_max=qo_max, kv_max=1500, num_qo_heads=hkv * group,
                               num_kv_heads=hkv, page_size=page, causal=causal, device=DEV, kv_min=qo_max)
    _full(b, 2048, theta, scale, num_ctas=9, decode_min_chunk=64, prefill_min_chunk=128, split_factor=3)


@pytest.mark.parametrize("qo,kv,causal", [
    ([32], [128], 1),           # one M tile, one KV tile
    ([100], [900], 1),          # 400 rows: two items, several KV tiles
    ([64, 33], [1000, 40], 1),  # two requests, ragged
    ([40], [300], 0),
])
def test_rope_tensor_core_tiles(qo, kv, causal):
    b = workloads.make_batch("tcr", "bf16", qo, kv, 8, 2, 16, causal, 500 + kv[0], DEV,
                             pool_pages=sum((k + 15) // 16 for k in kv) + 2)
    info = _full(b, 4096, 10000.0, 1.0)
    assert info.num_prefill_items > 0


def test_rope_with_window_sink_and_cap():
    b = workloads.make_batch("tcrv", "bf16", [64, 1, 1], [1000, 700, 300], 8, 2, 16, 1, 611, DEV, pool_pages=140)
    _full(b, 4096, 500000.0, 1.0, window=130, sink=4, cap=3.0)


def _sampled(b, cfg_kw, oracle_kw, rows, heads):
    o, lse, info, ws = gpu_run(b, cfg=_cfg(**cfg_kw))
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0
    rr, hh = np.repeat(rows, len(heads)), np.tile(heads, len(rows))
    o_ref, l_ref = oracle.attention_select(oracle_problem(b, **oracle_kw), rr, hh)
    err_o, err_l = compare(o[torch.as_tensor(rr), torch.as_tensor(hh)], lse[torch.as_tensor(rr), torch.as_tensor(hh)],
                           o_ref, l_ref)
    assert err_o <= O_TOL and err_l <= LSE_TOL, (err_o, err_l)


def test_rope_long_decode_sampled():
    """Llama-3-8B-shaped decode (positions up to 32767) with the Llama-3 theta."""
    b = workloads.llama8b_decode(device=DEV, batch=16)
    _sampled(b, dict(max_pos=32768, theta=500000.0), dict(rope=1, rope_theta=500000.0),
             np.arange(b.total_qo, dtype=np.int64), np.array([0, 9, 31]))


def test_rope_ragged_prefill_sampled():
    b = workloads.ragged_prefill(device=DEV, batch=4)
    rows = []
    for r in range(b.batch):
        q0, q1 = int(b.qo_indptr[r]), int(b.qo_indptr[r + 1])
        rows += [q0, (q0 + q1) // 2, q1 - 1]
    _sampled(b, dict(max_pos=8192, theta=10000.0), dict(rope=1, rope_theta=10000.0), np.array(rows, np.int64),
             np.array([0, 17, 31]))


def test_unfused_rotation_utility():
    """fi_rope_apply_k rotates every key of the plan's requests (key j at
    position j) into the copy, each element within one rounding of the cache
    type (bf16 keeps 8 significant bits) of the fp64 rotation; keys of no
    request are left alone."""
    b = workloads.random_batch(451, batch=5, qo_max=1, kv_max=900, num_qo_heads=8, num_kv_heads=2, page_size=16,
                               causal=0, device=DEV, kv_min=1)
    cfg = _cfg(2048)
    ws = fi.Workspace(cfg, device=DEV)
    info = fi.plan(ws, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, 8, 2, 128, 16, 0, b.num_pages)
    k_rot = torch.zeros_like(b.k)
    fi.rope_apply_k(ws, info, b.k, k_rot, torch.as_tensor(b.kv_indices, device=DEV), int(b.kv_lens().max()))
    torch.cuda.synchronize()
    k64, r64 = b.k.double().cpu().numpy(), k_rot.double().cpu().numpy()
    freq = 10000.0 ** (-2.0 * np.arange(64) / 128)
    used = np.zeros(b.k.shape[:2], bool)
    for r in range(b.batch):
        pages = b.kv_indices[b.kv_indptr[r]:b.kv_indptr[r + 1]]
        for j in range(int(b.kv_lens()[r])):
            pg, sl = int(pages[j // 16]), j % 16
            used[pg, sl] = True
            c, sn = np.cos(j * freq), np.sin(j * freq)
            x0, x1 = k64[pg, sl, :, :64], k64[pg, sl, :, 64:]
            want = np.concatenate([x0 * c - x1 * sn, x1 * c + x0 * sn], axis=-1)
            assert np.all(np.abs(r64[pg, sl] - want) <= 2.0 ** -8 * np.abs(want) + 1e-30), (r, j)
    assert np.all(r64[~used] == 0)

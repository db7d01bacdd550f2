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
    fi.rope_apply_k(ws, info, b.k, k_rot, torch.as_tensor(b.kv_indices, device=DEV))
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


def _rotated64(x64, pos, theta=10000.0):
    """fp64 RoPE of rows x64[..., 128] at positions pos (broadcast over the leading axes)."""
    ang = np.asarray(pos, np.float64)[..., None] * theta ** (-2.0 * np.arange(64) / 128)
    c, sn = np.cos(ang), np.sin(ang)
    while c.ndim < x64.ndim:
        c, sn = c[..., None, :], sn[..., None, :]
    x0, x1 = x64[..., :64], x64[..., 64:]
    return np.concatenate([x0 * c - x1 * sn, x1 * c + x0 * sn], axis=-1)


def test_unfused_query_rotation_utility():
    """fi_rope_apply_q rotates every query row (token t of a request at
    kv_len - qo_len + t), each element within one bf16 rounding of the fp64
    rotation; in place it gives the same bits as into a copy."""
    b = workloads.random_batch(452, batch=5, qo_max=40, kv_max=900, num_qo_heads=8, num_kv_heads=2, page_size=16,
                               causal=1, device=DEV, kv_min=40)
    ws = fi.Workspace(_cfg(2048), device=DEV)
    info = fi.plan(ws, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, 8, 2, 128, 16, 1, b.num_pages)
    q_rot = torch.zeros_like(b.q)
    fi.rope_apply_q(ws, info, b.q, q_rot)
    q_in_place = b.q.clone()
    fi.rope_apply_q(ws, info, q_in_place, q_in_place)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0
    assert torch.equal(q_rot, q_in_place)
    q64, r64 = b.q.double().cpu().numpy(), q_rot.double().cpu().numpy()
    kv = b.kv_lens()
    for r in range(b.batch):
        q0, q1 = int(b.qo_indptr[r]), int(b.qo_indptr[r + 1])
        pos = int(kv[r]) - (q1 - q0) + np.arange(q1 - q0)
        want = _rotated64(q64[q0:q1], pos)
        assert np.all(np.abs(r64[q0:q1] - want) <= 2.0 ** -8 * np.abs(want) + 1e-5), r


def test_rotation_utilities_past_the_list_capacity():
    """More requests than a rotation CTA lists in shared memory (1024): the
    passes walk the whole request table instead, with the same results --
    every key and query row against the fp64 rotation."""
    b = workloads.random_batch(453, batch=1100, qo_max=2, kv_max=40, num_qo_heads=8, num_kv_heads=2, page_size=16,
                               causal=1, device=DEV, kv_min=2)
    ws = fi.Workspace(_cfg(2048), device=DEV)
    info = fi.plan(ws, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, 8, 2, 128, 16, 1, b.num_pages)
    kvi = torch.as_tensor(b.kv_indices, device=DEV)
    k_rot, q_rot = torch.zeros_like(b.k), torch.zeros_like(b.q)
    fi.rope_apply_k(ws, info, b.k, k_rot, kvi)
    fi.rope_apply_q(ws, info, b.q, q_rot)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0
    k64, kr = b.k.double().cpu().numpy(), k_rot.double().cpu().numpy()
    q64, qr = b.q.double().cpu().numpy(), q_rot.double().cpu().numpy()
    kv = b.kv_lens()
    pg, sl, pos, tok, qpos = [], [], [], [], []
    for r in range(b.batch):
        pages = b.kv_indices[b.kv_indptr[r]:b.kv_indptr[r + 1]]
        j = np.arange(int(kv[r]))
        pg.append(pages[j // 16]); sl.append(j % 16); pos.append(j)
        q0, q1 = int(b.qo_indptr[r]), int(b.qo_indptr[r + 1])
        tok.append(np.arange(q0, q1)); qpos.append(int(kv[r]) - (q1 - q0) + np.arange(q1 - q0))
    pg, sl, pos = np.concatenate(pg), np.concatenate(sl), np.concatenate(pos)
    tok, qpos = np.concatenate(tok), np.concatenate(qpos)
    want_k, want_q = _rotated64(k64[pg, sl], pos), _rotated64(q64[tok], qpos)
    assert np.all(np.abs(kr[pg, sl] - want_k) <= 2.0 ** -8 * np.abs(want_k) + 1e-5)
    assert np.all(np.abs(qr[tok] - want_q) <= 2.0 ** -8 * np.abs(want_q) + 1e-5)


def _prerotated_pass_check(b, q_rot, k_rot):
    """The pass wrote the fp16 rotation (one fp16 rounding of the fp64 value;
    1e-5 absolute covers the fp32 arithmetic where the two products cancel)
    of exactly the prefill-class requests' query
    rows and keys, and left every other element of both buffers alone."""
    q64, k64 = b.q.double().cpu().numpy(), b.k.double().cpu().numpy()
    qr, kr = q_rot.double().cpu().numpy(), k_rot.double().cpu().numpy()
    kv, G = b.kv_lens(), b.num_qo_heads // b.num_kv_heads
    q_seen = np.zeros(qr.shape[0], bool)
    k_seen = np.zeros(kr.shape[:2], bool)
    for r in range(b.batch):
        q0, q1 = int(b.qo_indptr[r]), int(b.qo_indptr[r + 1])
        if (q1 - q0) * G <= 16:
            continue
        pos = int(kv[r]) - (q1 - q0) + np.arange(q1 - q0)
        want = _rotated64(q64[q0:q1], pos)
        assert np.all(np.abs(qr[q0:q1] - want) <= 2.0 ** -10 * np.abs(want) + 1e-5), r
        q_seen[q0:q1] = True
        pages = b.kv_indices[b.kv_indptr[r]:b.kv_indptr[r + 1]]
        for j in range(int(kv[r])):
            pg, sl = int(pages[j // b.page_size]), j % b.page_size
            want = _rotated64(k64[pg, sl], j)
            assert np.all(np.abs(kr[pg, sl] - want) <= 2.0 ** -10 * np.abs(want) + 1e-5), (r, j)
            k_seen[pg, sl] = True
    assert np.isnan(qr[~q_seen]).all() and np.isnan(kr[~k_seen]).all()


@pytest.mark.parametrize("qo,kv,causal,dtype", [
    ([100], [900], 1, "bf16"),           # 400 rows: two items sharing the pre-rotated keys
    ([64, 33, 1, 1], [1000, 40, 700, 300], 1, "bf16"),  # prefill-class and decode-class requests in one batch
    ([40], [300], 0, "fp16"),
])
def test_rope_prerotated_keys(qo, kv, causal, dtype):
    """Queries and keys of prefill-class requests rotated once into fp16
    copies before the kernel (the tensor cores read them there), decode-class
    requests rotated inside the kernel: against the oracle, and close to the fully
    fused run (the two walk the cos/sin table differently, so the fp16 keys
    may differ in their last bit)."""
    b = workloads.make_batch("tcp", dtype, qo, kv, 8, 2, 16, causal, 600 + kv[0], DEV,
                             pool_pages=sum((k + 15) // 16 for k in kv) + 2)
    cfg = _cfg(4096)
    ws = fi.Workspace(cfg, device=DEV)
    info = fi.plan(ws, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, 8, 2, 128, 16, causal, b.num_pages)
    kvi = torch.as_tensor(b.kv_indices, device=DEV)
    k_rot = torch.full(b.k.shape, float("nan"), dtype=torch.float16, device=DEV)
    q_rot = torch.full(b.q.shape, float("nan"), dtype=torch.float16, device=DEV)
    o = torch.full_like(b.q, float("nan"))
    lse = torch.full(b.q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    fi.run_rope_prerotated(ws, info, b.q, b.k, b.v, kvi, q_rot, k_rot, o, lse, b.sm_scale)
    o_f = torch.full_like(b.q, float("nan"))
    l_f = torch.full(b.q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    fi.run(ws, info, b.q, b.k, b.v, kvi, o_f, l_f, b.sm_scale)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0 and info.num_prefill_items > 0
    o_ref, l_ref = oracle.attention(oracle_problem(b, rope=1))
    n = b.total_qo
    err_o, err_l = compare(o[:n], lse[:n], o_ref, l_ref)
    assert err_o <= O_TOL and err_l <= LSE_TOL, (err_o, err_l)
    assert float((o[:n].float() - o_f[:n].float()).abs().max()) <= O_TOL
    assert float((lse[:n] - l_f[:n]).abs().max()) <= LSE_TOL
    _prerotated_pass_check(b, q_rot, k_rot)


def test_rope_prerotated_refuses_a_replanned_workspace_with_cuda_core_items():
    """A plan whose items all run on the tensor cores sends the pre-rotated
    run to the kernel without RoPE; if the workspace has since been re-planned
    with decode-class items (which only the RoPE kernel rotates), the kernel
    records FI_ERR_DEVICE_CHECK and writes nothing."""
    qo, kv = [64, 1], [1000, 300]
    b = workloads.make_batch("tcx", "bf16", qo, kv, 8, 2, 16, 1, 611, DEV, pool_pages=sum((k + 15) // 16 for k in kv) + 2)
    ws = fi.Workspace(_cfg(4096), device=DEV)
    qo_a, kv_a = np.array([0, 64], np.int32), np.array([0, 63], np.int32)  # request 0 alone: 256 rows
    info_a = fi.plan(ws, qo_a, kv_a, b.kv_indices[:63], np.array([1000 - 62 * 16], np.int32), 8, 2, 128, 16, 1,
                     b.num_pages)
    assert info_a.num_decode_items == 0
    info_b = fi.plan(ws, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, 8, 2, 128, 16, 1, b.num_pages)
    assert info_b.num_decode_items > 0
    kvi = torch.as_tensor(b.kv_indices, device=DEV)
    k_rot = torch.zeros(b.k.shape, dtype=torch.float16, device=DEV)
    q_rot = torch.zeros(b.q.shape, dtype=torch.float16, device=DEV)
    o = torch.full_like(b.q, float("nan"))
    lse = torch.full(b.q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    fi.run_rope_prerotated(ws, info_a, b.q, b.k, b.v, kvi, q_rot, k_rot, o, lse, b.sm_scale)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 6  # FI_ERR_DEVICE_CHECK
    assert torch.isnan(o).all() and torch.isnan(lse).all()


@pytest.mark.parametrize("path", ["fused", "prerotated"])
def test_rope_fp16_range_guard(path):
    """A bf16 key whose rotation leaves the fp16 range (bf16 holds 1.5e5,
    fp16 tops out at 65504) is reported as FI_ERR_DEVICE_CHECK by the role or
    pass that rotated it; the same batch in range reports nothing."""
    qo, kv = [64], [500]
    b = workloads.make_batch("tcg", "bf16", qo, kv, 8, 2, 16, 1, 612, DEV, pool_pages=(500 + 15) // 16 + 2)
    ws = fi.Workspace(_cfg(4096), device=DEV)
    info = fi.plan(ws, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, 8, 2, 128, 16, 1, b.num_pages)
    kvi = torch.as_tensor(b.kv_indices, device=DEV)
    k_rot = torch.zeros(b.k.shape, dtype=torch.float16, device=DEV)
    q_rot = torch.zeros(b.q.shape, dtype=torch.float16, device=DEV)
    o = torch.empty_like(b.q)
    lse = torch.empty(b.q.shape[:2], dtype=torch.float32, device=DEV)

    def go():
        if path == "fused":
            fi.run(ws, info, b.q, b.k, b.v, kvi, o, lse, b.sm_scale)
        else:
            fi.run_rope_prerotated(ws, info, b.q, b.k, b.v, kvi, q_rot, k_rot, o, lse, b.sm_scale)
        torch.cuda.synchronize()
        return fi.device_status(ws)

    assert go() == 0
    page = int(b.kv_indices[3])
    b.k[page, 5, 1, 7] = 1.5e5  # key 53 of the request, KV head 1, dim 7
    assert go() == 6
    fi.plan(ws, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, 8, 2, 128, 16, 1, b.num_pages)
    b.k[page, 5, 1, 7] = 1.0
    assert go() == 0  # a new plan clears the status word


def test_prerotated_run_refusals():
    """A plan made without RoPE, or rotation buffers off the 16-byte grid, are
    refused on the host before anything is enqueued (outputs untouched)."""
    b = workloads.make_batch("tcr2", "bf16", [40], [300], 8, 2, 16, 1, 613, DEV, pool_pages=(300 + 15) // 16 + 2)
    kvi = torch.as_tensor(b.kv_indices, device=DEV)
    o = torch.full_like(b.q, float("nan"))
    lse = torch.full(b.q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    k_rot = torch.zeros(b.k.shape, dtype=torch.float16, device=DEV)
    q_rot = torch.zeros(b.q.shape, dtype=torch.float16, device=DEV)
    ws_p = fi.Workspace(fi.default_plan_config(0), device=DEV)
    info_p = fi.plan(ws_p, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, 8, 2, 128, 16, 1, b.num_pages)
    with pytest.raises(fi.FIError) as e:
        fi.run_rope_prerotated(ws_p, info_p, b.q, b.k, b.v, kvi, q_rot, k_rot, o, lse, b.sm_scale)
    assert e.value.status == 1
    ws_r = fi.Workspace(_cfg(4096), device=DEV)
    info_r = fi.plan(ws_r, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, 8, 2, 128, 16, 1, b.num_pages)
    flat = torch.zeros(k_rot.numel() + 8, dtype=torch.float16, device=DEV)
    k_off = flat[1:1 + k_rot.numel()].view(k_rot.shape)  # 2 bytes off the 16-byte grid
    with pytest.raises(fi.FIError) as e:
        fi.run_rope_prerotated(ws_r, info_r, b.q, b.k, b.v, kvi, q_rot, k_off, o, lse, b.sm_scale)
    assert e.value.status == 4
    torch.cuda.synchronize()
    assert torch.isnan(o).all()


@pytest.mark.parametrize("page,qo,kv", [
    (8, [64, 0, 40], [300, 100, 200]),        # a request with no query rows (nothing to rotate for it)
    (64, [33, 5, 100], [1000, 700, 100]),     # pages of 64: a 32-row pass unit spans half a page
    (32, [20, 1, 48], [20, 600, 48]),         # qo_len == kv_len: positions start at 0
])
def test_rope_prerotated_page_sizes(page, qo, kv):
    """The pre-rotation pass at other page sizes and with empty or exactly
    causal requests: against the oracle, and its buffers hold exactly the
    fp16 rotation of the prefill-class rows and keys.  Outputs here reach
    |o| > 2, where half an ulp of the stored bf16 value (2^-7 = 0.0078) is
    nearly the whole flat bar by itself and the fp16 rounding of the rotated
    q and k adds about 5e-4: above |o| = 2 the bar adds the storage rounding
    (2^-8 |o_ref|), as the peaked-softmax parity test does above 4; below 2
    it is the flat 8e-3.  (The fully fused run gives the same bits.)"""
    b = workloads.make_batch("tcq", "bf16", qo, kv, 8, 2, page, 1, 620 + page, DEV,
                             pool_pages=sum((k + page - 1) // page for k in kv) + 2)
    ws = fi.Workspace(_cfg(4096), device=DEV)
    info = fi.plan(ws, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, 8, 2, 128, page, 1, b.num_pages)
    kvi = torch.as_tensor(b.kv_indices, device=DEV)
    k_rot = torch.full(b.k.shape, float("nan"), dtype=torch.float16, device=DEV)
    q_rot = torch.full(b.q.shape, float("nan"), dtype=torch.float16, device=DEV)
    o = torch.full_like(b.q, float("nan"))
    lse = torch.full(b.q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    fi.run_rope_prerotated(ws, info, b.q, b.k, b.v, kvi, q_rot, k_rot, o, lse, b.sm_scale)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0 and info.num_prefill_items > 0
    o_ref, l_ref = oracle.attention(oracle_problem(b, rope=1))
    n = b.total_qo
    err_o, err_l = compare(o[:n], lse[:n], o_ref, l_ref)
    assert err_l <= LSE_TOL, err_l
    err = np.abs(o[:n].float().cpu().numpy() - o_ref)
    bar = np.where(np.abs(o_ref) < 2.0, O_TOL, O_TOL + 2.0 ** -8 * np.abs(o_ref))
    assert (err <= bar).all(), float((err - bar).max())
    _prerotated_pass_check(b, q_rot, k_rot)


@pytest.mark.parametrize("qo,kv", [([64, 40], [900, 300]), ([64, 1, 40], [900, 500, 300])])
def test_rope_prerotated_with_window_sink_cap(qo, kv):
    """The pre-rotated run on a plan with RoPE, a sliding window, sinks and a
    soft-cap: all tensor-core items (the kernel without RoPE, cap and mask
    kept) and with a decode-class request (the full RoPE kernel)."""
    b = workloads.make_batch("tcw", "bf16", qo, kv, 8, 2, 16, 1, 640 + len(qo), DEV,
                             pool_pages=sum((k + 15) // 16 for k in kv) + 2)
    cfg = _cfg(4096, window_left=200, sink_tokens=4, logits_soft_cap=30.0)
    ws = fi.Workspace(cfg, device=DEV)
    info = fi.plan(ws, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, 8, 2, 128, 16, 1, b.num_pages)
    assert info.variant == 7
    kvi = torch.as_tensor(b.kv_indices, device=DEV)
    k_rot = torch.zeros(b.k.shape, dtype=torch.float16, device=DEV)
    q_rot = torch.zeros(b.q.shape, dtype=torch.float16, device=DEV)
    o = torch.full_like(b.q, float("nan"))
    lse = torch.full(b.q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    fi.run_rope_prerotated(ws, info, b.q, b.k, b.v, kvi, q_rot, k_rot, o, lse, b.sm_scale)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0
    o_ref, l_ref = oracle.attention(oracle_problem(b, 200, 4, 30.0, rope=1))
    n = b.total_qo
    err_o, err_l = compare(o[:n], lse[:n], o_ref, l_ref)
    assert err_o <= O_TOL and err_l <= LSE_TOL, (err_o, err_l)

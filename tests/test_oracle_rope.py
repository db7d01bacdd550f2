"""Pins of the oracle's RoPE against things other than itself.

Reading (the FlashInfer paper summary, section "주요 성능 테스트 결과 / 2. 커널 수준 성능", names a kernel
that fuses RoPE with attention but gives no formula): Llama-style rotary
embedding on q and k, dims i and i + d/2 rotated by (pos / scale) *
theta^(-2i/d), key j at position j, query token t at Lkv - Lq + t.

Pins:
* relative positions: RoPE scores depend only on the query-key position
  difference, so a request whose keys all move back by P positions (P junk
  keys in front, hidden by a sliding window) gives the same result;
* a query and a key both at position 0 are not rotated;
* the rotation as a complex product (x_i + i x_{i+d/2}) * exp(i a) in numpy,
  then torch SDPA in fp64, matches the oracle.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import oracle_problem


@pytest.mark.parametrize("theta,scale", [(10000.0, 1.0), (500000.0, 1.0), (10000.0, 4.0)])
def test_shifting_every_position_changes_nothing(theta, scale):
    kv, front = [9, 23, 40], 37
    a = workloads.make_batch("rope", "bf16", [1, 1, 1], kv, 4, 2, 4, 0, 5, pool_pages=None, poison=False)
    o_a, l_a = oracle.attention(oracle_problem(a, rope=1, rope_theta=theta, rope_scale=scale))
    for r, n in enumerate(kv):
        # the same query and keys, with `front` other keys in front: every position moves by `front`
        sub = workloads.make_batch("shifted", "bf16", [1], [n + front], 4, 2, 4, 0, 100 + r, pool_pages=None,
                                   poison=False)
        pa = torch.as_tensor(a.kv_indices[a.kv_indptr[r]:a.kv_indptr[r + 1]], dtype=torch.long)
        ka = a.k[pa].reshape(-1, 2, 128)[:n]
        va = a.v[pa].reshape(-1, 2, 128)[:n]
        ps = sub.kv_indices
        for j in range(n):
            jj = front + j
            sub.k[int(ps[jj // 4]), jj % 4] = ka[j]
            sub.v[int(ps[jj // 4]), jj % 4] = va[j]
        sub.q.copy_(a.q[r:r + 1])
        # the query sits at front + n - 1; a window of n - 1 shows it exactly the moved keys
        o_b, l_b = oracle.attention(oracle_problem(sub, window_left=n - 1, rope=1, rope_theta=theta,
                                                   rope_scale=scale))
        np.testing.assert_allclose(o_b[0], o_a[r], rtol=0, atol=1e-10)
        np.testing.assert_allclose(l_b[0], l_a[r], rtol=0, atol=1e-10)
        # not vacuous: RoPE does change the result of this request
        assert not np.allclose(o_a[r], oracle.attention(oracle_problem(a))[0][r], atol=1e-6)


def test_position_zero_is_not_rotated():
    b = workloads.make_batch("p0", "bf16", [1], [1], 4, 2, 4, 1, 9, pool_pages=None, poison=False)
    o0, l0 = oracle.attention(oracle_problem(b))
    o1, l1 = oracle.attention(oracle_problem(b, rope=1))
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


def _rope_complex(x: np.ndarray, pos: np.ndarray, theta: float, scale: float) -> np.ndarray:
    """x[..., pos_axis, d] rotated as complex numbers x_i + i x_{i+d/2}."""
    d = x.shape[-1]
    z = x[..., : d // 2] + 1j * x[..., d // 2:]
    freq = theta ** (-2.0 * np.arange(d // 2) / d)
    z = z * np.exp(1j * (pos[:, None] / scale) * freq[None, :])
    return np.concatenate([z.real, z.imag], axis=-1)


@pytest.mark.parametrize("causal,theta,scale", [(1, 10000.0, 1.0), (0, 500000.0, 2.0)])
def test_matches_complex_rotation_and_sdpa(causal, theta, scale):
    b = workloads.random_batch(71 + causal, batch=3, qo_max=5, kv_max=60, num_qo_heads=4, num_kv_heads=2,
                               page_size=4, causal=causal, kv_min=5)
    lq, lkv = np.diff(b.qo_indptr), b.kv_lens()
    keep = lq <= lkv
    assert keep.all()
    o, lse = oracle.attention(oracle_problem(b, rope=1, rope_theta=theta, rope_scale=scale))
    G = 2
    for r in range(b.batch):
        q0, q1 = int(b.qo_indptr[r]), int(b.qo_indptr[r + 1])
        pages = b.kv_indices[b.kv_indptr[r]:b.kv_indptr[r + 1]]
        idx = torch.as_tensor(pages, dtype=torch.long)
        k = b.k.double()[idx].reshape(-1, 2, 128)[:lkv[r]].numpy()            # [Lkv, Hkv, d]
        v = b.v.double()[idx].reshape(-1, 2, 128)[:lkv[r]]
        q = b.q.double()[q0:q1].numpy()                                       # [Lq, Hq, d]
        qpos = lkv[r] - lq[r] + np.arange(lq[r])
        kpos = np.arange(lkv[r])
        qr = _rope_complex(np.transpose(q, (1, 0, 2)), qpos, theta, scale)   # [Hq, Lq, d]
        kr = _rope_complex(np.transpose(k, (1, 0, 2)), kpos, theta, scale)   # [Hkv, Lkv, d]
        qq = torch.as_tensor(qr).unsqueeze(0)
        kk = torch.as_tensor(kr).repeat_interleave(G, dim=0).unsqueeze(0)
        vv = v.permute(1, 0, 2).repeat_interleave(G, dim=0).unsqueeze(0)
        t = torch.arange(lq[r]).unsqueeze(1)
        j = torch.arange(lkv[r]).unsqueeze(0)
        mask = (j <= lkv[r] - lq[r] + t) if causal else torch.ones(lq[r], lkv[r], dtype=torch.bool)
        out = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=b.sm_scale)
        ls = torch.logsumexp((qq @ kk.transpose(-1, -2) * b.sm_scale).masked_fill(~mask, float("-inf")), dim=-1)
        np.testing.assert_allclose(o[q0:q1], out[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-11)
        np.testing.assert_allclose(lse[q0:q1], ls[0].T.numpy(), rtol=0, atol=1e-11)

"""Seeded synthetic inputs shaped like the serving mixes of the FlashInfer pages.

This module only draws inputs (lengths, page tables, N(0,1) values, poison);
it holds none of the attention arithmetic and serves both the CUDA path and
the oracle.  Lengths and page permutations come from numpy's PCG64 generator
(seed = 1000 * workload + replan); values come from a seeded torch generator
on the device the tensors live on, drawn in fp32 and rounded once (RNE) to the
storage type.

Poison (so indexing and masking mistakes show as large errors):
  * pages of the pool that no request references are filled with NaN;
  * the slots past last_page_len of every last page hold +BIG in K and -BIG
    in V (BIG = 6e4 for fp16, 1e30 for bf16), finite so that a correctly
    masked slot contributes exactly 0.

Workloads (the serving mixes they stand in for, with their sizes):
  tiny_decode        fp16, 4 requests, qo 1, kv U{1..512}, 8/2 heads, page 16, 256-page pool
  llama8b_decode     bf16, 64 requests, qo 1, kv floor(exp U(ln 512, ln 32768)), 32/8 heads, page 16
  ragged_prefill     bf16, 16 requests, qo U{128..4096}, prefix U{0..2048}, causal, 32/8 heads, page 16
  shared_prefix      bf16, prefix 8192 tokens (dense, as pages of 16 with identity indices) + 64 branches
                     with private suffixes U{64..512} at page 1; also the flat page-1 layout
  continuous_batch   bf16, 8 chunked-prefill requests (qo 512, prefix U{0..16384}, causal) + 120 decode
                     requests with kv clip(zipf(1.2), 128, 65536); V stored with one extra padding head,
                     so K and V strides differ
  mla_decode         bf16 absorbed-MLA decode, 64 requests, qo 1, the llama8b_decode length mix, 128 heads,
                     latent 512 + RoPE key 64 per token, page 64
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

HEAD_DIM = 128
_BIG = {"fp16": 6.0e4, "bf16": 1.0e30}
_TORCH = {"fp16": torch.float16, "bf16": torch.bfloat16}


@dataclass
class PagedBatch:
    name: str
    dtype: str
    qo_indptr: np.ndarray
    kv_indptr: np.ndarray
    kv_indices: np.ndarray
    last_page_len: np.ndarray
    num_qo_heads: int
    num_kv_heads: int
    page_size: int
    causal: int
    sm_scale: float
    q: torch.Tensor          # [tokens, Hq, d]
    k: torch.Tensor          # [pages, P, Hkv, d] (may be a strided view)
    v: torch.Tensor
    k_base: torch.Tensor = field(repr=False, default=None)   # storage k is a view of
    v_base: torch.Tensor = field(repr=False, default=None)
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return len(self.qo_indptr) - 1

    @property
    def num_pages(self) -> int:
        return int(self.k.shape[0])

    @property
    def total_qo(self) -> int:
        return int(self.qo_indptr[-1])

    def kv_lens(self) -> np.ndarray:
        pages = np.diff(self.kv_indptr).astype(np.int64)
        return np.where(pages == 0, 0, (pages - 1) * self.page_size + self.last_page_len[:self.batch])

    def qo_lens(self) -> np.ndarray:
        return np.diff(self.qo_indptr).astype(np.int64)


def torch_dtype(name: str) -> torch.dtype:
    return _TORCH[name]


def _fill_normal(t: torch.Tensor, gen: torch.Generator, chunk: int = 1 << 26, std: float = 1.0) -> None:
    flat = t.view(-1)
    for s in range(0, flat.numel(), chunk):
        part = flat[s:s + chunk]
        x = torch.randn(part.numel(), generator=gen, device=t.device, dtype=torch.float32)
        part.copy_(x if std == 1.0 else x * std)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _pages_for(kv_lens: np.ndarray, page_size: int):
    n = (kv_lens + page_size - 1) // page_size
    indptr = np.zeros(len(kv_lens) + 1, dtype=np.int32)
    indptr[1:] = np.cumsum(n)
    last = np.where(n == 0, 1, kv_lens - (n - 1) * page_size).astype(np.int32)
    return indptr, last


def _poison(batch: PagedBatch) -> None:
    """NaN into unreferenced pages, +-BIG into the tails of last pages."""
    used = np.zeros(batch.num_pages, dtype=bool)
    nnz = int(batch.kv_indptr[-1])
    used[batch.kv_indices[:nnz]] = True
    unused = np.nonzero(~used)[0]
    big = _BIG[batch.dtype]
    with torch.no_grad():
        if unused.size:
            idx = torch.as_tensor(unused, device=batch.k.device, dtype=torch.long)
            batch.k.index_fill_(0, idx, float("nan"))
            batch.v.index_fill_(0, idx, float("nan"))
        P = batch.page_size
        for b in range(batch.batch):
            n = int(batch.kv_indptr[b + 1] - batch.kv_indptr[b])
            lpl = int(batch.last_page_len[b])
            if n == 0 or lpl == P:
                continue
            page = int(batch.kv_indices[batch.kv_indptr[b + 1] - 1])
            batch.k[page, lpl:] = big
            batch.v[page, lpl:] = -big


def make_batch(name: str, dtype: str, qo_lens, kv_lens, num_qo_heads: int, num_kv_heads: int, page_size: int,
               causal: int, seed: int, device="cpu", pool_pages: int | None = None, v_pad_heads: int = 0,
               q_tokens: int | None = None, poison: bool = True, rng: np.random.Generator | None = None,
               sm_scale: float | None = None) -> PagedBatch:
    """A paged batch with shuffled physical pages and N(0,1) values."""
    rng = rng if rng is not None else np.random.default_rng(seed)
    qo_lens = np.asarray(qo_lens, dtype=np.int64)
    kv_lens = np.asarray(kv_lens, dtype=np.int64)
    qo_indptr = np.zeros(len(qo_lens) + 1, dtype=np.int32)
    qo_indptr[1:] = np.cumsum(qo_lens)
    kv_indptr, last = _pages_for(kv_lens, page_size)
    nnz = int(kv_indptr[-1])
    pool = max(nnz, pool_pages or 0, 1)
    kv_indices = rng.permutation(pool)[:nnz].astype(np.int32)
    tdt = _TORCH[dtype]
    gen = _gen(device, seed)
    tokens = max(int(qo_indptr[-1]), q_tokens or 0, 1)
    q = torch.empty((tokens, num_qo_heads, HEAD_DIM), dtype=tdt, device=device)
    k_base = torch.empty((pool, page_size, num_kv_heads, HEAD_DIM), dtype=tdt, device=device)
    v_base = torch.empty((pool, page_size, num_kv_heads + v_pad_heads, HEAD_DIM), dtype=tdt, device=device)
    for t in (q, k_base, v_base):
        _fill_normal(t, gen)
    v = v_base[:, :, :num_kv_heads, :]
    b = PagedBatch(name, dtype, qo_indptr, kv_indptr, kv_indices, last, num_qo_heads, num_kv_heads, page_size,
                   int(causal), float(sm_scale if sm_scale is not None else 1.0 / np.sqrt(HEAD_DIM)), q, k_base,
                   v, k_base, v_base)
    if poison:
        _poison(b)
    return b


# ---------------------------------------------------------------- workloads


def tiny_decode(device="cpu", replan: int = 0) -> PagedBatch:
    seed = 1000 * 1 + replan
    rng = np.random.default_rng(seed)
    kv = rng.integers(1, 513, size=4)
    return make_batch("tiny_decode", "fp16", np.ones(4, np.int64), kv, 8, 2, 16, 0, seed, device,
                      pool_pages=256, rng=rng)


def llama8b_decode_lengths(rng: np.random.Generator, batch: int = 64) -> np.ndarray:
    return np.floor(np.exp(rng.uniform(np.log(512), np.log(32768), size=batch))).astype(np.int64)


def llama8b_decode(device="cpu", replan: int = 0, batch: int = 64) -> PagedBatch:
    seed = 1000 * 2 + replan
    rng = np.random.default_rng(seed)
    kv = llama8b_decode_lengths(rng, batch)
    return make_batch("llama8b_decode", "bf16", np.ones(batch, np.int64), kv, 32, 8, 16, 0, seed, device, rng=rng)


def ragged_prefill_lengths(rng: np.random.Generator, batch: int = 16, qo_max: int = 4096, prefix_max: int = 2048):
    qo = rng.integers(128, qo_max + 1, size=batch)
    prefix = rng.integers(0, prefix_max + 1, size=batch)
    return qo, prefix + qo


def ragged_prefill(device="cpu", replan: int = 0, batch: int = 16, qo_max: int = 4096,
                   prefix_max: int = 2048) -> PagedBatch:
    seed = 1000 * 3 + replan
    rng = np.random.default_rng(seed)
    qo, kv = ragged_prefill_lengths(rng, batch, qo_max, prefix_max)
    return make_batch("ragged_prefill", "bf16", qo, kv, 32, 8, 16, 1, seed, device, rng=rng)


def shared_prefix(device="cpu", replan: int = 0, prefix_len: int = 8192, branches: int = 64,
                  suffix_lo: int = 64, suffix_hi: int = 512, prefix_page: int = 16) -> dict:
    """The composable-format case.  One page-1 pool holds the prefix in its
    first prefix_len pages (contiguous) and the branches' suffix tokens on
    shuffled pages after it.  Returns three batches over that one pool:
      prefix -- 1 request whose queries are the branch tokens, KV = the dense
                prefix viewed as pages of `prefix_page` with identity indices;
      suffix -- one request per branch, qo 1, page-1 suffix pages;
      flat   -- one request per branch, qo 1, pages [0..prefix_len) + suffix."""
    seed = 1000 * 4 + replan
    rng = np.random.default_rng(seed)
    suf = rng.integers(suffix_lo, suffix_hi + 1, size=branches).astype(np.int64)
    nsuf = int(suf.sum())
    pool = prefix_len + nsuf
    tdt = _TORCH["bf16"]
    gen = _gen(device, seed)
    Hq, Hkv = 32, 8
    q = torch.empty((branches, Hq, HEAD_DIM), dtype=tdt, device=device)
    k_base = torch.empty((pool, 1, Hkv, HEAD_DIM), dtype=tdt, device=device)
    v_base = torch.empty((pool, 1, Hkv, HEAD_DIM), dtype=tdt, device=device)
    for t in (q, k_base, v_base):
        _fill_normal(t, gen)
    suffix_pages = (prefix_len + rng.permutation(nsuf)).astype(np.int32)
    ones = np.ones(branches, np.int64)
    scale = 1.0 / np.sqrt(HEAD_DIM)
    sind = np.zeros(branches + 1, np.int32)
    sind[1:] = np.cumsum(suf)
    suffix = PagedBatch("shared_prefix.suffix", "bf16", np.arange(branches + 1, dtype=np.int32), sind,
                        suffix_pages, np.ones(branches, np.int32), Hq, Hkv, 1, 0, scale, q, k_base, v_base,
                        k_base, v_base)
    npre = prefix_len // prefix_page
    pk = k_base[:prefix_len].view(npre, prefix_page, Hkv, HEAD_DIM)
    pv = v_base[:prefix_len].view(npre, prefix_page, Hkv, HEAD_DIM)
    prefix = PagedBatch("shared_prefix.prefix", "bf16", np.array([0, branches], np.int32),
                        np.array([0, npre], np.int32), np.arange(npre, dtype=np.int32),
                        np.array([prefix_page], np.int32), Hq, Hkv, prefix_page, 0, scale, q, pk, pv, k_base,
                        v_base, meta={"prefix_len": prefix_len})
    flat_idx = np.concatenate([np.concatenate([np.arange(prefix_len, dtype=np.int32),
                                               suffix_pages[sind[i]:sind[i + 1]]]) for i in range(branches)])
    find = np.zeros(branches + 1, np.int32)
    find[1:] = np.cumsum(suf + prefix_len)
    flat = PagedBatch("shared_prefix.flat", "bf16", np.arange(branches + 1, dtype=np.int32), find, flat_idx,
                      np.ones(branches, np.int32), Hq, Hkv, 1, 0, scale, q, k_base, v_base, k_base, v_base)
    del ones
    return {"prefix": prefix, "suffix": suffix, "flat": flat}


def continuous_batch_lengths(rng: np.random.Generator, n_prefill: int = 8, n_decode: int = 120,
                             chunk: int = 512, prefix_max: int = 16384, kv_max: int = 65536):
    prefix = rng.integers(0, prefix_max + 1, size=n_prefill)
    dec = np.clip(rng.zipf(1.2, size=n_decode), 128, kv_max)
    qo = np.concatenate([np.full(n_prefill, chunk), np.ones(n_decode, np.int64)])
    kv = np.concatenate([prefix + chunk, dec])
    return qo.astype(np.int64), kv.astype(np.int64)


def continuous_batch(device="cpu", replan: int = 0, pool_pages: int | None = None, q_tokens: int | None = None,
                     n_prefill: int = 8, n_decode: int = 120, chunk: int = 512, prefix_max: int = 16384,
                     kv_max: int = 65536, poison: bool = True) -> PagedBatch:
    seed = 1000 * 5 + replan
    rng = np.random.default_rng(seed)
    qo, kv = continuous_batch_lengths(rng, n_prefill, n_decode, chunk, prefix_max, kv_max)
    return make_batch("continuous_batch", "bf16", qo, kv, 32, 8, 16, 1, seed, device, pool_pages=pool_pages,
                      v_pad_heads=1, q_tokens=q_tokens, poison=poison, rng=rng)


def continuous_batch_capacity(replans: int = 10, **kw) -> tuple[int, int]:
    """Pool pages and query tokens that hold every one of the first `replans` draws."""
    pages = tokens = 0
    for r in range(replans):
        rng = np.random.default_rng(1000 * 5 + r)
        qo, kv = continuous_batch_lengths(rng, **kw)
        pages = max(pages, int(((kv + 15) // 16).sum()))
        tokens = max(tokens, int(qo.sum()))
    return pages, tokens


def random_batch(seed: int, batch: int, qo_max: int, kv_max: int, num_qo_heads: int, num_kv_heads: int,
                 page_size: int, causal: int, dtype: str = "bf16", device="cpu", kv_min: int = 0,
                 qo_min: int = 1, extra_pages: int = 3, v_pad_heads: int = 0) -> PagedBatch:
    """Small random batches for parity sweeps (edge cases included by the caller's ranges)."""
    rng = np.random.default_rng(seed)
    qo = rng.integers(qo_min, qo_max + 1, size=batch)
    kv = rng.integers(kv_min, kv_max + 1, size=batch)
    nnz = int(((kv + page_size - 1) // page_size).sum())
    return make_batch(f"random{seed}", dtype, qo, kv, num_qo_heads, num_kv_heads, page_size, causal, seed, device,
                      pool_pages=nnz + extra_pages, rng=rng, v_pad_heads=v_pad_heads)


def cascade_batch(seed: int, block_sizes, qo_max: int, kv_max: int, shared_max: int, num_qo_heads: int,
                  num_kv_heads: int, page_size: int, shared_page_size: int, causal: int, dtype: str = "bf16",
                  device="cpu", qo_min: int = 1, kv_min: int = 0, shared_min: int = 0, poison: bool = True) -> dict:
    """A two-level batch: requests grouped into consecutive blocks of
    block_sizes[s] requests, each block with its own shared keys (a pool of
    pages of shared_page_size, shuffled) and each request with its own keys
    (a pool of pages of page_size, shuffled).  Returns
      shared -- the blocks as a batch: block s owns the query rows of its
                requests and the block's pages;
      own    -- the requests' own batch (its q is the queries of both levels);
      flat   -- the same attention as one page-1 batch for the oracle: request
                r's keys are its block's keys followed by its own (gathered).
    With causal, every request holds at least as many own keys as queries."""
    rng = np.random.default_rng(seed)
    block_sizes = np.asarray(block_sizes, dtype=np.int64)
    B = int(block_sizes.sum())
    qo = rng.integers(qo_min, qo_max + 1, size=B)
    kv = rng.integers(kv_min, kv_max + 1, size=B)
    if causal:
        kv = np.maximum(kv, qo)
    skv = rng.integers(shared_min, shared_max + 1, size=len(block_sizes))
    own = make_batch(f"cascade{seed}.own", dtype, qo, kv, num_qo_heads, num_kv_heads, page_size, causal, seed,
                     device, pool_pages=int(((kv + page_size - 1) // page_size).sum()) + 2, rng=rng, poison=poison)
    first = np.concatenate([[0], np.cumsum(block_sizes)])
    sqo = own.qo_indptr[first].astype(np.int32)
    shared = make_batch(f"cascade{seed}.shared", dtype, np.diff(sqo), skv, num_qo_heads, num_kv_heads,
                        shared_page_size, 0, seed + 1, device,
                        pool_pages=int(((skv + shared_page_size - 1) // shared_page_size).sum()) + 2, rng=rng,
                        poison=poison)
    shared.q = own.q
    # flat: per request, its block's tokens then its own tokens, as pages of 1
    def tokens(b: PagedBatch, r: int):
        n = int(b.kv_lens()[r])
        j = np.arange(n)
        return b.kv_indices[b.kv_indptr[r] + j // b.page_size].astype(np.int64), j % b.page_size
    ks, vs, lens = [], [], []
    for s_ in range(len(block_sizes)):
        sp, ss = tokens(shared, s_)
        for r in range(int(first[s_]), int(first[s_ + 1])):
            op, os_ = tokens(own, r)
            idx = lambda a: torch.as_tensor(a, device=device, dtype=torch.long)  # noqa: E731
            ks.append(torch.cat([shared.k[idx(sp), idx(ss)], own.k[idx(op), idx(os_)]]))
            vs.append(torch.cat([shared.v[idx(sp), idx(ss)], own.v[idx(op), idx(os_)]]))
            lens.append(len(sp) + len(op))
    lens = np.asarray(lens, dtype=np.int64)
    tot = int(lens.sum())
    fk = torch.cat(ks).reshape(tot, 1, num_kv_heads, HEAD_DIM) if tot else own.k[:0, :1]
    fv = torch.cat(vs).reshape(tot, 1, num_kv_heads, HEAD_DIM) if tot else own.v[:0, :1]
    find = np.zeros(B + 1, np.int32)
    find[1:] = np.cumsum(lens)
    flat = PagedBatch(f"cascade{seed}.flat", dtype, own.qo_indptr, find, np.arange(tot, dtype=np.int32),
                      np.ones(B, np.int32), num_qo_heads, num_kv_heads, 1, causal, own.sm_scale, own.q, fk, fv,
                      fk, fv)
    return {"shared": shared, "own": own, "flat": flat}


def to_numpy_storage(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns (fp16/bf16) of a tensor, on the host, strides kept."""
    if t.dtype == torch.float32:
        return t.detach().cpu().numpy()
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def host_views(b: PagedBatch):
    """Host numpy storage of q, k, v with the same element strides as the device views."""
    q = to_numpy_storage(b.q.contiguous())
    kb = to_numpy_storage(b.k_base)
    vb = to_numpy_storage(b.v_base)
    k = np.lib.stride_tricks.as_strided(kb, shape=tuple(b.k.shape),
                                        strides=tuple(s * kb.itemsize for s in b.k.stride()))
    v = np.lib.stride_tricks.as_strided(vb, shape=tuple(b.v.shape),
                                        strides=tuple(s * vb.itemsize for s in b.v.stride()))
    return q, k, v


# ---------------------------------------------------------------- MLA decode inputs

MLA_DC = 512   # latent (compressed KV) dims
MLA_DR = 64    # decoupled RoPE key dims
MLA_Q_STD = (1.0 / 3.0) ** 0.5


@dataclass
class MlaBatch:
    """Absorbed-MLA decode inputs: one query token per request.
    q_nope [B, H, 512] is the query already multiplied by the absorbed key
    up-projection, q_pe [B, H, 64] its RoPE part; ckv [pages, P, 512] holds the
    latents and kpe [pages, P, 64] the RoPE keys, paged like the GQA cache."""
    name: str
    kv_indptr: np.ndarray
    kv_indices: np.ndarray
    last_page_len: np.ndarray
    num_heads: int
    page_size: int
    sm_scale: float
    q_nope: torch.Tensor
    q_pe: torch.Tensor
    ckv: torch.Tensor
    kpe: torch.Tensor
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return len(self.kv_indptr) - 1

    @property
    def num_pages(self) -> int:
        return int(self.ckv.shape[0])

    def kv_lens(self) -> np.ndarray:
        pages = np.diff(self.kv_indptr).astype(np.int64)
        return np.where(pages == 0, 0, (pages - 1) * self.page_size + self.last_page_len[:self.batch])


def make_mla_batch(name: str, kv_lens, num_heads: int, page_size: int, seed: int, device="cpu",
                   pool_pages: int | None = None, poison: bool = True, rng: np.random.Generator | None = None,
                   sm_scale: float | None = None) -> MlaBatch:
    """Shuffled physical pages, N(0,1) bf16 latents and RoPE keys, N(0,1/3)
    queries.  The default scale is that
    of the un-absorbed head, 1/sqrt(128 + 64).  Poison as for the GQA batches:
    NaN in unreferenced pages, +BIG in both caches past last_page_len."""
    rng = rng if rng is not None else np.random.default_rng(seed)
    kv_lens = np.asarray(kv_lens, dtype=np.int64)
    kv_indptr, last = _pages_for(kv_lens, page_size)
    nnz = int(kv_indptr[-1])
    pool = max(nnz, pool_pages or 0, 1)
    kv_indices = rng.permutation(pool)[:nnz].astype(np.int32)
    gen = _gen(device, seed)
    B = len(kv_lens)
    bf = torch.bfloat16
    q_nope = torch.empty((max(B, 1), num_heads, MLA_DC), dtype=bf, device=device)
    q_pe = torch.empty((max(B, 1), num_heads, MLA_DR), dtype=bf, device=device)
    ckv = torch.empty((pool, page_size, MLA_DC), dtype=bf, device=device)
    kpe = torch.empty((pool, page_size, MLA_DR), dtype=bf, device=device)
    # queries N(0, 1/3): with 576 contracted dims and scale 1/sqrt(192) the
    # logits then spread like those of the GQA workloads (unit variance)
    for t, std in ((q_nope, MLA_Q_STD), (q_pe, MLA_Q_STD), (ckv, 1.0), (kpe, 1.0)):
        _fill_normal(t, gen, std=std)
    b = MlaBatch(name, kv_indptr, kv_indices, last, num_heads, page_size,
                 float(sm_scale if sm_scale is not None else 1.0 / np.sqrt(128 + MLA_DR)), q_nope, q_pe, ckv, kpe)
    if poison:
        used = np.zeros(pool, dtype=bool)
        used[kv_indices] = True
        unused = np.nonzero(~used)[0]
        with torch.no_grad():
            if unused.size:
                idx = torch.as_tensor(unused, device=device, dtype=torch.long)
                ckv.index_fill_(0, idx, float("nan"))
                kpe.index_fill_(0, idx, float("nan"))
            for r in range(B):
                n = int(kv_indptr[r + 1] - kv_indptr[r])
                lpl = int(last[r])
                if n == 0 or lpl == page_size:
                    continue
                page = int(kv_indices[kv_indptr[r + 1] - 1])
                ckv[page, lpl:] = _BIG["bf16"]
                kpe[page, lpl:] = _BIG["bf16"]
    return b


def mla_decode(device="cpu", replan: int = 0, batch: int = 64, num_heads: int = 128,
               page_size: int = 64) -> MlaBatch:
    """DeepSeek-V3-shaped absorbed-MLA decode: 128 heads, latent 512 + RoPE
    64, page 64, the llama8b_decode length mix."""
    seed = 1000 * 6 + replan
    rng = np.random.default_rng(seed)
    kv = llama8b_decode_lengths(rng, batch)
    return make_mla_batch("mla_decode", kv, num_heads, page_size, seed, device, rng=rng)


def random_mla_batch(seed: int, batch: int, kv_max: int, num_heads: int, page_size: int, device="cpu",
                     kv_min: int = 0) -> MlaBatch:
    rng = np.random.default_rng(seed)
    kv = rng.integers(kv_min, kv_max + 1, size=batch)
    extra = int(rng.integers(0, 8))
    pool = int(((kv + page_size - 1) // page_size).sum()) + extra
    return make_mla_batch(f"random_mla{seed}", kv, num_heads, page_size, seed, device, pool_pages=pool, rng=rng)

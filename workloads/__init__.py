"""Seeded synthetic inputs for block-sparse paged attention.

This module only builds inputs: request lengths, a page pool laid out as a
paged (BSR) KV cache with a seeded permutation of physical pages, and N(0, 1)
values. It holds none of the attention arithmetic; the oracle and the CUDA
path both consume what it returns.

Recipe (numpy PCG64, ``default_rng(seed)``; every integer draw is inclusive):
1. lengths are drawn first, then the page permutation, then q, then K, then V;
2. values are float32 N(0, 1), rounded to the stated dtype (bf16 by
   round-to-nearest-even, or kept as fp32);
3. page slots that no request uses, and the tail of each last page beyond
   ``last_page_len``, are set to NaN in K and V, so any read of them shows up
   as NaN in the output.

The five named workloads follow the five benchmark shapes: a tiny fp32 paged
decode, a Llama-3-8B-shaped batched paged decode, a 70B-shaped page-size-1
("vector-sparse") decode with a contiguous twin, a ragged causal prefill, and a
shared-prefix decode split into a prefix view and a suffix view.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np
import torch

_TORCH_DTYPES = {"bf16": torch.bfloat16, "f32": torch.float32}


@dataclass
class PagedBatch:
    """Inputs of one attention call over a paged KV cache (host tensors)."""
    name: str
    dtype: str                 # "bf16" or "f32"
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    causal: bool
    sm_scale: float
    qo_indptr: np.ndarray      # int32 [B + 1]
    kv_indptr: np.ndarray      # int32 [B + 1]  (pages)
    kv_indices: np.ndarray     # int32 [total pages]
    last_page_len: np.ndarray  # int32 [B]
    q: torch.Tensor            # [n_tokens, H_qo, D]
    k_pages: torch.Tensor      # [num_pages, page_size, H_kv, D]
    v_pages: torch.Tensor
    meta: dict = field(default_factory=dict)
    window_left: int = -1    # sliding window (> 0) or none
    soft_cap: float = 0.0    # logits soft-cap c (> 0) or none

    @property
    def batch(self) -> int:
        return len(self.qo_indptr) - 1

    @property
    def qo_lens(self) -> np.ndarray:
        return np.diff(self.qo_indptr).astype(np.int64)

    @property
    def kv_lens(self) -> np.ndarray:
        npages = np.diff(self.kv_indptr).astype(np.int64)
        return np.where(npages > 0, (npages - 1) * self.page_size + self.last_page_len, 0)

    @property
    def is_decode(self) -> bool:
        return bool(np.all(self.qo_lens == 1))


def _round(x: np.ndarray, dtype: str) -> torch.Tensor:
    return torch.from_numpy(x).to(_TORCH_DTYPES[dtype])


def _normal(rng, shape, dtype):
    return _round(rng.standard_normal(size=shape, dtype=np.float32), dtype)


def _pages_for(kv_lens, page_size):
    npages = np.array([-(-int(n) // page_size) for n in kv_lens], np.int64)
    last = np.array([int(n) - (p - 1) * page_size if p > 0 else 0 for n, p in zip(kv_lens, npages)],
                    np.int32)
    return npages, last


def _poison(k, v, used_pages, npages_per_req, last, page_pool_ids, page_size):
    """NaN in unused pages and in the tail of every last page."""
    num_pages = k.shape[0]
    unused = np.ones(num_pages, bool)
    unused[used_pages] = False
    if unused.any():
        idx = torch.from_numpy(np.nonzero(unused)[0])
        k[idx] = float("nan")
        v[idx] = float("nan")
    for pages, n, lp in zip(page_pool_ids, npages_per_req, last):
        if n > 0 and lp < page_size:
            k[int(pages[-1]), int(lp):] = float("nan")
            v[int(pages[-1]), int(lp):] = float("nan")


def paged_batch(seed: int, qo_lens, kv_lens, num_qo_heads: int, num_kv_heads: int, head_dim: int,
                page_size: int, dtype: str = "bf16", causal: bool = False, sm_scale: float | None = None,
                extra_pages: int = 0, name: str = "random", rng=None, contiguous: bool = False) -> PagedBatch:
    """A batch with the given lengths; pages drawn as a seeded permutation of the pool.

    extra_pages adds unused (NaN) pages to the pool; contiguous=True lays the
    pages out in request order instead of permuting them.
    """
    rng = rng if rng is not None else np.random.default_rng(seed)
    qo_lens = np.asarray(qo_lens, np.int64)
    kv_lens = np.asarray(kv_lens, np.int64)
    B = len(qo_lens)
    npages, last = _pages_for(kv_lens, page_size)
    total = int(npages.sum())
    pool = total + extra_pages
    perm = np.arange(pool, dtype=np.int64) if contiguous else rng.permutation(pool)
    kv_indptr = np.zeros(B + 1, np.int32)
    kv_indptr[1:] = np.cumsum(npages)
    kv_indices = perm[:total].astype(np.int32)
    qo_indptr = np.zeros(B + 1, np.int32)
    qo_indptr[1:] = np.cumsum(qo_lens)
    n_tok = int(qo_indptr[-1])
    q = _normal(rng, (n_tok, num_qo_heads, head_dim), dtype)
    k = _normal(rng, (pool, page_size, num_kv_heads, head_dim), dtype)
    v = _normal(rng, (pool, page_size, num_kv_heads, head_dim), dtype)
    per_req = [kv_indices[kv_indptr[b]:kv_indptr[b + 1]] for b in range(B)]
    _poison(k, v, kv_indices, npages, last, per_req, page_size)
    return PagedBatch(name=name, dtype=dtype, num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads,
                      head_dim=head_dim, page_size=page_size, causal=causal,
                      sm_scale=(1.0 / math.sqrt(head_dim)) if sm_scale is None else sm_scale,
                      qo_indptr=qo_indptr, kv_indptr=kv_indptr, kv_indices=kv_indices,
                      last_page_len=last, q=q, k_pages=k, v_pages=v)


# ---------------------------------------------------------------------------
# The five benchmark workloads
# ---------------------------------------------------------------------------

def tiny_decode_f32() -> PagedBatch:
    """3 decode requests, KV 10/3/7 tokens, page size 4, a 16-page permuted pool,
    4 qo / 2 kv heads, head_dim 64, fp32, sm_scale 1/8 (seed 1)."""
    rng = np.random.default_rng(1)
    kv = np.array([10, 3, 7])
    npages, last = _pages_for(kv, 4)          # 3, 1, 2 pages
    perm = rng.permutation(16)
    kv_indptr = np.array([0, 3, 4, 6], np.int32)
    kv_indices = perm[:6].astype(np.int32)
    q = _normal(rng, (3, 4, 64), "f32")
    k = _normal(rng, (16, 4, 2, 64), "f32")
    v = _normal(rng, (16, 4, 2, 64), "f32")
    per_req = [kv_indices[kv_indptr[b]:kv_indptr[b + 1]] for b in range(3)]
    _poison(k, v, kv_indices, npages, last, per_req, 4)
    return PagedBatch(name="tiny_decode_f32", dtype="f32", num_qo_heads=4, num_kv_heads=2, head_dim=64,
                      page_size=4, causal=False, sm_scale=1.0 / 8, qo_indptr=np.arange(4, dtype=np.int32),
                      kv_indptr=kv_indptr, kv_indices=kv_indices, last_page_len=last, q=q, k_pages=k,
                      v_pages=v)


def batched_decode_lengths(batch: int = 64, seed: int = 2):
    """(generator after the draw, KV lengths) of the batched decode: U{512..8192}."""
    rng = np.random.default_rng(seed)
    return rng, rng.integers(512, 8192, size=batch, endpoint=True)


def batched_decode_bf16(batch: int = 64, seed: int = 2) -> PagedBatch:
    """Llama-3-8B layer shape: batch 64, KV ~ U{512..8192}, page 16, a pool sized to
    the total and permuted, 32 qo / 8 kv heads, head_dim 128, bf16."""
    rng, kv = batched_decode_lengths(batch, seed)
    b = paged_batch(seed, np.ones(batch, np.int64), kv, 32, 8, 128, 16, "bf16", rng=rng,
                    name="batched_decode_bf16")
    return b


def vector_sparse_decode_bf16(batch: int = 32, kv_len: int = 4096, seed: int = 3):
    """70B-like heads: batch 32 x 4096 tokens, page size 1 (every token slot of the
    131072-slot pool permuted), 64 qo / 8 kv heads, head_dim 128, bf16.

    Returns (permuted, contiguous): the same logical KV, once scattered and once
    laid out in request order (indices = arange)."""
    rng = np.random.default_rng(seed)
    n = batch * kv_len
    perm = rng.permutation(n)
    q = _normal(rng, (batch, 64, 128), "bf16")
    k_log = _normal(rng, (n, 1, 8, 128), "bf16")   # logical order: request-major
    v_log = _normal(rng, (n, 1, 8, 128), "bf16")
    kv_indptr = (np.arange(batch + 1, dtype=np.int64) * kv_len).astype(np.int32)
    last = np.ones(batch, np.int32)
    qo_indptr = np.arange(batch + 1, dtype=np.int32)
    # permuted: logical token t lives in slot perm[t]
    k_perm = torch.empty_like(k_log)
    v_perm = torch.empty_like(v_log)
    pt = torch.from_numpy(perm)
    k_perm[pt] = k_log
    v_perm[pt] = v_log
    common = dict(dtype="bf16", num_qo_heads=64, num_kv_heads=8, head_dim=128, page_size=1,
                  causal=False, sm_scale=1.0 / math.sqrt(128), qo_indptr=qo_indptr,
                  kv_indptr=kv_indptr, last_page_len=last, q=q)
    permuted = PagedBatch(name="vector_sparse_decode_bf16", kv_indices=perm.astype(np.int32),
                          k_pages=k_perm, v_pages=v_perm, **common)
    contiguous = PagedBatch(name="vector_sparse_decode_bf16_contiguous",
                            kv_indices=np.arange(n, dtype=np.int32), k_pages=k_log, v_pages=v_log,
                            **common)
    return permuted, contiguous


def bsr_prefill_bf16(seed: int = 7, n_row_blocks: int = 32, block_rows: int = 64, n_col_blocks: int = 512,
                     block_cols: int = 16, density: float = 0.25, num_qo_heads: int = 32, num_kv_heads: int = 8,
                     head_dim: int = 128):
    """A general block-sparse (BSR) attention: n_row_blocks row blocks of
    block_rows query rows; row block r attends to a seeded random subset (each
    column block kept with probability `density`, at least one) of the
    n_col_blocks column blocks of block_cols KV tokens, in a permuted order.
    The column blocks are the pages of the pool (page size = block_cols) and may
    be shared by several row blocks. Non-causal, bf16.

    As a batch: request r = row block r, qo_indptr steps by block_rows, the page
    list of request r is its column-block list (kv_indptr / kv_indices are the
    BSR row_ptr / col_indices), every page full."""
    rng = np.random.default_rng(seed)
    lists = []
    for _ in range(n_row_blocks):
        keep = np.flatnonzero(rng.random(n_col_blocks) < density)
        if keep.size == 0:
            keep = rng.integers(0, n_col_blocks, size=1)
        lists.append(rng.permutation(keep))
    row_ptr = np.zeros(n_row_blocks + 1, np.int32)
    row_ptr[1:] = np.cumsum([len(x) for x in lists])
    col_indices = np.concatenate(lists).astype(np.int32)
    n = n_row_blocks * block_rows
    q = _normal(rng, (n, num_qo_heads, head_dim), "bf16")
    k = _normal(rng, (n_col_blocks, block_cols, num_kv_heads, head_dim), "bf16")
    v = _normal(rng, (n_col_blocks, block_cols, num_kv_heads, head_dim), "bf16")
    return PagedBatch(name="bsr_prefill_bf16", dtype="bf16", num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads,
                      head_dim=head_dim, page_size=block_cols, causal=False, sm_scale=1.0 / math.sqrt(head_dim),
                      qo_indptr=(np.arange(n_row_blocks + 1) * block_rows).astype(np.int32), kv_indptr=row_ptr,
                      kv_indices=col_indices, last_page_len=np.full(n_row_blocks, block_cols, np.int32),
                      q=q, k_pages=k, v_pages=v)


def vector_sparse_prefill_bf16(length: int = 32768, seed: int = 6, num_qo_heads: int = 32, num_kv_heads: int = 8):
    """One causal prefill of `length` tokens (qo = kv), page size 1 with every
    token slot of the pool permuted, 32 qo / 8 kv heads, head_dim 128, bf16.

    Returns (permuted, contiguous): the same logical KV, once scattered and once
    laid out in order (indices = arange)."""
    rng = np.random.default_rng(seed)
    perm = rng.permutation(length)
    q = _normal(rng, (length, num_qo_heads, 128), "bf16")
    k_log = _normal(rng, (length, 1, num_kv_heads, 128), "bf16")
    v_log = _normal(rng, (length, 1, num_kv_heads, 128), "bf16")
    k_perm = torch.empty_like(k_log)
    v_perm = torch.empty_like(v_log)
    pt = torch.from_numpy(perm)
    k_perm[pt] = k_log
    v_perm[pt] = v_log
    ind = np.array([0, length], np.int32)
    common = dict(dtype="bf16", num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads, head_dim=128, page_size=1,
                  causal=True, sm_scale=1.0 / math.sqrt(128), qo_indptr=ind.copy(), kv_indptr=ind.copy(),
                  last_page_len=np.ones(1, np.int32), q=q)
    permuted = PagedBatch(name="vector_sparse_prefill_bf16", kv_indices=perm.astype(np.int32),
                          k_pages=k_perm, v_pages=v_perm, **common)
    contiguous = PagedBatch(name="vector_sparse_prefill_bf16_contiguous",
                            kv_indices=np.arange(length, dtype=np.int32), k_pages=k_log, v_pages=v_log, **common)
    return permuted, contiguous


def ragged_causal_prefill_lengths(batch: int = 16, seed: int = 4):
    """(generator after the draw, lengths) of the ragged causal prefill: qo = kv ~ U{128..2048}."""
    rng = np.random.default_rng(seed)
    return rng, rng.integers(128, 2048, size=batch, endpoint=True)


def ragged_causal_prefill_bf16(batch: int = 16, seed: int = 4) -> PagedBatch:
    """batch 16, qo = kv ~ U{128..2048}, ragged Q, page 16 permuted, 32 qo / 8 kv
    heads, head_dim 128, bf16, causal (bottom-right)."""
    rng, lens = ragged_causal_prefill_lengths(batch, seed)
    return paged_batch(seed, lens, lens, 32, 8, 128, 16, "bf16", causal=True, rng=rng,
                       name="ragged_causal_prefill_bf16")


@dataclass
class SharedPrefixBatch:
    """A shared-prefix decode batch and its two composable views over the same pages."""
    full: PagedBatch      # every request: prefix pages then its suffix pages
    prefix: PagedBatch    # one row block of all queries over the prefix pages, non-causal
    suffix: PagedBatch    # each request over its own suffix pages (decode)
    prefix_len: int
    suffix_lens: np.ndarray


def shared_prefix_suffix_lengths(batch: int = 64, outlier: int = 32768, suffix_lo: int = 64, suffix_hi: int = 1024,
                                 seed: int = 5):
    """(generator after the draw, suffix lengths) of the shared-prefix decode:
    U{suffix_lo..suffix_hi}, the last one the outlier."""
    rng = np.random.default_rng(seed)
    suffix = rng.integers(suffix_lo, suffix_hi, size=batch, endpoint=True)
    suffix[-1] = outlier
    return rng, suffix


def shared_prefix_decode_bf16(batch: int = 64, prefix_len: int = 8192, outlier: int = 32768,
                              suffix_lo: int = 64, suffix_hi: int = 1024, seed: int = 5,
                              num_qo_heads: int = 32, num_kv_heads: int = 8, head_dim: int = 128,
                              page_size: int = 16) -> SharedPrefixBatch:
    """64 decode requests sharing an 8192-token prefix (512 pages of 16); suffixes
    ~ U{64..1024} for the first 63 requests and 32768 tokens for the last one
    (the skewed outlier); 32 qo / 8 kv heads, head_dim 128, bf16."""
    rng, suffix = shared_prefix_suffix_lengths(batch, outlier, suffix_lo, suffix_hi, seed)
    assert prefix_len % page_size == 0
    n_prefix_pages = prefix_len // page_size
    s_pages, s_last = _pages_for(suffix, page_size)
    pool = n_prefix_pages + int(s_pages.sum())
    perm = rng.permutation(pool).astype(np.int32)
    prefix_pages = perm[:n_prefix_pages]
    s_indptr = np.zeros(batch + 1, np.int32)
    s_indptr[1:] = np.cumsum(s_pages)
    s_indices = perm[n_prefix_pages:]
    q = _normal(rng, (batch, num_qo_heads, head_dim), "bf16")
    k = _normal(rng, (pool, page_size, num_kv_heads, head_dim), "bf16")
    v = _normal(rng, (pool, page_size, num_kv_heads, head_dim), "bf16")
    per_req = [s_indices[s_indptr[b]:s_indptr[b + 1]] for b in range(batch)]
    _poison(k, v, perm, s_pages, s_last, per_req, page_size)
    full_indices = np.concatenate([np.concatenate([prefix_pages, p]) for p in per_req]).astype(np.int32)
    full_indptr = np.zeros(batch + 1, np.int32)
    full_indptr[1:] = np.cumsum(s_pages + n_prefix_pages)
    decode_qo = np.arange(batch + 1, dtype=np.int32)
    common = dict(dtype="bf16", num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads,
                  head_dim=head_dim, page_size=page_size, causal=False,
                  sm_scale=1.0 / math.sqrt(head_dim), q=q, k_pages=k, v_pages=v)
    full = PagedBatch(name="shared_prefix_full", qo_indptr=decode_qo, kv_indptr=full_indptr,
                      kv_indices=full_indices, last_page_len=s_last, **common)
    prefix = PagedBatch(name="shared_prefix_view", qo_indptr=np.array([0, batch], np.int32),
                        kv_indptr=np.array([0, n_prefix_pages], np.int32), kv_indices=prefix_pages.copy(),
                        last_page_len=np.array([page_size], np.int32), **common)
    suffix_view = PagedBatch(name="shared_prefix_suffix_view", qo_indptr=decode_qo, kv_indptr=s_indptr,
                             kv_indices=s_indices.copy(), last_page_len=s_last, **common)
    return SharedPrefixBatch(full=full, prefix=prefix, suffix=suffix_view, prefix_len=prefix_len,
                             suffix_lens=suffix.astype(np.int64))


WORKLOADS = {
    "tiny_decode_f32": tiny_decode_f32,
    "batched_decode_bf16": batched_decode_bf16,
    "vector_sparse_decode_bf16": vector_sparse_decode_bf16,
    "ragged_causal_prefill_bf16": ragged_causal_prefill_bf16,
    "shared_prefix_decode_bf16": shared_prefix_decode_bf16,
}


def scaled(batch: PagedBatch, **changes) -> PagedBatch:
    return replace(batch, **changes)


@dataclass
class Fp8KV:
    """An e4m3 copy of a batch's K / V pools: k = k_scale * k8, v = v_scale * v8."""
    k8: torch.Tensor   # uint8 codes (OCP e4m3), [num_pages, page_size, H_kv, D]
    v8: torch.Tensor
    k_scale: float
    v_scale: float


def fp8_kv(batch: PagedBatch) -> Fp8KV:
    """Per-pool scale = (largest finite |x|) / 448, the e4m3 maximum; values are
    divided by it in float32 and rounded to e4m3 by torch (nearest even,
    saturating casts are not used: |x / scale| <= 448 already). NaN poison
    stays NaN (code 0x7f / 0xff)."""
    out = []
    for t in (batch.k_pages, batch.v_pages):
        x = t.float()
        amax = float(torch.nan_to_num(x, nan=0.0).abs().max())
        scale = amax / 448.0 if amax > 0 else 1.0
        q = (x / scale).to(torch.float8_e4m3fn)
        out += [q.view(torch.uint8).contiguous(), scale]
    return Fp8KV(k8=out[0], v8=out[2], k_scale=out[1], v_scale=out[3])

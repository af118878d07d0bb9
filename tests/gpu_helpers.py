"""Shared helpers of the GPU parity tests: run the library on a workloads batch
and compare with the oracle at the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Acceptance bounds: O max-abs 1e-2 and LSE 1e-3 for bf16 inputs with fp32
# accumulation; 1e-5 for both with fp32 inputs.
TOL = {"bf16": (1e-2, 1e-3), "f32": (1e-5, 1e-5)}
TORCH = {"bf16": torch.bfloat16, "f32": torch.float32}


def lib():
    from block_sparse_paged_gb300 import build
    build.build()
    import block_sparse_paged_gb300 as bsp
    return bsp


def to_dev(batch, dev="cuda"):
    return (batch.q.to(dev), batch.k_pages.to(dev), batch.v_pages.to(dev),
            torch.from_numpy(np.ascontiguousarray(batch.kv_indices, np.int32)).to(dev))


def run_batch(bsp, batch, mode=None, num_ctas=None, dev_tensors=None, max_batch=None, max_qo=None, sink=None,
              chunks_per_cta=1):
    """Plan + run through the library; returns (O, LSE) on the host and the runner."""
    mode = mode or ("decode" if batch.is_decode else "prefill")
    pa = bsp.PagedAttention(mode, batch.num_qo_heads, batch.num_kv_heads, batch.head_dim, batch.page_size,
                            batch.causal, TORCH[batch.dtype], max_batch=max_batch or batch.batch,
                            max_qo_tokens=max_qo or int(batch.qo_indptr[-1]), num_ctas=num_ctas,
                            window_left=batch.window_left, logits_soft_cap=batch.soft_cap,
                            chunks_per_cta=chunks_per_cta)
    qo = None if mode == "decode" and batch.is_decode else batch.qo_indptr
    pa.plan(batch.kv_indptr, batch.last_page_len, qo_indptr=qo)
    q, k, v, idx = dev_tensors or to_dev(batch)
    sk = None if sink is None else torch.as_tensor(np.asarray(sink, np.float32)).to(q.device)
    out, lse = pa.run(q, k, v, idx, batch.sm_scale, sink=sk)
    torch.cuda.synchronize()
    return out, lse, pa


def compare(out, lse, O_ref, L_ref, dtype, rows=None, rounding_aware=False):
    """Element-wise check of (out, lse) against the oracle's fp64 (O_ref, L_ref).

    bf16 outputs are compared after the GPU's cast: the bound on O is the
    stated 1e-2 plus the cast's own rounding, at most |O_ref| * 2^-8 (half a
    bf16 ulp; 8 significant bits). A row with two visible keys can reach
    |O| ~ 2, where the cast alone is up to 0.0078.

    rounding_aware instead bounds O by max(1e-2, |O_ref| * 2^-8) for bf16, for
    states that are not attention outputs (merge inputs of any magnitude)."""
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        tok, head = rows
        o, l = o[tok, head], l[tok, head]
    tol_o, tol_l = TOL[dtype]
    empty = np.isneginf(L_ref)
    assert np.array_equal(np.isneginf(l), empty), "empty-state rows differ"
    assert np.all(o[empty] == 0)
    fin = ~empty
    if rounding_aware and dtype == "bf16":
        excess = np.abs(o - O_ref) - np.maximum(tol_o, np.abs(O_ref) * 2.0 ** -8)
        assert excess.max() <= 0, f"O error beyond the bf16 rounding bound by {excess.max()}"
        tol_o = np.inf
    elif dtype == "bf16" and o.size:
        excess = np.abs(o - O_ref) - (tol_o + np.abs(O_ref) * 2.0 ** -8)
        assert excess.max() <= 0, f"O error beyond 1e-2 + the bf16 cast bound by {excess.max()}"
        tol_o = np.inf
    err_o = np.abs(o - O_ref).max() if o.size else 0.0
    err_l = np.abs(l[fin] - L_ref[fin]).max() if fin.any() else 0.0
    assert np.isfinite(o).all(), "non-finite output"
    assert err_o <= tol_o, f"O max-abs error {err_o} > {tol_o}"
    assert err_l <= tol_l, f"LSE max-abs error {err_l} > {tol_l}"
    return err_o, err_l


def oracle_full(batch, num_threads=0, sink=None):
    return oracle.attention_of(batch, num_threads=num_threads, sink=sink)


def sample_rows(batch, n, seed):
    """n (token, head) pairs: every head of the longest and shortest request,
    then seeded random pairs."""
    rng = np.random.default_rng(seed)
    kv = batch.kv_lens
    n_tok = int(batch.qo_indptr[-1])
    toks, heads = [], []
    for b in (int(np.argmax(kv)), int(np.argmin(kv))):
        t = int(batch.qo_indptr[b + 1]) - 1
        toks += [t] * batch.num_qo_heads
        heads += list(range(batch.num_qo_heads))
    extra = max(0, n - len(toks))
    toks += list(rng.integers(0, n_tok, size=extra))
    heads += list(rng.integers(0, batch.num_qo_heads, size=extra))
    return np.array(toks, np.int64), np.array(heads, np.int32)

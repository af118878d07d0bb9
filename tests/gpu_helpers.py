"""Shared helpers of the GPU parity tests: run the library on a workloads batch
and compare with the oracle at the stated tolerances."""
from __future__ import annotations

import os
import time

import numpy as np
import torch

import oracle

# Acceptance bounds: O max-abs 1e-2 and LSE 1e-3 for bf16 inputs with fp32
# accumulation; 1e-5 for both with fp32 inputs.
TOL = {"bf16": (1e-2, 1e-3), "f32": (1e-5, 1e-5)}
TORCH = {"bf16": torch.bfloat16, "f32": torch.float32}

# One record per compare() call, printed at the end of the session (conftest):
# which test, how many (token, head) rows were compared, how many of them have
# an element above the plain 1e-2 (bf16) or 1e-5 (fp32) bound, the largest
# errors, and the oracle's time for the compared rows when the caller timed it.
PARITY_LOG: list[dict] = []


def lib():
    from block_sparse_paged_gb300 import build
    build.build()
    import block_sparse_paged_gb300 as bsp
    return bsp


def to_dev(batch, dev="cuda"):
    return (batch.q.to(dev), batch.k_pages.to(dev), batch.v_pages.to(dev),
            torch.from_numpy(np.ascontiguousarray(batch.kv_indices, np.int32)).to(dev))


def run_batch(bsp, batch, mode=None, num_ctas=None, dev_tensors=None, max_batch=None, max_qo=None, sink=None,
              chunks_per_cta=1, **kw):
    """Plan + run through the library; returns (O, LSE) on the host and the runner."""
    mode = mode or ("decode" if batch.is_decode else "prefill")
    pa = bsp.PagedAttention(mode, batch.num_qo_heads, batch.num_kv_heads, batch.head_dim, batch.page_size,
                            batch.causal, TORCH[batch.dtype], max_batch=max_batch or batch.batch,
                            max_qo_tokens=max_qo or int(batch.qo_indptr[-1]), num_ctas=num_ctas,
                            window_left=batch.window_left, logits_soft_cap=batch.soft_cap,
                            chunks_per_cta=chunks_per_cta, **kw)
    qo = None if mode == "decode" and batch.is_decode else batch.qo_indptr
    pa.plan(batch.kv_indptr, batch.last_page_len, qo_indptr=qo)
    q, k, v, idx = dev_tensors or to_dev(batch)
    sk = None if sink is None else torch.as_tensor(np.asarray(sink, np.float32)).to(q.device)
    out, lse = pa.run(q, k, v, idx, batch.sm_scale, sink=sk)
    torch.cuda.synchronize()
    return out, lse, pa


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Half a bf16 ulp at the binade of |x|: 2^(floor(log2 |x|) - 8) (bf16 keeps 8
    significant bits), 0 where x = 0. Exact: frexp gives |x| = m 2^e with m in
    [0.5, 1), so floor(log2 |x|) = e - 1."""
    _, e = np.frexp(np.abs(x))
    return np.where(x != 0, np.ldexp(1.0, e - 9), 0.0)


def compare(out, lse, O_ref, L_ref, dtype, rows=None, rounding_aware=False, oracle_s=None, label=None):
    """Element-wise check of (out, lse) against the oracle's fp64 (O_ref, L_ref).

    bf16 outputs are compared after the GPU's cast to bf16, so the bound on
    each element of O is the stated 1e-2 plus the cast's own rounding, half a
    bf16 ulp at the binade of O_ref: 2^(floor(log2 |O_ref|) - 8). LSE (fp32)
    keeps 1e-3; fp32 outputs keep 1e-5 for both.

    rounding_aware bounds O by max(1e-2, half_ulp + |O_ref| 2^-20) instead, for
    merged states that are not attention outputs (inputs of any magnitude): the
    cast plus the fp32 merge arithmetic's relative error.

    rows = (token, head) index arrays selects the compared rows of out / lse
    (O_ref / L_ref then hold just those rows). Each call appends a record to
    PARITY_LOG."""
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        tok, head = rows
        o, l = o[tok, head], l[tok, head]
    tol_o, tol_l = TOL[dtype]
    empty = np.isneginf(L_ref)
    assert np.array_equal(np.isneginf(l), empty), "empty-state rows differ"
    assert np.all(o[empty] == 0)
    assert np.isfinite(o).all(), "non-finite output"
    fin = ~empty
    err = np.abs(o - O_ref)
    if dtype == "bf16":
        hu = half_ulp_bf16(O_ref)
        bound = np.maximum(tol_o, hu + np.abs(O_ref) * 2.0 ** -20) if rounding_aware else tol_o + hu
    else:
        bound = np.full(err.shape, tol_o)
    row_err = err.reshape(err.shape[:-1] + (-1,)).max(axis=-1) if err.ndim else err
    err_o = float(err.max()) if err.size else 0.0
    err_l = float(np.abs(l[fin] - L_ref[fin]).max()) if fin.any() else 0.0
    rec = {"test": label or os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0],
           "rows": int(row_err.size), "rows_above_plain_tol": int((row_err > tol_o).sum()),
           "max_err_o": err_o, "max_err_lse": err_l, "oracle_s": oracle_s}
    if err.size:
        i = np.unravel_index(int(np.argmax(err - bound)), err.shape)
        rec["worst"] = {"o_ref": float(O_ref[i]), "o_gpu": float(o[i]), "bound": float(bound[i])}
    PARITY_LOG.append(rec)
    if err.size:
        excess = float((err - bound).max())
        assert excess <= 0, f"O error beyond its bound by {excess} (max error {err_o})"
    assert err_l <= tol_l, f"LSE max-abs error {err_l} > {tol_l}"
    return err_o, err_l


def oracle_full(batch, num_threads=0, sink=None):
    return oracle.attention_of(batch, num_threads=num_threads, sink=sink)


def timed(fn, *a, **k):
    """(result, seconds) of one call."""
    t0 = time.perf_counter()
    r = fn(*a, **k)
    return r, time.perf_counter() - t0


def stratified_rows(batch, stride: int, seed: int, tile_positions: int | None = None):
    """(token, head) pairs: for every request and every query head, every
    stride-th query position (a seeded phase per request and head) plus every
    position of the request's first and last query tile (tile_positions
    positions, the prefill tile of 256 packed rows / g by default).
    At least 1/stride of the rows of every (request, head)."""
    g = batch.num_qo_heads // batch.num_kv_heads
    tp = tile_positions or max(1, 256 // g)
    rng = np.random.default_rng(seed)
    toks, heads = [], []
    for b in range(batch.batch):
        q0, q1 = int(batch.qo_indptr[b]), int(batch.qo_indptr[b + 1])
        n = q1 - q0
        if n == 0:
            continue
        pos = np.arange(n)
        edge = (pos < tp) | (pos >= ((n - 1) // tp) * tp)
        for h in range(batch.num_qo_heads):
            sel = pos[edge | ((pos + int(rng.integers(stride))) % stride == 0)]
            toks.append(q0 + sel)
            heads.append(np.full(sel.size, h, np.int32))
    return np.concatenate(toks).astype(np.int64), np.concatenate(heads)

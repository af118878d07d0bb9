"""Oracle for block-sparse paged attention: plain, slow, fp64, CPU only.

TEST INFRASTRUCTURE ONLY. The product package never imports this module; only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
do. It shares no code with the CUDA path.

- ``attention.c``: the attention definition and the exact state merge, in C,
  fp64, one output at a time (loaded here through ctypes).
- ``plan.py``: the load-balanced plan in plain Python.
- ``fp8.py``: values of e4m3 KV codes (for the e4m3 KV-cache decode).

``build()`` compiles ``attention.c`` with gcc into ``liboracle.so`` next to it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from . import fp8 as fp8  # noqa: F401  (re-export)
from . import plan as plan  # noqa: F401  (re-export)

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "attention.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")


def compile_source(src: str, out: str) -> str:
    """gcc -O2 -fopenmp a C oracle source into a shared library."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                           "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the C oracle next to its source. Returns the library path."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(SOURCE):
        compile_source(SOURCE, _LIB_PATH)
    return _LIB_PATH


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


class COracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i32, i64, f64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        lib.oracle_attention_rows.argtypes = [i32, i32, i32, i32, i32, i32, f64, i32, f64, vp,
                                              vp, vp, vp, vp, vp, vp, vp, i64, vp, vp, vp, vp, i32]
        lib.oracle_attention_rows.restype = ctypes.c_int
        lib.oracle_merge_states.argtypes = [i64, i32, vp, vp, vp, vp, vp, vp]
        lib.oracle_merge_states.restype = None
        lib.oracle_physical_row.argtypes = [vp, vp, i32, i32, i64]
        lib.oracle_physical_row.restype = i64
        lib.oracle_num_threads_available.argtypes = []
        lib.oracle_num_threads_available.restype = ctypes.c_int
        self.lib = lib

    def num_threads_available(self) -> int:
        return int(self.lib.oracle_num_threads_available())

    def physical_row(self, kv_indptr, kv_indices, page_size: int, b: int, t: int) -> int:
        """eq 7: physical token row of logical token t of request b."""
        ip, ix = _c(kv_indptr, np.int32), _c(kv_indices, np.int32)
        return int(self.lib.oracle_physical_row(_ptr(ip), _ptr(ix), page_size, b, t))

    def attention_rows(self, q, k_pages, v_pages, qo_indptr, kv_indptr, kv_indices, last_page_len,
                       num_qo_heads: int, num_kv_heads: int, page_size: int, causal: bool,
                       sm_scale: float, sel_token, sel_head, num_threads: int = 0,
                       window_left: int = -1, soft_cap: float = 0.0, sink=None):
        """(O [n, D], LSE [n]) in fp64 for the selected (token, head) pairs.
        sink: None or one logit per query head (the attention-sink variant).

        q: [n_tokens, H_qo, D]; k_pages, v_pages: [num_pages, page_size, H_kv, D],
        any float dtype (converted to float32, which holds bf16 and fp32 exactly).
        """
        q = _c(q, np.float32)
        k = _c(k_pages, np.float32)
        v = _c(v_pages, np.float32)
        D = q.shape[-1]
        qi, ki, kx, lp = (_c(a, np.int32) for a in (qo_indptr, kv_indptr, kv_indices, last_page_len))
        st, sh = _c(sel_token, np.int64), _c(sel_head, np.int32)
        n = st.shape[0]
        o = np.zeros((n, D), np.float64)
        lse = np.zeros((n,), np.float64)
        sk = None
        if sink is not None:
            sk = _c(sink, np.float64)
            if sk.shape != (num_qo_heads,):
                raise ValueError("sink must hold one value per query head")
        rc = self.lib.oracle_attention_rows(len(qi) - 1, num_qo_heads, num_kv_heads, D, page_size,
                                            int(bool(causal)), float(sm_scale), int(window_left), float(soft_cap),
                                            None if sk is None else _ptr(sk), _ptr(qi), _ptr(ki), _ptr(kx), _ptr(lp),
                                            _ptr(q), _ptr(k), _ptr(v), n, _ptr(st), _ptr(sh),
                                            _ptr(o), _ptr(lse), int(num_threads))
        if rc != 0:
            raise ValueError("oracle_attention_rows rejected its input")
        return o, lse

    def attention(self, q, k_pages, v_pages, qo_indptr, kv_indptr, kv_indices, last_page_len,
                  num_qo_heads: int, num_kv_heads: int, page_size: int, causal: bool,
                  sm_scale: float, num_threads: int = 0, window_left: int = -1, soft_cap: float = 0.0,
                  sink=None):
        """All outputs: O [n_tokens, H_qo, D] and LSE [n_tokens, H_qo], fp64."""
        n_tok = int(np.asarray(qo_indptr)[-1])
        tok = np.repeat(np.arange(n_tok, dtype=np.int64), num_qo_heads)
        head = np.tile(np.arange(num_qo_heads, dtype=np.int32), n_tok)
        o, lse = self.attention_rows(q, k_pages, v_pages, qo_indptr, kv_indptr, kv_indices,
                                     last_page_len, num_qo_heads, num_kv_heads, page_size, causal,
                                     sm_scale, tok, head, num_threads, window_left, soft_cap, sink)
        D = o.shape[-1]
        return o.reshape(n_tok, num_qo_heads, D), lse.reshape(n_tok, num_qo_heads)

    def merge_states(self, o_a, lse_a, o_b, lse_b):
        """Stable merge of two arrays of states: O [..., D], LSE [...], fp64."""
        o_a = _c(o_a, np.float64)
        o_b = _c(o_b, np.float64)
        la = _c(lse_a, np.float64)
        lb = _c(lse_b, np.float64)
        D = o_a.shape[-1]
        o = np.zeros(o_a.shape, np.float64)
        lse = np.zeros(la.shape, np.float64)
        self.lib.oracle_merge_states(la.size, D, _ptr(o_a), _ptr(la), _ptr(o_b), _ptr(lb),
                                     _ptr(o), _ptr(lse))
        return o, lse


_default: COracle | None = None


def default() -> COracle:
    global _default
    if _default is None:
        _default = COracle(build())
    return _default


def num_threads_available() -> int:
    return default().num_threads_available()


def physical_row(*a, **k):
    return default().physical_row(*a, **k)


def attention_rows(*a, **k):
    return default().attention_rows(*a, **k)


def attention(*a, **k):
    return default().attention(*a, **k)


def merge_states(*a, **k):
    return default().merge_states(*a, **k)


def attention_of(batch, num_threads: int = 0, k=None, v=None, **kw):
    """All outputs of a workloads.PagedBatch (K / V value arrays may be passed in)."""
    k = batch.k_pages.float().numpy() if k is None else k
    v = batch.v_pages.float().numpy() if v is None else v
    return default().attention(batch.q.float().numpy(), k, v, batch.qo_indptr, batch.kv_indptr,
                               batch.kv_indices, batch.last_page_len, batch.num_qo_heads,
                               batch.num_kv_heads, batch.page_size, batch.causal, batch.sm_scale,
                               num_threads=num_threads, window_left=getattr(batch, "window_left", -1),
                               soft_cap=getattr(batch, "soft_cap", 0.0), **kw)


def attention_rows_of(batch, sel_token, sel_head, num_threads: int = 0, k_f32=None, v_f32=None):
    """Selected outputs of a workloads.PagedBatch (K/V float32 copies may be passed in)."""
    k = batch.k_pages.float().numpy() if k_f32 is None else k_f32
    v = batch.v_pages.float().numpy() if v_f32 is None else v_f32
    return default().attention_rows(batch.q.float().numpy(), k, v, batch.qo_indptr, batch.kv_indptr,
                                    batch.kv_indices, batch.last_page_len, batch.num_qo_heads,
                                    batch.num_kv_heads, batch.page_size, batch.causal,
                                    batch.sm_scale, sel_token, sel_head, num_threads,
                                    getattr(batch, "window_left", -1), getattr(batch, "soft_cap", 0.0))

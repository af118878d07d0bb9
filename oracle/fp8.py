"""Oracle decoding of e4m3 (FP8) KV codes: plain numpy, fp64.

TEST INFRASTRUCTURE ONLY. The product path converts codes in its own kernel;
the two share no code. Only tests, the package's smoke check and the bench's
CPU-baseline leg import this module.

The pages run decode over an e4m3 KV cache (FlashInfer: A Customizable
Attention Engine for LLM Serving, App. G.4 Table 8, the "e4m3" rows) without
defining the format or its scaling. Reading taken here: the E4M3 encoding of
the OCP 8-bit floating point specification (1 sign bit, 4 exponent bits with
bias 7, 3 mantissa bits; no infinities; exponent and mantissa all ones is NaN;
largest finite value 448), and one scale per pool, so that a stored code c
of K stands for k_scale * value(c) (same for V).
"""
from __future__ import annotations

import numpy as np


def e4m3_value(code: int) -> float:
    """The value of one code, written out case by case from the format."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:  # subnormal: no implicit leading one, exponent fixed at 1 - bias
        return sign * (m / 8.0) * 2.0 ** (1 - 7)
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


# one entry per code; built from e4m3_value, so it is that function, tabulated
_TABLE = np.array([e4m3_value(c) for c in range(256)], np.float64)


def e4m3_to_float(codes) -> np.ndarray:
    """fp64 values of an array of e4m3 codes (uint8, any shape)."""
    c = np.asarray(codes)
    if c.dtype != np.uint8:
        raise TypeError("e4m3 codes must be uint8")
    return _TABLE[c]


def dequantize(codes, scale: float) -> np.ndarray:
    """scale * value(code), fp64: the K or V a stored e4m3 pool stands for."""
    return e4m3_to_float(codes) * float(scale)

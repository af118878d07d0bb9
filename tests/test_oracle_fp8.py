"""The oracle's e4m3 decoding against values the format fixes, against a
library routine, and planted mistakes in copies of it (all on the CPU).

The format is OCP E4M3 (bias 7, 3 mantissa bits, no infinities, S.1111.111
NaN, largest finite 448), the reading the oracle states for the e4m3 KV-cache
rows of FlashInfer: A Customizable Attention Engine for LLM Serving, App. G.4
Table 8."""
import math
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from oracle import fp8 as ofp8


def _codes():
    return np.arange(256, dtype=np.uint8)


# (code, value) pairs worked out by hand from the format
CLOSED_FORMS = [
    (0x00, 0.0), (0x38, 1.0), (0xB8, -1.0), (0x40, 2.0), (0x3C, 1.5), (0x30, 0.5),
    (0x7E, 448.0), (0xFE, -448.0), (0x78, 256.0), (0x08, 2.0 ** -6), (0x07, 7 * 2.0 ** -9),
    (0x01, 2.0 ** -9), (0x81, -(2.0 ** -9)), (0x11, 1.125 * 2.0 ** -5), (0x5A, 1.25 * 2.0 ** 4),
]


def pin_closed_forms(mod):
    vals = mod.e4m3_to_float(np.array([c for c, _ in CLOSED_FORMS], np.uint8))
    for (c, want), got in zip(CLOSED_FORMS, vals):
        assert got == want, f"code {c:#04x}: {got} != {want}"
    neg0 = mod.e4m3_to_float(np.array([0x80], np.uint8))[0]
    assert neg0 == 0.0 and math.copysign(1.0, neg0) == -1.0


def pin_nan_and_order(mod):
    v = mod.e4m3_to_float(_codes())
    nan = np.isnan(v)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF], "exactly S.1111.111 is NaN"
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0), "positive codes increase with their value"
    assert np.array_equal(v[0x80:0xFF], -pos), "the sign bit negates"
    # within a binade e >= 1 the step is 2^(e - 7) / 8; subnormals step by 2^-9
    for e in range(1, 16):
        lo = e << 3
        hi = min(lo + 8, 0x7F)
        assert np.all(np.diff(v[lo:hi]) == 2.0 ** (e - 7) / 8)
    assert np.all(np.diff(v[0:9]) == 2.0 ** -9)


def pin_library(mod):
    """torch's float8_e4m3fn is the same format: all 256 codes agree."""
    lib = torch.from_numpy(_codes()).view(torch.float8_e4m3fn).double().numpy()
    v = mod.e4m3_to_float(_codes())
    assert np.array_equal(np.isnan(lib), np.isnan(v))
    fin = ~np.isnan(v)
    assert np.array_equal(lib[fin], v[fin])


def pin_dequantize(mod):
    c = np.array([[0x38, 0x7E], [0x81, 0x00]], np.uint8)
    got = mod.dequantize(c, 0.25)
    assert np.array_equal(got, np.array([[0.25, 112.0], [-(2.0 ** -11), 0.0]]))


PINS = [pin_closed_forms, pin_nan_and_order, pin_library, pin_dequantize]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(ofp8)


def test_uint8_only():
    with pytest.raises(TypeError):
        ofp8.e4m3_to_float(np.array([1, 2], np.int32))


MUTATIONS = [
    ("bias_8", "2.0 ** (e - 7)", "2.0 ** (e - 8)"),
    ("subnormal_exponent", "2.0 ** (1 - 7)", "2.0 ** (0 - 7)"),
    ("subnormal_implicit_one", "return sign * (m / 8.0) * 2.0 ** (1 - 7)",
     "return sign * (1.0 + m / 8.0) * 2.0 ** (1 - 7)"),
    ("nan_all_ones_exponent", "if e == 0xF and m == 0x7:", "if e == 0xF:"),
    ("mantissa_width", "(1.0 + m / 8.0) * 2.0 ** (e - 7)", "(1.0 + m / 16.0) * 2.0 ** (e - 7)"),
    ("sign_dropped", "sign = -1.0 if code & 0x80 else 1.0", "sign = 1.0"),
    ("scale_dropped", "return e4m3_to_float(codes) * float(scale)", "return e4m3_to_float(codes)"),
]

_RUN = """
import sys, importlib.util
sys.path[:0] = [{tests!r}, {root!r}]
spec = importlib.util.spec_from_file_location("fp8_mutant", {path!r})
mod = importlib.util.module_from_spec(spec)
spec.loader.exec_module(mod)
import test_oracle_fp8 as t
caught = []
for pin in t.PINS:
    try:
        pin(mod)
    except (AssertionError, ValueError):
        caught.append(pin.__name__)
print(",".join(caught))
sys.exit(0 if caught else 3)
"""


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(name, old, new, tmp_path):
    src = open(ofp8.__file__).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = tmp_path / "fp8_mutant.py"
    path.write_text(src.replace(old, new))
    tests_dir = os.path.dirname(os.path.abspath(__file__))
    code = _RUN.format(tests=tests_dir, root=os.path.dirname(tests_dir), path=str(path))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode != 3, f"no pin caught the planted mistake {name}"
    assert r.returncode == 0, r.stderr[-2000:]

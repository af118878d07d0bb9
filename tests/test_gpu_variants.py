"""Attention variants (FlashInfer 原理 overview, ⑧; FlashInfer: Making Attention
Fit the Serving Workload, eq 8): sliding window, logits soft-cap and attention
sink, on the decode and prefill paths, against the oracle on the same seeded
inputs."""
import numpy as np
import pytest

import workloads
from gpu_helpers import compare, lib, oracle_full, run_batch, timed

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bsp():
    return lib()


def with_variant(b, window_left=-1, soft_cap=0.0):
    b.window_left, b.soft_cap = window_left, soft_cap
    return b


DECODE = [
    # (seed, kv lens, H_qo, H_kv, D, page, dtype, window, cap, num_ctas)
    (91, [3000, 17, 900, 4100, 1, 250], 32, 8, 128, 16, "bf16", 700, 0.0, 29),     # window, splits
    (92, [3000, 17, 900, 4100, 1, 250], 32, 8, 128, 16, "bf16", -1, 1.5, 29),      # soft-cap
    (93, [2000, 64, 1500], 64, 8, 128, 1, "bf16", 333, 2.0, 11),                   # both, page size 1
    (94, [700, 5, 1200], 16, 4, 64, 4, "f32", 100, 3.0, 9),                        # fp32 path
]


@pytest.mark.parametrize("case", DECODE, ids=[f"decode{c[0]}" for c in DECODE])
def test_decode_variants(bsp, case):
    seed, kv, hq, hk, D, ps, dt, w, cap, C = case
    b = with_variant(workloads.paged_batch(seed, [1] * len(kv), kv, hq, hk, D, ps, dt, extra_pages=2), w, cap)
    O, L = oracle_full(b)
    out, lse, pa = run_batch(bsp, b, num_ctas=C)
    compare(out, lse, O, L, dt)
    assert pa.check_device_error() == 0


PREFILL = [
    # (seed, qo lens, kv lens, H_qo, H_kv, page, causal, window, cap, num_ctas)
    (95, [300, 65, 1000], [300, 65, 1000], 32, 8, 16, True, 150, 0.0, 13),
    (96, [300, 65, 1000], [300, 65, 1000], 32, 8, 16, True, -1, 1.5, 13),
    (97, [200, 90], [700, 90], 16, 4, 1, True, 77, 2.5, 7),      # page size 1, qo < kv, both
    (98, [128, 300], [128, 500], 32, 8, 32, False, 100, 0.0, 9),  # non-causal window
    # a tile spans 256 (g = 1) or 128 (g = 2) positions: late rows' windows start
    # past a whole 128-key tile that earlier rows of the same tile still see
    (99, [400, 70], [400, 900], 16, 16, 16, True, 40, 0.0, 11),
    (100, [300, 129], [300, 129], 16, 8, 16, True, 64, 1.0, 5),
]


@pytest.mark.parametrize("case", PREFILL, ids=[f"prefill{c[0]}" for c in PREFILL])
def test_prefill_variants(bsp, case):
    seed, qo, kv, hq, hk, ps, causal, w, cap, C = case
    b = with_variant(workloads.paged_batch(seed, qo, kv, hq, hk, 128, ps, "bf16", causal=causal, extra_pages=2),
                     w, cap)
    O, L = oracle_full(b)
    out, lse, pa = run_batch(bsp, b, mode="prefill", num_ctas=C)
    compare(out, lse, O, L, "bf16")
    assert pa.check_device_error() == 0


def test_prefill_window_full_size(bsp):
    """The ragged causal prefill workload with a 512-token window and a soft-cap
    of 30: every output row against the oracle."""
    b = with_variant(workloads.ragged_causal_prefill_bf16(), 512, 30.0)
    out, lse, pa = run_batch(bsp, b, mode="prefill")
    (O, L), t = timed(oracle_full, b)
    compare(out, lse, O, L, "bf16", oracle_s=t)


def sinks(h, seed):
    """Per-head sink logits around the scale of the scores, one of them -inf."""
    x = np.random.default_rng(seed).uniform(-2.0, 4.0, size=h)
    x[h // 2] = -np.inf
    return x


SINK_DECODE = [
    # (seed, kv lens, H_qo, H_kv, D, page, dtype, num_ctas): splits, an empty request
    (121, [3000, 0, 900, 4100, 1, 250], 32, 8, 128, 16, "bf16", 29),
    (122, [700, 5, 0, 1200], 16, 4, 64, 4, "f32", 9),
    (123, [2000, 64, 0, 1500], 64, 8, 128, 1, "bf16", 11),
]


@pytest.mark.parametrize("case", SINK_DECODE, ids=[f"sink_decode{c[0]}" for c in SINK_DECODE])
def test_decode_sink(bsp, case):
    seed, kv, hq, hk, D, ps, dt, C = case
    b = workloads.paged_batch(seed, [1] * len(kv), kv, hq, hk, D, ps, dt, extra_pages=2)
    sk = sinks(hq, seed)
    O, L = oracle_full(b, sink=sk)
    out, lse, pa = run_batch(bsp, b, num_ctas=C, sink=sk)
    compare(out, lse, O, L, dt)
    assert pa.check_device_error() == 0


SINK_PREFILL = [
    # (seed, qo lens, kv lens, H_qo, H_kv, page, causal, window, num_ctas): split rows go
    # through the merge kernel, whole rows through the epilogue
    (124, [300, 65, 1000], [300, 65, 1000], 32, 8, 16, True, -1, 13),
    (125, [200, 90], [700, 90], 16, 4, 1, True, 77, 7),
    (126, [128, 300], [128, 500], 32, 8, 32, False, -1, 80),   # 40 merge entries
]


@pytest.mark.parametrize("case", SINK_PREFILL, ids=[f"sink_prefill{c[0]}" for c in SINK_PREFILL])
def test_prefill_sink(bsp, case):
    seed, qo, kv, hq, hk, ps, causal, w, C = case
    b = with_variant(workloads.paged_batch(seed, qo, kv, hq, hk, 128, ps, "bf16", causal=causal, extra_pages=2), w)
    sk = sinks(hq, seed)
    O, L = oracle_full(b, sink=sk)
    out, lse, pa = run_batch(bsp, b, mode="prefill", num_ctas=C, sink=sk)
    compare(out, lse, O, L, "bf16")
    assert pa.check_device_error() == 0

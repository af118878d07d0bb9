"""The oracle against its pins, and planted mistakes in copies of the oracle
that the pins must catch (all on the CPU)."""
import os
import subprocess
import sys

import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_mod):
    pin(oracle_mod.default())


# Each mutation is a plausible slip in the oracle's C source: (name, old, new).
MUTATIONS = [
    ("gqa_head_mapping", "const int32_t hk = h / g;", "const int32_t hk = h % H_kv;"),
    ("dropped_scale", "sc[j] = sm_scale * acc;", "sc[j] = acc;"),
    ("causal_off_by_one", "int64_t lim = i + kv_len - qo_len + 1;", "int64_t lim = i + kv_len - qo_len;"),
    ("causal_top_left", "int64_t lim = i + kv_len - qo_len + 1;", "int64_t lim = i + 1;"),
    ("page_index_mod", "kv_indices[kv_indptr[b] + t / page_size]", "kv_indices[kv_indptr[b] + t % page_size]"),
    ("page_offset_dropped", "return page * page_size + t % page_size;", "return page * page_size;"),
    ("last_page_ignored", "return (npages - 1) * page_size + last_page_len[b];", "return npages * page_size;"),
    ("lse_missing_max", "const double lse = m + log(z);", "const double lse = log(z);"),
    ("unnormalised_output", "const double p = exp(sc[j] - lse);", "const double p = exp(sc[j] - m);"),
    ("v_reads_k", "const float *vv = v_pages +", "const float *vv = k_pages +"),
    ("q_head_transposed", "const float *qv = q + (tok * H_qo + h) * (int64_t)D;",
     "const float *qv = q + (h * H_qo + tok % H_qo) * (int64_t)D;"),
    ("merge_weights_swapped", "o[d] = (a * oa[d] + bb * ob[d]) / (a + bb);",
     "o[d] = (bb * oa[d] + a * ob[d]) / (a + bb);"),
    ("merge_lse_missing_max", "lse_out[s] = m + log(a + bb);", "lse_out[s] = log(a + bb);"),
    ("merge_empty_passes_wrong_side", "for (int32_t d = 0; d < D; ++d) o[d] = oa[d];\n            lse_out[s] = la;",
     "for (int32_t d = 0; d < D; ++d) o[d] = ob[d];\n            lse_out[s] = lb;"),
    ("soft_cap_scale_dropped", "sc[j] = soft_cap * tanh(sc[j] / soft_cap);", "sc[j] = tanh(sc[j]);"),
    ("window_off_by_one", "j0 = i + kv_len - qo_len - window_left;", "j0 = i + kv_len - qo_len - window_left + 1;"),
    ("merge_naive_average", "o[d] = (a * oa[d] + bb * ob[d]) / (a + bb);", "o[d] = 0.5 * (oa[d] + ob[d]);"),
    ("sink_left_out_of_normaliser", "if (sink) z += exp(sink[h] - m);", "if (sink) z += 0.0;"),
    ("sink_of_kv_head", "if (sink) z += exp(sink[h] - m);", "if (sink) z += exp(sink[hk] - m);"),
    ("sink_empty_row_stays_empty", "lse_out[s] = sink ? sink[h] : -INFINITY;", "lse_out[s] = -INFINITY;"),
]


_RUN_PINS = """
import sys
sys.path[:0] = [{tests!r}, {root!r}]
import oracle, oracle_pins
mutant = oracle.COracle({lib!r})
caught = []
for pin in oracle_pins.ALL_PINS:
    try:
        pin(mutant)
    except (AssertionError, ValueError):
        caught.append(pin.__name__)
print(",".join(caught))
sys.exit(0 if caught else 3)
"""


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(name, old, new, tmp_path):
    """The pins run in a child process: a mutant may also read out of bounds and
    crash, which counts as caught."""
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mutant_src = tmp_path / "attention_mutant.c"
    mutant_src.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(mutant_src), str(tmp_path / "libmutant.so"))
    tests_dir = os.path.dirname(os.path.abspath(__file__))
    code = _RUN_PINS.format(tests=tests_dir, root=os.path.dirname(tests_dir), lib=lib)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode != 3, f"no pin caught the planted mistake {name}"
    assert r.returncode == 0 or r.returncode < 0, r.stderr[-2000:]


def test_thread_count_applies_to_one_call_only():
    """A call with an explicit thread count leaves the default for later calls
    (all available threads) unchanged, and the result does not depend on it."""
    import numpy as np
    import workloads
    b = workloads.paged_batch(5, [1, 1, 1], [100, 300, 7], 8, 2, 64, 16, "bf16")
    n = oracle.num_threads_available()
    O1, L1 = oracle.attention_of(b, num_threads=1)
    assert oracle.num_threads_available() == n
    O2, L2 = oracle.attention_of(b)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)

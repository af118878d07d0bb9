"""General block-sparse (BSR) attention with row blocks of B_r > 1 query rows
(engineering walkthrough §IV.3-IV.4, §V.1): each row block is a ragged query
group whose page list is its BSR row, run through the prefill path (non-causal)
and compared with the oracle on the same seeded inputs."""
import pytest
import torch

import oracle
import workloads
from gpu_helpers import compare, lib, oracle_full, run_batch, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bsp():
    return lib()


@pytest.mark.parametrize("case", [
    # (seed, row blocks, B_r, column blocks, B_c, density, H_qo, H_kv, num_ctas)
    (71, 6, 16, 40, 16, 0.3, 32, 8, 13),     # B_r = 16
    (72, 5, 64, 24, 8, 0.5, 16, 4, 7),       # B_c = 8
    (73, 4, 40, 30, 1, 0.4, 8, 8, 9),        # B_c = 1 (cp.async gather), ragged row blocks of 40
    (74, 3, 300, 20, 32, 0.6, 32, 8, 5),     # a row block spans several query tiles
], ids=["br16_bc16", "br64_bc8", "br40_bc1", "br300_bc32"])
def test_bsr_small(bsp, case):
    seed, nrb, br, ncb, bc, dens, hq, hk, C = case
    b = workloads.bsr_prefill_bf16(seed, nrb, br, ncb, bc, dens, hq, hk)
    O, L = oracle_full(b)
    out, lse, pa = run_batch(bsp, b, mode="prefill", num_ctas=C)
    compare(out, lse, O, L, "bf16")
    assert pa.check_device_error() == 0


def test_bsr_full_size(bsp):
    """32 row blocks of 64 rows over 512 column blocks of 16 tokens at 25%
    density: sampled rows against the oracle, two runs bitwise equal."""
    b = workloads.bsr_prefill_bf16()
    out, lse, pa = run_batch(bsp, b, mode="prefill")
    tok, head = sample_rows(b, 256, 24)
    O, L = oracle.attention_rows_of(b, tok, head)
    compare(out, lse, O, L, "bf16", rows=(tok, head))
    out2, lse2, _ = run_batch(bsp, b, mode="prefill")
    assert torch.equal(out, out2) and torch.equal(lse, lse2)

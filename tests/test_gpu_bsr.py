"""General block-sparse (BSR) attention with row blocks of B_r > 1 query rows
(engineering walkthrough §IV.3-IV.4, §V.1): each row block is a ragged query
group whose page list is its BSR row, run through the prefill path (non-causal)
and compared with the oracle on the same seeded inputs."""
import pytest
import torch

import workloads
from gpu_helpers import compare, lib, oracle_full, run_batch, timed

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
    density: every output row against the oracle, two runs bitwise equal."""
    b = workloads.bsr_prefill_bf16()
    out, lse, pa = run_batch(bsp, b, mode="prefill")
    (O, L), t = timed(oracle_full, b)
    compare(out, lse, O, L, "bf16", oracle_s=t)
    out2, lse2, _ = run_batch(bsp, b, mode="prefill")
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def variable_block_sparse(seed, row_sizes, col_sizes, density, hq, hk, D=128):
    """Variable block sparse: row block i has row_sizes[i] queries, column block
    j covers col_sizes[j] consecutive KV tokens; row block i attends to a seeded
    random subset of column blocks. Expressed with page size 1: the page list of
    row block i is the token slots of its column blocks."""
    import math
    import numpy as np
    rng = np.random.default_rng(seed)
    starts = np.concatenate([[0], np.cumsum(col_sizes)])
    n_kv = int(starts[-1])
    lists = []
    for _ in row_sizes:
        keep = np.flatnonzero(rng.random(len(col_sizes)) < density)
        if keep.size == 0:
            keep = np.array([0])
        lists.append(np.concatenate([np.arange(starts[j], starts[j + 1]) for j in keep]))
    kv_indptr = np.zeros(len(row_sizes) + 1, np.int32)
    kv_indptr[1:] = np.cumsum([len(x) for x in lists])
    qo_indptr = np.zeros(len(row_sizes) + 1, np.int32)
    qo_indptr[1:] = np.cumsum(row_sizes)
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(int(qo_indptr[-1]), hq, D, generator=gen).to(torch.bfloat16)
    k = torch.randn(n_kv, 1, hk, D, generator=gen).to(torch.bfloat16)
    v = torch.randn(n_kv, 1, hk, D, generator=gen).to(torch.bfloat16)
    return workloads.PagedBatch(name="variable_block_sparse", dtype="bf16", num_qo_heads=hq, num_kv_heads=hk,
                                head_dim=D, page_size=1, causal=False, sm_scale=1.0 / math.sqrt(D),
                                qo_indptr=qo_indptr, kv_indptr=kv_indptr, kv_indices=np.concatenate(lists).astype(np.int32),
                                last_page_len=np.ones(len(row_sizes), np.int32), q=q, k_pages=k, v_pages=v)


def test_variable_block_sparse(bsp):
    """Row blocks of 7..90 queries, column blocks of 3..61 tokens: the page-size-1
    gather covers any block sizes; against the oracle."""
    b = variable_block_sparse(75, [7, 90, 33, 64, 12], [3, 61, 17, 40, 5, 29, 33, 8], 0.5, 16, 4)
    O, L = oracle_full(b)
    out, lse, pa = run_batch(bsp, b, mode="prefill", num_ctas=11)
    compare(out, lse, O, L, "bf16")
    assert pa.check_device_error() == 0

"""GPU parity at the limits the header allows, against the fp64 oracle.

The largest batch (65,535 sequences, the grid's limit), the largest block of
packed rows per KV head (q_len * Hq / Hkv = 4096), very large and odd query
groups, and sequences whose rows see no key at all.  Large batches are
checked on a seeded sample of sequences (always including the first and
the last) and for finite output everywhere.
"""
import math

import numpy as np
import pytest
import torch

from sliding_window_speculative_gb300 import inputs
from tests.helpers import compare, forced_kernel, oracle_reference, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sliding_window_speculative_gb300 import build
    build.build()
    yield


def _sample(B, n, seed):
    rng = np.random.default_rng(seed)
    return sorted(set(rng.choice(B, size=min(n, B), replace=False).tolist()) | {0, B - 1})


@pytest.mark.parametrize("D,q_len,kernel", [(64, 1, "plan"), (128, 8, "plan"), (128, 8, "simt")])
def test_largest_batch(D, q_len, kernel):
    """65,535 sequences of 9..40 cached rows (window 16)."""
    B = 65535
    lens = inputs.context_lengths(B, 9, 40, seed=D + q_len)
    case = inputs.make_case("max_batch", B, 2, 1, D, q_len, 16, lens, 40, seed=5,
                            device="cuda", gen_device="cuda")
    with forced_kernel(kernel):
        out, lse = run_gpu(case)
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    seqs = _sample(B, 48, D)
    ref_o, ref_l = oracle_reference(case, seqs)
    compare(out[seqs], lse[seqs], ref_o, ref_l, f"B=65535 D{D} q{q_len} {kernel}")
    del case, out, lse
    torch.cuda.empty_cache()


@pytest.mark.parametrize("kernel", ["plan", "tc", "simt"])
def test_largest_row_block(kernel):
    """q_len 512 at 16 / 2 heads: 4096 packed rows per KV head."""
    case = inputs.make_case("max_rows", 2, 16, 2, 128, 512, 188, [512, 1400], 1536, seed=6,
                            outliers=True, device="cuda")
    with forced_kernel(kernel):
        out, lse = run_gpu(case)
    ref_o, ref_l = oracle_reference(case)
    compare(out, lse, ref_o, ref_l, f"4096 rows per KV head, {kernel}")


@pytest.mark.parametrize("Hq,Hkv,q_len", [(64, 1, 8), (48, 4, 3), (48, 4, 1), (12, 1, 17)])
@pytest.mark.parametrize("kernel", ["plan", "simt", "tc", "rows", "pairs"])
def test_large_and_odd_query_groups(Hq, Hkv, q_len, kernel):
    """G = 64 and G = 12 query heads per KV head, head_dim 128 and 256."""
    for D in (128, 256):
        lens = [q_len, 150, 333]
        case = inputs.make_case("groups", 3, Hq, Hkv, D, q_len, 100, lens, 384, seed=Hq + D,
                                outliers=True, device="cuda")
        with forced_kernel(kernel):
            out, lse = run_gpu(case)
            out3, lse3 = run_gpu(case, num_splits=3)
        ref_o, ref_l = oracle_reference(case)
        compare(out, lse, ref_o, ref_l, f"G={Hq // Hkv} q{q_len} D{D} {kernel}")
        compare(out3, lse3, ref_o, ref_l, f"G={Hq // Hkv} q{q_len} D{D} {kernel}, 3 splits")


@pytest.mark.parametrize("kernel", ["simt", "tc", "rows", "pairs"])
def test_sequences_with_no_visible_key(kernel):
    """seq_len 0 (nothing cached) and rows entirely before position 0: every
    such row gives out = 0 and lse = -inf; the other sequences are exact."""
    q_len = 8
    case = inputs.make_case("empty", 4, 8, 2, 128, q_len, 50, [0, 60, 0, 200], 256,
                            q_pos=[0, 52, -20, 192], seed=8, device="cuda")
    with forced_kernel(kernel):
        for splits in (0, 2):
            out, lse = run_gpu(case, splits)
            assert torch.all(out[0] == 0) and torch.all(lse[0] == -math.inf)
            assert torch.all(out[2] == 0) and torch.all(lse[2] == -math.inf)
            ref_o, ref_l = oracle_reference(case)
            compare(out, lse, ref_o, ref_l, f"empty sequences, {kernel}, {splits} splits")

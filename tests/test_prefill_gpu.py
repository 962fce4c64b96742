"""GPU parity of sliding-window prefill chunks (blocks of up to 512 query
rows, MAX_NUM_BATCHED_TOKENS in the pages' manifest) through the same entry
points as the verify blocks.  A work item reads only the windows of its own
draft rows, so these cases also check that narrowing: a row tile that read
too few keys fails the oracle comparison, and the count probe pins every
row's key count exactly."""
import math

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


@pytest.fixture(params=["simt", "tc", "rows", "pairs"])
def kernel(request):
    with forced_kernel(request.param):
        yield request.param


@pytest.mark.parametrize("D,q_len,window", [(64, 100, 37), (128, 256, 188), (256, 512, 188),
                                            (256, 200, 37), (128, 512, 600)])
@pytest.mark.parametrize("splits", [0, 5])
def test_prefill_chunk(D, q_len, window, splits, kernel):
    # a chunk at the start of a prompt (q_pos 0), one in the middle of a
    # longer context, and one clipped by the cache end
    lens = [q_len, q_len + 333, 1024]
    case = inputs.make_case("prefill", 3, 8, 2, D, q_len, window, lens, 1024, seed=31,
                            outliers=True, device="cuda")
    out, lse = run_gpu(case, splits)
    ref_o, ref_l = oracle_reference(case)
    compare(out, lse, ref_o, ref_l, f"prefill D{D} q{q_len} W{window} {splits} splits {kernel}")


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("q_len", [128, 512])
def test_prefill_count_probe(q_len, D, kernel):
    """K = 0: lse = ln |K(p)| for every row, with |K(p)| = min(W, p + 1) near
    the start of the sequence and W further on."""
    window = 188
    lens = [q_len, q_len + 50]
    case = inputs.make_case("count", 2, 8, 2, D, q_len, window, lens, 1024, seed=7,
                            device="cuda")
    case.k_cache.zero_()
    _, lse = run_gpu(case)
    for b, (sl, qp) in enumerate(zip(case.seq_lens_host, case.q_pos_host)):
        got = lse[b].double().cpu()
        for i in range(q_len):
            p = qp + i
            n = min(p, sl - 1) - max(0, p - window + 1) + 1
            assert torch.all((got[i] - math.log(n)).abs() < min(1e-3, 0.5 * math.log1p(1 / n))), \
                (b, i, n, got[i])


def test_prefill_with_fused_append():
    """A 256-token prefill chunk whose K/V rows are appended by the same call."""
    from tests.test_append_gpu import check_contiguous
    for kernel in ("simt", "tc", "rows"):
        with forced_kernel(kernel):
            case = inputs.make_case("prefill", 2, 8, 2, 256, 256, 188, [256, 700], 1024, seed=3,
                                    device="cuda")
            check_contiguous(case, 0, f"prefill append {kernel}")

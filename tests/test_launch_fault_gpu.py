"""Injected launch failures: the host's launch-error path, with no GPU fault.

`swa_set_debug_options(fail_launch=n)` makes the n-th kernel launch the
library makes not happen and report a launch error to its call.  For every
kernel, for the merge launch of split plans, for the fused append and for
greedy acceptance:

- the call returns SWA_ERR_CUDA naming the launch that failed;
- nothing of that call reached its outputs (or, for the fused append, the
  cache);
- the control is back to 0, the CUDA context still works, and the next
  call gives the same bits as before the failure, which match the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import sliding_window_speculative_gb300 as swa
from sliding_window_speculative_gb300 import inputs
from tests.helpers import compare, oracle_reference, run_gpu
from tests.test_append_gpu import take_block

pytestmark = pytest.mark.gpu

SENTINEL = 7.0


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sliding_window_speculative_gb300 import build
    build.build()
    yield
    swa.swa_set_debug_options()


def _q64(device):
    return inputs.make_case("q64", 3, 8, 2, 256, 64, 188, [64, 300, 1000], 1024, seed=21,
                            outliers=True, device=device)


# (kernel, workload, forced splits, failing launch, text of the failing launch)
CASES = [
    ("simt", lambda d: inputs.tiny(8, device=d), 0, 1, "attention kernel launch"),
    ("simt", lambda d: inputs.tiny(8, device=d), 3, 2, "merge kernel launch"),
    ("tc", lambda d: inputs.single_stream(device=d), 0, 1, "tensor-core kernel launch"),
    ("tc", lambda d: inputs.single_stream(device=d), 5, 2, "merge kernel launch"),
    ("rows", _q64, 0, 1, "tensor-core kernel launch"),
    ("rows", _q64, 3, 2, "merge kernel launch"),
    ("pairs", _q64, 0, 1, "tensor-core kernel launch"),
    ("pairs", _q64, 3, 2, "merge kernel launch"),
]


@pytest.mark.parametrize("kernel,make,splits,nth,what", CASES,
                         ids=[f"{c[0]}-splits{c[2]}-launch{c[3]}" for c in CASES])
def test_injected_launch_failure(kernel, make, splits, nth, what):
    case = make("cuda")
    try:
        swa.swa_set_debug_options(force_kernel=kernel)
        ref_out, ref_lse = run_gpu(case, splits)
        out = torch.full_like(ref_out, SENTINEL)
        lse = torch.full_like(ref_lse, SENTINEL)
        swa.swa_set_debug_options(force_kernel=kernel, fail_launch=nth)
        with pytest.raises(swa.SwaError) as e:
            swa.swa_verify_attn(case.q, case.k_cache, case.v_cache, case.seq_lens, case.q_pos,
                                case.window, case.scale, out=out, lse=lse, num_splits=splits)
        assert e.value.status == swa.SWA_ERR_CUDA
        assert what in str(e.value) and what in swa.swa_last_error()
        assert swa.swa_get_debug_options()["fail_launch"] == 0
        torch.cuda.synchronize()
        # with the first launch withheld nothing ran; with the merge withheld
        # the attention kernel wrote only its partials (workspace)
        assert torch.all(out == SENTINEL) and torch.all(lse == SENTINEL)
        again_out, again_lse = run_gpu(case, splits)
        assert torch.equal(again_out, ref_out) and torch.equal(again_lse, ref_lse)
    finally:
        swa.swa_set_debug_options()
    ref_o, ref_l = oracle_reference(case)
    compare(again_out, again_lse, ref_o, ref_l, f"after an injected failure, {kernel}")


@pytest.mark.parametrize("kernel", ["simt", "tc"])
def test_injected_launch_failure_leaves_the_cache(kernel):
    """The fused append's only launch withheld: the cache keeps its poisoned
    rows (no append happened), then the next call appends and attends."""
    case = inputs.single_stream(device="cuda")
    k_new, v_new = take_block(case)
    k0, v0 = case.k_cache.clone(), case.v_cache.clone()
    try:
        swa.swa_set_debug_options(force_kernel=kernel, fail_launch=1)
        with pytest.raises(swa.SwaError) as e:
            swa.swa_append_verify_attn(case.q, k_new, v_new, case.k_cache, case.v_cache,
                                       case.seq_lens, case.q_pos, case.window, case.scale)
        assert e.value.status == swa.SWA_ERR_CUDA and "launch" in str(e.value)
        torch.cuda.synchronize()
        assert torch.equal(case.k_cache, k0) and torch.equal(case.v_cache, v0)
        swa.swa_set_debug_options(force_kernel=kernel)
        out, lse = swa.swa_append_verify_attn(case.q, k_new, v_new, case.k_cache, case.v_cache,
                                              case.seq_lens, case.q_pos, case.window, case.scale)
        torch.cuda.synchronize()
    finally:
        swa.swa_set_debug_options()
    # the append wrote back the rows take_block read out (single_stream's
    # block ends at seq_len), so the cache is the original one again
    for b in range(case.q.shape[0]):
        qp, n = case.q_pos_host[b], case.q.shape[1]
        assert torch.equal(case.k_cache[b, :, qp:qp + n], k_new[b].transpose(0, 1))
        assert torch.equal(case.v_cache[b, :, qp:qp + n], v_new[b].transpose(0, 1))
    ref_o, ref_l = oracle_reference(case)
    compare(out, lse, ref_o, ref_l, f"append after an injected failure, {kernel}")


def test_injected_launch_failure_accept():
    """Greedy acceptance's launch withheld: outputs untouched, then a normal
    call."""
    g = torch.Generator(device="cpu").manual_seed(23)
    logits = torch.randn((4, 8, 4096), generator=g).to(torch.bfloat16).cuda()
    draft = torch.randint(0, 4096, (4, 7), generator=g, dtype=torch.int32).cuda()
    arg = torch.full((4, 8), -5, dtype=torch.int32, device="cuda")
    acc = torch.full((4,), -5, dtype=torch.int32, device="cuda")
    try:
        swa.swa_set_debug_options(fail_launch=1)
        with pytest.raises(swa.SwaError) as e:
            swa.swa_greedy_accept(logits, draft, argmax=arg, accepted=acc)
        assert e.value.status == swa.SWA_ERR_CUDA and "acceptance kernel launch" in str(e.value)
        torch.cuda.synchronize()
        assert torch.all(arg == -5) and torch.all(acc == -5)
    finally:
        swa.swa_set_debug_options()
    a2, c2 = swa.swa_greedy_accept(logits, draft)
    torch.cuda.synchronize()
    ref_am, ref_acc = oracle.greedy_accept(logits.cpu().double().numpy(),
                                           draft.cpu().numpy().astype(np.int64))
    assert np.array_equal(a2.cpu().numpy(), ref_am) and np.array_equal(c2.cpu().numpy(), ref_acc)

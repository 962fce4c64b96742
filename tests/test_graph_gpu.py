"""Verify calls captured in a CUDA graph and checked against the oracle.

The pages credit the single-graph decode step (ONEGRAPH=1 in "The Fast Gemma
Challenge: our verified-SOTA recipe, in full", section "What each piece does,
and why") with removing launch overhead.  Inside a graph, a plan that splits
the keys runs the attention kernel and the log-sum-exp merge kernel chained
by programmatic dependent launch.  Each call here is captured once and
replayed three times; new query rows (and, for the fused append, new K/V
block rows) are written into the captured buffers before every replay, and
every replay is compared with the fp64 oracle on that replay's inputs.
"""
import numpy as np
import pytest
import torch

from sliding_window_speculative_gb300 import inputs
from tests.helpers import compare, forced_kernel, oracle_reference
from tests.test_append_gpu import expected_cache, f64, take_block
from tests.test_paged_gpu import paginate

pytestmark = pytest.mark.gpu

REPLAYS = 3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sliding_window_speculative_gb300 import build
    build.build()
    yield


def _capture(call):
    """One call outside capture (grows the workspace), then the graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            call(s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return g


def _fresh(t, step, scale=1.0):
    """Overwrite tensor t in place with seeded N(0, scale^2) bf16 values."""
    g = torch.Generator().manual_seed(1000 + step)
    t.copy_((scale * torch.randn(t.shape, generator=g)).to(t.dtype))


def _plan(case, splits):
    import sliding_window_speculative_gb300 as swa
    return swa.swa_plan(swa.dims_of(case.q, case.k_cache, splits), case.window,
                        torch.cuda.get_device_properties(0).multi_processor_count)


def _replay_and_check(g, case, out, lse, what, before=None):
    prev = None
    for step in range(REPLAYS):
        _fresh(case.q, step)
        if before is not None:
            before(step)
        torch.cuda.synchronize()
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        ref_o, ref_l = oracle_reference(case)
        compare(out, lse, ref_o, ref_l, f"{what}, replay {step}")
        if prev is not None:
            assert not torch.equal(out, prev), f"{what}: replay {step} repeated the last output"
        prev = out.clone()


@pytest.mark.parametrize("name,splits,kernel,want", [
    # decode over the whole 4096-key context: 64 CUDA-core chunks + merge
    ("window_vs_full_w4096", 0, "plan", 1),
    # the single-stream verify block split in five: key-major tensor-core + merge
    ("single_stream", 5, "plan", 2),
    # the same with the rows-major tensor-core kernel, and on CTA pairs
    ("single_stream", 3, "rows", 3),
    ("single_stream", 3, "pairs", 4),
    # a 64-sequence batch split in two
    ("batched", 2, "plan", 2),
])
def test_graph_split_plan_matches_oracle(name, splits, kernel, want):
    from sliding_window_speculative_gb300 import swa_verify_attn
    case = {"window_vs_full_w4096": lambda: inputs.window_vs_full(4096, device="cuda"),
            "single_stream": lambda: inputs.single_stream(device="cuda"),
            "batched": lambda: inputs.batched(device="cuda")}[name]()
    with forced_kernel(kernel):
        plan = _plan(case, splits)
        assert plan["merge"] == 1 and plan["num_splits"] > 1 and plan["kernel"] == want, plan
        out = torch.empty_like(case.q)
        lse = torch.empty(case.q.shape[:3], dtype=torch.float32, device="cuda")
        g = _capture(lambda s: swa_verify_attn(case.q, case.k_cache, case.v_cache, case.seq_lens,
                                               case.q_pos, case.window, case.scale, out=out,
                                               lse=lse, num_splits=splits, stream=s))
        _replay_and_check(g, case, out, lse, f"graph {name} {splits} splits {kernel}")


@pytest.mark.parametrize("kernel", ["simt", "tc", "rows"])
def test_graph_paged_split_matches_oracle(kernel):
    from sliding_window_speculative_gb300 import swa_verify_attn_paged
    case = inputs.single_stream(device="cuda")
    kp, vp, table = paginate(case, 16)
    with forced_kernel(kernel):
        assert _plan(case, 4)["merge"] == 1
        out = torch.empty_like(case.q)
        lse = torch.empty(case.q.shape[:3], dtype=torch.float32, device="cuda")
        g = _capture(lambda s: swa_verify_attn_paged(case.q, kp, vp, table, case.seq_lens,
                                                     case.q_pos, case.window, case.scale,
                                                     out=out, lse=lse, num_splits=4, stream=s))
        _replay_and_check(g, case, out, lse, f"graph paged, 4 splits, {kernel}")


@pytest.mark.parametrize("kernel", ["simt", "tc", "rows"])
def test_graph_fused_append_split_matches_oracle(kernel):
    """Each replay appends a new block (fresh K/V rows) and attends over it:
    the cache rows must equal the oracle's append, and the attention the
    oracle's on that cache."""
    from sliding_window_speculative_gb300 import swa_append_verify_attn
    case = inputs.single_stream(device="cuda")
    k_blk, v_blk = take_block(case)
    k_new = torch.empty_like(k_blk)
    v_new = torch.empty_like(v_blk)
    with forced_kernel(kernel):
        assert _plan(case, 3)["merge"] == 1
        out = torch.empty_like(case.q)
        lse = torch.empty(case.q.shape[:3], dtype=torch.float32, device="cuda")
        k_new.copy_(k_blk)
        v_new.copy_(v_blk)
        g = _capture(lambda s: swa_append_verify_attn(case.q, k_new, v_new, case.k_cache,
                                                      case.v_cache, case.seq_lens, case.q_pos,
                                                      case.window, case.scale, out=out, lse=lse,
                                                      num_splits=3, stream=s))
        want = {}

        def new_block(step):
            _fresh(k_new, 10 + step)
            _fresh(v_new, 20 + step)
            want["k"] = expected_cache(case.k_cache, k_new, case)
            want["v"] = expected_cache(case.v_cache, v_new, case)

        prev = None
        for step in range(REPLAYS):
            _fresh(case.q, step)
            new_block(step)
            torch.cuda.synchronize()
            out.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            assert np.array_equal(f64(case.k_cache), want["k"]), f"{kernel} replay {step}: K"
            assert np.array_equal(f64(case.v_cache), want["v"]), f"{kernel} replay {step}: V"
            ref_o, ref_l = oracle_reference(case)
            compare(out, lse, ref_o, ref_l, f"graph fused append, 3 splits, {kernel}, "
                                            f"replay {step}")
            if prev is not None:
                assert not torch.equal(out, prev)
            prev = out.clone()

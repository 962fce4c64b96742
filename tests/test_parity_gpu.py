"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Element-by-element on the named workloads (every output for the small ones,
a seeded subset of sequences at the full bandwidth-stress size), forced
split counts, ragged and degenerate shapes, and bit-exact probes of the
window mask.
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


@pytest.fixture(params=["simt", "tc", "rows", "pairs"])
def kernel(request):
    """Runs the test once per kernel: the CUDA-core chunk kernel, the
    key-major tensor-core kernel, the rows-major tensor-core kernel and its
    CTA-pair form (shapes a tensor-core kernel does not cover fall back:
    head_dim 64 to the CUDA-core kernel, head_dim 128 under "pairs" to the
    one-CTA rows-major kernel)."""
    with forced_kernel(request.param):
        yield request.param


def _check(case, num_splits=0, seqs=None, what=None):
    out, lse = run_gpu(case, num_splits)
    ref_o, ref_l = oracle_reference(case, seqs)
    if seqs is not None:
        out, lse = out[list(seqs)], lse[list(seqs)]
    return compare(out, lse, ref_o, ref_l, what or case.name)


# ------------------------------------------------------------ named workloads

@pytest.mark.parametrize("q_len", [1, 8])
@pytest.mark.parametrize("splits", [0, 1, 2, 3])
def test_tiny(q_len, splits, kernel):
    _check(inputs.tiny(q_len, device="cuda"), splits)


@pytest.mark.parametrize("splits", [0, 1, 2, 5, 13])
def test_single_stream(splits, kernel):
    _check(inputs.single_stream(device="cuda"), splits)


@pytest.mark.parametrize("window", [188, 4096])
def test_window_vs_full(window, kernel):
    _check(inputs.window_vs_full(window, device="cuda"))


def test_batched(kernel):
    _check(inputs.batched(device="cuda"))


STRESS = [(w, q) for w in (188, 512, 1024) for q in (1, 8, 64)]


@pytest.mark.parametrize("window,q_len", STRESS)
def test_stress_full_size_sampled(window, q_len, kernel):
    """Full bandwidth-stress size (512 sequences, cache 32768); the oracle
    checks a seeded subset of 12 sequences (plus the shortest and longest)."""
    case = inputs.stress(window, q_len)
    rng = np.random.default_rng(window * 100 + q_len)
    seqs = set(rng.choice(512, size=12, replace=False).tolist())
    seqs.add(int(np.argmin(case.seq_lens_host)))
    seqs.add(int(np.argmax(case.seq_lens_host)))
    _check(case, seqs=sorted(seqs))
    del case
    torch.cuda.empty_cache()


# -------------------------------------------------------- shapes and edges

@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (6, 2), (16, 2), (8, 1)])
@pytest.mark.parametrize("q_len", [1, 3, 8, 17])
def test_ragged_shapes(D, Hq, Hkv, q_len, kernel):
    lens = [q_len, 5 + q_len, 100, 301, 77]
    case = inputs.make_case("ragged", 5, Hq, Hkv, D, q_len, 37, lens, 320, seed=11,
                            outliers=True, device="cuda")
    _check(case)
    _check(case, num_splits=4, what="ragged/4 splits")


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (16, 2)])
def test_max_draft_block(Hq, Hkv, kernel):
    """q_len 64 (the verify maximum); 16/2 heads gives 512 packed rows."""
    case = inputs.make_case("maxq", 3, Hq, Hkv, 256, 64, 188, [64, 300, 1000], 1024, seed=12,
                            outliers=True, device="cuda")
    _check(case)


@pytest.mark.parametrize("window", [1, 2, 63, 64, 65, 5000])
def test_window_sizes(window, kernel):
    case = inputs.make_case("win", 2, 8, 2, 128, 8, window, [200, 33], 256, seed=13,
                            device="cuda")
    _check(case)
    _check(case, num_splits=3, what=f"W{window}/3 splits")


def test_single_row_sequence(kernel):
    case = inputs.make_case("one", 1, 8, 2, 256, 1, 188, [1], 16, q_pos=[0], seed=14,
                            device="cuda")
    _check(case)


def test_nan_in_unseen_rows_never_reaches_output(kernel):
    """Rows before the window and past seq_len hold NaN (an unwritten cache)."""
    case = inputs.make_case("nan", 4, 8, 2, 256, 8, 188, [100, 1000, 4000, 9], 4096, seed=15,
                            device="cuda", fill="window", margin=0, poison="nan")
    for splits in (0, 1, 3, 7):
        out, lse = run_gpu(case, splits)
        assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    _check(case)


def test_rows_past_seq_len_and_before_zero(kernel):
    """Device preconditions broken on purpose: q_pos < 0 gives rows with no
    key (out 0, lse -inf); rows past seq_len see keys up to seq_len - 1."""
    case = inputs.make_case("defensive", 3, 4, 2, 64, 8, 10, [20, 12, 6], 24,
                            q_pos=[-3, 8, 2], seed=16, device="cuda")
    out, lse = run_gpu(case)
    assert torch.all(out[0, :3] == 0) and torch.all(lse[0, :3] == -math.inf)
    _check(case)


def test_deterministic(kernel):
    case = inputs.batched(device="cuda")
    a = run_gpu(case)
    b = run_gpu(case)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_lse_optional():
    from sliding_window_speculative_gb300 import swa_verify_attn
    case = inputs.single_stream(device="cuda")
    out, lse = swa_verify_attn(case.q, case.k_cache, case.v_cache, case.seq_lens, case.q_pos,
                               case.window, case.scale, want_lse=False)
    torch.cuda.synchronize()
    assert lse is None
    ref, _ = run_gpu(case)
    assert torch.equal(out, ref)


# ----------------------------------------------- bit-exact window probes

@pytest.mark.parametrize("window,q_len", [(188, 8), (188, 1), (16, 8), (1, 4), (512, 64)])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_count_probe(window, q_len, splits, kernel):
    """K = 0 makes every score 0, so lse = ln |K(p)| exactly: an off-by-one
    window (|K| = W + 1) moves lse by ln((W+1)/W) > 1e-3 for W <= 999."""
    lens = [window + q_len + 40, window // 2 + q_len, q_len]
    case = inputs.make_case("count", 3, 8, 2, 128, q_len, window, lens, max(lens) + 8,
                            seed=17, device="cuda")
    case.k_cache.zero_()
    _, lse = run_gpu(case, splits)
    for b, (sl, qp) in enumerate(zip(case.seq_lens_host, case.q_pos_host)):
        for i in range(q_len):
            p = qp + i
            n = min(p, sl - 1) - max(0, p - window + 1) + 1
            got = lse[b, i].double().cpu()
            assert torch.all((got - math.log(n)).abs() < min(1e-3, 0.5 * math.log1p(1 / n))), \
                (b, i, n, got)


@pytest.mark.parametrize("offset,inside", [(-188, False), (-187, True), (0, True), (1, False)])
def test_edge_probe(offset, inside, kernel):
    """One spike key at p + offset carries a marker value; rows see it only
    when it lies in (p - W, p]."""
    W, q_len = 188, 8
    case = inputs.make_case("edge", 1, 8, 2, 256, q_len, W, [1000], 1000, seed=18,
                            device="cuda")
    q_row = 3
    p = case.q_pos_host[0] + q_row
    j = p + offset
    case.k_cache.zero_()
    case.v_cache.zero_()
    # score of the spike for every query row: large positive
    case.q.fill_(1.0)
    case.k_cache[0, :, j] = 1.0
    case.v_cache[0, :, j] = 7.0
    out, _ = run_gpu(case)
    val = out[0, q_row].float()
    if inside:
        assert torch.all(val > 6.0), val.max()
    else:
        assert torch.all(val == 0.0), val.abs().max()


# ----------------------------------------------------- workspace contract

@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_workspace_caller_owned_and_capture():
    import sliding_window_speculative_gb300 as swa
    case = inputs.single_stream(device="cuda")
    dims = swa.dims_of(case.q, case.k_cache, num_splits=8)
    need = swa.swa_workspace_bytes(dims, case.window)
    assert need > 0
    ref, _ = run_gpu(case, 8)
    small = torch.empty(need // 8, dtype=torch.uint8, device="cuda")
    swa.swa_set_workspace(small)
    with pytest.raises(swa.SwaError) as e:
        run_gpu(case, 8)
    assert e.value.status == swa.SWA_ERR_WORKSPACE
    big = torch.empty(need, dtype=torch.uint8, device="cuda")
    swa.swa_set_workspace(big)
    out, _ = run_gpu(case, 8)
    assert torch.equal(out, ref)
    swa.swa_set_workspace(None)
    swa.swa_release_workspace()
    # capture with an empty library-owned workspace is refused, not allocated
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with pytest.raises(swa.SwaError) as e:
        with torch.cuda.graph(g, stream=s):
            swa.swa_verify_attn(case.q, case.k_cache, case.v_cache, case.seq_lens, case.q_pos,
                                case.window, case.scale, num_splits=8)
    assert e.value.status == swa.SWA_ERR_WORKSPACE


def test_graph_replay_matches_eager(kernel):
    import sliding_window_speculative_gb300 as swa
    case = inputs.single_stream(device="cuda")
    ref, ref_l = run_gpu(case)          # grows the workspace outside capture
    out = torch.empty_like(ref)
    lse = torch.empty_like(ref_l)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        swa.swa_verify_attn(case.q, case.k_cache, case.v_cache, case.seq_lens, case.q_pos,
                            case.window, case.scale, out=out, lse=lse)
    for _ in range(3):
        out.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref) and torch.equal(lse, ref_l)


def test_no_device_faults_recorded():
    import sliding_window_speculative_gb300 as swa
    run_gpu(inputs.tiny(8, device="cuda"))
    assert swa.swa_read_device_errors() == 0

"""GPU parity of the fused KV append + verify (swa_append_verify_attn).

Each case starts from a seeded workload whose cache already holds the
verify block's rows.  The test reads those rows out as k_new / v_new,
overwrites them in the cache with poison (K = 1e4, V = -1e4: a key read
before its append lands dominates the softmax and wrecks the output), and
calls the fused entry point.  Then

- the cache (with its guard bands) equals the oracle's append of the rows
  into the poisoned cache, bit for bit, and nothing else changed;
- out / lse agree with the oracle's attention over the original cache.
"""
import numpy as np
import pytest
import torch

import oracle
from sliding_window_speculative_gb300 import inputs
from tests.helpers import compare, forced_kernel, oracle_reference
from tests.test_paged_gpu import paginate

pytestmark = pytest.mark.gpu

POISON_K, POISON_V = 1.0e4, -1.0e4


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sliding_window_speculative_gb300 import build
    build.build()
    yield


@pytest.fixture(params=["simt", "tc", "rows"])
def kernel(request):
    with forced_kernel(request.param):
        yield request.param


def take_block(case):
    """k_new / v_new [B, q_len, Hkv, D] read from the cache at q_pos + i (rows
    past the cache end stay zero), then those cache rows set to poison."""
    B, q_len = case.q.shape[:2]
    Hkv, L, D = case.k_cache.shape[1:]
    k_new = torch.zeros((B, q_len, Hkv, D), dtype=torch.bfloat16, device=case.q.device)
    v_new = torch.zeros_like(k_new)
    for b, qp in enumerate(case.q_pos_host):
        n = max(0, min(q_len, L - qp))
        k_new[b, :n] = case.k_cache[b, :, qp:qp + n].transpose(0, 1)
        v_new[b, :n] = case.v_cache[b, :, qp:qp + n].transpose(0, 1)
        case.k_cache[b, :, qp:qp + n] = POISON_K
        case.v_cache[b, :, qp:qp + n] = POISON_V
    return k_new, v_new


def f64(t):
    return t.to(torch.float64).cpu().numpy()


def expected_cache(cache, rows, case):
    return oracle.append_rows(f64(cache), f64(rows), case.q_pos_host, case.seq_lens_host)


def run_append(case, k_new, v_new, num_splits=0, block_table=None, k_cache=None, v_cache=None):
    from sliding_window_speculative_gb300 import swa_append_verify_attn
    out, lse = swa_append_verify_attn(
        case.q, k_new, v_new, case.k_cache if k_cache is None else k_cache,
        case.v_cache if v_cache is None else v_cache, case.seq_lens, case.q_pos, case.window,
        case.scale, block_table=block_table, num_splits=num_splits)
    torch.cuda.synchronize()
    return out, lse


def check_contiguous(case, num_splits, what):
    ref_o, ref_l = oracle_reference(case)
    k_new, v_new = take_block(case)
    exp_k = expected_cache(case.k_cache, k_new, case)
    exp_v = expected_cache(case.v_cache, v_new, case)
    guard_k = case.k_buf.clone()
    n = case.k_cache.numel()
    off = case.k_cache.data_ptr() - case.k_buf.data_ptr()
    out, lse = run_append(case, k_new, v_new, num_splits)
    assert np.array_equal(f64(case.k_cache), exp_k), f"{what}: K cache"
    assert np.array_equal(f64(case.v_cache), exp_v), f"{what}: V cache"
    lo = off // 2
    assert torch.equal(case.k_buf[:lo], guard_k[:lo]), f"{what}: guard band before the cache"
    assert torch.equal(case.k_buf[lo + n:], guard_k[lo + n:]), f"{what}: guard band after"
    compare(out, lse, ref_o, ref_l, what)


@pytest.mark.parametrize("splits", [0, 3])
def test_single_stream_append(splits, kernel):
    case = inputs.single_stream(device="cuda")
    check_contiguous(case, splits, f"single_stream append, {splits} splits, {kernel}")


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("q_len", [1, 8, 17, 64])
def test_ragged_batch_append(D, q_len, kernel):
    lens = [q_len, 5 + q_len, 100, 301, 77 + q_len]
    for splits in (0, 4):
        case = inputs.make_case("ragged", 5, 8, 2, D, q_len, 37, lens, 384, seed=11,
                                outliers=True, device="cuda")
        check_contiguous(case, splits, f"append D{D} q{q_len} {splits} splits {kernel}")


def test_append_clips_rows_past_seq_len(kernel):
    """q_pos + q_len > seq_len (outside the documented preconditions): rows
    at or past seq_len, or past the cache end, are not written."""
    q_len = 8
    lens = [100, 60, 384]
    q_pos = [95, 56, 380]         # blocks run 3, 4 and 4 rows past seq_len
    case = inputs.make_case("clip", 3, 8, 2, 128, q_len, 37, lens, 384, q_pos=q_pos, seed=3,
                            device="cuda")
    check_contiguous(case, 0, f"append clipped, {kernel}")


@pytest.mark.parametrize("page_size", [8, 16, 64])
@pytest.mark.parametrize("q_len", [8, 64])
def test_paged_append(page_size, q_len, kernel):
    lens = [q_len, 5 + q_len, 100, 301, 77 + q_len]
    case = inputs.make_case("paged", 5, 8, 2, 256, q_len, 188, lens, 384, seed=13,
                            outliers=True, device="cuda")
    ref_o, ref_l = oracle_reference(case)
    k_new, v_new = take_block(case)
    exp_k = expected_cache(case.k_cache, k_new, case)
    exp_v = expected_cache(case.v_cache, v_new, case)
    kp, vp, table = paginate(case, page_size, poison=3.0)
    used = torch.zeros(kp.shape[0], dtype=torch.bool)
    used[table.flatten().long().cpu()] = True
    spare_k = kp[~used.to(kp.device)].clone()
    out, lse = run_append(case, k_new, v_new, block_table=table, k_cache=kp, v_cache=vp)
    # the pool read back through the table is the oracle's appended cache
    B, Hkv, L, D = case.k_cache.shape
    nb = L // page_size
    k_back = kp[table.long()].permute(0, 2, 1, 3, 4).reshape(B, Hkv, L, D)
    v_back = vp[table.long()].permute(0, 2, 1, 3, 4).reshape(B, Hkv, L, D)
    assert nb == table.shape[1]
    assert np.array_equal(f64(k_back), exp_k), f"paged {page_size} q{q_len}: K pool"
    assert np.array_equal(f64(v_back), exp_v), f"paged {page_size} q{q_len}: V pool"
    assert torch.equal(kp[~used.to(kp.device)], spare_k), "a page outside the tables changed"
    compare(out, lse, ref_o, ref_l, f"paged append {page_size} q{q_len} {kernel}")


def test_append_in_cuda_graph():
    """Captured once, replayed with new block contents: each replay writes
    that step's rows and attends over them."""
    from sliding_window_speculative_gb300 import swa_append_verify_attn
    case = inputs.single_stream(device="cuda")
    ref_o, ref_l = oracle_reference(case)
    k_blk, v_blk = take_block(case)
    k_new = torch.zeros_like(k_blk)
    v_new = torch.zeros_like(v_blk)
    out = torch.empty_like(case.q)
    lse = torch.empty(case.q.shape[:3], dtype=torch.float32, device="cuda")
    args = (case.q, k_new, v_new, case.k_cache, case.v_cache, case.seq_lens, case.q_pos,
            case.window, case.scale)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        swa_append_verify_attn(*args, out=out, lse=lse, stream=s)   # outside capture first
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            swa_append_verify_attn(*args, out=out, lse=lse, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    # replay 1: a block of zeros; replay 2: the real rows
    g.replay()
    torch.cuda.synchronize()
    qp = case.q_pos_host[0]
    assert torch.count_nonzero(case.k_cache[0, :, qp:qp + 8]) == 0
    k_new.copy_(k_blk)
    v_new.copy_(v_blk)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(case.k_cache[0, :, qp:qp + 8], k_blk[0].transpose(0, 1))
    compare(out, lse, ref_o, ref_l, "append in a CUDA graph")


def test_append_rejects_bad_arguments():
    import sliding_window_speculative_gb300 as swa
    case = inputs.single_stream(device="cuda")
    k_new, v_new = take_block(case)
    lib = swa.load_library()
    dims = swa.dims_of(case.q, case.k_cache)
    args = [case.q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), case.k_cache.data_ptr(),
            case.v_cache.data_ptr(), None, case.seq_lens.data_ptr(), case.q_pos.data_ptr(),
            case.window, case.scale, torch.empty_like(case.q).data_ptr(), None]
    import ctypes
    for i, bad in ((1, None), (2, None), (1, k_new.data_ptr() + 2)):
        a = list(args)
        a[i] = bad
        st = lib.swa_append_verify_attn(*a, ctypes.byref(dims), None)
        assert st == swa.SWA_ERR_INVALID_ARG, (i, st)

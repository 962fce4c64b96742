"""Prepared calls: an entry point validated and marshalled once, then
re-issued every step on buffers whose contents change (the serving loop's
shape).  Each re-issue must give the bits of the ordinary call on the same
contents, and meet the parity bar against the fp64 oracle."""
import pytest
import torch

import sliding_window_speculative_gb300 as swa
from sliding_window_speculative_gb300 import inputs
from tests.helpers import compare, oracle_reference
from tests.test_append_gpu import take_block
from tests.test_paged_gpu import paginate

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sliding_window_speculative_gb300 import build
    build.build()
    yield


def _fresh(t, step):
    g = torch.Generator().manual_seed(500 + step)
    t.copy_(torch.randn(t.shape, generator=g).to(t.dtype))


@pytest.mark.parametrize("name,splits", [("single_stream", 0), ("single_stream", 4),
                                         ("batched", 0), ("window_vs_full_w4096", 0)])
def test_prepared_verify(name, splits):
    case = {"single_stream": lambda: inputs.single_stream(device="cuda"),
            "batched": lambda: inputs.batched(device="cuda"),
            "window_vs_full_w4096": lambda: inputs.window_vs_full(4096, device="cuda")}[name]()
    call = swa.prepare(swa.swa_verify_attn, case.q, case.k_cache, case.v_cache, case.seq_lens,
                       case.q_pos, case.window, case.scale, num_splits=splits)
    for step in range(3):
        _fresh(case.q, step)
        out, lse = call()
        torch.cuda.synchronize()
        ref_out, ref_lse = swa.swa_verify_attn(case.q, case.k_cache, case.v_cache, case.seq_lens,
                                               case.q_pos, case.window, case.scale,
                                               num_splits=splits)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
        o, l_ = oracle_reference(case)
        compare(out, lse, o, l_, f"prepared {name} {splits} splits, step {step}")


def test_prepared_noalloc_and_paged():
    case = inputs.single_stream(device="cuda")
    out = torch.empty_like(case.q)
    lse = torch.empty(case.q.shape[:3], dtype=torch.float32, device="cuda")
    na = swa.prepare("swa_verify_attn_noalloc", case.q, case.k_cache, case.v_cache,
                     case.seq_lens, case.q_pos, case.window, case.scale, out, lse, num_splits=3)
    kp, vp, table = paginate(case, 16)
    pg = swa.prepare(swa.swa_verify_attn_paged, case.q, kp, vp, table, case.seq_lens, case.q_pos,
                     case.window, case.scale)
    for step in range(2):
        _fresh(case.q, step)
        o, l_ = oracle_reference(case)
        na()
        p_out, p_lse = pg()
        torch.cuda.synchronize()
        compare(out, lse, o, l_, f"prepared noalloc, step {step}")
        compare(p_out, p_lse, o, l_, f"prepared paged, step {step}")


def test_prepared_fused_append():
    """The end-to-end step's call: each step's block rows are written into
    k_new / v_new, the prepared fused append stores them and attends."""
    case = inputs.single_stream(device="cuda")
    k_blk, v_blk = take_block(case)
    k_new, v_new = torch.empty_like(k_blk), torch.empty_like(v_blk)
    call = swa.prepare(swa.swa_append_verify_attn, case.q, k_new, v_new, case.k_cache,
                       case.v_cache, case.seq_lens, case.q_pos, case.window, case.scale,
                       num_splits=0)
    p0, n = case.q_pos_host[0], case.q.shape[1]
    for step in range(3):
        _fresh(case.q, step)
        _fresh(k_new, 10 + step)
        _fresh(v_new, 20 + step)
        out, lse = call()
        torch.cuda.synchronize()
        assert torch.equal(case.k_cache[:, :, p0:p0 + n], k_new.transpose(1, 2))
        assert torch.equal(case.v_cache[:, :, p0:p0 + n], v_new.transpose(1, 2))
        o, l_ = oracle_reference(case)
        compare(out, lse, o, l_, f"prepared fused append, step {step}")


def test_prepare_rejects_bad_arguments_up_front():
    case = inputs.tiny(8, device="cuda")
    with pytest.raises(TypeError):
        swa.prepare(swa.swa_verify_attn, case.q.float(), case.k_cache, case.v_cache,
                    case.seq_lens, case.q_pos, case.window, case.scale)
    with pytest.raises(ValueError):
        swa.prepare("swa_greedy_accept", case.q)
    # an error the library finds is raised at call time
    call = swa.prepare(swa.swa_verify_attn, case.q, case.k_cache, case.v_cache, case.seq_lens,
                       case.q_pos, 0, case.scale)
    with pytest.raises(swa.SwaError) as e:
        call()
    assert e.value.status == swa.SWA_ERR_INVALID_ARG

"""GPU parity of the paged cache (block tables): the same workloads as the
contiguous tests, their caches scattered over a shuffled page pool whose
unused pages hold poison, through swa_verify_attn_paged against the oracle
run on the contiguous cache."""
import math

import pytest
import torch

from sliding_window_speculative_gb300 import inputs
from tests.helpers import compare, forced_kernel, oracle_reference

pytestmark = pytest.mark.gpu


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


def paginate(case, page_size, spare=5, seed=0, poison=float("nan")):
    """Pool [num_pages, Hkv, page_size, D] holding case's caches in shuffled
    pages, block table [B, L / page_size]; spare pages hold poison."""
    B, Hkv, L, D = case.k_cache.shape
    assert L % page_size == 0
    nb = L // page_size
    num = B * nb + spare
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(num, generator=g)
    table = perm[:B * nb].view(B, nb).to(torch.int32)
    kp = torch.full((num, Hkv, page_size, D), poison, dtype=torch.bfloat16, device=case.q.device)
    vp = torch.full_like(kp, poison)
    kc = case.k_cache.view(B, Hkv, nb, page_size, D)
    vc = case.v_cache.view(B, Hkv, nb, page_size, D)
    for b in range(B):
        for k in range(nb):
            kp[table[b, k]] = kc[b, :, k]
            vp[table[b, k]] = vc[b, :, k]
    return kp, vp, table.to(case.q.device)


def run_paged(case, page_size, num_splits=0, **kw):
    from sliding_window_speculative_gb300 import swa_verify_attn_paged
    kp, vp, table = paginate(case, page_size, **kw)
    out, lse = swa_verify_attn_paged(case.q, kp, vp, table, case.seq_lens, case.q_pos,
                                     case.window, case.scale, num_splits=num_splits)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("page_size", [8, 16, 64, 256])
@pytest.mark.parametrize("splits", [0, 3])
def test_single_stream_paged(page_size, splits, kernel):
    case = inputs.single_stream(device="cuda")
    out, lse = run_paged(case, page_size, splits)
    ref_o, ref_l = oracle_reference(case)
    compare(out, lse, ref_o, ref_l, f"paged {page_size}, {splits} splits, {kernel}")


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("q_len", [1, 8, 17, 64])
def test_ragged_batch_paged(D, q_len, kernel):
    lens = [q_len, 5 + q_len, 100, 301, 77 + q_len]
    case = inputs.make_case("ragged", 5, 8, 2, D, q_len, 37, lens, 384, seed=11, outliers=True,
                            device="cuda")
    ref_o, ref_l = oracle_reference(case)
    for page_size, splits in ((16, 0), (32, 4)):
        out, lse = run_paged(case, page_size, splits, seed=page_size)
        compare(out, lse, ref_o, ref_l, f"ragged D{D} q{q_len} page {page_size}")


@pytest.mark.parametrize("splits", [0, 3])
def test_count_probe_paged(splits, kernel):
    """K = 0: lse = ln |K(p)| exactly; chunk starts inside a page (split
    plans) must not add or drop a key."""
    window, q_len = 188, 8
    lens = [window + q_len + 40, window // 2 + q_len, q_len]
    case = inputs.make_case("count", 3, 8, 2, 128, q_len, window, lens, 320, seed=17,
                            device="cuda")
    case.k_cache.zero_()
    _, lse = run_paged(case, 16, splits)
    for b, (sl, qp) in enumerate(zip(case.seq_lens_host, case.q_pos_host)):
        for i in range(q_len):
            p = qp + i
            n = min(p, sl - 1) - max(0, p - window + 1) + 1
            got = lse[b, i].double().cpu()
            assert torch.all((got - math.log(n)).abs() < min(1e-3, 0.5 * math.log1p(1 / n))), \
                (b, i, n, got)


def test_paged_rejects_bad_tables():
    import sliding_window_speculative_gb300 as swa
    case = inputs.single_stream(device="cuda")
    kp, vp, table = paginate(case, 16)
    with pytest.raises(swa.SwaError) as e:   # pages of 12 rows: not a multiple of 8
        swa.swa_verify_attn_paged(case.q, kp.view(-1, 2, 12, 256)[:100], vp.view(-1, 2, 12, 256)[:100],
                                  table, case.seq_lens, case.q_pos, case.window, case.scale)
    assert e.value.status == swa.SWA_ERR_INVALID_ARG


def ring_pool(case, ring, page_size):
    """A window-sized ring per sequence, written as a block table: logical
    row j lives in slot j mod ring, logical page k in ring page k mod
    (ring / page_size). The ring holds each sequence's most recent `ring`
    rows; older rows were overwritten, so a read outside the window span
    picks up the wrong row and fails the parity check."""
    B, Hkv, L, D = case.k_cache.shape
    assert ring % page_size == 0 and L % page_size == 0
    rp = ring // page_size
    kp = torch.empty((B * rp, Hkv, page_size, D), dtype=torch.bfloat16, device=case.q.device)
    vp = torch.empty_like(kp)
    for b, sl in enumerate(case.seq_lens_host):
        for j in range(max(0, sl - ring), sl):
            s = j % ring
            kp[b * rp + s // page_size, :, s % page_size] = case.k_cache[b, :, j]
            vp[b * rp + s // page_size, :, s % page_size] = case.v_cache[b, :, j]
    k = torch.arange(L // page_size, dtype=torch.int32) % rp
    table = (torch.arange(B, dtype=torch.int32)[:, None] * rp + k[None, :]).to(case.q.device)
    return kp, vp, table


@pytest.mark.parametrize("q_len", [8, 64])
@pytest.mark.parametrize("page_size", [8, 64, 256])
def test_window_ring_as_block_table(q_len, page_size, kernel):
    """A cache of 256 slots (>= W + q_len - 1 = 251) serves positions far
    past its length; spans that wrap the ring cross from its last slot to
    its first."""
    from sliding_window_speculative_gb300 import swa_verify_attn_paged
    window = 188
    lens = [4096, 4000 + q_len, 1000, 256 + 3, window + q_len - 5, q_len]
    case = inputs.make_case("ring", len(lens), 8, 2, 256, q_len, window, lens, 4096, seed=23,
                            outliers=True, device="cuda")
    kp, vp, table = ring_pool(case, 256, page_size)
    out, lse = swa_verify_attn_paged(case.q, kp, vp, table, case.seq_lens, case.q_pos,
                                     case.window, case.scale)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle_reference(case)
    compare(out, lse, ref_o, ref_l, f"ring 256, page {page_size}, q{q_len}, {kernel}")

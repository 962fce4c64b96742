"""GPU parity of the fused greedy verification (argmax + accepted prefix)
through the C ABI against the oracle, bit-exact (token ids and counts)."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sliding_window_speculative_gb300 import build
    build.build()
    yield


def _case(B, q_len, V, seed, kind="normal", keep=False, accept=None):
    """Logits (bf16, device), drafts that accept `accept[b]` rows of the
    oracle's argmax (random per sequence if None), optional keep set."""
    g = torch.Generator().manual_seed(seed)
    if kind == "normal":
        x = torch.randn((B, q_len, V), generator=g)
    elif kind == "ties":          # small integers: many equal maxima
        x = torch.randint(-2, 3, (B, q_len, V), generator=g).float()
    else:                         # NaN / -inf sprinkled, some rows all -inf
        x = torch.randn((B, q_len, V), generator=g)
        m = torch.rand((B, q_len, V), generator=g)
        x[m < 0.05] = float("nan")
        x[(m >= 0.05) & (m < 0.1)] = float("-inf")
        x[:, 0, :] = float("-inf")
    logits = x.to(torch.bfloat16)
    keep_ids = torch.randperm(4 * V, generator=g)[:V].to(torch.int32) if keep else None
    ref_am, _ = oracle.greedy_accept(logits.double().numpy(), np.zeros((B, max(q_len - 1, 0))),
                                     None if keep_ids is None else keep_ids.numpy())
    rng = np.random.default_rng(seed)
    n = rng.integers(0, q_len, size=B) if accept is None else np.array(accept)
    draft = ref_am[:, :-1].copy()
    for b in range(B):
        if n[b] < q_len - 1:
            draft[b, n[b]] += 1 + rng.integers(0, 5)   # first mismatch at row n[b]
    ref_am2, ref_acc = oracle.greedy_accept(logits.double().numpy(), draft,
                                            None if keep_ids is None else keep_ids.numpy())
    assert np.array_equal(ref_am2, ref_am)
    return logits, keep_ids, torch.from_numpy(draft).to(torch.int32), ref_am, ref_acc


def _run(logits, keep_ids, draft):
    import sliding_window_speculative_gb300 as swa
    dev = "cuda"
    d = draft.to(dev) if draft.shape[1] > 0 else None
    am, acc = swa.swa_greedy_accept(logits.to(dev), d,
                                    None if keep_ids is None else keep_ids.to(dev))
    torch.cuda.synchronize()
    return am.cpu().numpy(), acc.cpu().numpy()


@pytest.mark.parametrize("B,q_len,V,kind,keep", [
    (1, 8, 262144, "normal", False),   # one verify block over a Gemma-size vocabulary
    (1, 8, 12000, "normal", True),     # a pruned LM head's keep set
    (64, 8, 4000, "normal", False),
    (3, 64, 1000, "ties", False),
    (2, 1, 7, "normal", False),        # q_len 1: nothing to accept
    (5, 5, 13, "special", True),       # odd vocabulary: rows off the 16-byte grid
    (4, 8, 1, "normal", False),        # one logit per row
    (7, 3, 8193, "ties", True),
])
def test_accept_matches_oracle(B, q_len, V, kind, keep):
    logits, keep_ids, draft, ref_am, ref_acc = _case(B, q_len, V, seed=B * 1000 + q_len, kind=kind,
                                                     keep=keep)
    for _ in range(2):   # the second call finds the scratch cleared by the first
        am, acc = _run(logits, keep_ids, draft)
        assert np.array_equal(am, ref_am)
        assert np.array_equal(acc, ref_acc)


def test_accept_every_prefix_length():
    q_len = 8
    logits, keep_ids, draft, ref_am, ref_acc = _case(q_len, q_len, 3000, seed=3,
                                                     accept=list(range(q_len)))
    am, acc = _run(logits, keep_ids, draft)
    assert acc.tolist() == list(range(q_len - 1)) + [q_len - 1]
    assert np.array_equal(am, ref_am)


def test_accept_scratch_grows_and_graph_replays():
    import sliding_window_speculative_gb300 as swa
    small = _case(1, 4, 500, seed=1)
    big = _case(300, 8, 700, seed=2)
    for logits, keep_ids, draft, ref_am, ref_acc in (small, big, small):
        am, acc = _run(logits, keep_ids, draft)
        assert np.array_equal(am, ref_am) and np.array_equal(acc, ref_acc)
    logits, keep_ids, draft, ref_am, ref_acc = big
    lg, dr = logits.cuda(), draft.cuda()
    am = torch.empty((300, 8), dtype=torch.int32, device="cuda")
    acc = torch.empty((300,), dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        swa.swa_greedy_accept(lg, dr, None, am, acc)
    for _ in range(3):
        am.zero_()
        acc.fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(am.cpu().numpy(), ref_am)
        assert np.array_equal(acc.cpu().numpy(), ref_acc)


def _signed_zero_logits(B, q_len, V, zeros, seed):
    """bf16 logits of negative values in [-4, -1] with the row maximum held
    as signed zeros at the given (column, sign) places of every row."""
    g = torch.Generator().manual_seed(seed)
    x = -1.0 - 3.0 * torch.rand((B, q_len, V), generator=g)
    for col, sign in zeros:
        x[:, :, col] = -0.0 if sign < 0 else 0.0
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("B,q_len,V,zeros,keep", [
    # -0.0 first, +0.0 later, in different threads of one CTA (8 logits per
    # 16-byte load: columns 0 and 8 belong to neighbouring threads)
    (1, 2, 4000, [(0, -1), (8, +1)], False),
    # the same across warps of one CTA
    (2, 3, 4000, [(3, -1), (1029, +1), (2047, -1)], False),
    # across CTAs of a 262,144-column row (chunks of 4096 logits)
    (1, 8, 262144, [(5, -1), (200000, +1)], False),
    (1, 8, 262144, [(70000, -1), (70008, +1), (262143, +1)], False),
    # +0.0 first, -0.0 later: still the first column
    (1, 4, 262144, [(9, +1), (100000, -1)], False),
    # through a keep set
    (3, 5, 262144, [(4100, -1), (4108, +1), (150000, +1)], True),
])
def test_accept_signed_zero_ties(B, q_len, V, zeros, keep):
    """-0.0 and +0.0 are equal maxima: the first column wins, wherever the
    two sit (threads, warps, CTAs), bit-exactly as the oracle says."""
    logits = _signed_zero_logits(B, q_len, V, zeros, seed=V + len(zeros))
    assert torch.signbit(logits[0, 0, zeros[0][0]]).item() == (zeros[0][1] < 0)
    g = torch.Generator().manual_seed(7)
    keep_ids = torch.randperm(2 * V, generator=g)[:V].to(torch.int32) if keep else None
    ref_am, _ = oracle.greedy_accept(logits.double().numpy(), np.zeros((B, q_len - 1)),
                                     None if keep_ids is None else keep_ids.numpy())
    first = zeros[0][0]
    want = keep_ids[first].item() if keep else first
    assert (ref_am == want).all()
    draft = torch.from_numpy(ref_am[:, :-1].copy()).to(torch.int32)
    _, ref_acc = oracle.greedy_accept(logits.double().numpy(), draft.numpy(),
                                      None if keep_ids is None else keep_ids.numpy())
    for _ in range(2):
        am, acc = _run(logits, keep_ids, draft)
        assert np.array_equal(am, ref_am)
        assert np.array_equal(acc, ref_acc)


def test_accept_random_signed_zero_maxima():
    """Rows whose maximum is zero at several random columns of random sign."""
    B, q_len, V = 16, 8, 50000
    g = torch.Generator().manual_seed(21)
    x = -1.0 - torch.rand((B, q_len, V), generator=g)
    cols = torch.randint(0, V, (B, q_len, 6), generator=g)
    signs = torch.randint(0, 2, (B, q_len, 6), generator=g)
    for b in range(B):
        for i in range(q_len):
            for c, s in zip(cols[b, i].tolist(), signs[b, i].tolist()):
                x[b, i, c] = -0.0 if s else 0.0
    logits = x.to(torch.bfloat16)
    ref_am, _ = oracle.greedy_accept(logits.double().numpy(), np.zeros((B, q_len - 1)), None)
    assert np.array_equal(ref_am, cols.min(dim=2).values.numpy())
    draft = torch.from_numpy(ref_am[:, :-1].copy()).to(torch.int32)
    am, acc = _run(logits, None, draft)
    assert np.array_equal(am, ref_am)
    assert (acc == q_len - 1).all()

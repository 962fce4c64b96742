"""The seeded input recipe on the CPU: shapes, positions, context draws,
the 1% outlier keys, poison outside the visible rows, and determinism."""
import math

import torch

from sliding_window_speculative_gb300 import inputs


def test_same_seed_same_tensors_other_seed_differs():
    a = inputs.make_case("a", 2, 8, 2, 64, 8, 16, [40, 30], 48, seed=5, outliers=True)
    b = inputs.make_case("b", 2, 8, 2, 64, 8, 16, [40, 30], 48, seed=5, outliers=True)
    c = inputs.make_case("c", 2, 8, 2, 64, 8, 16, [40, 30], 48, seed=6, outliers=True)
    for x, y in ((a.q, b.q), (a.k_buf, b.k_buf), (a.v_buf, b.v_buf)):
        assert torch.equal(x, y)
    assert not torch.equal(a.q, c.q) and not torch.equal(a.k_cache, c.k_cache)


def test_named_workload_shapes_and_positions():
    t1, t8 = inputs.tiny(1), inputs.tiny(8)
    assert t1.q.shape == (1, 1, 2, 64) and t1.q_pos_host == [39] and t1.seq_lens_host == [40]
    assert t8.q.shape == (1, 8, 2, 64) and t8.q_pos_host == [32] and t8.window == 16
    s = inputs.single_stream()
    assert s.q.shape == (1, 8, 8, 256) and s.k_cache.shape == (1, 2, 4096, 256)
    assert s.q_pos_host == [4088] and s.window == 188
    assert s.scale == 1.0 / math.sqrt(256)
    w = inputs.window_vs_full(4096, base=s)
    assert w.q_pos_host == [4095] and torch.equal(w.q[:, 0], s.q[:, -1])
    assert w.k_cache.data_ptr() == s.k_cache.data_ptr()
    bt = inputs.batched(device="cpu")
    assert bt.q.shape == (64, 8, 8, 256)
    assert all(qp == sl - 8 for qp, sl in zip(bt.q_pos_host, bt.seq_lens_host))


def test_context_lengths_are_inclusive_uniform_integers():
    lens = inputs.context_lengths(20000, 200, 4096)
    assert min(lens) >= 200 and max(lens) <= 4096
    assert abs(sum(lens) / len(lens) - 2148) < 40          # mean of U[200, 4096]
    small = inputs.context_lengths(2000, 0, 3)
    assert set(small) == {0, 1, 2, 3}                      # both ends drawn
    assert inputs.context_lengths(5, 1, 9, seed=1) == inputs.context_lengths(5, 1, 9, seed=1)


def test_one_percent_of_key_entries_scaled_by_eight():
    # |8x| > 5 for x ~ N(0, 1) has probability P(|x| > 0.625) = 0.532, while an
    # unscaled entry exceeds 5 with probability 6e-7: the share of keys above
    # 5 is 1% x 0.532
    s = inputs.single_stream()
    k = s.k_cache[0, :, :4096].float()
    share = (k.abs() > 5).float().mean().item()
    assert abs(share - 0.01 * 0.532) < 0.1 * 0.01 * 0.532
    v = s.v_cache[0, :, :4096].float()
    assert (v.abs() > 5).float().mean().item() < 1e-5      # values carry no outliers
    assert (s.q.float().abs() > 5).sum().item() == 0


def test_poison_outside_the_visible_rows():
    case = inputs.make_case("p", 2, 4, 2, 64, 4, 8, [20, 12], 32, seed=3, fill="window",
                            margin=2)
    for b, (sl, qp) in enumerate(zip(case.seq_lens_host, case.q_pos_host)):
        st = max(0, qp - case.window + 1 - 2)
        assert torch.all(case.k_cache[b, :, sl:] == inputs.POISON_K)
        assert torch.all(case.v_cache[b, :, sl:] == inputs.POISON_V)
        assert torch.all(case.v_cache[b, :, :st] == inputs.POISON_V)
        assert torch.all(case.v_cache[b, :, st:sl].abs() < 100)
    # guard bands before and after the cache
    D = 64
    off = (case.v_cache.data_ptr() - case.v_buf.data_ptr()) // 2
    assert off == 64 * D
    assert torch.all(case.v_buf[:off] == inputs.POISON_V)
    assert torch.all(case.v_buf[off + case.v_cache.numel():] == inputs.POISON_V)
    nan = inputs.make_case("n", 1, 4, 2, 64, 4, 8, [20], 32, seed=3, poison="nan")
    assert torch.isnan(nan.k_cache[0, :, :16 - 8 + 1]).all()   # before the first visible row
    assert torch.isnan(nan.k_cache[0, :, 20:]).all()
    assert not torch.isnan(nan.k_cache[0, :, 16 - 8 + 1:20]).any()

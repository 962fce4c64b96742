"""Pins of the fp64 oracle against things other than itself.

Each test fixes the oracle to a fact the windowed-attention definition or
plain mathematics settles: hand-worked examples, an independent brute-force
evaluation, reduction to full causal attention (a library routine), closed
forms, invariants, and the split-KV merge identity.  A plausible slip in the
oracle (window off by one, lost causality, wrong GQA head map, a dropped
max-subtraction term, a transposed operand) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from sliding_window_speculative_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")


def f64(t):
    return t.to(torch.float64).cpu().numpy()


def oracle_case(case, **kw):
    return oracle.attention(f64(case.q), f64(case.k_cache), f64(case.v_cache),
                            case.seq_lens_host, case.q_pos_host, case.window, case.scale, **kw)


# --------------------------------------------------------------- hand worked

def _load_golden():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("c", _load_golden(), ids=lambda c: c["name"])
def test_hand_worked_examples(c):
    B, q_len, Hq, Hkv, D = c["B"], c["q_len"], c["Hq"], c["Hkv"], c["D"]
    q = np.array(c["q"], dtype=np.float64)
    T = c["seq_lens"][0]
    if c.get("k_zero"):
        k = np.zeros((B, Hkv, T, D))
        v = np.zeros((B, Hkv, T, D))
        for g, row in enumerate(c["v_const"]):
            v[:, g, :, :] = np.array(row)
    else:
        k = np.zeros((B, Hkv, T, D))
        k[..., 0] = np.array(c["k_log_weights"])
        v = np.array(c["v"], dtype=np.float64)
    out, lse = oracle.attention(q, k, v, c["seq_lens"], c["q_pos"], c["window"], c["scale"])
    np.testing.assert_allclose(out, np.array(c["out"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(c["lse"]), rtol=0, atol=1e-12)


# --------------------------------------------------- independent brute force

def brute_force(q, k, v, seq_lens, q_pos, window, scale):
    """Separately written evaluation: per-element loops, no max subtraction,
    weights exp(s) / sum exp(s) taken literally."""
    B, q_len, Hq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    out = np.zeros_like(q)
    lse = np.zeros((B, q_len, Hq))
    for b in range(B):
        for i in range(q_len):
            p = q_pos[b] + i
            for h in range(Hq):
                keys = [j for j in range(seq_lens[b]) if p - window < j <= p]
                e = []
                for j in keys:
                    s = 0.0
                    for d in range(D):
                        s += q[b, i, h, d] * k[b, h // G, j, d]
                    e.append(math.exp(scale * s))
                z = sum(e)
                lse[b, i, h] = math.log(z)
                for d in range(D):
                    out[b, i, h, d] = sum(e[t] * v[b, h // G, j, d] for t, j in enumerate(keys)) / z
    return out, lse


@pytest.mark.parametrize("q_len", [1, 8])
def test_brute_force_tiny(q_len):
    case = inputs.tiny(q_len)
    out, lse = oracle_case(case)
    bo, bl = brute_force(f64(case.q), f64(case.k_cache), f64(case.v_cache),
                         case.seq_lens_host, case.q_pos_host, case.window, case.scale)
    np.testing.assert_allclose(out, bo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, bl, rtol=0, atol=1e-12)


def test_brute_force_gqa_batch_ragged():
    """Several sequences of different lengths, G=3, positions near the start
    (window clipped at 0) and at the end."""
    case = inputs.make_case("bf", 3, 6, 2, 16, 5, 7, [5, 12, 30], 32, q_pos=[0, 4, 25],
                            seed=3, outliers=True)
    out, lse = oracle_case(case)
    bo, bl = brute_force(f64(case.q), f64(case.k_cache), f64(case.v_cache),
                         case.seq_lens_host, case.q_pos_host, case.window, case.scale)
    np.testing.assert_allclose(out, bo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, bl, rtol=0, atol=1e-12)


def test_brute_force_prefill_block():
    """A prefill-sized block (more rows than the window): rows near the
    start see the whole prefix, later rows slide; G=2, ragged lengths."""
    case = inputs.make_case("pf", 2, 4, 2, 8, 40, 9, [40, 47], 48, seed=12, outliers=True)
    out, lse = oracle_case(case)
    bo, bl = brute_force(f64(case.q), f64(case.k_cache), f64(case.v_cache),
                         case.seq_lens_host, case.q_pos_host, case.window, case.scale)
    np.testing.assert_allclose(out, bo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, bl, rtol=0, atol=1e-12)


def test_prefill_recipe():
    """The prefill workload's block is the last q_len positions of each
    sequence, contexts within [q_len, max_len]."""
    case = inputs.prefill(64, batch=5, device="cpu", max_len=256)
    assert case.q.shape == (5, 64, 8, 256)
    for sl, qp in zip(case.seq_lens_host, case.q_pos_host):
        assert 64 <= sl <= 256 and qp == sl - 64


# ------------------------------------------- W >= context: full causal (SDPA)

@pytest.mark.parametrize("D,Hq,Hkv,ctx,q_len", [(64, 2, 1, 40, 8), (256, 8, 2, 300, 8),
                                                 (128, 4, 4, 97, 64)])
def test_full_window_is_causal_attention(D, Hq, Hkv, ctx, q_len):
    case = inputs.make_case("full", 1, Hq, Hkv, D, q_len, 4096, [ctx], ctx, seed=1,
                            outliers=True)
    out, lse = oracle_case(case)
    q = case.q.to(torch.float64).permute(0, 2, 1, 3)               # [B, Hq, q, D]
    k = case.k_cache.to(torch.float64).repeat_interleave(Hq // Hkv, dim=1)
    v = case.v_cache.to(torch.float64).repeat_interleave(Hq // Hkv, dim=1)
    pos = case.q_pos_host[0] + torch.arange(q_len)
    mask = torch.arange(ctx)[None, :] <= pos[:, None]               # causal
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask,
                                                           scale=case.scale)
    np.testing.assert_allclose(out, ref.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-11)
    s = torch.einsum("bhqd,bhkd->bhqk", q, k) * case.scale
    ref_lse = torch.logsumexp(s.masked_fill(~mask, -math.inf), dim=-1)
    np.testing.assert_allclose(lse, ref_lse.permute(0, 2, 1).numpy(), rtol=0, atol=1e-11)


# ----------------------------------------------------- q_len = 1 is decode

def test_draft_row_equals_decode():
    case = inputs.single_stream()
    out8, lse8 = oracle_case(case)
    for i in (0, 3, 7):
        c1 = inputs.make_case("d", 1, 8, 2, 256, 1, case.window, case.seq_lens_host, 4096,
                              q_pos=[case.q_pos_host[0] + i], q=case.q[:, i:i + 1],
                              kv=(case.k_buf, case.v_buf, case.k_cache, case.v_cache))
        out1, lse1 = oracle_case(c1)
        np.testing.assert_array_equal(out1[:, 0], out8[:, i])
        np.testing.assert_array_equal(lse1[:, 0], lse8[:, i])


# ------------------------------------------------ weights: sum 1, mask exact

@pytest.mark.parametrize("window,q_len,q_pos", [(16, 8, 32), (16, 1, 39), (1, 4, 10),
                                                (40, 8, 32), (5, 3, 0)])
def test_weights_sum_to_one_and_vanish_outside_window(window, q_len, q_pos):
    """V = identity (V[j] = e_j) turns the output into the weight vector."""
    ctx, D = 40, 64
    case = inputs.make_case("w", 1, 2, 1, D, q_len, window, [ctx], ctx, q_pos=[q_pos], seed=2)
    v = np.zeros((1, 1, ctx, D))
    for j in range(ctx):
        v[0, 0, j, j] = 1.0
    out, _ = oracle.attention(f64(case.q), f64(case.k_cache), v, [ctx], [q_pos], window,
                              case.scale)
    for i in range(q_len):
        p = q_pos + i
        for h in range(2):
            w = out[0, i, h]
            assert abs(w.sum() - 1.0) < 1e-12
            inside = [j for j in range(D) if max(0, p - window + 1) <= j <= min(p, ctx - 1)]
            outside = [j for j in range(D) if j not in inside]
            assert np.all(w[outside] == 0.0)
            assert np.all(w[inside] > 0.0)
            assert len(inside) == min(window, p + 1)


def test_constant_value_row_is_returned():
    case = inputs.single_stream()
    v = np.zeros(f64(case.v_cache).shape)
    row = np.linspace(-3, 5, 256)
    v[:] = row
    out, _ = oracle.attention(f64(case.q), f64(case.k_cache), v, case.seq_lens_host,
                              case.q_pos_host, case.window, case.scale)
    np.testing.assert_allclose(out, np.broadcast_to(row, out.shape), rtol=0, atol=1e-12)


def test_zero_keys_closed_form():
    """K = 0: every score is 0, so out is the mean of V over the window and
    lse = ln |K(p)|."""
    case = inputs.make_case("z", 2, 4, 2, 32, 8, 10, [30, 7], 30, q_pos=[22, 0], seed=4)
    v = f64(case.v_cache)
    out, lse = oracle.attention(f64(case.q), np.zeros(v.shape), v, case.seq_lens_host,
                                case.q_pos_host, case.window, case.scale)
    for b in range(2):
        for i in range(8):
            p = case.q_pos_host[b] + i
            lo, hi = max(0, p - 9), min(p, case.seq_lens_host[b] - 1)
            for h in range(4):
                np.testing.assert_allclose(out[b, i, h], v[b, h // 2, lo:hi + 1].mean(0),
                                           rtol=0, atol=1e-12)
                assert abs(lse[b, i, h] - math.log(hi - lo + 1)) < 1e-12


def test_value_shift_invariance():
    case = inputs.tiny(8)
    out, _ = oracle_case(case)
    shift = np.linspace(1, 2, 64)
    out2, _ = oracle.attention(f64(case.q), f64(case.k_cache), f64(case.v_cache) + shift,
                               case.seq_lens_host, case.q_pos_host, case.window, case.scale)
    np.testing.assert_allclose(out2, out + shift, rtol=0, atol=1e-12)


def test_scale_enters_as_product_with_scores():
    """Doubling q and halving scale leaves the result; doubling scale alone
    sharpens it (lse changes)."""
    case = inputs.tiny(8)
    out, lse = oracle_case(case)
    out2, lse2 = oracle.attention(2 * f64(case.q), f64(case.k_cache), f64(case.v_cache),
                                  case.seq_lens_host, case.q_pos_host, case.window,
                                  case.scale / 2)
    np.testing.assert_allclose(out2, out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-12)
    _, lse3 = oracle.attention(f64(case.q), f64(case.k_cache), f64(case.v_cache),
                               case.seq_lens_host, case.q_pos_host, case.window,
                               case.scale * 2)
    assert np.max(np.abs(lse3 - lse)) > 0.1


# --------------------------------------------------------- LSE merge (a8)

@pytest.mark.parametrize("nsplit", [1, 2, 3, 7])
def test_split_merge_identity(nsplit):
    case = inputs.make_case("m", 2, 8, 2, 64, 8, 20, [60, 33], 60, seed=5, outliers=True)
    out, lse = oracle_case(case)
    rng = np.random.default_rng(nsplit)
    B = 2
    cuts = []
    for b in range(B):
        lo = max(0, case.q_pos_host[b] - case.window + 1)
        hi = case.seq_lens_host[b]
        inner = np.sort(rng.choice(np.arange(lo + 1, hi), size=nsplit - 1, replace=False))
        cuts.append([lo, *inner.tolist(), hi])
    ms, ls, accs = [], [], []
    for s in range(nsplit):
        m, l, acc = oracle.partial(f64(case.q), f64(case.k_cache), f64(case.v_cache),
                                   case.seq_lens_host, case.q_pos_host, case.window,
                                   case.scale, [c[s] for c in cuts], [c[s + 1] for c in cuts])
        ms.append(m.reshape(-1))
        ls.append(l.reshape(-1))
        accs.append(acc.reshape(-1, 64))
    mo, ml = oracle.lse_merge(np.stack(ms), np.stack(ls), np.stack(accs))
    np.testing.assert_allclose(mo.reshape(out.shape), out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ml.reshape(lse.shape), lse, rtol=0, atol=1e-12)


def test_merge_of_empty_partials():
    m = np.array([[-np.inf], [-np.inf]])
    l = np.zeros((2, 1))
    acc = np.zeros((2, 1, 4))
    out, lse = oracle.lse_merge(m, l, acc)
    assert np.all(out == 0) and lse[0] == -np.inf
    m = np.array([[-np.inf], [0.5]])
    l = np.array([[0.0], [2.0]])
    acc = np.zeros((2, 1, 4))
    acc[1, 0] = [2, 4, 6, 8]
    out, lse = oracle.lse_merge(m, l, acc)
    np.testing.assert_allclose(out[0], [1, 2, 3, 4], atol=1e-15)
    assert abs(lse[0] - (0.5 + math.log(2.0))) < 1e-15


# ------------------------------------------------------------ edge cases

def test_row_without_keys_is_zero_with_minus_inf_lse():
    """Rows before position 0 (q_pos < 0) have an empty window."""
    case = inputs.make_case("e", 1, 2, 1, 16, 4, 3, [10], 10, q_pos=[-2], seed=6)
    out, lse = oracle_case(case)
    assert np.all(out[0, :2] == 0) and np.all(lse[0, :2] == -np.inf)
    assert np.all(np.isfinite(lse[0, 2:]))


def test_slice_must_cover_window():
    case = inputs.tiny(8)
    k = f64(case.k_cache)[:, :, 30:]
    v = f64(case.v_cache)[:, :, 30:]
    with pytest.raises(ValueError):
        oracle.attention(f64(case.q), k, v, [40], [32], 16, case.scale, base=[30])
    out, lse = oracle.attention(f64(case.q), f64(case.k_cache)[:, :, 17:],
                                f64(case.v_cache)[:, :, 17:], [40], [32], 16, case.scale,
                                base=[17])
    ref, rl = oracle_case(case)
    np.testing.assert_array_equal(out, ref)
    np.testing.assert_array_equal(lse, rl)


def test_threads_do_not_change_result():
    case = inputs.make_case("t", 4, 8, 2, 64, 8, 30, [50, 40, 64, 31], 64, seed=7)
    a = oracle_case(case, threads=1)
    b = oracle_case(case, threads=5)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


# ------------------------------------------------- greedy verification (accept)

def _load_accept_golden():
    path = os.path.join(os.path.dirname(__file__), "golden", "accept_cases.json")
    with open(path) as f:
        return json.load(f)["cases"]


def _num(x):
    return float(x) if not isinstance(x, str) else {"nan": np.nan, "-inf": -np.inf,
                                                     "inf": np.inf}[x]


@pytest.mark.parametrize("case", _load_accept_golden(), ids=lambda c: c["name"])
def test_accept_hand_worked_examples(case):
    logits = np.array([[[_num(x) for x in row] for row in seq] for seq in case["logits"]])
    B, q_len, _ = logits.shape
    draft = np.array(case["draft"], dtype=np.int64).reshape(B, q_len - 1)
    am, acc = oracle.greedy_accept(logits, draft, case["keep"])
    assert am.tolist() == case["argmax"], case["derivation"]
    assert acc.tolist() == case["accepted"], case["derivation"]


def test_accept_matches_numpy_argmax_and_prefix_count():
    # NaN-free rows reduce to numpy's argmax (first maximum) and a plain
    # prefix count; ties are forced by drawing small integers
    rng = np.random.default_rng(7)
    for B, q_len, V in [(3, 8, 50), (2, 1, 7), (1, 64, 300), (4, 5, 1)]:
        logits = rng.integers(-3, 4, size=(B, q_len, V)).astype(np.float64)
        ref_am = np.argmax(logits, axis=2)
        for k in range(q_len):
            draft = np.where(np.arange(q_len - 1)[None, :] < k, ref_am[:, :-1],
                             ref_am[:, :-1] + 1 if V > 1 else ref_am[:, :-1] - 1)
            am, acc = oracle.greedy_accept(logits, draft)
            assert np.array_equal(am, ref_am)
            assert np.all(acc == min(k, q_len - 1))


def test_accept_keep_set_is_a_relabelling():
    rng = np.random.default_rng(8)
    logits = rng.standard_normal((2, 8, 40))
    keep = rng.permutation(1000)[:40]
    am0, _ = oracle.greedy_accept(logits, np.zeros((2, 7), dtype=np.int64))
    am1, acc1 = oracle.greedy_accept(logits, keep[am0[:, :-1]], keep)
    assert np.array_equal(am1, keep[am0])
    assert np.all(acc1 == 7)                 # drafts taken from the argmax: all accepted


# ------------------------------------------------------------ fused KV append

def _load_append_golden():
    path = os.path.join(os.path.dirname(__file__), "golden", "append_cases.json")
    with open(path) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _load_append_golden(), ids=lambda c: c["name"])
def test_append_hand_worked_examples(case):
    got = oracle.append_rows(np.array(case["cache"], dtype=np.float64),
                             np.array(case["rows"], dtype=np.float64), case["q_pos"],
                             case["seq_lens"])
    assert np.array_equal(got, np.array(case["expected"], dtype=np.float64)), case["derivation"]


def test_append_restores_a_cleared_block():
    # A seeded case's cache already holds its block's rows; blanking them and
    # appending the rows read back out gives the cache back exactly, so
    # attention over the appended cache is the attention of the case itself.
    case = inputs.make_case("append", 3, 8, 2, 64, 8, 16, [40, 8, 25], 48, seed=5)
    k, v = f64(case.k_cache), f64(case.v_cache)
    B, Hkv, L, D = k.shape
    rows_k = np.zeros((B, 8, Hkv, D))
    rows_v = np.zeros((B, 8, Hkv, D))
    k0, v0 = k.copy(), v.copy()
    for b, qp in enumerate(case.q_pos_host):
        rows_k[b] = k[b, :, qp:qp + 8].transpose(1, 0, 2)
        rows_v[b] = v[b, :, qp:qp + 8].transpose(1, 0, 2)
        k0[b, :, qp:qp + 8] = 7.0
        v0[b, :, qp:qp + 8] = -7.0
    k1 = oracle.append_rows(k0, rows_k, case.q_pos_host, case.seq_lens_host)
    v1 = oracle.append_rows(v0, rows_v, case.q_pos_host, case.seq_lens_host)
    assert np.array_equal(k1, k) and np.array_equal(v1, v)
    assert np.all(k0[0, :, case.q_pos_host[0]] == 7.0)   # the input is not modified


def test_append_writes_nothing_outside_the_block():
    rng = np.random.default_rng(9)
    cache = rng.standard_normal((2, 3, 20, 4))
    rows = rng.standard_normal((2, 5, 3, 4))
    got = oracle.append_rows(cache, rows, [4, 15], [9, 20])
    mask = np.zeros(cache.shape, dtype=bool)
    mask[0, :, 4:9] = True
    mask[1, :, 15:20] = True
    assert np.array_equal(got[~mask], cache[~mask])
    assert np.array_equal(got[0, :, 4:9], rows[0].transpose(1, 0, 2))
    assert np.array_equal(got[1, :, 15:20], rows[1].transpose(1, 0, 2))

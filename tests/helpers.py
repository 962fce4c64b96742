"""Shared test plumbing: host copies of window slices for the oracle, the
tolerance check, and a GPU-path runner."""
import math

import numpy as np
import torch

import oracle

# Tolerances of the parity bar: max abs 2e-2, max rel 2e-2 (relative to
# max(|ref|, 1e-2)), lse within 1e-3 abs.
ATOL = 2e-2
RTOL = 2e-2
REL_FLOOR = 1e-2
LSE_ATOL = 1e-3


def host_slices(case, seqs=None, margin=64):
    """fp64 host copies of q and of each sequence's cache rows
    [max(0, q_pos - W + 1 - margin), seq_len), padded to one length.
    Returns (q, k, v, base, seq_lens, q_pos) for the oracle."""
    seqs = list(range(case.q.shape[0])) if seqs is None else list(seqs)
    spans = case.span(margin)
    T = max(spans[b][1] - spans[b][0] for b in seqs)
    Hkv, D = case.k_cache.shape[1], case.k_cache.shape[3]
    k = np.zeros((len(seqs), Hkv, max(T, 1), D))
    v = np.zeros_like(k)
    for n, b in enumerate(seqs):
        st, sl = spans[b]
        k[n, :, :sl - st] = case.k_cache[b, :, st:sl].to(torch.float64).cpu().numpy()
        v[n, :, :sl - st] = case.v_cache[b, :, st:sl].to(torch.float64).cpu().numpy()
    q = case.q[seqs].to(torch.float64).cpu().numpy()
    base = [spans[b][0] for b in seqs]
    return (q, k, v, base, [case.seq_lens_host[b] for b in seqs],
            [case.q_pos_host[b] for b in seqs])


def oracle_reference(case, seqs=None, margin=64):
    q, k, v, base, sl, qp = host_slices(case, seqs, margin)
    return oracle.attention(q, k, v, sl, qp, case.window, case.scale, base=base)


def run_gpu(case, num_splits=0):
    from sliding_window_speculative_gb300 import swa_verify_attn
    out, lse = swa_verify_attn(case.q, case.k_cache, case.v_cache, case.seq_lens, case.q_pos,
                               case.window, case.scale, num_splits=num_splits)
    torch.cuda.synchronize()
    return out, lse


def compare(out_gpu, lse_gpu, out_ref, lse_ref, what=""):
    """Assert the parity bar; returns (max_abs, max_rel, max_lse)."""
    o = out_gpu.to(torch.float64).cpu().numpy()
    l = lse_gpu.to(torch.float64).cpu().numpy()
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    err = np.abs(o - out_ref)
    rel = err / np.maximum(np.abs(out_ref), REL_FLOOR)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(fin, np.isfinite(l)), f"{what}: empty-row pattern differs"
    assert np.all(l[~fin] == -np.inf)
    lerr = np.abs(l[fin] - lse_ref[fin]) if fin.any() else np.zeros(1)
    max_abs, max_rel, max_lse = float(err.max()), float(rel.max()), float(lerr.max())
    worst = np.unravel_index(int(np.argmax(err)), err.shape)
    msg = (f"{what}: max_abs {max_abs:.3e} at {tuple(int(x) for x in worst)}, "
           f"max_rel {max_rel:.3e}, max_lse {max_lse:.3e}")
    assert max_abs <= ATOL and max_rel <= RTOL and max_lse <= LSE_ATOL, msg
    return max_abs, max_rel, max_lse


def ln_count(n):
    return math.log(n)

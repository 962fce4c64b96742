"""Host copies of a workload's window slices for the fp64 oracle.

TEST INFRASTRUCTURE ONLY, like the rest of this package: used by ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``.  It
only copies data (bf16 widened exactly to float64); no arithmetic of the
method happens here.
"""
import numpy as np
import torch


def host_slices(case, seqs=None, margin=64):
    """fp64 host copies of q and of each sequence's cache rows
    [max(0, q_pos - W + 1 - margin), seq_len), padded to one length.
    Returns (q, k, v, base, seq_lens, q_pos) for ``oracle.attention``: row t
    of sequence n's slice holds key position base[n] + t."""
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

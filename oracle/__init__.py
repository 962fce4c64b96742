"""fp64 CPU oracle for sliding-window verify attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The CUDA
library never calls it and it shares no code with the CUDA library.

It follows "The Fast Gemma Challenge: our verified-SOTA recipe, in full",
section "What each piece does, and why" (sliding window: attend to the most
recent W tokens), with the window read as (p-W, p], and the split-KV verify
partial/merge of the manifest entry SPLITKV_VERIFY on the same page.  The
arithmetic lives in ``swa_oracle.c``; this module only marshals arrays.

Every function takes numpy float64 arrays (callers widen bf16 exactly) and
int64 index arrays, and returns float64 arrays.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _bind(path):
    """Load an oracle shared library and declare its signatures."""
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int64)
    i64 = ctypes.c_int64
    lib.oracle_swa_attention.argtypes = [dp, dp, dp, ip, ip, ip, i64, i64, i64, i64,
                                         i64, i64, i64, ctypes.c_double, dp, dp,
                                         ctypes.c_int]
    lib.oracle_swa_attention.restype = ctypes.c_int
    lib.oracle_swa_partial.argtypes = [dp, dp, dp, ip, ip, ip, i64, i64, i64, i64,
                                       i64, i64, i64, ctypes.c_double, ip, ip, dp, dp,
                                       dp, ctypes.c_int]
    lib.oracle_swa_partial.restype = ctypes.c_int
    lib.oracle_lse_merge.argtypes = [dp, dp, dp, i64, i64, i64, dp, dp]
    lib.oracle_lse_merge.restype = ctypes.c_int
    lib.oracle_greedy_accept.argtypes = [dp, ip, ip, i64, i64, i64, ip, ip]
    lib.oracle_greedy_accept.restype = ctypes.c_int
    lib.oracle_append_rows.argtypes = [dp, dp, ip, ip, i64, i64, i64, i64, i64]
    lib.oracle_append_rows.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(_build.build())
    return _lib


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64))


def _dp(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _ip(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def default_threads():
    return max(1, os.cpu_count() or 1)


def _check(rc, what):
    if rc == 1:
        raise ValueError(f"{what}: invalid shape")
    if rc == 2:
        raise ValueError(f"{what}: a key inside a query's window lies outside the given K/V slice")
    if rc != 0:
        raise RuntimeError(f"{what}: status {rc}")


def _shapes(q, k, v):
    B, q_len, Hq, D = q.shape
    Bk, Hkv, T, Dk = k.shape
    if Bk != B or Dk != D or v.shape != k.shape:
        raise ValueError("q / k / v shapes disagree")
    return B, q_len, Hq, Hkv, D, T


def attention(q, k, v, seq_lens, q_pos, window, scale, base=None, threads=None):
    """Windowed attention by the definition.

    q [B, q_len, Hq, D]; k, v [B, Hkv, T, D] with row t of sequence b at
    absolute position base[b] + t (base defaults to 0, i.e. the whole cache).
    Returns (out [B, q_len, Hq, D], lse [B, q_len, Hq]) in float64, lse in
    natural log.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, q_len, Hq, Hkv, D, T = _shapes(q, k, v)
    base = _i64(np.zeros(B) if base is None else base)
    seq_lens, q_pos = _i64(seq_lens), _i64(q_pos)
    out = np.zeros((B, q_len, Hq, D))
    lse = np.zeros((B, q_len, Hq))
    rc = _load().oracle_swa_attention(_dp(q), _dp(k), _dp(v), _ip(base), _ip(seq_lens),
                                      _ip(q_pos), B, q_len, Hq, Hkv, D, T, int(window),
                                      float(scale), _dp(out), _dp(lse),
                                      threads or default_threads())
    _check(rc, "attention")
    return out, lse


def partial(q, k, v, seq_lens, q_pos, window, scale, c_lo, c_hi, base=None, threads=None):
    """Split-KV partial over absolute key range [c_lo[b], c_hi[b]).

    Returns (m, l, acc): m, l [B, q_len, Hq]; acc [B, q_len, Hq, D].
    m is the running max of the scaled scores (natural units), l the sum of
    exp(s - m), acc the unnormalised sum of exp(s - m) * v.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, q_len, Hq, Hkv, D, T = _shapes(q, k, v)
    base = _i64(np.zeros(B) if base is None else base)
    seq_lens, q_pos = _i64(seq_lens), _i64(q_pos)
    c_lo, c_hi = _i64(c_lo), _i64(c_hi)
    m = np.zeros((B, q_len, Hq))
    l = np.zeros((B, q_len, Hq))
    acc = np.zeros((B, q_len, Hq, D))
    rc = _load().oracle_swa_partial(_dp(q), _dp(k), _dp(v), _ip(base), _ip(seq_lens),
                                    _ip(q_pos), B, q_len, Hq, Hkv, D, T, int(window),
                                    float(scale), _ip(c_lo), _ip(c_hi), _dp(m), _dp(l),
                                    _dp(acc), threads or default_threads())
    _check(rc, "partial")
    return m, l, acc


def lse_merge(m, l, acc):
    """Merge n partials: m, l [n, rows]; acc [n, rows, D] -> (out [rows, D], lse [rows])."""
    m, l, acc = _f64(m), _f64(l), _f64(acc)
    n, rows, D = acc.shape
    if m.shape != (n, rows) or l.shape != (n, rows):
        raise ValueError("partial shapes disagree")
    out = np.zeros((rows, D))
    lse = np.zeros(rows)
    rc = _load().oracle_lse_merge(_dp(m), _dp(l), _dp(acc), n, rows, D, _dp(out), _dp(lse))
    _check(rc, "lse_merge")
    return out, lse


def greedy_accept(logits, draft, keep=None):
    """Greedy verification of draft blocks.

    logits [B, q_len, V] (any real dtype, widened to float64), draft
    [B, q_len - 1] token ids, keep [V] token ids of the logits' columns or
    None.  Returns (argmax [B, q_len], accepted [B]) as int64: the first
    column of the largest logit per row (mapped through keep), and the length
    of the longest prefix of rows whose argmax equals the drafted token.
    """
    logits = _f64(logits)
    B, q_len, V = logits.shape
    draft = _i64(np.asarray(draft).reshape(B, max(q_len - 1, 0)))
    keep_a = None if keep is None else _i64(keep)
    if keep_a is not None and keep_a.shape != (V,):
        raise ValueError("keep must have one token id per logit column")
    argmax = np.zeros((B, q_len), dtype=np.int64)
    accepted = np.zeros(B, dtype=np.int64)
    rc = _load().oracle_greedy_accept(_dp(logits), _ip(keep_a) if keep_a is not None else None,
                                      _ip(draft), B, q_len, V, _ip(argmax), _ip(accepted))
    _check(rc, "greedy_accept")
    return argmax, accepted


def append_rows(cache, rows, q_pos, seq_lens):
    """The cache after a verify block's new rows are written.

    cache [B, Hkv, L, D], rows [B, q_len, Hkv, D] (widened to float64),
    q_pos / seq_lens [B].  Returns a new float64 cache in which position
    q_pos[b] + i of every KV head holds rows[b, i] wherever
    0 <= q_pos[b] + i < min(seq_lens[b], L); the input is not modified.
    """
    out = np.array(cache, dtype=np.float64, order="C", copy=True)
    rows = _f64(rows)
    B, Hkv, L, D = out.shape
    if rows.ndim != 4 or rows.shape[0] != B or rows.shape[2:] != (Hkv, D):
        raise ValueError("rows must be [B, q_len, Hkv, D] matching the cache")
    q_len = rows.shape[1]
    q_pos, seq_lens = _i64(q_pos), _i64(seq_lens)
    rc = _load().oracle_append_rows(_dp(out), _dp(rows), _ip(q_pos), _ip(seq_lens), B, q_len,
                                    Hkv, L, D)
    _check(rc, "append_rows")
    return out

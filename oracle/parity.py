"""The parity bar between the CUDA path and the fp64 oracle.

TEST INFRASTRUCTURE ONLY, like the rest of this package: used by ``tests/``
and ``__graft_entry__.smoke()``.  Tolerances of the verify attention: max
abs error 2e-2; max relative error 2e-2, relative to max(|ref|, 1e-2) so
that outputs near zero do not dominate the measure; log-sum-exp within 1e-3
absolute; rows without a visible key must agree exactly (out 0, lse -inf).
"""
import numpy as np
import torch

ATOL = 2e-2
RTOL = 2e-2
REL_FLOOR = 1e-2
LSE_ATOL = 1e-3


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

"""Shared test plumbing: the oracle on a workload's window slices, the
tolerance check, a GPU-path runner and the kernel override."""
import contextlib

import torch

import oracle
from oracle.parity import ATOL, LSE_ATOL, REL_FLOOR, RTOL, compare  # noqa: F401
from oracle.slices import host_slices  # noqa: F401  (re-exported for the tests)


def oracle_reference(case, seqs=None, margin=64):
    q, k, v, base, sl, qp = host_slices(case, seqs, margin)
    return oracle.attention(q, k, v, sl, qp, case.window, case.scale, base=base)


def run_gpu(case, num_splits=0):
    from sliding_window_speculative_gb300 import swa_verify_attn
    out, lse = swa_verify_attn(case.q, case.k_cache, case.v_cache, case.seq_lens, case.q_pos,
                               case.window, case.scale, num_splits=num_splits)
    torch.cuda.synchronize()
    return out, lse


@contextlib.contextmanager
def forced_kernel(name):
    """Every call inside runs kernel `name` ("simt", "tc", "rows", or "plan")
    where the shape allows, through the library's test controls."""
    from sliding_window_speculative_gb300 import swa_set_debug_options
    swa_set_debug_options(force_kernel=name)
    try:
        yield name
    finally:
        swa_set_debug_options()

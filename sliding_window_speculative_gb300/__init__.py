"""Sliding-window split-KV verify attention on GB300 (sm_103a).

The compute lives in the CUDA library ``libswa.so`` (C ABI, include/swa.h);
this package is its thin Python binding plus the seeded synthetic input
generators (``inputs``).  The library is loaded on first use and a missing
build raises: there is no CPU path.
"""
from ._binding import (SWA_ERR_CUDA, SWA_ERR_INVALID_ARG, SWA_ERR_UNSUPPORTED,  # noqa: F401
                       SWA_ERR_WORKSPACE, SWA_OK, PreparedCall, SwaDebugOptions, SwaDims,
                       SwaError, SwaPaged, dims_of, load_library, make_dims, swa_append_verify_attn,
                       swa_get_debug_options, swa_greedy_accept, swa_last_error, swa_plan,
                       swa_read_debug_checks, swa_read_device_errors, swa_release_workspace,
                       swa_set_debug_options,
                       swa_set_workspace, swa_verify_attn, swa_verify_attn_noalloc,
                       swa_verify_attn_paged, swa_version, swa_workspace_bytes, prepare)

__all__ = [
    # the C entry points of include/swa.h, same names
    "swa_verify_attn", "swa_verify_attn_noalloc", "swa_verify_attn_paged",
    "swa_append_verify_attn", "swa_greedy_accept", "swa_workspace_bytes", "swa_set_workspace",
    "swa_release_workspace", "swa_plan", "swa_last_error", "swa_read_device_errors",
    "swa_read_debug_checks", "swa_version",
    # a call validated once and re-issued (serving loops)
    "prepare", "PreparedCall",
    # test and sweep controls
    "swa_set_debug_options", "swa_get_debug_options",
    # structs and helpers
    "SwaDims", "SwaPaged", "SwaDebugOptions", "SwaError", "make_dims", "dims_of",
    "load_library",
]

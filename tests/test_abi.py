"""C-ABI checks that need no GPU: the library loads, exports every entry
point include/swa.h declares, rejects bad arguments before touching CUDA,
and its split plan / workspace arithmetic hold their invariants."""
import ctypes
import os
import re

import pytest

import sliding_window_speculative_gb300 as swa
from sliding_window_speculative_gb300 import build
from tests.helpers import forced_kernel

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "swa.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return swa.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(swa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("swa_verify_attn", "swa_workspace_bytes", "swa_set_workspace",
                     "swa_last_error"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in swa.h but not exported"


def test_binding_uses_the_c_names():
    for name in declared_functions():
        assert hasattr(swa, name), f"binding lacks {name}"


def test_version(lib):
    assert "sm_103a" in swa.swa_version()
    assert "debug-checks" not in swa.swa_version()


def test_debug_checks_only_in_the_debug_build(lib):
    """The release library answers swa_read_debug_checks with
    SWA_ERR_UNSUPPORTED (no CUDA call); the SWA_DEBUG_CHECKS build exports
    the same symbols and names itself in its version."""
    c = ctypes.c_uint32(5)
    assert lib.swa_read_debug_checks(ctypes.byref(c)) == swa.SWA_ERR_UNSUPPORTED and c.value == 0
    assert "SWA_DEBUG_CHECKS" in swa.swa_last_error()
    assert lib.swa_read_debug_checks(None) == swa.SWA_ERR_INVALID_ARG
    dbg_path = build.build(debug_checks=True)
    dbg = ctypes.CDLL(dbg_path)
    for name in declared_functions():
        assert hasattr(dbg, name), f"{name} not exported by the debug build"
    dbg.swa_version.restype = ctypes.c_char_p
    assert dbg.swa_version().decode() == "swa 0.1.0 sm_103a debug-checks"
    dbg.swa_read_debug_checks.argtypes = [ctypes.c_void_p]
    assert dbg.swa_read_debug_checks(None) == swa.SWA_ERR_INVALID_ARG


def _call_raw(lib, dims, window=188, q=16, k=32, v=48, sl=64, qp=128, out=256, lse=None,
              scale=0.0625):
    d = swa.make_dims(*dims) if isinstance(dims, tuple) else dims
    return lib.swa_verify_attn(q, k, v, sl, qp, window, scale, out, lse,
                               ctypes.byref(d) if d is not None else None, None)


GOOD = (2, 8, 8, 2, 256, 4096, 0)


@pytest.mark.parametrize("dims,window,code", [
    ((0, 8, 8, 2, 256, 4096, 0), 188, swa.SWA_ERR_INVALID_ARG),     # batch 0
    ((2, 0, 8, 2, 256, 4096, 0), 188, swa.SWA_ERR_INVALID_ARG),     # q_len 0
    ((2, 513, 8, 2, 256, 4096, 0), 188, swa.SWA_ERR_INVALID_ARG),   # q_len > 512
    ((2, 8, 8, 3, 256, 4096, 0), 188, swa.SWA_ERR_INVALID_ARG),     # Hq % Hkv
    ((2, 8, 8, 0, 256, 4096, 0), 188, swa.SWA_ERR_INVALID_ARG),     # Hkv 0
    ((2, 8, 8, 2, 96, 4096, 0), 188, swa.SWA_ERR_UNSUPPORTED),      # head_dim
    ((2, 8, 8, 2, 256, 0, 0), 188, swa.SWA_ERR_INVALID_ARG),        # max_len
    ((2, 8, 8, 2, 256, 4096, -1), 188, swa.SWA_ERR_INVALID_ARG),    # splits
    (GOOD, 0, swa.SWA_ERR_INVALID_ARG),                              # window 0
    ((2, 64, 512, 1, 256, 4096, 0), 188, swa.SWA_ERR_UNSUPPORTED),  # R > 4096
])
def test_invalid_dims_rejected_before_cuda(lib, dims, window, code):
    assert _call_raw(lib, dims, window) == code
    assert swa.swa_last_error() != ""


def test_null_and_misaligned_pointers(lib):
    assert _call_raw(lib, None) == swa.SWA_ERR_INVALID_ARG
    assert _call_raw(lib, GOOD, q=None) == swa.SWA_ERR_INVALID_ARG
    assert _call_raw(lib, GOOD, out=None) == swa.SWA_ERR_INVALID_ARG
    assert _call_raw(lib, GOOD, k=40) == swa.SWA_ERR_INVALID_ARG     # 8-byte aligned only
    assert _call_raw(lib, GOOD, sl=66) == swa.SWA_ERR_INVALID_ARG    # int32 misaligned
    assert _call_raw(lib, GOOD, scale=float("nan")) == swa.SWA_ERR_INVALID_ARG
    assert _call_raw(lib, GOOD, scale=float("inf")) == swa.SWA_ERR_INVALID_ARG


def test_workspace_bytes(lib):
    d = swa.make_dims(*GOOD)
    assert swa.swa_workspace_bytes(d, 188) > 0
    assert swa.swa_workspace_bytes(swa.make_dims(0, 8, 8, 2, 256, 4096), 188) == 0
    one = swa.make_dims(2, 8, 8, 2, 256, 4096, 1)
    assert swa.swa_workspace_bytes(one, 188) == 0


@pytest.mark.parametrize("B,q_len,Hq,Hkv,D,L,W", [
    (1, 8, 8, 2, 256, 4096, 188), (1, 1, 8, 2, 256, 4096, 188), (1, 1, 8, 2, 256, 4096, 4096),
    (64, 8, 8, 2, 256, 4096, 188), (512, 64, 8, 2, 256, 32768, 1024), (1, 1, 2, 1, 64, 40, 16),
    (3, 64, 16, 2, 256, 1024, 188), (7, 5, 6, 2, 128, 300, 5000),
    (1, 512, 8, 2, 256, 4096, 188), (2, 300, 8, 2, 64, 1024, 37), (1, 512, 8, 2, 128, 8192, 4096),
    (4, 200, 16, 2, 256, 2048, 600),
    # large query groups and odd head ratios, the largest batch
    (1, 8, 64, 1, 128, 1024, 188), (3, 1, 32, 1, 256, 512, 188), (2, 64, 64, 1, 256, 2048, 188),
    (5, 3, 48, 4, 128, 777, 100), (65535, 1, 8, 2, 256, 16, 8), (2, 17, 24, 8, 64, 300, 50),
    (4, 64, 128, 2, 128, 1024, 1024),
])
@pytest.mark.parametrize("sms", [1, 148, 152])
def test_plan_invariants(lib, B, q_len, Hq, Hkv, D, L, W, sms):
    dims = swa.make_dims(B, q_len, Hq, Hkv, D, L)
    p = swa.swa_plan(dims, W, sms)
    span = min(W + q_len - 1, L)
    R = q_len * Hq // Hkv
    assert 1 <= p["num_splits"] <= 64
    assert p["num_splits"] * p["chunk_keys"] >= span               # chunks cover the span
    assert (p["num_splits"] - 1) * p["chunk_keys"] < span          # no empty trailing chunk
    assert p["row_tiles"] * p["rows_per_tile"] >= R
    units = p["num_splits"] * Hkv * p["row_tiles"] * B
    if p["kernel"] == 1:
        assert p["grid_ctas"] == units
    elif p["kernel"] == 4:                  # persistent grid of CTA pairs over the work items
        assert p["grid_ctas"] % 2 == 0 and 2 <= p["grid_ctas"] <= 2 * min(units, max(1, sms // 2))
        assert D == 256 and R > 128
        assert p["rows_per_tile"] == 2 * (128 // (Hq // Hkv)) * (Hq // Hkv)
    else:                                   # persistent grid over the work items
        assert p["kernel"] in (2, 3) and 1 <= p["grid_ctas"] <= min(units, sms)
        # rows-major above 32 packed rows (on CTA pairs above 128 at head_dim
        # 256), unless the key-major items fit in one wave of the SMs or are
        # small (8 or 16 rows)
        assert p["kernel"] == (3 if R > 32 and not (D == 256 and R > 128) else 2) or (
            p["kernel"] == 2 and (p["rows_per_tile"] <= 16 or units <= sms))
        assert p["rows_per_tile"] <= (128 if p["kernel"] == 3 else 64)
        assert p["rows_per_tile"] % (Hq // Hkv) == 0
    assert p["merge"] == (1 if p["num_splits"] > 1 else 0)
    assert p["workspace_bytes"] <= swa.swa_workspace_bytes(dims, W)
    if p["num_splits"] > 1:
        assert p["workspace_bytes"] == B * Hkv * p["num_splits"] * R * (D + 2) * 4


def test_plan_kernel_choice(lib):
    q8 = swa.make_dims(1, 8, 8, 2, 256, 4096)
    assert swa.swa_plan(q8, 188, 152)["kernel"] == 2            # 32 packed rows: tensor cores
    q1 = swa.make_dims(1, 1, 8, 2, 256, 4096)
    assert swa.swa_plan(q1, 188, 152)["kernel"] == 1            # 4 rows, 2 units: CUDA cores
    q1_big = swa.make_dims(76, 1, 8, 2, 256, 4096)              # 152 units: tensor cores
    assert swa.swa_plan(q1_big, 188, 152)["kernel"] == 2
    assert swa.swa_plan(swa.make_dims(75, 1, 8, 2, 256, 4096), 188, 152)["kernel"] == 2
    assert swa.swa_plan(swa.make_dims(37, 1, 8, 2, 256, 4096), 188, 152)["kernel"] == 1
    d64 = swa.make_dims(1, 8, 2, 1, 64, 40)
    assert swa.swa_plan(d64, 16, 152)["kernel"] == 1            # head_dim 64: CUDA cores
    q64 = swa.swa_plan(swa.make_dims(512, 64, 8, 2, 256, 32768), 1024, 152)
    assert q64["kernel"] == 4 and q64["row_tiles"] == 1 and q64["rows_per_tile"] == 256
    assert q64["grid_ctas"] == 152
    q64 = swa.swa_plan(swa.make_dims(512, 64, 8, 2, 128, 32768), 1024, 152)
    assert q64["kernel"] == 3 and q64["row_tiles"] == 2 and q64["rows_per_tile"] == 128
    q16 = swa.swa_plan(swa.make_dims(128, 16, 8, 2, 256, 4096), 188, 152)
    assert q16["kernel"] == 3 and q16["row_tiles"] == 1 and q16["rows_per_tile"] == 64
    q16 = swa.swa_plan(swa.make_dims(64, 16, 8, 2, 256, 4096), 188, 152)   # one wave
    assert q16["kernel"] == 2 and q16["row_tiles"] == 1 and q16["rows_per_tile"] == 64
    with forced_kernel("simt"):
        assert swa.swa_plan(q8, 188, 152)["kernel"] == 1
    with forced_kernel("tc"):
        assert swa.swa_plan(q1, 188, 152)["kernel"] == 2
        assert swa.swa_plan(d64, 16, 152)["kernel"] == 1
    with forced_kernel("rows"):
        assert swa.swa_plan(q1, 188, 152)["kernel"] == 3
    with forced_kernel("pairs"):
        p = swa.swa_plan(q1, 188, 152)
        assert p["kernel"] == 4 and p["grid_ctas"] == 4 and p["rows_per_tile"] == 256
        assert swa.swa_plan(swa.make_dims(1, 8, 8, 2, 128, 4096), 188, 152)["kernel"] == 3
        assert swa.swa_plan(d64, 16, 152)["kernel"] == 1
    assert swa.swa_plan(q8, 188, 152)["kernel"] == 2  # back to the plan's choice


def test_plan_forced_splits(lib):
    with forced_kernel("simt"):
        dims = swa.make_dims(1, 8, 8, 2, 256, 4096, 5)
        p = swa.swa_plan(dims, 188, 152)
        assert p["num_splits"] == 5 and p["chunk_keys"] == 39
        dims = swa.make_dims(1, 8, 8, 2, 256, 4096, 500)
        assert swa.swa_plan(dims, 188, 152)["num_splits"] <= 64


def test_debug_options_round_trip_and_validation(lib):
    """The test controls replace environment variables: the library reads
    none.  Defaults, a round trip, range checks and the reset."""
    assert swa.swa_get_debug_options() == {"force_kernel": 0, "pdl": 1, "wait_limit_cycles": 0,
                                           "withhold_fill": -1, "rows_per_item": 0,
                                           "fail_launch": 0, "reserved": 0}
    swa.swa_set_debug_options(force_kernel="rows", pdl=0, wait_limit_cycles=100000,
                              withhold_fill=3, rows_per_item=64, fail_launch=2)
    try:
        assert swa.swa_get_debug_options() == {"force_kernel": 3, "pdl": 0,
                                               "wait_limit_cycles": 100000, "withhold_fill": 3,
                                               "rows_per_item": 64, "fail_launch": 2,
                                               "reserved": 0}
    finally:
        swa.swa_set_debug_options()
    assert swa.swa_get_debug_options()["force_kernel"] == 0
    assert swa.swa_get_debug_options()["fail_launch"] == 0
    for bad in ({"force_kernel": 5}, {"force_kernel": -1}, {"pdl": 2},
                {"wait_limit_cycles": -5}, {"withhold_fill": -2}, {"rows_per_item": -1},
                {"fail_launch": -1}):
        with pytest.raises(swa.SwaError) as e:
            swa.swa_set_debug_options(**bad)
        assert e.value.status == swa.SWA_ERR_INVALID_ARG
    # the reserved field must stay 0 (raw C call)
    opt = swa._binding.SwaDebugOptions(0, 1, 0, -1, 0, 0, 7)
    assert lib.swa_set_debug_options(ctypes.byref(opt)) == swa.SWA_ERR_INVALID_ARG
    assert lib.swa_set_debug_options(None) == swa.SWA_OK
    assert lib.swa_get_debug_options(None) == swa.SWA_ERR_INVALID_ARG


def test_rows_per_item_override(lib):
    """The sweep override of rows per item: rounded to whole query groups,
    capped per kernel, ignored for CUDA-core plans and forced splits."""
    q64 = swa.make_dims(512, 64, 8, 2, 256, 32768)
    assert swa.swa_plan(q64, 188, 152)["rows_per_tile"] == 256  # CTA pairs: no override
    swa.swa_set_debug_options(rows_per_item=64)
    assert swa.swa_plan(q64, 188, 152)["rows_per_tile"] == 256
    swa.swa_set_debug_options()
    try:
        for want, got in ((64, 64), (32, 32), (30, 28), (3, 4), (500, 128)):
            swa.swa_set_debug_options(force_kernel="rows", rows_per_item=want)
            p = swa.swa_plan(q64, 188, 152)
            assert p["kernel"] == 3 and p["rows_per_tile"] == got, (want, p)
            assert p["row_tiles"] == -(-64 // (got // 4))
        swa.swa_set_debug_options(rows_per_item=48)
        q8 = swa.make_dims(64, 8, 8, 2, 256, 4096)
        p = swa.swa_plan(q8, 188, 152)
        assert p["kernel"] == 2 and p["rows_per_tile"] == 32      # all 32 rows, below the cap
        swa.swa_set_debug_options(rows_per_item=16)
        assert swa.swa_plan(q8, 188, 152)["rows_per_tile"] == 16
        assert swa.swa_plan(swa.make_dims(64, 8, 8, 2, 256, 4096, 3), 188, 152)["rows_per_tile"] == 32
        d64 = swa.make_dims(1, 8, 2, 1, 64, 40)
        assert swa.swa_plan(d64, 16, 152)["kernel"] == 1
    finally:
        swa.swa_set_debug_options()


def test_library_reads_no_environment():
    """No source of the CUDA library calls getenv: test and sweep controls
    go through swa_set_debug_options only."""
    csrc = os.path.join(ROOT, "sliding_window_speculative_gb300", "csrc")
    for name in os.listdir(csrc):
        text = open(os.path.join(csrc, name)).read()
        assert "getenv" not in text, name


def test_plan_splits_long_spans_of_one_sequence(lib):
    # a W=188 span (two 128-key tiles) stays one chunk on the tensor-core
    # path: a split's merge costs more than the tile it saves
    p = swa.swa_plan(swa.make_dims(1, 8, 8, 2, 256, 4096), 188, 152)
    assert p["kernel"] == 2 and p["num_splits"] == 1
    # a full-context decode spreads over the SMs in chunks of >= 128 keys
    p = swa.swa_plan(swa.make_dims(1, 8, 8, 2, 256, 4096), 4096, 152)
    assert p["kernel"] == 2 and p["num_splits"] == 32 and p["chunk_keys"] == 128
    # the CUDA-core path (q_len 1, one sequence) still splits W=188
    p = swa.swa_plan(swa.make_dims(1, 1, 8, 2, 256, 4096), 188, 152)
    assert p["kernel"] == 1 and p["num_splits"] > 1


def test_binding_rejects_cpu_tensors(lib):
    import torch
    q = torch.zeros(1, 8, 8, 256, dtype=torch.bfloat16)
    k = torch.zeros(1, 2, 64, 256, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        swa.swa_verify_attn(q, k, k, torch.zeros(1, dtype=torch.int32),
                            torch.zeros(1, dtype=torch.int32), 188, 0.0625)


def test_greedy_accept_rejects_bad_arguments(lib):
    # validated on the host before any CUDA call
    vp = ctypes.c_void_p
    dummy = vp(16)
    cases = [
        (None, None, dummy, dummy, dummy, 1, 8, 100),       # logits NULL
        (dummy, None, None, dummy, dummy, 1, 8, 100),       # draft NULL with q_len 8
        (dummy, None, dummy, None, dummy, 1, 8, 100),       # argmax NULL
        (dummy, None, dummy, dummy, dummy, 0, 8, 100),      # batch 0
        (dummy, None, dummy, dummy, dummy, 1, 65, 100),     # q_len above 64
        (dummy, None, dummy, dummy, dummy, 1, 8, 0),        # empty vocabulary
        (vp(17), None, dummy, dummy, dummy, 1, 8, 100),     # logits not 2-byte aligned
        (dummy, vp(18), dummy, dummy, dummy, 1, 8, 100),    # keep_ids not 4-byte aligned
    ]
    for args in cases:
        st = lib.swa_greedy_accept(*args, None)
        assert st == swa.SWA_ERR_INVALID_ARG, args
        assert swa.swa_last_error()


def test_append_verify_rejects_bad_arguments(lib):
    # validated on the host before any CUDA call
    d = swa.make_dims(*GOOD)

    def call(kn=16, vn=32, paged=None, q=48):
        return lib.swa_append_verify_attn(q, kn, vn, 64, 80, paged, 96, 112, 188, 0.0625, 128,
                                          None, ctypes.byref(d), None)

    assert call(kn=None) == swa.SWA_ERR_INVALID_ARG
    assert call(vn=None) == swa.SWA_ERR_INVALID_ARG
    assert call(kn=24) == swa.SWA_ERR_INVALID_ARG        # 8-byte aligned only
    assert call(q=None) == swa.SWA_ERR_INVALID_ARG
    bad_page = swa.SwaPaged(160, 4096 // 12, 12, 100)    # pages of 12 rows
    assert call(paged=ctypes.byref(bad_page)) == swa.SWA_ERR_INVALID_ARG
    short = swa.SwaPaged(160, 10, 16, 100)               # max_len != max_blocks * page_size
    assert call(paged=ctypes.byref(short)) == swa.SWA_ERR_INVALID_ARG
    assert swa.swa_last_error()


def test_paged_verify_rejects_bad_tables(lib):
    # every case fails on the host, before any CUDA call
    d = swa.make_dims(*GOOD)                              # max_len 4096, Hkv 2

    def call(paged, q=48):
        return lib.swa_verify_attn_paged(q, 16, 32, ctypes.byref(paged) if paged else None,
                                         96, 112, 188, 0.0625, 128, None, ctypes.byref(d), None)

    assert call(None) == swa.SWA_ERR_INVALID_ARG                       # no description
    assert call(swa.SwaPaged(None, 256, 16, 100)) == swa.SWA_ERR_INVALID_ARG   # no table
    assert call(swa.SwaPaged(162, 256, 16, 100)) == swa.SWA_ERR_INVALID_ARG    # table misaligned
    assert call(swa.SwaPaged(160, 1024, 4, 100)) == swa.SWA_ERR_INVALID_ARG    # pages of 4 rows
    assert call(swa.SwaPaged(160, 0, 16, 100)) == swa.SWA_ERR_INVALID_ARG      # no blocks
    assert call(swa.SwaPaged(160, 256, 16, 0)) == swa.SWA_ERR_INVALID_ARG      # empty pool
    assert call(swa.SwaPaged(160, 128, 16, 100)) == swa.SWA_ERR_INVALID_ARG    # 2048 != max_len
    # 2^20 pages x 2 KV heads x 1024 rows = 2^31 pool rows
    assert call(swa.SwaPaged(160, 4, 1024, 1 << 20)) == swa.SWA_ERR_UNSUPPORTED
    assert call(swa.SwaPaged(160, 256, 16, 100), q=None) == swa.SWA_ERR_INVALID_ARG
    assert "page" in swa.swa_last_error() or "NULL" in swa.swa_last_error()


def test_plan_prefill_chunk_reads_row_windows(lib):
    # a 512-row prefill chunk at W = 188: an item's rows see W + 63 keys (CTA
    # pairs, 256 rows) or W + 31 (one-CTA rows-major, 128 rows), so no split
    # although the whole span is 699 keys; at W = 4096 the row tiles'
    # windows are split to reach the SMs
    p = swa.swa_plan(swa.make_dims(1, 512, 8, 2, 256, 4096), 188, 152)
    assert p["kernel"] == 4 and p["row_tiles"] == 8 and p["num_splits"] == 1
    with forced_kernel("rows"):
        p = swa.swa_plan(swa.make_dims(1, 512, 8, 2, 256, 4096), 188, 152)
        assert p["kernel"] == 3 and p["row_tiles"] == 16 and p["num_splits"] == 1
    p = swa.swa_plan(swa.make_dims(1, 512, 8, 2, 128, 8192), 4096, 152)
    assert p["num_splits"] > 1 and p["chunk_keys"] < 4096 + 31


def test_plan_few_units_prefer_small_key_major_items(lib):
    # few (sequence, KV head) units: the key-major kernel with 8- or 16-row
    # items, even above 32 packed rows (8 rows only while those items fill at
    # most a sixteenth of the SMs); full batches keep the rows-major kernel
    for B, q_len, rows in ((1, 8, 8), (1, 16, 16), (1, 64, 16), (2, 8, 16), (8, 16, 16),
                           (16, 8, 16), (24, 8, 32)):
        p = swa.swa_plan(swa.make_dims(B, q_len, 8, 2, 256, 4096), 188, 152)
        assert p["kernel"] == 2 and p["rows_per_tile"] == rows, (B, q_len, p)
        assert p["grid_ctas"] <= 152
    # 33..128 rows: the key-major kernel while its items (up to 64 rows) fit
    # in one wave of the SMs, else the rows-major kernel; above 128 rows the
    # CTA pairs unless the key-major items are small
    for B, q_len in ((16, 16), (64, 16), (8, 32), (32, 32), (1, 64), (2, 64)):
        p = swa.swa_plan(swa.make_dims(B, q_len, 8, 2, 256, 4096), 188, 152)
        assert p["kernel"] == 2 and p["grid_ctas"] <= 152, (B, q_len, p)
    for B, q_len in ((4, 64), (16, 64), (1, 512), (2, 512)):
        p = swa.swa_plan(swa.make_dims(B, q_len, 8, 2, 256, 4096), 188, 152)
        assert p["kernel"] == 4, (B, q_len, p)
    for B, q_len in ((512, 16), (512, 64), (128, 16), (64, 32), (32, 64), (64, 512)):
        p = swa.swa_plan(swa.make_dims(B, q_len, 8, 2, 256, 4096), 188, 152)
        # (on CTA pairs above 128 packed rows)
        assert p["kernel"] == (4 if q_len * 4 > 128 else 3), (B, q_len, p)
    p = swa.swa_plan(swa.make_dims(64, 8, 8, 2, 256, 4096), 188, 152)
    assert p["kernel"] == 2 and p["rows_per_tile"] == 32


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    from sliding_window_speculative_gb300 import _binding
    monkeypatch.setattr(_binding, "_lib", None)
    with pytest.raises(ImportError, match="no CPU fallback"):
        _binding.load_library(str(tmp_path / "libswa.so"))


def test_last_error_is_per_thread(lib):
    import threading
    got = {}
    barrier = threading.Barrier(2)

    def worker(name, dims, window):
        assert _call_raw(lib, dims, window) == swa.SWA_ERR_INVALID_ARG
        barrier.wait()          # both calls have failed before either reads
        got[name] = swa.swa_last_error()

    t1 = threading.Thread(target=worker, args=("batch", (0, 8, 8, 2, 256, 4096, 0), 188))
    t2 = threading.Thread(target=worker, args=("window", GOOD, 0))
    t1.start(); t2.start(); t1.join(); t2.join()
    assert "batch" in got["batch"] and "window" in got["window"]
    assert got["batch"] != got["window"]

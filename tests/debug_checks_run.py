"""Child process of tests/test_debug_checks_gpu.py: loads the library built
with SWA_DEBUG_CHECKS (before anything else loads the release one), runs
each case and prints one JSON line per case:
{"name", "count" (out-of-range attempts the library counted), "ok", "detail"}.

Valid inputs must count nothing and match the oracle.  Invalid device-side
inputs: a sequence length past the cache (clamped in every build) and a
block-table page outside the pool.  The bad page points at guard pages
allocated past the pool the call is given, filled with marker values (K =
30, V = 1000) that would dominate any output that read them, so even an
unchecked access would stay inside memory the test owns and show.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from sliding_window_speculative_gb300 import _binding  # noqa: E402

_binding.load_library(_binding.DEBUG_LIB_PATH)

import sliding_window_speculative_gb300 as swa  # noqa: E402
from sliding_window_speculative_gb300 import inputs  # noqa: E402
from tests.helpers import compare, oracle_reference, run_gpu  # noqa: E402
from tests.test_append_gpu import take_block  # noqa: E402

GUARD_K, GUARD_V = 30.0, 1000.0
KERNELS = ("simt", "tc", "rows", "pairs")


def record(name, fn):
    swa.swa_read_debug_checks()  # clear
    try:
        detail = fn() or ""
        ok = True
    except Exception as e:  # reported to the parent test
        ok, detail = False, repr(e)[:400]
    count = swa.swa_read_debug_checks()
    print(json.dumps({"name": name, "count": count, "ok": ok, "detail": detail}), flush=True)


def pool_with_guards(case, page_size, guards=3):
    """Pool [B * nb + guards, Hkv, page_size, D]: the cache in pages
    0 .. B * nb - 1 (block k of sequence b in page b * nb + 3k mod nb, so
    tables are not the identity and page 0 holds sequence 0's first block,
    whose rows are all below its length: the page a debug check reads in
    place of a bad one), then guard pages of marker values.  Returns
    (k pool, v pool, table, pages the call is given)."""
    B, Hkv, L, D = case.k_cache.shape
    nb = L // page_size
    assert nb % 3 != 0
    n = B * nb
    kp = torch.empty((n + guards, Hkv, page_size, D), dtype=torch.bfloat16, device="cuda")
    vp = torch.empty_like(kp)
    kp[n:] = GUARD_K
    vp[n:] = GUARD_V
    table = torch.empty((B, nb), dtype=torch.int32)
    kc = case.k_cache.view(B, Hkv, nb, page_size, D)
    vc = case.v_cache.view(B, Hkv, nb, page_size, D)
    for b in range(B):
        for k in range(nb):
            pg = b * nb + (3 * k) % nb
            table[b, k] = pg
            kp[pg] = kc[b, :, k]
            vp[pg] = vc[b, :, k]
    return kp, vp, table.cuda(), n


def paged_call(case, kp, vp, table, n, **kw):
    out, lse = swa.swa_verify_attn_paged(case.q, kp[:n], vp[:n], table, case.seq_lens,
                                         case.q_pos, case.window, case.scale, **kw)
    torch.cuda.synchronize()
    return out, lse


def cases(kernel):
    d = 128 if kernel == "simt" else 256
    q_len = 64 if kernel in ("rows", "pairs") else 8
    lens = [q_len + 300, q_len + 40, 512]
    return inputs.make_case("dbg", 3, 8, 2, d, q_len, 188, lens, 512, seed=31, outliers=True,
                            device="cuda")


def main():
    for kernel in KERNELS:
        swa.swa_set_debug_options(force_kernel=kernel)

        # ---- valid inputs: nothing counted, oracle parity
        case = cases(kernel)
        ref_o, ref_l = oracle_reference(case)

        def plain():
            for splits in (0, 3):
                out, lse = run_gpu(case, splits)
                compare(out, lse, ref_o, ref_l, f"debug build, {kernel}, {splits} splits")
        record(f"{kernel}/valid contiguous", plain)

        def paged():
            kp, vp, table, n = pool_with_guards(case, 64)
            out, lse = paged_call(case, kp, vp, table, n)
            compare(out, lse, ref_o, ref_l, f"debug build, {kernel}, paged")
            assert torch.all(kp[n:] == GUARD_K) and torch.all(vp[n:] == GUARD_V)
        if kernel != "pairs":  # (a paged call takes the one-CTA kernel)
            record(f"{kernel}/valid paged", paged)

        if kernel not in ("rows", "pairs"):
            def append():
                c2 = cases(kernel)
                k_new, v_new = take_block(c2)
                out, lse = swa.swa_append_verify_attn(c2.q, k_new, v_new, c2.k_cache,
                                                      c2.v_cache, c2.seq_lens, c2.q_pos,
                                                      c2.window, c2.scale)
                torch.cuda.synchronize()
                compare(out, lse, ref_o, ref_l, f"debug build, {kernel}, fused append")
            record(f"{kernel}/valid fused append", append)

        # ---- a sequence length past the cache (clamped to max_len in every build)
        def long_seq():
            c3 = cases(kernel)
            c3.seq_lens[2] = 512 + 40
            out, lse = run_gpu(c3, 0)
            compare(out, lse, ref_o, ref_l, f"debug build, {kernel}, seq_len past the cache")
        record(f"{kernel}/seq_len past the cache", long_seq)

        # ---- a page outside the pool, in sequence 0's window (block 4 of 64-row
        # pages holds positions 256..319, inside every row's window)
        def bad_page():
            kp, vp, table, n = pool_with_guards(case, 64)
            table[0, 4] = n + 1
            out, lse = paged_call(case, kp, vp, table, n)
            assert torch.isfinite(out).all() and float(out[0].float().abs().max()) < 100.0, \
                "sequence 0 read the guard page"
            compare(out[1:], lse[1:], ref_o[1:], ref_l[1:], f"debug build, {kernel}, bad page")
            assert torch.all(kp[n:] == GUARD_K) and torch.all(vp[n:] == GUARD_V)
        if kernel != "pairs":
            record(f"{kernel}/page outside the pool", bad_page)

        if kernel not in ("rows", "pairs"):
            def bad_page_append():
                c4 = cases(kernel)
                k_new, v_new = take_block(c4)
                kp, vp, table, n = pool_with_guards(c4, 64)
                # the block holding sequence 0's new rows (positions q_pos ..)
                table[0, int(c4.q_pos_host[0]) // 64] = n + 2
                out, lse = swa.swa_append_verify_attn(c4.q, k_new, v_new, kp[:n], vp[:n],
                                                      c4.seq_lens, c4.q_pos, c4.window, c4.scale,
                                                      block_table=table)
                torch.cuda.synchronize()
                assert torch.all(kp[n:] == GUARD_K) and torch.all(vp[n:] == GUARD_V), \
                    "a store reached a guard page"
                assert float(out[0].float().abs().max()) < 100.0
                compare(out[1:], lse[1:], ref_o[1:], ref_l[1:],
                        f"debug build, {kernel}, fused append, bad page")
            record(f"{kernel}/fused append into a page outside the pool", bad_page_append)
    swa.swa_set_debug_options()


if __name__ == "__main__":
    assert swa.swa_version().endswith("debug-checks"), swa.swa_version()
    main()

"""The boundary from plain C: a C11 program that includes include/swa.h,
links libswa.so and makes the host-only calls (version, plan, workspace
size, argument validation).  No GPU is needed and no Python type crosses
the boundary."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "swa.h"

int main(void) {
    const char *v = swa_version();
    if (v == NULL || strstr(v, "sm_103a") == NULL) return 10;
    swa_dims d = {1, 8, 8, 2, 256, 4096, 0};
    swa_plan_info p;
    if (swa_plan(&d, 188, 152, &p) != SWA_OK) return 11;
    if (p.kernel != 2 || p.num_splits != 1 || p.merge != 0) return 12;
    if (p.row_tiles * p.rows_per_tile < 8 * 4) return 13;
    if (swa_workspace_bytes(&d, 188) < (size_t)p.workspace_bytes) return 14;
    /* rejected on the host before any CUDA call */
    swa_dims bad = d;
    bad.head_dim = 96;
    if (swa_verify_attn((void *)16, (void *)32, (void *)48, (const int32_t *)64,
                        (const int32_t *)80, 188, 0.0625f, (void *)96, NULL, &bad,
                        NULL) != SWA_ERR_UNSUPPORTED) return 15;
    if (strstr(swa_last_error(), "head_dim") == NULL) return 16;
    printf("%s | kernel %d splits %d chunk %d rows %d x %d grid %d\n", v, p.kernel,
           p.num_splits, p.chunk_keys, p.row_tiles, p.rows_per_tile, p.grid_ctas);
    return 0;
}
"""


def test_plain_c_program_uses_the_library(tmp_path):
    from sliding_window_speculative_gb300 import build
    lib = build.build()
    src = tmp_path / "consumer.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "consumer"
    libdir = os.path.dirname(lib)
    r = subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        str(src), "-o", str(exe), "-L", libdir, "-l:libswa.so",
                        "-Wl,-rpath," + libdir], capture_output=True, text=True)
    if r.returncode != 0:
        pytest.fail("gcc: " + r.stderr)
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, (run.returncode, run.stdout, run.stderr)
    assert "kernel 2" in run.stdout


LAYOUT = r"""
#include <stddef.h>
#include <stdio.h>
#include "swa.h"
#define F(T, f) printf(#T "." #f " %zu %zu\n", offsetof(T, f), sizeof(((T *)0)->f))
int main(void) {
    printf("swa_dims %zu\nswa_paged %zu\nswa_plan_info %zu\nswa_debug_options %zu\n",
           sizeof(swa_dims), sizeof(swa_paged), sizeof(swa_plan_info),
           sizeof(swa_debug_options));
    F(swa_dims, batch); F(swa_dims, q_len); F(swa_dims, num_q_heads);
    F(swa_dims, num_kv_heads); F(swa_dims, head_dim); F(swa_dims, max_len);
    F(swa_dims, num_splits);
    F(swa_paged, block_table); F(swa_paged, max_blocks); F(swa_paged, page_size);
    F(swa_paged, num_pages);
    F(swa_plan_info, kernel); F(swa_plan_info, num_splits); F(swa_plan_info, chunk_keys);
    F(swa_plan_info, row_tiles); F(swa_plan_info, rows_per_tile); F(swa_plan_info, grid_ctas);
    F(swa_plan_info, merge); F(swa_plan_info, workspace_bytes);
    F(swa_debug_options, force_kernel); F(swa_debug_options, pdl);
    F(swa_debug_options, wait_limit_cycles); F(swa_debug_options, withhold_fill);
    F(swa_debug_options, rows_per_item); F(swa_debug_options, fail_launch);
    F(swa_debug_options, reserved);
    return 0;
}
"""


def test_binding_structs_match_the_c_layout(tmp_path):
    """The ctypes mirrors of the header's structs have the C compiler's
    size, field offsets and field sizes."""
    import ctypes

    from sliding_window_speculative_gb300 import _binding
    src = tmp_path / "layout.c"
    src.write_text(LAYOUT)
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o",
                    str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout
    mirrors = {"swa_dims": _binding.SwaDims, "swa_paged": _binding.SwaPaged,
               "swa_plan_info": _binding.SwaPlanInfo,
               "swa_debug_options": _binding.SwaDebugOptions}
    seen = 0
    for line in out.splitlines():
        parts = line.split()
        if "." not in parts[0]:
            assert ctypes.sizeof(mirrors[parts[0]]) == int(parts[1]), line
        else:
            struct, field = parts[0].split(".")
            desc = getattr(mirrors[struct], field)
            assert (desc.offset, desc.size) == (int(parts[1]), int(parts[2])), line
        seen += 1
    assert seen == 4 + 7 + 4 + 8 + 7


def _prototypes():
    """(return type, name, [parameter types]) of every function include/swa.h
    declares, comments removed."""
    import re
    text = open(os.path.join(ROOT, "include", "swa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"#[^\n]*\n", "\n", text)
    protos = []
    for ret, name, params in re.findall(r"([A-Za-z_][\w \*]*?)\s*\b(swa_\w+)\s*\(([^)]*)\)\s*;",
                                        text):
        ps = [p.strip() for p in params.split(",") if p.strip() and p.strip() != "void"]
        types = [re.sub(r"\s*\b\w+$", "", p) if not p.endswith("*") else p for p in ps]
        protos.append((ret.strip(), name, types))
    return protos


def test_binding_signatures_match_the_header():
    """Every declared function's ctypes argtypes / restype agree with the
    header's parameter types: pointers as pointers, int32_t as c_int32,
    float as c_float, size_t as c_size_t."""
    import ctypes

    from sliding_window_speculative_gb300 import build, load_library
    build.build()
    lib = load_library()
    protos = _prototypes()
    assert len(protos) >= 12
    for ret, name, types in protos:
        fn = getattr(lib, name)
        assert fn.argtypes is not None and len(fn.argtypes) == len(types), (name, types)
        for c_t, py_t in zip(types, fn.argtypes):
            if "*" in c_t or c_t == "swa_stream_t":
                assert py_t in (ctypes.c_void_p, ctypes.c_char_p) or \
                    issubclass(py_t, ctypes._Pointer), (name, c_t, py_t)
            else:
                want = {"int32_t": ctypes.c_int32, "float": ctypes.c_float,
                        "size_t": ctypes.c_size_t}[c_t]
                assert py_t is want, (name, c_t, py_t)
        want_ret = {"swa_status": ctypes.c_int, "size_t": ctypes.c_size_t,
                    "const char *": ctypes.c_char_p}[ret]
        assert fn.restype is want_ret, (name, ret, fn.restype)

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

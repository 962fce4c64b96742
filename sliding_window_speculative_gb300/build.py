"""Builds the CUDA library ``libswa.so`` in-tree for sm_103a with nvcc.

One shared object, C ABI only (include/swa.h).  Translation units compile in
parallel; the CUDA runtime is linked statically so the library needs only
the driver at run time.  ``libswa_debug.so`` is the same library built with
SWA_DEBUG_CHECKS (out-of-range index attempts on device-side inputs counted,
swa_read_debug_checks); ``build_all`` makes both at once.
"""
import concurrent.futures as cf
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libswa.so")
DEBUG_LIB = os.path.join(HERE, "libswa_debug.so")
BUILD_DIR = os.path.join(HERE, "_build")

SOURCES = ["swa_api.cu", "swa_tc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I" + os.path.join(ROOT, "include")]


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(ROOT, "include", "swa.h"))
    files.append(os.path.abspath(__file__))
    return files


def _target(debug_checks):
    """(library, object directory, extra nvcc flags) of one variant."""
    if debug_checks:
        return DEBUG_LIB, BUILD_DIR + "_debug", ["-DSWA_DEBUG_CHECKS"]
    return LIB, BUILD_DIR, []


def up_to_date(debug_checks=False):
    lib = _target(debug_checks)[0]
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force=False, verbose=False, extra=(), debug_checks=False):
    lib, build_dir, defs = _target(debug_checks)
    if not force and up_to_date(debug_checks):
        return lib
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *defs, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + ".tmp%d" % os.getpid()
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    os.replace(tmp, lib)
    return lib


def build_all(force=False):
    """Both variants, their translation units compiling side by side."""
    with cf.ThreadPoolExecutor(max_workers=2) as ex:
        libs = list(ex.map(lambda d: build(force=force, debug_checks=d), (False, True)))
    return libs


if __name__ == "__main__":
    if "--debug-checks" in sys.argv:
        print(build(force="--force" in sys.argv, debug_checks=True))
    else:
        print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                    extra=["-Xptxas", "-v"] if "-v" in sys.argv else ()))

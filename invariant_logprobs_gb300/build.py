"""Builds the CUDA library librz.so in-tree for sm_103a with nvcc.

Each .cu translation unit is compiled in parallel, then linked into one
shared object next to this file (static CUDA runtime; the driver API is
reached through the runtime's entry-point query, so the library loads on
machines without a GPU driver as well).
"""

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "librz.so")
# the debug build: every device bounds check compiled in (-DRZ_CHECKS)
BUILD_CHECKS = os.path.join(HERE, "_build_checks")
LIB_CHECKS = os.path.join(HERE, "librz_checks.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE]


def _nvcc():
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.sep not in c or os.path.exists(c)):
            return c
    return "nvcc"


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _stale(obj, src):
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    deps = [src] + [os.path.join(CSRC, f) for f in os.listdir(CSRC)
                    if f.endswith((".cuh", ".h"))]
    deps.append(os.path.join(HERE, "..", "include", "rz.h"))
    return any(os.path.getmtime(d) > t for d in deps if os.path.exists(d))


def _compile(src, flags, build_dir, force):
    obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
    if not force and not _stale(obj, src):
        return obj, ""
    cmd = [_nvcc()] + ARCH + NVCC_FLAGS + flags + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
    return obj, r.stderr


def build(verbose=False, extra=(), checks=False):
    """Compile every .cu under csrc/ and link librz.so (with checks=True the
    debug build librz_checks.so, device bounds checks compiled in); returns
    the library's path.  Objects are rebuilt when a source is newer, or
    always when extra flags are given."""
    build_dir, lib = (BUILD_CHECKS, LIB_CHECKS) if checks else (BUILD, LIB)
    os.makedirs(build_dir, exist_ok=True)
    flags = list(extra) + (["-DRZ_CHECKS"] if checks else [])
    srcs = sources()
    with ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(lambda s: _compile(s, flags, build_dir, bool(extra)), srcs))
    objs = [o for o, _ in results]
    if verbose:
        for _, log in results:
            if log:
                sys.stderr.write(log)
    need_link = (not os.path.exists(lib) or
                 any(os.path.getmtime(o) > os.path.getmtime(lib) for o in objs))
    if need_link:
        tmp = lib + ".tmp"
        cmd = [_nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-cudart", "static",
                                                                  "-ldl", "-lpthread", "-lrt"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    v = "-v" in sys.argv
    ex = ["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else []
    print(build(verbose=v or bool(ex), extra=ex, checks="--checks" in sys.argv))

"""Build libs4.so for sm_103a with nvcc (no cmake, no torch extension machinery).

Each source under csrc/ (CUDA .cu files and the host-only hippo.cpp) is
compiled in parallel to a position-independent object and the objects are
linked into lib/libs4.so inside the package.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "lib")
OBJDIR = os.path.join(PKG, "_build")
LIB = os.path.join(LIBDIR, "libs4.so")
SOURCES = ["s4_api.cu", "cauchy.cu", "fft_rows.cu", "fft_cluster.cu", "fft_fourstep.cu", "s4_noalloc.cu", "recurrent.cu", "bordered.cu",
           "hippo.cpp"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
GENDIR = os.path.join(OBJDIR, "gen")
FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC, "-I", GENDIR]


def nvcc() -> str:
    for cand in [os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]:
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(extra_deps, lib=LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + extra_deps
    return any(os.path.getmtime(d) > t for d in deps)


CHECKED_LIB = os.path.join(LIBDIR, "libs4_checked.so")


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, bounds_check: bool = False) -> str:
    """Compile (if needed) and return the path of libs4.so; with bounds_check,
    the separate test build libs4_checked.so (-DS4_BOUNDS_CHECK: every index of
    the instrumented kernels compared with its buffer's extent)."""
    deps = [os.path.join(INCLUDE, "s4.h"), os.path.abspath(__file__),
            os.path.join(PKG, "gen_twiddles.py")]
    lib_path = CHECKED_LIB if bounds_check else LIB
    objdir = os.path.join(OBJDIR, "checked") if bounds_check else OBJDIR
    if not force and not _stale(deps, lib_path):
        return lib_path
    os.makedirs(LIBDIR, exist_ok=True)
    os.makedirs(GENDIR, exist_ok=True)
    os.makedirs(objdir, exist_ok=True)
    sys.path.insert(0, PKG)
    import gen_twiddles
    gen_twiddles.generate(os.path.join(GENDIR, "s4_twiddles.cuh"))
    gen_twiddles.generate_tan(os.path.join(GENDIR, "s4_tan.cuh"))
    cc = nvcc()
    extra = (["-Xptxas", "-v"] if ptxas_info else []) + (["-DS4_BOUNDS_CHECK"] if bounds_check else [])

    def compile_one(src):
        obj = os.path.join(objdir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    for src, _, r in results:
        if verbose or ptxas_info:
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    tmp = lib_path + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[o for _, o, _ in results], "-lcudart_static", "-lrt", "-ldl", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                bounds_check="--bounds-check" in sys.argv))

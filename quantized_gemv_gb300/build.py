"""Compile libmk.so (the decode engine's C-ABI library) for sm_103a, in-tree.

Each .cu translation unit is compiled in parallel into _build/, then linked into
quantized_gemv_gb300/libmk.so. The same sources compiled with -DMK_DEBUG_BOUNDS give
libmk_debug.so, the bounds-checking debug build (out-of-range accesses are skipped and reported in
the step's status instead of faulting). Rebuilds only when a source or header is newer than the
library.
"""
import concurrent.futures as cf
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmk.so")
LIB_DEBUG = os.path.join(HERE, "libmk_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "-I", os.path.join(ROOT, "include"), "-I", CSRC]
VARIANTS = {LIB: [], LIB_DEBUG: ["-DMK_DEBUG_BOUNDS"]}


def _nvcc():
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.sep not in c or os.path.exists(c)):
            return c
    return "nvcc"


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(lib):
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        [os.path.join(ROOT, "include", "mk.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Build both libraries where stale; return the path of the plain one (debug=True: of the
    bounds-checking one)."""
    todo = [lib for lib in VARIANTS if force or _stale(lib)]
    if todo:
        nvcc = _nvcc()

        def compile_one(job):
            lib, src = job
            out = os.path.join(BUILD, "debug" if lib == LIB_DEBUG else "plain")
            os.makedirs(out, exist_ok=True)
            obj = os.path.join(out, os.path.basename(src) + ".o")
            cmd = [nvcc, *ARCH, *FLAGS, *VARIANTS[lib], "-c", src, "-o", obj]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
            return lib, obj, r.stderr

        jobs = [(lib, src) for lib in todo for src in sources()]
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            results = list(ex.map(compile_one, jobs))
        if verbose:
            for _, _, err in results:
                sys.stderr.write(err)
        for lib in todo:
            tmp = lib + f".tmp{os.getpid()}"
            cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *[o for l, o, _ in results if l == lib], "-lcudart"]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"link failed:\n{r.stderr}")
            os.replace(tmp, lib)
    return LIB_DEBUG if debug else LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

"""Build libdsa.so (the C-ABI library) from csrc/*.cu with nvcc for sm_103a, in tree.

Each translation unit compiles in parallel to _build/*.o, then one shared-library link.  The
library statically links the CUDA runtime, so it only needs the NVIDIA driver at run time.

The same sources compiled with -DDSA_TEST_HOOKS give libdsa_testhooks.so (objects in
_build_hooks/): a test build whose device-side waits give up after 20 ms instead of 1 s and that
exports dsa_test_inject_stall() (include/dsa_testhooks.h).  Only the failure-handling tests load
it; the product path never does.
"""
import concurrent.futures as cf
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libdsa.so")
OBJ_HOOKS = os.path.join(PKG, "_build_hooks")
LIB_HOOKS = os.path.join(PKG, "libdsa_testhooks.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-I", INCLUDE,
                "-I", CSRC, "--expt-relaxed-constexpr"]


def _nvcc():
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.sep not in c or os.path.exists(c)):
            return c
    return "nvcc"


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        [os.path.join(INCLUDE, "dsa.h"), os.path.abspath(__file__)]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra=(), hooks: bool = False) -> str:
    """Build libdsa.so, or with hooks=True the test build libdsa_testhooks.so."""
    lib, objdir = (LIB_HOOKS, OBJ_HOOKS) if hooks else (LIB, OBJ)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(objdir, exist_ok=True)
    nvcc = _nvcc()
    extra = list(extra) + (["-DDSA_TEST_HOOKS=1"] if hooks else [])
    jobs = []
    for src in sources():
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        jobs.append(([nvcc, *FLAGS, *extra, "-c", src, "-o", obj], obj))

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode:
            raise RuntimeError("nvcc failed: " + " ".join(cmd))
        return r

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        list(ex.map(run, [j[0] for j in jobs]))
    tmp = lib + ".%d.tmp" % os.getpid()
    run([nvcc, *ARCH, "-shared", "-o", tmp, *[j[1] for j in jobs]])
    os.replace(tmp, lib)
    return lib


def build_all(force: bool = False) -> None:
    """Both libraries, their translation units compiled in parallel."""
    with cf.ThreadPoolExecutor(max_workers=2) as ex:
        list(ex.map(lambda h: build(force=force, hooks=h), (False, True)))


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra=["-Xptxas", "-v"] if "--ptxas" in sys.argv else [],
                hooks="--hooks" in sys.argv))

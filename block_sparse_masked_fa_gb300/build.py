"""Builds the CUDA library libfa_gb300.so in-tree with nvcc for sm_103a.

Translation units are compiled in parallel, then linked into one shared
library with the static CUDA runtime (the library does not link libcuda; the
tensor-map encoder is fetched through the runtime's driver entry point).
"""
from __future__ import annotations

import concurrent.futures
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfa_gb300.so")
# The test library: the same sources with FA_TEST_HOOKS (short device wait
# limit, a hook that starves one wait, fa_test_hook exported).  Built only by
# the test that uses it; never loaded by the package.
HOOKS_BUILD = os.path.join(PKG, "_build_hooks")
HOOKS_LIB = os.path.join(PKG, "libfa_gb300_hooks.so")
SOURCES = ["api.cu", "builder.cu", "fwd.cu", "bwd.cu", "decode.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _needs_rebuild(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(ROOT, "include", "fa.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build_test_hooks(force: bool = False) -> str:
    """Builds libfa_gb300_hooks.so, the library of the device-timeout tests."""
    return build(force=force, extra_flags=("-DFA_TEST_HOOKS",), build_dir=HOOKS_BUILD, lib=HOOKS_LIB)


def build(force: bool = False, verbose: bool = False, extra_flags=(), build_dir: str = BUILD,
          lib: str = LIB) -> str:
    if not force and not _needs_rebuild(lib):
        return lib
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = lib + ".tmp"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results], "-cudart", "static"],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

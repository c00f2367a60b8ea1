"""Builds libgdn.so in-tree with nvcc for sm_103a (one -gencode, translation units compiled
in parallel, static CUDA runtime).  Run as ``python -m chunked_prefill_gb300.build``."""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libgdn.so")
BUILD = os.path.join(ROOT, "_build")
# checked variant (-DGDN_CHECK): every output store tests its index against the tensor's
# extent and records ERR_BOUNDS instead of writing out of range; for tests, not for timing
LIB_CHECK = os.path.join(HERE, "libgdn_check.so")
BUILD_CHECK = os.path.join(ROOT, "_build_check")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                   "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), *extra]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(lib) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
    deps.append(os.path.join(ROOT, "include", "gdn.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_v: bool = False,
          checked: bool = False) -> str:
    lib, bdir = (LIB_CHECK, BUILD_CHECK) if checked else (LIB, BUILD)
    os.makedirs(bdir, exist_ok=True)
    srcs = sources()
    objs = [os.path.join(bdir, os.path.basename(s) + ".o") for s in srcs]
    if not force and not _stale(lib):
        return lib
    extra = (["-Xptxas", "-v"] if ptxas_v else []) + (["-DGDN_CHECK"] if checked else [])

    def compile_one(so):
        src, obj = so
        cmd = [nvcc(), *flags(extra), "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        return r.stderr

    with ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        logs = list(ex.map(compile_one, zip(srcs, objs)))
    if ptxas_v:
        for s, log in zip(srcs, logs):
            print(f"== {os.path.basename(s)}\n{log}")
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_v="-v" in sys.argv,
                checked="--checked" in sys.argv))

"""Build the CUDA library in-tree: nvcc, sm_103a only, translation units in parallel.

    python -m async_copy_pipelined_gb300.buildlib [--force] [--verbose]

Produces ``async_copy_pipelined_gb300/_build/libpipelined_gemm.so`` (git-ignored).
``-Xptxas -v`` resource lines (registers, spills, shared memory per kernel)
are written next to it in ``ptxas.log``.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import contextlib
import fcntl
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libpipelined_gemm.so"
LIB_PATH = os.path.join(OUT_DIR, LIB_NAME)
INCLUDE = os.path.join(ROOT, "include")

GENCODE = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-std=c++17", "-O3", "-lineinfo", *GENCODE, "-Xcompiler", "-fPIC,-O2",
              "-Xptxas", "-v", "--expt-relaxed-constexpr", f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: set NVCC or put the CUDA toolkit on PATH")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _compile(src: str) -> tuple[str, str]:
    obj = os.path.join(OUT_DIR, os.path.basename(src).replace(".cu", ".o"))
    cmd = [nvcc(), *NVCC_FLAGS, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


@contextlib.contextmanager
def _build_lock():
    """One build at a time per tree (several ranks of one job may call build())."""
    os.makedirs(OUT_DIR, exist_ok=True)
    with open(os.path.join(OUT_DIR, ".build.lock"), "w") as f:
        fcntl.flock(f, fcntl.LOCK_EX)
        try:
            yield
        finally:
            fcntl.flock(f, fcntl.LOCK_UN)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB_PATH
    with _build_lock():
        if not force and up_to_date():  # another process built it while we waited
            return LIB_PATH
        return _build_locked(verbose)


def _build_locked(verbose: bool) -> str:
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        results = list(ex.map(_compile, srcs))
    logs = "\n".join(f"== {os.path.basename(o)}\n{err}" for o, err in results)
    with open(os.path.join(OUT_DIR, "ptxas.log"), "w") as f:
        f.write(logs)
    if verbose:
        print(logs)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc(), "-shared", *GENCODE, "-o", tmp, *[o for o, _ in results], "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    args = ap.parse_args(argv)
    path = build(force=args.force, verbose=args.verbose)
    print(path)


if __name__ == "__main__":
    sys.exit(main())

"""Build step for the CUDA library ``libi8conv.so`` (sm_103a only).

Compiles every ``csrc/*.cu`` translation unit in parallel with nvcc, then
links them into ``_lib/libi8conv.so`` next to this file.  Run it directly or
through ``__graft_entry__.build()``.  Rebuilds only when a source is newer
than the library or the build flavour changed.

``--pipeline-trace`` (or I8C_PIPELINE_TRACE=1 in the environment) builds the
pipeline-analysis flavour: the kernels also record per-wait cycle counts and
per-CTA timestamps in the plan's trace buffer (see pipeline_trace.py).  It is
for analysis only; build again without it for normal use.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIBDIR = os.path.join(HERE, "_lib")
OBJDIR = os.path.join(LIBDIR, "obj")
LIB = os.path.join(LIBDIR, "libi8conv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libi8conv.so")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


STAMP = os.path.join(LIBDIR, "flavour")


def _flavour(trace: bool) -> str:
    return "pipeline-trace" if trace else "release"


def up_to_date(trace: bool = False) -> bool:
    if not os.path.exists(LIB) or not os.path.exists(STAMP):
        return False
    with open(STAMP) as fh:
        if fh.read().strip() != _flavour(trace):
            return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _compile(src: str, verbose: bool, trace: bool = False) -> str:
    obj = os.path.join(OBJDIR, os.path.basename(src).replace(".cu", ".o"))
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *(["-DI8C_PIPELINE_TRACE"] if trace else []), "-c", src, "-o", obj]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False, trace: bool | None = None) -> str:
    if trace is None:
        trace = os.environ.get("I8C_PIPELINE_TRACE", "") not in ("", "0")
    if not force and up_to_date(trace):
        return LIB
    os.makedirs(OBJDIR, exist_ok=True)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, trace), srcs))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(STAMP, "w") as fh:
        fh.write(_flavour(trace))
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                trace=True if "--pipeline-trace" in sys.argv else None))

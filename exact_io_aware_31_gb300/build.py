"""Build the in-tree CUDA library ``libfa.so`` for sm_103a with nvcc.

Each translation unit compiles in its own nvcc process (in parallel), then one
link step produces ``exact_io_aware_31_gb300/libfa.so``.  The CUDA runtime is
linked statically, so the library loads on a host without a GPU driver (the
driver is only needed once a call reaches the device).

    python -m exact_io_aware_31_gb300.build [--force] [--verbose]
"""

from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "libfa.so")
OBJDIR = os.path.join(PKG, "_build")
SOURCES = ["fa_api.cu", "fa_fwd.cu", "fa_bwd.cu", "fa_bwd_dq.cu", "fa_decode.cu", "fa_noalloc.cu"]
HEADERS = ["fa_common.cuh", "fa_kernels.h", "sm103_ptx.cuh", "exp2_poly.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I" + os.path.join(ROOT, "include")]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfa.so")
    return exe


def _inputs_mtime() -> float:
    paths = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(ROOT, "include", "fa.h"),
                                                                   os.path.abspath(__file__)]
    return max(os.path.getmtime(p) for p in paths)


TRACE_OUT = os.path.join(PKG, "libfa_trace.so")


def up_to_date(out: str = OUT) -> bool:
    return os.path.exists(out) and os.path.getmtime(out) >= _inputs_mtime()


def build(force: bool = False, verbose: bool = False, extra_flags=None, trace: bool = False, out: str = None) -> str:
    """Compile and link libfa.so if any input changed; returns its path.

    ``trace=True`` builds the phase-tracing variant ``libfa_trace.so``
    (-DFA_TRACE) instead; the default library never contains tracing.
    ``out`` (with ``extra_flags``) builds a tuning variant at another path.
    """
    custom = out is not None
    out = out or (TRACE_OUT if trace else OUT)
    if not force and not custom and up_to_date(out):
        return out
    objdir = (out + ".objs") if custom else OBJDIR + ("_trace" if trace else "")
    os.makedirs(objdir, exist_ok=True)
    exe = nvcc()
    flags = FLAGS + list(extra_flags or []) + (["-DFA_TRACE"] if trace else [])
    if verbose:
        flags = flags + ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [exe] + ARCH + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = out + ".tmp"
    cmd = [exe] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true", help="print ptxas register/spill/smem usage")
    ap.add_argument("--trace", action="store_true", help="build the phase-tracing variant libfa_trace.so")
    args = ap.parse_args()
    print(build(force=args.force, verbose=args.verbose, trace=args.trace))

"""Build the in-tree CUDA library ``libfa.so`` for sm_103a with nvcc.

Each translation unit compiles in its own nvcc process (in parallel), then one
link step produces ``exact_io_aware_31_gb300/libfa.so``.  The CUDA runtime is
linked statically, so the library loads on a host without a GPU driver (the
driver is only needed once a call reaches the device).

A library is reused only when the SHA-256 digest of everything that went into
it matches the digest stored beside it (``libfa.so.sha256``): every source,
every header those sources include (found by following their ``#include "…"``
lines, so no list can go stale), the compiler flags, the nvcc version and this
file.  File times play no part, so a library copied from another machine or
built from other sources is never taken for a current one.

    python -m exact_io_aware_31_gb300.build [--force] [--verbose]
"""

from __future__ import annotations

import argparse
import functools
import hashlib
import os
import re
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(PKG, "libfa.so")
OBJDIR = os.path.join(PKG, "_build")
SOURCES = ["fa_api.cu", "fa_fwd.cu", "fa_bwd.cu", "fa_bwd_dq.cu", "fa_decode.cu", "fa_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]
STAMP_SUFFIX = ".sha256"
TRACE_OUT = os.path.join(PKG, "libfa_trace.so")

_INCLUDE_RE = re.compile(r'^\s*#\s*include\s+"([^"]+)"', re.M)


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfa.so")
    return exe


@functools.lru_cache(maxsize=None)
def _nvcc_version() -> str:
    try:
        return subprocess.run([nvcc(), "--version"], capture_output=True, text=True).stdout
    except (OSError, RuntimeError):
        return "nvcc unavailable"


def build_inputs(csrc: str = CSRC, sources=tuple(SOURCES)) -> list[str]:
    """Every file that goes into the library: the sources and, transitively, the
    headers they include with ``#include "…"`` (resolved beside the including
    file).  A quoted include that resolves to no file is an error."""
    seen, order = set(), []
    stack = [os.path.realpath(os.path.join(csrc, s)) for s in sources]
    while stack:
        path = stack.pop()
        if path in seen:
            continue
        if not os.path.exists(path):
            raise RuntimeError(f"build input not found: {path}")
        seen.add(path)
        order.append(path)
        with open(path, encoding="utf-8") as f:
            text = f.read()
        for inc in _INCLUDE_RE.findall(text):
            stack.append(os.path.realpath(os.path.join(os.path.dirname(path), inc)))
    return sorted(order)


def inputs_digest(flags=(), csrc: str = CSRC, sources=tuple(SOURCES)) -> str:
    """SHA-256 over the build inputs' names and contents, the flags, nvcc's version and this file."""
    h = hashlib.sha256()
    base = os.path.dirname(os.path.realpath(csrc))
    for path in build_inputs(csrc, sources):
        h.update(os.path.relpath(path, base).encode() + b"\0")
        with open(path, "rb") as f:
            h.update(f.read())
        h.update(b"\0")
    h.update("\0".join(ARCH + FLAGS + list(flags)).encode())
    h.update(_nvcc_version().encode())
    with open(os.path.abspath(__file__), "rb") as f:
        h.update(f.read())
    return h.hexdigest()


def up_to_date(out: str = OUT, flags=(), csrc: str = CSRC) -> bool:
    """True when ``out`` exists and its stored digest equals the current inputs' digest."""
    stamp = out + STAMP_SUFFIX
    if not (os.path.exists(out) and os.path.exists(stamp)):
        return False
    with open(stamp) as f:
        return f.read().strip() == inputs_digest(flags, csrc)


def build(force: bool = False, verbose: bool = False, extra_flags=None, trace: bool = False, out: str = None) -> str:
    """Compile and link libfa.so unless a library built from the same inputs is present; returns its path.

    ``trace=True`` builds the phase-tracing variant ``libfa_trace.so``
    (-DFA_TRACE) instead; the default library never contains tracing.
    ``out`` (with ``extra_flags``) builds a variant at another path.
    """
    out = out or (TRACE_OUT if trace else OUT)
    flags = list(extra_flags or []) + (["-DFA_TRACE"] if trace else [])
    digest = inputs_digest(flags)
    stamp = out + STAMP_SUFFIX
    if not force and os.path.exists(out) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return out
    objdir = OBJDIR + "_" + os.path.basename(out).replace(".", "_")
    os.makedirs(objdir, exist_ok=True)
    exe = nvcc()
    cflags = FLAGS + ["-I" + INCLUDE] + flags
    if verbose:
        cflags = cflags + ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [exe] + ARCH + cflags + ["-c", os.path.join(CSRC, src), "-o", obj]
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
    if os.path.exists(stamp):
        os.unlink(stamp)
    os.replace(tmp, out)
    with open(stamp, "w") as f:
        f.write(digest + "\n")
    sys.stderr.write(f"built {os.path.basename(out)} ({len(SOURCES)} translation units, inputs {digest[:16]})\n")
    return out


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true", help="print ptxas register/spill/smem usage")
    ap.add_argument("--trace", action="store_true", help="build the phase-tracing variant libfa_trace.so")
    args = ap.parse_args()
    print(build(force=args.force, verbose=args.verbose, trace=args.trace))

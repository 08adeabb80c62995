"""The library is rebuilt whenever anything it is built from changes (CPU only).

``build.build()`` reuses ``libfa.so`` only if the SHA-256 digest of its inputs
(every source, every header reached through ``#include "…"``, the flags and
the compiler version) equals the digest stored beside it.  These tests work
on a copy of the sources, so they neither compile nor touch the real library.
"""

import os
import re
import shutil

import pytest

from exact_io_aware_31_gb300 import build


@pytest.fixture
def tree(tmp_path):
    """A copy of the package's csrc/ and the repository's include/ in the same relative layout."""
    pkg = tmp_path / "pkg"
    shutil.copytree(build.CSRC, pkg / "csrc")
    shutil.copytree(build.INCLUDE, tmp_path / "include")
    return pkg / "csrc"


def _stamp(out, digest):
    out.write_bytes(b"not a real library")
    (out.parent / (out.name + build.STAMP_SUFFIX)).write_text(digest + "\n")


def test_every_included_header_is_a_build_input():
    inputs = {os.path.basename(p) for p in build.build_inputs()}
    for name in os.listdir(build.CSRC):
        path = os.path.join(build.CSRC, name)
        if not name.endswith((".cu", ".cuh", ".h")):
            continue
        for inc in re.findall(r'^\s*#\s*include\s+"([^"]+)"', open(path).read(), flags=re.M):
            if name in build.SOURCES or name in inputs:
                assert os.path.basename(inc) in inputs, (name, inc)
    for header in ("fa_dropout.cuh", "fa_common.cuh", "sm103_ptx.cuh", "fa_kernels.h", "fa_context.h", "fa.h"):
        assert header in inputs, header


@pytest.mark.parametrize("edit", ["fa_dropout.cuh", "sm103_ptx.cuh", "fa_bwd.cu", "fa.h"])
def test_editing_any_input_makes_the_library_stale(tree, tmp_path, edit):
    out = tmp_path / "libfa.so"
    _stamp(out, build.inputs_digest((), csrc=str(tree)))
    assert build.up_to_date(str(out), (), csrc=str(tree))
    target = tree / edit if edit != "fa.h" else tmp_path / "include" / "fa.h"
    target.write_text(target.read_text() + "\n// edited\n")
    assert not build.up_to_date(str(out), (), csrc=str(tree))


def test_flags_and_missing_stamp_make_the_library_stale(tree, tmp_path):
    out = tmp_path / "libfa.so"
    digest = build.inputs_digest((), csrc=str(tree))
    _stamp(out, digest)
    assert not build.up_to_date(str(out), ("-DFA_TRACE",), csrc=str(tree))
    os.unlink(str(out) + build.STAMP_SUFFIX)
    assert not build.up_to_date(str(out), (), csrc=str(tree))


def test_file_times_do_not_matter(tree, tmp_path):
    """A library newer than its sources but built from other ones is stale; an old one from the same is current."""
    out = tmp_path / "libfa.so"
    _stamp(out, "0" * 64)
    os.utime(out, (4e9, 4e9))
    assert not build.up_to_date(str(out), (), csrc=str(tree))
    _stamp(out, build.inputs_digest((), csrc=str(tree)))
    os.utime(out, (1.0, 1.0))
    assert build.up_to_date(str(out), (), csrc=str(tree))


def test_a_missing_include_is_an_error(tree):
    (tree / "fa_dropout.cuh").unlink()
    with pytest.raises(RuntimeError, match="build input not found"):
        build.inputs_digest((), csrc=str(tree))

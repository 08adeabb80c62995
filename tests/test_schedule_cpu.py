"""The persistent schedule's host-visible helpers (CPU, compiled with g++).

``fa_common.cuh`` declares ``snake_unit``, ``split_unit`` and
``block_major_order`` for host and device.  A small C++ driver built from that
header checks, over many problem shapes and grid sizes, that:

* the snake order hands every unit position in [0, total) to exactly one
  (round, CTA) pair, alternating direction by round;
* ``split_unit`` is a bijection from positions onto (slice, block) pairs in
  both orders, slice-major keeping one slice's blocks consecutive;
* block-major is chosen only for causal shapes with N >= 4096 and fewer than
  16 units per CTA.
"""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_io_aware_31_gb300", "csrc")

DRIVER = r"""
#include <cstdio>
#include <vector>
#include "fa_common.cuh"
using namespace fa;
static int fail(const char* what, int a, int b, int c) {
  std::printf("FAIL %s %d %d %d\n", what, a, b, c);
  return 1;
}
int main() {
  const int BHs[] = {1, 2, 3, 16, 32, 1024};
  const int blks[] = {1, 2, 7, 8, 32, 128};
  const int grids[] = {1, 5, 148, 152};
  for (int BH : BHs) for (int nblk : blks) for (int g : grids) {
    const int total = BH * nblk;
    const int grid = total < g ? total : g;
    std::vector<int> seen(total, 0);
    for (int r = 0; r * grid < total; ++r)
      for (int c = 0; c < grid; ++c) {
        const int p = snake_unit(r, c, grid);
        if (p < r * grid || p >= (r + 1) * grid) return fail("snake round", r, c, p);
        if ((r & 1) == 0 && p != r * grid + c) return fail("snake even", r, c, p);
        if ((r & 1) == 1 && p != r * grid + grid - 1 - c) return fail("snake odd", r, c, p);
        if (p < total) ++seen[p];
      }
    for (int p = 0; p < total; ++p)
      if (seen[p] != 1) return fail("snake cover", BH, nblk, p);
    for (int bm = 0; bm < 2; ++bm) {
      std::vector<int> hit(total, 0);
      for (int p = 0; p < total; ++p) {
        int bh = -1, blk = -1;
        split_unit(p, BH, nblk, bm != 0, bh, blk);
        if (bh < 0 || bh >= BH || blk < 0 || blk >= nblk) return fail("split range", p, bh, blk);
        ++hit[bh * nblk + blk];
        if (!bm && (bh != p / nblk || blk != p % nblk)) return fail("slice-major", p, bh, blk);
        if (bm && (blk != p / BH || bh != p % BH)) return fail("block-major", p, bh, blk);
      }
      for (int x = 0; x < total; ++x)
        if (hit[x] != 1) return fail("split bijection", BH, nblk, x);
    }
  }
  const int Ns[] = {1, 1024, 4095, 4096, 16384};
  for (int N : Ns) for (int causal = 0; causal < 2; ++causal)
    for (int units : {100, 2431, 2432, 5000}) {
      const bool want = causal && N >= 4096 && units < 16 * 152;
      if (block_major_order(causal != 0, units, 152, N) != want) return fail("block-major choice", N, causal, units);
    }
  std::printf("OK\n");
  return 0;
}
"""


def test_schedule_helpers(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    src = tmp_path / "sched.cpp"
    src.write_text(DRIVER)
    exe = tmp_path / "sched"
    r = subprocess.run([gxx, "-std=c++17", "-O1", "-D__host__=", "-D__device__=", "-I", CSRC, str(src), "-o",
                        str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "OK", out.stdout + out.stderr

"""Failure detection on the GPU without faulting it (needs a GB300).

Every wait inside the kernels is bounded (1 s).  A test-only build of the
library (-DFA_TEST_HOOKS, built next to the real one, never loaded by the
product) can make the forward's first softmax warpgroup withhold one "P
ready" arrival, so the MMA warp's wait runs out.  The kernel must then record
FA_ERR_DEVICE_TIMEOUT in the status word, leave cleanly (drain its copies,
free tensor memory), and the very next call must run normally and correctly.
Nothing here traps, asserts on the device or spins without a limit.
"""

import ctypes
import math
import os
import time

import pytest
import torch

import exact_io_aware_31_gb300 as fa
from exact_io_aware_31_gb300 import build
from tests.gpu_util import require_gpu
from workloads import make_inputs

pytestmark = pytest.mark.gpu

HOOKS_LIB = os.path.join(os.path.dirname(fa.LIB_PATH), "libfa_testhooks.so")


@pytest.fixture(scope="module")
def hooks():
    require_gpu()
    path = build.build(extra_flags=["-DFA_TEST_HOOKS"], out=HOOKS_LIB, force=True)
    lib = ctypes.CDLL(path)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
    lib.fa_get_device_status.argtypes = [vp]
    lib.fa_test_withhold_arrival.argtypes = [i]
    return lib


def test_withheld_arrival_times_out_then_next_call_is_clean(hooks):
    B, H, N, d, causal = 1, 2, 512, 64, True
    scale = 1.0 / math.sqrt(d)
    q, k, v, _ = (t.cuda() for t in make_inputs(B, H, N, d, seed=77))
    ref_o, ref_lse = fa.forward(q, k, v, scale, causal)       # the product library
    torch.cuda.synchronize()
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), device="cuda", dtype=torch.float32)
    s = torch.cuda.current_stream().cuda_stream

    def call():
        return hooks.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
                            scale, int(causal), s)

    assert hooks.fa_get_device_status(s) == fa.FA_OK
    assert hooks.fa_test_withhold_arrival(1) == 0
    try:
        t0 = time.time()
        assert call() == fa.FA_OK                          # the launch itself is fine
        st = hooks.fa_get_device_status(s)                 # synchronises, reads and clears
        elapsed = time.time() - t0
    finally:
        assert hooks.fa_test_withhold_arrival(0) == 0
    assert st == fa.FA_ERR_DEVICE_TIMEOUT, fa.fa_status_string(st)
    assert elapsed < 30.0                                   # bounded: a few 1 s limits at most
    assert hooks.fa_get_device_status(s) == fa.FA_OK        # the word was cleared
    # the context is healthy: a normal call succeeds and matches the product library
    assert call() == fa.FA_OK
    assert hooks.fa_get_device_status(s) == fa.FA_OK
    torch.cuda.synchronize()
    assert float((o.float() - ref_o.float()).abs().max()) <= 1e-2
    assert float((lse - ref_lse).abs().max()) <= 1e-3

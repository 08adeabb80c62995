"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory (needs a GB300).

Some callers cannot call cudaMalloc (an allocator hook, a plug-in that must
not touch the process's memory pool), so they cannot supply fa_bwd's
workspace; fa_bwd_noalloc uses a scratch array the library owns instead.
These tests call it through the C ABI and check its gradients against
fa_bwd's on the same inputs, twice in a row (the scratch keeps the previous
call's contents, which must not leak into the next result), with the
gradient tolerance the other GPU tests use.  This file sorts last so a run
that stops at the first failure has already run every other test.
"""

import math

import numpy as np
import pytest
import torch

import exact_io_aware_31_gb300 as fa
from tests.gpu_util import TOL_GRAD_REL, f64, require_gpu
from workloads import make_inputs

pytestmark = pytest.mark.gpu

CASES = [(1, 2, 256, 64, False), (2, 3, 777, 128, True), (1, 4, 1000, 64, True)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _ptrs(*ts):
    return [t.data_ptr() for t in ts]


@pytest.mark.parametrize("B,H,N,d,causal", CASES, ids=[f"b{b}h{h}n{n}d{d}{'c' if c else ''}" for b, h, n, d, c in CASES])
def test_noalloc_matches_workspace_backward_twice(B, H, N, d, causal):
    scale = 1.0 / math.sqrt(d)
    stream = torch.cuda.current_stream().cuda_stream
    q, k, v, do = (t.cuda() for t in make_inputs(B, H, N, d, seed=4000 + N + d))
    o, lse = fa.forward(q, k, v, scale, causal)
    ref = fa.backward(q, k, v, o, lse, do, scale, causal)
    torch.cuda.synchronize()
    for call in range(2):
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        st = fa.fa_bwd_noalloc(*_ptrs(q, k, v, o, do, lse, dq, dk, dv), B, H, N, d, scale, int(causal), stream)
        assert st == fa.FA_OK, fa.fa_status_string(st)
        assert fa.fa_get_device_status(stream) == fa.FA_OK
        for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            gr, rr = f64(g), f64(r)
            assert np.all(np.isfinite(gr)), (call, name)
            err = float(np.abs(gr - rr).max())
            assert err <= TOL_GRAD_REL * float(np.abs(rr).max()), (call, name, err)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # B*H*N*d = 32M elements needs a 128 MiB dQ accumulator, beyond the 64 MiB scratch;
    # the call must refuse before touching any pointer.
    B, H, N, d = 1, 64, 4096, 128
    assert fa.fa_bwd_workspace_size(B, H, N, d) > fa.NOALLOC_SCRATCH_BYTES
    a = 1 << 20
    st = fa.fa_bwd_noalloc(a, a, a, a, a, a, a, a, a, B, H, N, d, 0.1, 0, None)
    assert st == fa.FA_ERR_WORKSPACE
    assert fa.fa_bwd_noalloc(a, a, a, a, a, a, a, a, a, 1, 1, 16, 96, 0.1, 0, None) == fa.FA_ERR_UNSUPPORTED

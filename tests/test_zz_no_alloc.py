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


def _compare(grads, ref, what):
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        gr, rr = f64(g) if isinstance(g, torch.Tensor) else g, f64(r)
        assert np.all(np.isfinite(gr)), (what, name)
        err = float(np.abs(gr - rr).max())
        assert err <= TOL_GRAD_REL * float(np.abs(rr).max()), (what, name, err)


def test_noalloc_at_its_size_limit():
    """B2 H8 N8064 d128 is the largest such shape that fits the scratch: same gradients as fa_bwd, twice."""
    B, H, N, d, causal = 2, 8, 8064, 128, True
    assert fa.fa_bwd_workspace_size(B, H, N, d) <= fa.NOALLOC_SCRATCH_BYTES
    assert fa.fa_bwd_workspace_size(B, H, N + 1, d) > fa.NOALLOC_SCRATCH_BYTES
    scale = 1.0 / math.sqrt(d)
    stream = torch.cuda.current_stream().cuda_stream
    q, k, v, do = (t.cuda() for t in make_inputs(B, H, N, d, seed=4321))
    o, lse = fa.forward(q, k, v, scale, causal)
    ref = fa.backward(q, k, v, o, lse, do, scale, causal)
    for call in range(2):
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        st = fa.fa_bwd_noalloc(*_ptrs(q, k, v, o, do, lse, dq, dk, dv), B, H, N, d, scale, int(causal), stream)
        assert st == fa.FA_OK, fa.fa_status_string(st)
        assert fa.fa_get_device_status(stream) == fa.FA_OK
        _compare((dq, dk, dv), ref, f"limit call {call}")


class _Driver:
    """The few CUDA driver calls a caller with a context of its own would make (ctypes, no allocation by the library)."""

    def __init__(self):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libcuda.so.1")

    def __call__(self, name, *args):
        r = getattr(self.lib, name)(*args)
        assert r == 0, f"{name} returned CUresult {r}"


def test_noalloc_in_a_caller_created_context():
    """A caller that runs the library under its own driver-API context (not the primary one torch uses).

    The scratch's device address is looked up per context, so the first call in
    the new context must use that context's copy of the array; the primary
    context's calls before and after keep working.  Buffers here belong to the
    caller (cuMemAlloc in its context); the entry point itself allocates nothing.
    """
    B, H, N, d, causal = 1, 2, 640, 64, True
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = (t.cuda() for t in make_inputs(B, H, N, d, seed=4777))
    o, lse = fa.forward(q, k, v, scale, causal)
    ref = fa.backward(q, k, v, o, lse, do, scale, causal)
    stream = torch.cuda.current_stream().cuda_stream
    dq0, dk0, dv0 = (torch.empty_like(q) for _ in range(3))
    assert fa.fa_bwd_noalloc(*_ptrs(q, k, v, o, do, lse, dq0, dk0, dv0), B, H, N, d, scale, int(causal),
                             stream) == fa.FA_OK
    torch.cuda.synchronize()
    host_in = [t.cpu().contiguous() for t in (q, k, v, o, do, lse)]
    drv = _Driver()
    c = drv.c
    dev = c.c_int(0)
    drv("cuDeviceGet", c.byref(dev), torch.cuda.current_device())
    ctx = c.c_void_p()
    drv("cuCtxCreate_v2", c.byref(ctx), 0, dev)  # the new context is now current on this thread
    bufs = []
    try:
        def alloc(nbytes):
            p = c.c_uint64()
            drv("cuMemAlloc_v2", c.byref(p), c.c_size_t(nbytes))
            bufs.append(p)
            return p.value
        dev_in = []
        for t in host_in:
            nbytes = t.numel() * t.element_size()
            p = alloc(nbytes)
            drv("cuMemcpyHtoD_v2", c.c_uint64(p), c.c_void_p(t.data_ptr()), c.c_size_t(nbytes))
            dev_in.append(p)
        nbytes = q.numel() * 2
        outs = [alloc(nbytes) for _ in range(3)]
        for call in range(2):
            st = fa.fa_bwd_noalloc(*dev_in, *outs, B, H, N, d, scale, int(causal), None)
            assert st == fa.FA_OK, fa.fa_status_string(st)
            assert fa.fa_get_device_status(None) == fa.FA_OK
            got = []
            for p in outs:
                h = torch.empty(q.shape, dtype=torch.bfloat16)
                drv("cuMemcpyDtoH_v2", c.c_void_p(h.data_ptr()), c.c_uint64(p), c.c_size_t(nbytes))
                got.append(h)
            _compare(got, ref, f"own context call {call}")
    finally:
        for p in bufs:
            drv("cuMemFree_v2", p)
        drv("cuCtxDestroy_v2", ctx)
    # back in torch's primary context: the cached address there still serves
    dq1, dk1, dv1 = (torch.full_like(q, float("nan")) for _ in range(3))
    torch.cuda.set_device(torch.cuda.current_device())
    assert fa.fa_bwd_noalloc(*_ptrs(q, k, v, o, do, lse, dq1, dk1, dv1), B, H, N, d, scale, int(causal),
                             stream) == fa.FA_OK
    assert fa.fa_get_device_status(stream) == fa.FA_OK
    _compare((dq1, dk1, dv1), ref, "primary context after")

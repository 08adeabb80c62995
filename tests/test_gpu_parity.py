"""GPU vs oracle parity through the C ABI (needs a GB300).

* Small shapes, compared element by element with the full fp64 oracle: several
  128-row tiles plus ragged tails (N = 1, 127, 129, 300, 777, 1000), both head
  dims, both masks, batched heads.
* Stress inputs: queries x8 (score rows spanning dozens of units, so the
  running maximum moves and the lazy rescale fires), one spiked key per head,
  sorted keys (the maximum keeps growing along the row).  Their rows are
  dominated by single keys, so the bounds add the bf16 effects that then
  surface: one ulp of |O| on the output, and the first-order effect of D being
  formed from the stored bf16 O on dQ and dK (tests/gpu_util.py).
* scale = 0 (uniform attention, closed form).
"""

import math

import numpy as np
import pytest

import oracle
from tests.gpu_util import (assert_fwd_close, assert_grads_close, d_rounding_allowance, require_gpu, run_bwd,
                            run_fwd)
from workloads import make_inputs

pytestmark = pytest.mark.gpu

SMALL = [
    (1, 2, 256, 64, False), (1, 2, 256, 64, True), (1, 2, 256, 128, False), (1, 2, 256, 128, True),
    (1, 1, 1, 64, False), (1, 1, 1, 128, True), (1, 1, 127, 64, True), (1, 1, 128, 128, False),
    (1, 1, 129, 64, False), (1, 1, 129, 128, True), (2, 3, 777, 64, False), (2, 3, 777, 128, True),
    (1, 2, 1000, 128, True), (1, 1, 300, 64, True), (3, 1, 513, 128, False), (1, 2, 640, 64, True),
    # d = 64 forward with the second MMA issuer (non-causal N >= 1024, causal N >= 2048), ragged tails
    (1, 1, 1100, 64, False), (1, 1, 2100, 64, True),
    # causal N >= 4096 with few units per CTA: the block-major unit order
    (1, 2, 4096, 128, True),
]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _oracle_case(q, k, v, do, scale, causal):
    qd, kd, vd, dod = (t.double().numpy() for t in (q, k, v, do))
    o_ref, lse_ref = oracle.attention_forward(qd, kd, vd, scale, causal)
    dq_r, dk_r, dv_r, _ = oracle.attention_backward(qd, kd, vd, dod, scale, causal)
    return o_ref, lse_ref, (dq_r, dk_r, dv_r)


@pytest.mark.parametrize("B,H,N,d,causal", SMALL, ids=[f"b{b}h{h}n{n}d{d}{'c' if c else ''}" for b, h, n, d, c in SMALL])
def test_small_forward_backward(B, H, N, d, causal):
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = make_inputs(B, H, N, d, seed=2000 + N + d + causal)
    qg, kg, vg, o, lse = run_fwd(q, k, v, scale, causal)
    grads = run_bwd(qg, kg, vg, o, lse, do, scale, causal)
    o_ref, lse_ref, g_ref = _oracle_case(q, k, v, do, scale, causal)
    assert_fwd_close(o, lse, o_ref, lse_ref, f"{(B, H, N, d, causal)}")
    assert_grads_close(grads, g_ref, f"{(B, H, N, d, causal)}")


STRESS = [("wide", 512, 64, False), ("wide", 512, 128, True), ("spike", 384, 64, True),
          ("spike", 640, 128, False), ("sorted", 512, 64, False), ("sorted", 700, 128, True)]


@pytest.mark.parametrize("stress,N,d,causal", STRESS, ids=[f"{s}-n{n}d{d}{'c' if c else ''}" for s, n, d, c in STRESS])
def test_stress_inputs(stress, N, d, causal):
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = make_inputs(1, 2, N, d, seed=3000 + N, stress=stress)
    qg, kg, vg, o, lse = run_fwd(q, k, v, scale, causal)
    grads = run_bwd(qg, kg, vg, o, lse, do, scale, causal)
    o_ref, lse_ref, g_ref = _oracle_case(q, k, v, do, scale, causal)
    assert_fwd_close(o, lse, o_ref, lse_ref, stress, o_rel=2.0 ** -8)
    extra = d_rounding_allowance(q.double().numpy(), k.double().numpy(), do.double().numpy(), o_ref, lse_ref,
                                 scale, causal)
    assert_grads_close(grads, g_ref, stress, extra=extra)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_scale_is_uniform_attention(causal):
    q, k, v, do = make_inputs(1, 2, 300, 64, seed=11)
    qg, kg, vg, o, lse = run_fwd(q, k, v, 0.0, causal)
    vd = v.double().numpy()
    n = vd.shape[2]
    if causal:
        cnt = np.arange(1, n + 1, dtype=np.float64)
        o_ref = np.cumsum(vd, axis=2) / cnt[None, None, :, None]
        lse_ref = np.broadcast_to(np.log(cnt), (1, 2, n))
    else:
        o_ref = np.broadcast_to(vd.mean(axis=2, keepdims=True), vd.shape)
        lse_ref = np.full((1, 2, n), math.log(n))
    assert_fwd_close(o, lse, o_ref, lse_ref, "scale=0")
    grads = run_bwd(qg, kg, vg, o, lse, do, 0.0, causal)
    _, _, g_ref = _oracle_case(q, k, v, do, 0.0, causal)
    assert_grads_close(grads, g_ref, "scale=0")


SPLIT = [(2, 2, 300, 64, True), (1, 3, 513, 64, False), (1, 2, 300, 128, True), (2, 1, 257, 128, False)]


@pytest.mark.parametrize("B,H,N,d,causal", SPLIT, ids=[f"b{b}h{h}n{n}d{d}{'c' if c else ''}" for b, h, n, d, c in SPLIT])
def test_split_phases_match_oracle(B, H, N, d, causal):
    """fa_bwd_preprocess -> fa_bwd_dkdv -> fa_bwd_dq_convert on one workspace.

    The workspace starts as garbage (0xAB bytes): the preprocess must reset the
    dQ accumulator.  Run twice on the same workspace, so a finished call's
    accumulator is reset too.
    """
    import torch

    import exact_io_aware_31_gb300 as fa
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = make_inputs(B, H, N, d, seed=4100 + N + d + causal)
    qg, kg, vg, o, lse = run_fwd(q, k, v, scale, causal)
    dog = do.cuda()
    nbytes = fa.fa_bwd_workspace_size(B, H, N, d)
    ws = torch.full((nbytes,), 0xAB, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    _, _, g_ref = _oracle_case(q, k, v, do, scale, causal)
    for rep in range(2):
        dq, dk, dv = (torch.full_like(qg, float("nan")) for _ in range(3))
        assert fa.fa_bwd_preprocess(o.data_ptr(), dog.data_ptr(), lse.data_ptr(), B, H, N, d, ws.data_ptr(), nbytes,
                                    s) == fa.FA_OK
        assert fa.fa_bwd_dkdv(qg.data_ptr(), kg.data_ptr(), vg.data_ptr(), dog.data_ptr(), dk.data_ptr(),
                              dv.data_ptr(), B, H, N, d, scale, int(causal), ws.data_ptr(), nbytes, s) == fa.FA_OK
        assert fa.fa_bwd_dq_convert(dq.data_ptr(), B, H, N, d, scale, ws.data_ptr(), nbytes, s) == fa.FA_OK
        assert fa.fa_get_device_status(s) == fa.FA_OK
        assert_grads_close((dq, dk, dv), g_ref, f"split {(B, H, N, d, causal)} rep {rep}")


NEG = [(1, 2, 300, 64, False), (1, 2, 300, 64, True), (2, 1, 777, 128, False), (1, 2, 1000, 128, True),
       (1, 1, 1100, 64, False), (1, 2, 4096, 128, True)]


@pytest.mark.parametrize("B,H,N,d,causal", NEG, ids=[f"b{b}h{h}n{n}d{d}{'c' if c else ''}" for b, h, n, d, c in NEG])
def test_negative_scale(B, H, N, d, causal):
    """scale = -1/sqrt(d): the forward and backward match the oracle (S is formed negated on the tensor core)."""
    scale = -1.0 / math.sqrt(d)
    q, k, v, do = make_inputs(B, H, N, d, seed=7100 + N + d + causal)
    qg, kg, vg, o, lse = run_fwd(q, k, v, scale, causal)
    grads = run_bwd(qg, kg, vg, o, lse, do, scale, causal)
    o_ref, lse_ref, g_ref = _oracle_case(q, k, v, do, scale, causal)
    assert_fwd_close(o, lse, o_ref, lse_ref, f"scale<0 {(B, H, N, d, causal)}")
    assert_grads_close(grads, g_ref, f"scale<0 {(B, H, N, d, causal)}")

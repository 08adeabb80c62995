"""Deterministic backward (fa_bwd_deterministic) vs the oracle, and run-to-run bitwise equality (needs a GB300).

Same tolerances as fa_bwd: each gradient within 2e-2 of its reference's max-abs.
Shapes: both head dims and masks, ragged tails (N = 1, 129, 300, 777), several
query and key tiles; the full-size workloads on sampled (b, h) slices.  Every
case runs twice and the two results must match bit for bit (no reduction
order varies between runs).
"""

import math

import numpy as np
import pytest
import torch

import exact_io_aware_31_gb300 as fa
import oracle
from tests.gpu_util import assert_grads_close, require_gpu, run_fwd
from workloads import BY_NAME, GPT2_MEDIUM, LONG_SEQ, make_inputs, workload_inputs

pytestmark = pytest.mark.gpu

CASES = [(1, 2, 256, 64, False), (1, 2, 256, 64, True), (1, 2, 256, 128, False), (1, 2, 256, 128, True),
         (1, 1, 1, 64, True), (1, 1, 129, 128, True), (2, 3, 777, 64, False), (2, 2, 300, 128, True),
         (1, 2, 1000, 64, True), (3, 1, 513, 128, False)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _twice(qg, kg, vg, o, lse, dog, scale, causal):
    a = fa.backward(qg, kg, vg, o, lse, dog, scale, causal, deterministic=True)
    b = fa.backward(qg, kg, vg, o, lse, dog, scale, causal, deterministic=True)
    assert fa.fa_get_device_status(torch.cuda.current_stream().cuda_stream) == fa.FA_OK
    for x, y, name in zip(a, b, ("dq", "dk", "dv")):
        assert torch.equal(x, y), f"{name} differs between two runs"
    return a


@pytest.mark.parametrize("B,H,N,d,causal", CASES, ids=[f"b{b}h{h}n{n}d{d}{'c' if c else ''}" for b, h, n, d, c in CASES])
def test_deterministic_matches_oracle_and_repeats_bitwise(B, H, N, d, causal):
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = make_inputs(B, H, N, d, seed=6000 + N + d + causal)
    qg, kg, vg, o, lse = run_fwd(q, k, v, scale, causal)
    grads = _twice(qg, kg, vg, o, lse, do.cuda(), scale, causal)
    qd, kd, vd, dod = (t.double().numpy() for t in (q, k, v, do))
    dq_r, dk_r, dv_r, _ = oracle.attention_backward(qd, kd, vd, dod, scale, causal)
    assert_grads_close(grads, (dq_r, dk_r, dv_r), f"deterministic {(B, H, N, d, causal)}")


@pytest.mark.parametrize("w", [GPT2_MEDIUM, LONG_SEQ, BY_NAME["sweep_b16_h16_n1024_d128_causal"]],
                         ids=lambda w: w.name)
def test_deterministic_full_workloads_sampled_heads(w):
    q, k, v, do = workload_inputs(w)
    qg, kg, vg, o, lse = run_fwd(q, k, v, w.scale, w.causal)
    dq, dk, dv = _twice(qg, kg, vg, o, lse, do.cuda(), w.scale, w.causal)
    rng = np.random.default_rng(w.seed)
    for _ in range(1 if w.N > 4096 else 2):
        b, h = int(rng.integers(w.B)), int(rng.integers(w.H))
        sl = lambda t: t[b:b + 1, h:h + 1]
        qd, kd, vd, dod = (sl(t).double().numpy() for t in (q, k, v, do))
        dq_r, dk_r, dv_r, _ = oracle.attention_backward(qd, kd, vd, dod, w.scale, w.causal)
        assert_grads_close((sl(dq), sl(dk), sl(dv)), (dq_r, dk_r, dv_r), f"{w.name} slice {(b, h)}")


@pytest.mark.parametrize("d,causal", [(64, True), (128, False)])
def test_deterministic_negative_scale(d, causal):
    scale = -1.0 / math.sqrt(d)
    q, k, v, do = make_inputs(1, 2, 400, d, seed=6500 + d)
    qg, kg, vg, o, lse = run_fwd(q, k, v, scale, causal)
    grads = _twice(qg, kg, vg, o, lse, do.cuda(), scale, causal)
    qd, kd, vd, dod = (t.double().numpy() for t in (q, k, v, do))
    dq_r, dk_r, dv_r, _ = oracle.attention_backward(qd, kd, vd, dod, scale, causal)
    assert_grads_close(grads, (dq_r, dk_r, dv_r), f"deterministic scale<0 {(d, causal)}")

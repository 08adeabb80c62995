"""Parity at the measured workloads' full sizes (needs a GB300).

Each workload runs once on the GPU at its full size, in the same launch
configuration ``bench.py`` times.  The oracle then checks:

* every output row of two sampled (b, h) slices (first and last) for the
  forward, and the complete gradients of one sampled slice for the backward
  (exact oracle on that slice; every slice is independent);
* on ALL slices, properties that hold at any size: finite outputs, lse not
  below the largest visible score's lower bound ln(1), rows of dK summing to
  0 and rows of dV summing to the rows of dO (within tolerance).
"""

import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_util import (TOL_GRAD_REL, assert_fwd_close, assert_grads_close, f64, require_gpu, run_bwd,
                            run_fwd)

pytestmark = pytest.mark.gpu

FULL = [workloads.TINY, workloads.GPT2_MEDIUM, workloads.LLAMA7B_LAYER, workloads.LLAMA7B_LAYER_NC,
        workloads.LONG_SEQ]
SWEEP = workloads.sweep()


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _check_workload(w, bwd_slices=1):
    q, k, v, do = workloads.workload_inputs(w)
    scale = w.scale
    qg, kg, vg, o, lse = run_fwd(q, k, v, scale, w.causal)
    BH = w.B * w.H
    picks = [(0, 0), (w.B - 1, w.H - 1)] if BH > 1 else [(0, 0)]
    for b, h in picks:
        o_ref, lse_ref = oracle.attention_forward_head_rows(
            q[b, h].double().numpy(), k[b, h].double().numpy(), v[b, h].double().numpy(),
            np.arange(w.N), scale, w.causal)
        assert_fwd_close(o[b, h], lse[b, h], o_ref, lse_ref, f"{w.name} fwd slice {(b, h)}")
    assert bool(torch.isfinite(o.float()).all()) and bool(torch.isfinite(lse).all())
    if not w.backward:
        return
    dq, dk, dv = run_bwd(qg, kg, vg, o, lse, do, scale, w.causal)
    for b, h in picks[:bwd_slices]:
        dq_r, dk_r, dv_r, _, _, _ = oracle.attention_backward_head(
            q[b, h].double().numpy(), k[b, h].double().numpy(), v[b, h].double().numpy(),
            do[b, h].double().numpy(), scale, w.causal)
        assert_grads_close((dq[b, h], dk[b, h], dv[b, h]), (dq_r, dk_r, dv_r), f"{w.name} bwd slice {(b, h)}")
    # identities on every slice: sum_j dK_j = 0, sum_j dV_j = sum_i dO_i
    dk_sum = dk.double().sum(dim=2)
    dv_sum = dv.double().sum(dim=2)
    do_sum = do.cuda().double().sum(dim=2)
    dk_scale = dk.double().abs().amax().item()
    dv_scale = dv.double().abs().amax().item()
    # each column sum adds N bf16-rounded terms: allow N * half-ulp of the largest entry on top
    slack = w.N * 2.0 ** -8
    assert dk_sum.abs().amax().item() <= TOL_GRAD_REL * dk_scale * slack + 1e-3
    assert (dv_sum - do_sum).abs().amax().item() <= TOL_GRAD_REL * dv_scale * slack + 1e-3
    for t in (dq, dk, dv):
        assert bool(torch.isfinite(t.float()).all())


@pytest.mark.parametrize("w", FULL, ids=[w.name for w in FULL])
def test_workload_full_size(w):
    _check_workload(w)


@pytest.mark.parametrize("w", SWEEP, ids=[w.name for w in SWEEP])
def test_sweep_full_size(w):
    _check_workload(w)


@pytest.mark.parametrize("w", [workloads.GPT2_MEDIUM, workloads.LONG_SEQ], ids=lambda w: w.name)
def test_zero_queries_closed_form_all_slices(w):
    """Q = 0 gives uniform attention over visible keys on every slice at full size."""
    _, k, v, _ = workloads.workload_inputs(w)
    q = torch.zeros_like(k)
    _, _, _, o, lse = run_fwd(q, k, v, w.scale, w.causal)
    vg = v.cuda().double()
    n = w.N
    if w.causal:
        cnt = torch.arange(1, n + 1, device="cuda", dtype=torch.float64)
        o_ref = torch.cumsum(vg, dim=2) / cnt[None, None, :, None]
        lse_ref = torch.log(cnt)[None, None, :]
    else:
        o_ref = vg.mean(dim=2, keepdim=True)
        lse_ref = torch.full((1, 1, 1), math.log(n), device="cuda", dtype=torch.float64)
    assert (o.double() - o_ref).abs().amax().item() <= 1e-2
    assert (lse.double() - lse_ref).abs().amax().item() <= 1e-3

"""Helpers shared by the GPU tests: run the library, compare with the oracle."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import exact_io_aware_31_gb300 as fa
from exact_io_aware_31_gb300 import build

# Tolerances of GPU vs oracle on the same seeded bf16 inputs:
#   O max-abs 1e-2, lse max-abs 1e-3, each gradient max-abs <= 2e-2 * max|gradient_ref|.
TOL_O = 1e-2
TOL_LSE = 1e-3
TOL_GRAD_REL = 2e-2


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    fa.load_library()


def run_fwd(q, k, v, scale, causal):
    qg, kg, vg = (t.cuda() for t in (q, k, v))
    o, lse = fa.forward(qg, kg, vg, scale, causal)
    assert fa.fa_get_device_status(torch.cuda.current_stream().cuda_stream) == fa.FA_OK
    return qg, kg, vg, o, lse


def run_bwd(qg, kg, vg, o, lse, do, scale, causal):
    dq, dk, dv = fa.backward(qg, kg, vg, o, lse, do.cuda(), scale, causal)
    assert fa.fa_get_device_status(torch.cuda.current_stream().cuda_stream) == fa.FA_OK
    return dq, dk, dv


def f64(t):
    return t.detach().double().cpu().numpy()


def assert_fwd_close(o, lse, o_ref, lse_ref, what="", o_rel=0.0):
    """O within TOL_O (+ o_rel * |O_ref| elementwise), lse within TOL_LSE.

    ``o_rel`` is 0 for N(0, 1) inputs.  Stress inputs whose rows are dominated
    by one key produce |O| up to ~4, where one bf16 ulp of the stored output
    is 2^-6; they pass o_rel = 2^-8 (one bf16 rounding of the output plus one
    of the dominant probability) on top of the absolute bound.
    """
    diff = np.abs(f64(o) - o_ref)
    excess = diff - (TOL_O + o_rel * np.abs(o_ref))
    eo = float(diff.max()) if o_ref.size else 0.0
    el = float(np.abs(f64(lse) - lse_ref).max()) if lse_ref.size else 0.0
    assert np.all(np.isfinite(f64(o))), what
    assert (not o_ref.size) or float(excess.max()) <= 0.0, f"{what} O max abs error {eo}"
    assert el <= TOL_LSE, f"{what} lse max abs error {el}"
    return eo, el


def assert_grads_close(grads, refs, what="", extra=None):
    """Each gradient within 2e-2 of its reference's max-abs.

    Where a reference vanishes identically (N = 1 gives dQ = dK = 0 exactly),
    the bound uses the largest reference gradient of the call instead.
    ``extra`` optionally adds an elementwise allowance per gradient (see
    :func:`d_rounding_allowance`).
    """
    scale_all = max(float(np.abs(r).max()) for r in refs)
    errs = []
    for idx, (name, g, r) in enumerate(zip(("dq", "dk", "dv"), grads, refs)):
        gmax = float(np.abs(r).max())
        ref_scale = gmax if gmax > 0 else scale_all
        diff = np.abs(f64(g) - r)
        bound = TOL_GRAD_REL * ref_scale + (extra[idx] if extra is not None else 0.0)
        e = float(diff.max())
        assert np.all(np.isfinite(f64(g))), f"{what} {name} not finite"
        assert float((diff - bound).max()) <= 0.0, f"{what} {name} error {e} vs max|ref| {gmax}"
        errs.append(e / ref_scale)
    return errs


def d_rounding_allowance(q, k, do, o_ref, lse_ref, scale, causal):
    """First-order effect on the gradients of forming D = rowsum(dO * O) from the stored bf16 O.

    The method keeps only O (bf16) and lse, so D carries O's rounding:
    |dD_i| <= 2^-9 sum_c |dO_ic O_ic|.  It enters dS_ij = P_ij (dP_ij - D_i)
    unchanged, hence dQ_i by scale * dD_i * sum_j P_ij |K_j| and dK_j by
    scale * sum_i P_ij dD_i |Q_i|; dV does not see D.  Negligible for N(0, 1)
    inputs, it matters where one key dominates a row (dP_ij - D_i cancels).
    """
    B, H, N, d = q.shape
    exq = np.zeros((B, H, N, d))
    exk = np.zeros((B, H, N, d))
    for b in range(B):
        for h in range(H):
            s = scale * (q[b, h] @ k[b, h].T)
            if causal:
                s[np.triu_indices(N, 1)] = -np.inf
            p = np.exp(s - lse_ref[b, h][:, None])
            dD = 2.0 ** -9 * np.sum(np.abs(do[b, h] * o_ref[b, h]), axis=1)
            exq[b, h] = scale * dD[:, None] * (p @ np.abs(k[b, h]))
            exk[b, h] = scale * (p.T @ (dD[:, None] * np.abs(q[b, h])))
    return (exq, exk, 0.0)

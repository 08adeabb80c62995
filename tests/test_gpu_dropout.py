"""Dropout forward / backward vs the dropout oracle (needs a GB300).

* The keep mask, exactly: with V the identity (N = d, no mask) row i of O is
  P_i o M_i / (1 - p), so O is exactly 0 where the mask drops and positive
  where it keeps; the zero pattern must equal the oracle's mask bit for bit.
* O, lse and the three gradients against the oracle, several shapes, both
  masks and head dims, rates 0.1 .. 0.5.  Kept probabilities are amplified by
  1 / (1 - p), so the O bound is 1e-2 / (1 - p); gradients keep the usual
  2e-2 of max|ref|.
* p = 0 gives the plain forward bit for bit and the plain backward within
  tolerance (its dQ adds in a run-dependent order).
"""

import math

import numpy as np
import pytest
import torch

import exact_io_aware_31_gb300 as fa
from oracle import dropout as dr
from tests.gpu_util import TOL_LSE, TOL_O, assert_grads_close, f64, require_gpu
from workloads import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _fwd(q, k, v, scale, causal, p, seed, off):
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), device="cuda", dtype=torch.float32)
    s = torch.cuda.current_stream().cuda_stream
    assert fa.fa_fwd_dropout(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
                             scale, int(causal), p, seed, off, s) == fa.FA_OK
    assert fa.fa_get_device_status(s) == fa.FA_OK
    return o, lse


def _bwd(q, k, v, o, lse, do, scale, causal, p, seed, off):
    B, H, N, d = q.shape
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert fa.fa_bwd_dropout(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                             dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, scale, int(causal), p, seed, off,
                             ws.data_ptr(), ws.numel(), s) == fa.FA_OK
    assert fa.fa_get_device_status(s) == fa.FA_OK
    return dq, dk, dv


@pytest.mark.parametrize("d,p", [(64, 0.1), (64, 0.5), (128, 0.25)])
def test_keep_mask_bit_exact(d, p):
    B, H, N = 2, 3, d
    q, k, _, _ = make_inputs(B, H, N, d, seed=7000 + d)
    v = torch.eye(d, dtype=torch.bfloat16).expand(B, H, N, d).contiguous()
    seed, off = 0x1234_5678_9ABC_DEF0, 11
    o, _ = _fwd(q.cuda(), k.cuda(), v.cuda(), 1.0 / math.sqrt(d), False, p, seed, off)
    kept = (o.float() != 0).cpu().numpy()
    mask = dr.dropout_keep_mask(B, H, N, N, p, seed, off)
    assert np.array_equal(kept, mask)
    assert abs(mask.mean() - (1 - p)) <= 5 * math.sqrt(p * (1 - p) / mask.size)


CASES = [(1, 2, 256, 64, False, 0.1), (1, 2, 256, 128, True, 0.2), (2, 3, 300, 64, True, 0.5),
         (1, 1, 129, 128, False, 0.3), (1, 2, 1000, 64, True, 0.1), (2, 1, 513, 128, True, 0.15),
         # d = 64 forward with the second MMA issuer
         (1, 1, 1100, 64, False, 0.2), (1, 1, 2100, 64, True, 0.1)]


@pytest.mark.parametrize("B,H,N,d,causal,p", CASES,
                         ids=[f"b{b}h{h}n{n}d{d}{'c' if c else ''}p{p}" for b, h, n, d, c, p in CASES])
def test_dropout_matches_oracle(B, H, N, d, causal, p):
    scale = 1.0 / math.sqrt(d)
    seed, off = 4242 + N, 3
    q, k, v, do = make_inputs(B, H, N, d, seed=7100 + N + d)
    qg, kg, vg, dog = (t.cuda() for t in (q, k, v, do))
    o, lse = _fwd(qg, kg, vg, scale, causal, p, seed, off)
    qd, kd, vd, dod = (t.double().numpy() for t in (q, k, v, do))
    o_ref, lse_ref, _ = dr.attention_forward_dropout(qd, kd, vd, scale, causal, p, seed, off)
    assert float(np.abs(f64(o) - o_ref).max()) <= TOL_O / (1 - p)
    assert float(np.abs(f64(lse) - lse_ref).max()) <= TOL_LSE
    grads = _bwd(qg, kg, vg, o, lse, dog, scale, causal, p, seed, off)
    g_ref = dr.attention_backward_dropout(qd, kd, vd, dod, scale, causal, p, seed, off)
    assert_grads_close(grads, g_ref, f"dropout {(B, H, N, d, causal, p)}")


def test_zero_rate_is_the_plain_path():
    q, k, v, do = (t.cuda() for t in make_inputs(1, 2, 300, 64, seed=71))
    o0, l0 = fa.forward(q, k, v, 0.125, True)
    o1, l1 = _fwd(q, k, v, 0.125, True, 0.0, 5, 0)
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    g0 = fa.backward(q, k, v, o0, l0, do, 0.125, True)
    g1 = _bwd(q, k, v, o1, l1, do, 0.125, True, 0.0, 5, 0)
    for a, b in zip(g0, g1):
        assert float((a.float() - b.float()).abs().max()) <= 2e-2 * float(a.float().abs().max())

"""Pins of the oracle's analytic backward (CPU only).

The pages give no gradient formulas (only that the backward recomputes S and P
from Q, K, V and the saved statistics: blog.teqners.com, "The backward pass:
recompute instead of read").  The oracle's chain-rule gradients are pinned by:

* central finite differences of L = sum(O * dO) in fp64 on tiny inputs;
* PyTorch autograd through fp64 ``scaled_dot_product_attention`` on CPU;
* identities: sum_j dS_ij = 0 so sum_j dK_j = 0; sum_j dV_j = sum_i dO_i;
  D = rowsum(dO * O) = rowsum(P * dP).
"""

import math

import numpy as np
import pytest
import torch

from oracle import attention_backward, attention_backward_head, attention_backward_head_rows, attention_forward


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).normal(scale=scale, size=shape)


def _loss(q, k, v, do, scale, causal):
    o, _ = attention_forward(q, k, v, scale, causal)
    return float(np.sum(o * do))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,d", [(1, 4), (3, 4), (8, 8), (16, 4)])
def test_gradients_match_central_differences(n, d, causal):
    q, k, v, do = (_rand((1, 1, n, d), s) for s in (101, 102, 103, 104))
    scale = 1.0 / math.sqrt(d)
    dq, dk, dv, _ = attention_backward(q, k, v, do, scale, causal)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = dict(q=q, k=k, v=v)
            args_m = dict(q=q, k=k, v=v)
            args_p[name], args_m[name] = xp, xm
            num[idx] = (_loss(args_p["q"], args_p["k"], args_p["v"], do, scale, causal)
                        - _loss(args_m["q"], args_m["k"], args_m["v"], do, scale, causal)) / (2 * h)
        err = np.max(np.abs(num - g)) / max(1e-12, np.max(np.abs(g)))
        if np.max(np.abs(g)) < 1e-12:           # e.g. dk with a single key is exactly 0
            assert np.max(np.abs(num)) < 1e-8, name
        else:
            assert err < 1e-6, (name, err)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,d", [(5, 8), (70, 16), (129, 32)])
def test_gradients_match_torch_autograd_fp64(n, d, causal):
    q, k, v, do = (_rand((2, 2, n, d), s) for s in (111, 112, 113, 114))
    scale = 1.0 / math.sqrt(d)
    dq, dk, dv, _ = attention_backward(q, k, v, do, scale, causal, row_block=48)
    tq, tk, tv = (torch.from_numpy(a.copy()).requires_grad_(True) for a in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    out.backward(torch.from_numpy(do))
    for g, t in ((dq, tq), (dk, tk), (dv, tv)):
        assert np.max(np.abs(g - t.grad.numpy())) < 1e-11


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_identities(causal):
    n, d = 64, 16
    q, k, v, do = (_rand((n, d), s, 1.5) for s in (121, 122, 123, 124))
    scale = 0.3
    dq, dk, dv, D, o, lse = attention_backward_head(q, k, v, do, scale, causal)
    assert np.max(np.abs(dk.sum(axis=0))) < 1e-11
    assert np.max(np.abs(dv.sum(axis=0) - do.sum(axis=0))) < 1e-11
    s = scale * (q @ k.T)
    if causal:
        s[np.triu_indices(n, 1)] = -np.inf
    p = np.exp(s - lse[:, None])
    dp = do @ v.T
    assert np.max(np.abs(D - np.sum(p * dp, axis=1))) < 1e-12
    ds = p * (dp - D[:, None])
    assert np.max(np.abs(ds.sum(axis=1))) < 1e-12


def test_batched_backward_equals_per_head():
    q, k, v, do = (_rand((2, 2, 20, 8), s) for s in (131, 132, 133, 134))
    dq, dk, dv, D = attention_backward(q, k, v, do, 0.5, True)
    for b in range(2):
        for h in range(2):
            hq, hk, hv, hD, _, _ = attention_backward_head(q[b, h], k[b, h], v[b, h], do[b, h], 0.5, True)
            assert np.array_equal(hq, dq[b, h]) and np.array_equal(hk, dk[b, h])
            assert np.array_equal(hv, dv[b, h]) and np.array_equal(hD, D[b, h])


@pytest.mark.parametrize("causal", [False, True])
def test_row_contributions_match_torch_autograd(causal):
    """dQ rows are autograd's rows; dK, dV contributions summed over a partition of the rows are autograd's."""
    n, d = 150, 16
    q, k, v, do = (_rand((n, d), s) for s in (141, 142, 143, 144))
    scale = 0.4
    tq, tk, tv = (torch.from_numpy(a.copy()).requires_grad_(True) for a in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(tq[None, None], tk[None, None], tv[None, None],
                                                           is_causal=causal, scale=scale)
    out.backward(torch.from_numpy(do)[None, None])
    dk_sum, dv_sum = np.zeros_like(k), np.zeros_like(v)
    order = np.random.default_rng(5).permutation(n)
    for part in (order[:37], order[37:90], order[90:]):
        dq_r, dk_p, dv_p = attention_backward_head_rows(q, k, v, do, part, scale, causal)
        assert np.max(np.abs(dq_r - tq.grad.numpy()[part])) < 1e-11
        dk_sum += dk_p
        dv_sum += dv_p
    assert np.max(np.abs(dk_sum - tk.grad.numpy())) < 1e-11
    assert np.max(np.abs(dv_sum - tv.grad.numpy())) < 1e-11


"""Pins of the oracle's forward (CPU only).

Each test ties ``oracle.attention_forward`` (three-pass) or
``oracle.attention_forward_tiled`` (online softmax + rescaled accumulator) to
something other than itself:

* PyTorch's fp64 ``scaled_dot_product_attention`` on CPU (a library routine
  computing the same definition) and SciPy's ``logsumexp``;
* a scalar pure-Python brute force that normalises plain exp weights without
  any max subtraction (a different route to the same numbers);
* closed forms: Q = 0 gives uniform attention, N = 1 returns V, causal row 0
  returns V_0, constant V rows return that row, a dominating key returns its V;
* invariants: rows of P sum to 1, a shift of every key moves every score of a
  row by the same constant, joint permutation of keys and values, scale vs Q;
* the exactness check of lensaml.com "FlashAttention" Step 6 (d = 8, 4 tiles
  of 4 keys agree with standard attention to rounding, printed as 2.2e-16).
"""

import math

import numpy as np
import pytest
import scipy.special
import torch

from oracle import (attention_forward, attention_forward_head_rows,
                    attention_forward_tiled, scores, softmax_three_pass)


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).normal(scale=scale, size=shape)


def _sdpa(q, k, v, scale, causal):
    t = [torch.from_numpy(np.ascontiguousarray(a)) for a in (q, k, v)]
    return torch.nn.functional.scaled_dot_product_attention(
        t[0], t[1], t[2], is_causal=causal, scale=scale).numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,d", [(1, 4), (7, 8), (64, 16), (130, 64)])
def test_forward_matches_torch_sdpa_fp64(n, d, causal):
    q, k, v = (_rand((2, 3, n, d), s) for s in (1, 2, 3))
    scale = 1.0 / math.sqrt(d)
    o, lse = attention_forward(q, k, v, scale, causal)
    assert np.max(np.abs(o - _sdpa(q, k, v, scale, causal))) < 1e-12
    for b in range(2):
        for h in range(3):
            s = scale * (q[b, h] @ k[b, h].T)
            if causal:
                s[np.triu_indices(n, 1)] = -np.inf
            ref = scipy.special.logsumexp(s, axis=1)
            assert np.max(np.abs(lse[b, h] - ref)) < 1e-12


def test_forward_matches_scalar_brute_force():
    rng = np.random.default_rng(11)
    n, d = 6, 3
    q, k, v = (rng.normal(size=(1, 1, n, d)) for _ in range(3))
    scale = 0.7
    for causal in (False, True):
        o, lse = attention_forward(q, k, v, scale, causal)
        for i in range(n):
            w, total = [], 0.0
            for j in range(n):
                if causal and j > i:
                    w.append(0.0)
                    continue
                dot = sum(q[0, 0, i, c] * k[0, 0, j, c] for c in range(d))
                e = math.exp(scale * dot)               # no max subtraction
                w.append(e)
                total += e
            for c in range(d):
                ref = sum(w[j] * v[0, 0, j, c] for j in range(n)) / total
                assert abs(o[0, 0, i, c] - ref) < 1e-13
            assert abs(lse[0, 0, i] - math.log(total)) < 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_give_uniform_attention(causal):
    n, d = 37, 8
    q = np.zeros((1, 1, n, d))
    k, v = _rand((1, 1, n, d), 5), _rand((1, 1, n, d), 6)
    o, lse = attention_forward(q, k, v, 0.3, causal)
    for i in range(n):
        vis = i + 1 if causal else n
        assert np.allclose(o[0, 0, i], v[0, 0, :vis].mean(axis=0), atol=1e-14)
        assert abs(lse[0, 0, i] - math.log(vis)) < 1e-14


def test_single_key_returns_v():
    q, k, v = (_rand((2, 2, 1, 16), s) for s in (1, 2, 3))
    o, lse = attention_forward(q, k, v, 0.25, False)
    assert np.array_equal(o, v)
    assert np.allclose(lse, 0.25 * np.sum(q * k, axis=-1), atol=1e-15)


def test_causal_first_row_returns_v0():
    q, k, v = (_rand((1, 2, 20, 8), s) for s in (4, 5, 6))
    o, lse = attention_forward(q, k, v, 0.5, True)
    assert np.array_equal(o[:, :, 0], v[:, :, 0])
    assert np.allclose(lse[:, :, 0], 0.5 * np.sum(q[:, :, 0] * k[:, :, 0], axis=-1), atol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_value_rows_return_that_row(causal):
    n, d = 50, 8
    q, k = _rand((1, 1, n, d), 8, 3.0), _rand((1, 1, n, d), 9, 3.0)
    c = np.linspace(-2, 2, d)
    v = np.broadcast_to(c, (1, 1, n, d)).copy()
    o, _ = attention_forward(q, k, v, 1.0, causal)
    assert np.max(np.abs(o - c)) < 1e-13


def test_dominating_key_selects_its_value():
    n, d = 12, 4
    q = np.zeros((1, 1, n, d))
    q[..., 0] = 1.0
    k = np.zeros((1, 1, n, d))
    k[0, 0, 5, 0] = 200.0                 # score 200 for key 5, 0 for the rest
    v = _rand((1, 1, n, d), 10)
    o, _ = attention_forward(q, k, v, 1.0, False)
    assert np.allclose(o[0, 0], v[0, 0, 5][None, :], atol=1e-80)


@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows_sum_to_one(causal):
    q, k = _rand((40, 8), 12, 2.0), _rand((40, 8), 13, 2.0)
    s = scores(q, k, 0.9, causal)
    p, _, _ = softmax_three_pass(s)
    assert np.max(np.abs(p.sum(axis=1) - 1.0)) < 1e-14
    if causal:
        assert np.all(p[np.triu_indices(40, 1)] == 0.0)


@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_moves_lse_by_row_constant(causal):
    n, d = 33, 16
    q, k, v = (_rand((1, 2, n, d), s) for s in (21, 22, 23))
    u = _rand((d,), 24)
    scale = 0.4
    o1, lse1 = attention_forward(q, k, v, scale, causal)
    o2, lse2 = attention_forward(q, k + u, v, scale, causal)
    assert np.max(np.abs(o1 - o2)) < 1e-12
    assert np.max(np.abs((lse2 - lse1) - scale * (q @ u))) < 1e-12


def test_joint_key_value_permutation_noncausal():
    n, d = 29, 8
    q, k, v = (_rand((1, 1, n, d), s) for s in (31, 32, 33))
    perm = np.random.default_rng(34).permutation(n)
    o1, lse1 = attention_forward(q, k, v, 0.35, False)
    o2, lse2 = attention_forward(q, k[:, :, perm], v[:, :, perm], 0.35, False)
    assert np.max(np.abs(o1 - o2)) < 1e-13
    assert np.max(np.abs(lse1 - lse2)) < 1e-13


def test_scale_equals_scaled_queries():
    q, k, v = (_rand((1, 1, 24, 8), s) for s in (41, 42, 43))
    o1, lse1 = attention_forward(q, k, v, 0.125, True)
    o2, lse2 = attention_forward(0.125 * q, k, v, 1.0, True)
    assert np.max(np.abs(o1 - o2)) < 1e-13
    assert np.max(np.abs(lse1 - lse2)) < 1e-13


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("block", [1, 3, 16, 64, 128])
def test_tiled_online_equals_three_pass(block, causal):
    # the tolerance this library holds its two oracle forms to: 1e-12
    q, k, v = (_rand((1, 2, 150, 32), s, 2.0) for s in (51, 52, 53))
    o3, lse3 = attention_forward(q, k, v, 1 / math.sqrt(32), causal)
    ot, lset = attention_forward_tiled(q, k, v, 1 / math.sqrt(32), causal, block)
    assert np.max(np.abs(o3 - ot)) < 1e-12
    assert np.max(np.abs(lse3 - lset)) < 1e-12


def test_exactness_check_shape_of_step6():
    # lensaml.com Step 6: d = 8, keys split into 4 tiles of up to 4 keys; the tiled
    # output differs from standard attention by rounding only (2.2e-16 printed).
    q, k, v = (_rand((1, 1, 16, 8), s) for s in (61, 62, 63))
    o3, _ = attention_forward(q, k, v, 1 / math.sqrt(8), False)
    ot, _ = attention_forward_tiled(q, k, v, 1 / math.sqrt(8), False, 4)
    assert np.max(np.abs(o3 - ot)) < 4 * np.finfo(np.float64).eps


def test_tiled_handles_large_score_range():
    # rows whose maximum grows block after block exercise every rescale step
    n, d = 96, 8
    q = _rand((1, 1, n, d), 71, 8.0)
    k = np.sort(_rand((1, 1, n, d), 72, 8.0), axis=2)
    v = _rand((1, 1, n, d), 73)
    o3, lse3 = attention_forward(q, k, v, 1.0, True)
    ot, lset = attention_forward_tiled(q, k, v, 1.0, True, 7)
    assert np.all(np.isfinite(o3))
    assert np.max(np.abs(o3 - ot)) < 1e-12
    assert np.max(np.abs(lse3 - lset)) < 1e-10


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_rows_equal_full_forward(causal):
    q, k, v = (_rand((1, 1, 90, 16), s) for s in (81, 82, 83))
    o, lse = attention_forward(q, k, v, 0.25, causal, row_block=32)
    rows = np.array([0, 1, 31, 32, 33, 89])
    orow, lrow = attention_forward_head_rows(q[0, 0], k[0, 0], v[0, 0], rows, 0.25, causal)
    assert np.max(np.abs(orow - o[0, 0, rows])) < 1e-15
    assert np.max(np.abs(lrow - lse[0, 0, rows])) < 1e-15


@pytest.mark.parametrize("causal", [False, True])
def test_negative_scale_matches_sdpa_and_negated_queries(causal):
    """A negative scale is the positive one on negated queries; without a mask torch's SDPA agrees.

    (torch's CPU SDPA returns NaN for a negative scale under its causal mask:
    it masks before scaling, so a masked -inf times the scale becomes +inf.
    The scale multiplies Q K^T before the mask here.)
    """
    q, k, v = (_rand((1, 2, 40, 8), s) for s in (51, 52, 53))
    o1, lse1 = attention_forward(q, k, v, -0.3, causal)
    o2, lse2 = attention_forward(-q, k, v, 0.3, causal)
    assert np.max(np.abs(o1 - o2)) < 1e-13 and np.max(np.abs(lse1 - lse2)) < 1e-13
    if not causal:
        assert np.max(np.abs(o1 - _sdpa(q, k, v, -0.3, causal))) < 1e-12

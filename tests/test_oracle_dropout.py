"""Pins of the dropout oracle (CPU).

* Philox4x32-10 reproduces the generator's published known-answer vectors
  (tests/golden/philox4x32_10_kat.txt); a wrong multiplier, a missing key
  bump or one round short fails them.
* The keep mask: keep fraction within 5 standard deviations of 1 - p; the same
  (seed, offset) gives the same mask, another offset or seed another one; p = 0
  keeps everything.
* p = 0 reduces the dropout forward and backward to the plain oracle exactly.
* The backward matches central finite differences of the dropout forward
  (fixed mask) on tiny inputs, and D = rowsum(dO o O) = rowsum(P o dP).
"""

import os

import numpy as np
import pytest

import oracle
from oracle import dropout as dr

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def _kats():
    out = []
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        w = [int(x, 16) for x in line.split()]
        out.append((w[0:4], w[4:6], w[6:10]))
    return out


def test_philox_known_answers():
    for ctr, key, exp in _kats():
        got = [int(x) for x in dr.philox4x32(*ctr, *key)]
        assert got == exp


def test_philox_planted_mistakes_fail_the_known_answers():
    ctr, key, exp = _kats()[2]
    assert [int(x) for x in dr.philox4x32(*ctr, *key, rounds=9)] != exp
    saved = dr._W0
    try:
        dr._W0 = 0
        assert [int(x) for x in dr.philox4x32(*ctr, *key)] != exp
    finally:
        dr._W0 = saved
    saved = dr._M0
    try:
        dr._M0 = 0xD2511F55
        assert [int(x) for x in dr.philox4x32(*ctr, *key)] != exp
    finally:
        dr._M0 = saved


@pytest.mark.parametrize("p", [0.1, 0.25, 0.5])
def test_keep_fraction(p):
    m = dr.dropout_keep_mask(1, 2, 128, 256, p, seed=1234, offset=7)
    n = m.size
    frac = m.mean()
    assert abs(frac - (1 - p)) <= 5 * np.sqrt(p * (1 - p) / n)


def test_mask_is_a_function_of_seed_and_offset():
    a = dr.dropout_keep_mask(2, 2, 64, 64, 0.3, seed=99, offset=0)
    assert np.array_equal(a, dr.dropout_keep_mask(2, 2, 64, 64, 0.3, seed=99, offset=0))
    assert not np.array_equal(a, dr.dropout_keep_mask(2, 2, 64, 64, 0.3, seed=99, offset=1))
    assert not np.array_equal(a, dr.dropout_keep_mask(2, 2, 64, 64, 0.3, seed=98, offset=0))
    assert dr.dropout_keep_mask(1, 1, 16, 16, 0.0, seed=5, offset=0).all()
    assert dr.keep_threshold(0.0) == 0 and dr.keep_threshold(1.0) == 0xFFFFFFFF


@pytest.mark.parametrize("causal", [False, True])
def test_zero_rate_is_the_plain_oracle(causal):
    rng = np.random.default_rng(1)
    q, k, v, do = (rng.standard_normal((1, 2, 40, 8)) for _ in range(4))
    o, lse, _ = dr.attention_forward_dropout(q, k, v, 0.3, causal, 0.0, seed=3, offset=0)
    o_ref, lse_ref = oracle.attention_forward(q, k, v, 0.3, causal)
    assert np.max(np.abs(o - o_ref)) < 1e-14 and np.max(np.abs(lse - lse_ref)) < 1e-14
    g = dr.attention_backward_dropout(q, k, v, do, 0.3, causal, 0.0, seed=3, offset=0)
    g_ref = oracle.attention_backward(q, k, v, do, 0.3, causal)[:3]
    for a, b in zip(g, g_ref):
        assert np.max(np.abs(a - b)) < 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_finite_differences(causal):
    rng = np.random.default_rng(2)
    B, H, N, d = 1, 1, 8, 4
    q, k, v, do = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    p, seed, off, scale = 0.3, 11, 2, 0.7

    def loss(qq, kk, vv):
        return float(np.sum(dr.attention_forward_dropout(qq, kk, vv, scale, causal, p, seed, off)[0] * do))

    dq, dk, dv = dr.attention_backward_dropout(q, k, v, do, scale, causal, p, seed, off)
    h = 1e-6
    for t, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(t)
        for idx in np.ndindex(t.shape):
            t[idx] += h
            lp = loss(q, k, v)
            t[idx] -= 2 * h
            lm = loss(q, k, v)
            t[idx] += h
            num[idx] = (lp - lm) / (2 * h)
        assert np.max(np.abs(num - g)) <= 1e-6 * max(1.0, np.max(np.abs(g)))


def test_dsum_identity_with_dropout():
    rng = np.random.default_rng(4)
    q, k, v, do = (rng.standard_normal((1, 1, 32, 8)) for _ in range(4))
    o, _, m = dr.attention_forward_dropout(q, k, v, 0.5, True, 0.2, seed=8, offset=1)
    s = oracle.scores(q[0, 0], k[0, 0], 0.5, True)
    pr, _, _ = oracle.softmax_three_pass(s)
    dp = (do[0, 0] @ v[0, 0].T) * m[0, 0] / 0.8
    assert np.max(np.abs(np.sum(pr * dp, axis=1) - np.sum(do[0, 0] * o[0, 0], axis=1))) < 1e-12

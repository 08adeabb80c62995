"""Pins of the split-KV (decode) oracle, on the CPU.

Each check ties ``oracle.decode`` to something other than itself:
* a pure-Python loop over the visibility rule (brute force, tiny sizes);
* PyTorch's fp64 ``scaled_dot_product_attention`` with an explicit boolean mask;
* closed forms: Q = 0 gives the mean of the visible values and ln(#visible);
  one query under the bottom-right mask sees every key;
* Nq = Nk reduces to the square oracle (itself pinned elsewhere);
* merging per-split partials reproduces the full result to 1e-12, for even,
  uneven, empty and fully masked splits ([T] rescale rule);
* planted mistakes in the merge are caught.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle.decode import attention_forward_rect, merge_partials, split_bounds, split_partials


def _rand(shape, rng):
    return rng.standard_normal(shape)


def _brute(q, k, v, scale, causal):
    B, H, nq, d = q.shape
    nk = k.shape[2]
    o = np.zeros((B, H, nq, v.shape[3]))
    lse = np.zeros((B, H, nq))
    for b in range(B):
        for h in range(H):
            for i in range(nq):
                vis = [j for j in range(nk) if (not causal) or j <= i + nk - nq]
                s = [scale * sum(q[b, h, i, c] * k[b, h, j, c] for c in range(d)) for j in vis]
                m = max(s)
                e = [math.exp(x - m) for x in s]
                tot = sum(e)
                for jj, j in enumerate(vis):
                    o[b, h, i] += e[jj] / tot * v[b, h, j]
                lse[b, h, i] = m + math.log(tot)
    return o, lse


@pytest.mark.parametrize("nq,nk,causal", [(1, 5, True), (1, 5, False), (3, 7, True), (3, 7, False), (4, 4, True),
                                           (2, 9, True)])
def test_rect_matches_brute_force(nq, nk, causal):
    rng = np.random.default_rng(nq * 31 + nk)
    q, k, v = _rand((1, 2, nq, 4), rng), _rand((1, 2, nk, 4), rng), _rand((1, 2, nk, 3), rng)
    o, lse = attention_forward_rect(q, k, v, 0.7, causal)
    ob, lb = _brute(q, k, v, 0.7, causal)
    assert np.max(np.abs(o - ob)) < 1e-12
    assert np.max(np.abs(lse - lb)) < 1e-12


@pytest.mark.parametrize("nq,nk,causal", [(1, 300, True), (8, 300, True), (5, 129, False), (16, 16, True)])
def test_rect_matches_torch_sdpa_with_explicit_mask(nq, nk, causal):
    rng = np.random.default_rng(7 + nq + nk)
    q, k, v = _rand((2, 3, nq, 16), rng), _rand((2, 3, nk, 16), rng), _rand((2, 3, nk, 16), rng)
    scale = 0.25
    o, _ = attention_forward_rect(q, k, v, scale, causal)
    i = np.arange(nq)[:, None]
    j = np.arange(nk)[None, :]
    allowed = torch.from_numpy((j <= i + nk - nq) if causal else np.ones((nq, nk), dtype=bool))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), attn_mask=allowed, scale=scale)
    assert np.max(np.abs(o - ref.numpy())) < 1e-12


@pytest.mark.parametrize("causal", [True, False])
def test_rect_zero_queries_closed_form(causal):
    rng = np.random.default_rng(3)
    nq, nk = 6, 50
    q = np.zeros((1, 1, nq, 8))
    k, v = _rand((1, 1, nk, 8), rng), _rand((1, 1, nk, 8), rng)
    o, lse = attention_forward_rect(q, k, v, 0.3, causal)
    for i in range(nq):
        cnt = (i + nk - nq + 1) if causal else nk
        assert np.max(np.abs(o[0, 0, i] - v[0, 0, :cnt].mean(axis=0))) < 1e-12
        assert abs(lse[0, 0, i] - math.log(cnt)) < 1e-12


def test_single_query_causal_sees_every_key():
    rng = np.random.default_rng(5)
    q, k, v = _rand((2, 2, 1, 8), rng), _rand((2, 2, 77, 8), rng), _rand((2, 2, 77, 8), rng)
    a = attention_forward_rect(q, k, v, 0.5, True)
    b = attention_forward_rect(q, k, v, 0.5, False)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_square_case_is_the_square_oracle():
    rng = np.random.default_rng(11)
    q, k, v = _rand((1, 2, 40, 8), rng), _rand((1, 2, 40, 8), rng), _rand((1, 2, 40, 8), rng)
    for causal in (True, False):
        a = attention_forward_rect(q, k, v, 0.4, causal)
        b = oracle.attention_forward(q, k, v, 0.4, causal)
        assert np.max(np.abs(a[0] - b[0])) < 1e-13 and np.max(np.abs(a[1] - b[1])) < 1e-13


def test_split_bounds_cover_the_keys_in_whole_tiles():
    for nk in (1, 127, 128, 129, 1000, 4096):
        for s in (1, 2, 3, 7, 40):
            bounds = split_bounds(nk, s)
            assert len(bounds) == s
            assert bounds[0][0] == 0 and bounds[-1][1] == nk
            for (a0, b0), (a1, b1) in zip(bounds, bounds[1:]):
                assert b0 == a1 or (a1 == b1)          # contiguous (empty splits allowed)
            for a, b in bounds:
                assert a % 128 == 0 and (b == nk or b % 128 == 0 or b == a)


@pytest.mark.parametrize("nq,nk,splits,causal", [(1, 1000, 4, True), (4, 1000, 7, True), (8, 300, 3, True),
                                                  (3, 513, 5, False), (2, 100, 4, True), (8, 130, 2, True)])
def test_merge_of_partials_is_the_full_result(nq, nk, splits, causal):
    rng = np.random.default_rng(nq * 1000 + nk + splits)
    q, k, v = _rand((1, 2, nq, 16), rng), _rand((1, 2, nk, 16), rng), _rand((1, 2, nk, 16), rng)
    q *= 3.0  # wide score rows: the per-split maxima differ a lot
    bounds = split_bounds(nk, splits)
    o_s, lse_s = split_partials(q, k, v, 0.25, causal, bounds)
    o, lse = merge_partials(o_s, lse_s)
    o_ref, lse_ref = attention_forward_rect(q, k, v, 0.25, causal)
    assert np.max(np.abs(o - o_ref)) < 1e-12
    assert np.max(np.abs(lse - lse_ref)) < 1e-12


def test_merge_handles_empty_and_masked_splits():
    # Nq = 8 against 130 keys in 2 splits: split 1 holds keys 128..129, which
    # queries 0..5 cannot see (j <= i + 122); their partial is empty.
    rng = np.random.default_rng(9)
    q, k, v = _rand((1, 1, 8, 8), rng), _rand((1, 1, 130, 8), rng), _rand((1, 1, 130, 8), rng)
    bounds = split_bounds(130, 2)
    o_s, lse_s = split_partials(q, k, v, 0.5, True, bounds)
    assert np.all(np.isneginf(lse_s[1, 0, 0, :6])) and np.all(o_s[1, 0, 0, :6] == 0.0)
    o, lse = merge_partials(o_s, lse_s)
    o_ref, lse_ref = attention_forward_rect(q, k, v, 0.5, True)
    assert np.max(np.abs(o - o_ref)) < 1e-12 and np.max(np.abs(lse - lse_ref)) < 1e-12


def test_planted_merge_mistakes_are_caught():
    rng = np.random.default_rng(13)
    q, k, v = _rand((1, 1, 2, 8), rng) * 3, _rand((1, 1, 600, 8), rng), _rand((1, 1, 600, 8), rng)
    o_s, lse_s = split_partials(q, k, v, 0.5, False, split_bounds(600, 3))
    o_ref, _ = attention_forward_rect(q, k, v, 0.5, False)
    m = np.max(lse_s, axis=0)
    # (a) weights without the rescale to the common maximum, plain average of the partials
    bad_a = o_s.mean(axis=0)
    # (b) a dropped normalisation
    w = np.exp(lse_s - m[None])
    bad_b = np.sum(w[..., None] * o_s, axis=0)
    assert np.max(np.abs(bad_a - o_ref)) > 1e-3
    assert np.max(np.abs(bad_b - o_ref)) > 1e-3

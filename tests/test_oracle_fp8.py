"""Pins of the FP8 (E4M3) oracle (CPU).

* e4m3_decode equals PyTorch's own float8_e4m3fn -> float32 conversion on all
  256 codes (NaN codes in the same places): a wrong bias, mantissa width or
  subnormal rule fails it.
* Points fixed by the format's definition: 1.0, 448 (largest), 2^-6 (smallest
  normal), 2^-9 (smallest subnormal), -2.0, signed zeros, the two NaN codes;
  finite codes increase with the code below the NaN code.
* attention_forward_fp8: moving a factor between scale and a descale changes
  nothing; k_descale = 0 is uniform attention (the mean of the visible V rows)
  with lse = ln(#visible); on exactly representable inputs it is the plain
  oracle on those values.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8


def test_decode_matches_torch_on_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)
    got = fp8.e4m3_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


@pytest.mark.parametrize("code,value", [(0x38, 1.0), (0x7E, 448.0), (0x08, 2.0 ** -6), (0x01, 2.0 ** -9),
                                        (0xC0, -2.0), (0x00, 0.0), (0x3C, 1.5), (0x07, 7 * 2.0 ** -9)])
def test_decode_fixed_points(code, value):
    assert fp8.e4m3_decode(np.array([code], dtype=np.uint8))[0] == value


def test_decode_nan_sign_and_order():
    v = fp8.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert v[0x80] == 0.0 and math.copysign(1.0, v[0x80]) == -1.0
    assert np.all(np.diff(v[:0x7F]) > 0)
    assert np.array_equal(v[0x80:0xFF], -v[:0x7F])


def _codes(rng, shape):
    c = rng.integers(0, 256, size=shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x30  # no NaN inputs
    return c


@pytest.mark.parametrize("causal", [False, True])
def test_descale_moves_into_scale(causal):
    rng = np.random.default_rng(3)
    q8, k8 = _codes(rng, (1, 2, 20, 16)), _codes(rng, (1, 2, 20, 16))
    v = rng.standard_normal((1, 2, 20, 16))
    o1, l1 = fp8.attention_forward_fp8(q8, k8, 0.5, 0.25, v, 0.125, causal)
    o2, l2 = fp8.attention_forward_fp8(q8, k8, 1.0, 1.0, v, 0.125 * 0.125, causal)
    assert np.allclose(o1, o2, rtol=0, atol=1e-12) and np.allclose(l1, l2, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_key_descale_is_uniform_attention(causal):
    rng = np.random.default_rng(4)
    n = 12
    q8, k8 = _codes(rng, (1, 1, n, 8)), _codes(rng, (1, 1, n, 8))
    v = rng.standard_normal((1, 1, n, 8))
    o, lse = fp8.attention_forward_fp8(q8, k8, 1.0, 0.0, v, 0.35, causal)
    for i in range(n):
        vis = i + 1 if causal else n
        assert np.allclose(o[0, 0, i], v[0, 0, :vis].mean(axis=0), atol=1e-12)
        assert abs(lse[0, 0, i] - math.log(vis)) <= 1e-12


def test_representable_inputs_equal_the_plain_oracle():
    rng = np.random.default_rng(5)
    q8, k8 = _codes(rng, (2, 1, 33, 16)), _codes(rng, (2, 1, 33, 16))
    v = rng.standard_normal((2, 1, 33, 16))
    o, lse = fp8.attention_forward_fp8(q8, k8, 0.75, 2.0, v, 0.2, True)
    q = torch.from_numpy(q8).view(torch.float8_e4m3fn).to(torch.float64).numpy() * 0.75
    k = torch.from_numpy(k8).view(torch.float8_e4m3fn).to(torch.float64).numpy() * 2.0
    o_ref, lse_ref = oracle.attention_forward(q, k, v, 0.2, True)
    assert np.allclose(o, o_ref, rtol=0, atol=1e-12) and np.allclose(lse, lse_ref, rtol=0, atol=1e-12)


def test_fp8_input_generator_codes():
    """The seeded E4M3 inputs the GPU tests and the bench share: no NaN codes,
    the largest |x| lands on code 448, and every decoded value is x rounded to
    E4M3 (relative error <= 2^-4 in the normal range, absolute <= 2^-10 times
    the descale below it)."""
    import workloads
    q8, k8, qs, ks, v = workloads.make_fp8_inputs(1, 2, 300, 128, seed=11, stress="wide")
    q, k, _, _ = workloads.make_inputs(1, 2, 300, 128, seed=11, stress="wide")
    assert v.dtype == torch.bfloat16 and q8.dtype == torch.uint8 and k8.dtype == torch.uint8
    for codes, x, ds in ((q8, q, qs), (k8, k, ks)):
        c = codes.numpy()
        assert not np.any((c & 0x7F) == 0x7F)
        dec = fp8.e4m3_decode(c)
        xs = x.double().numpy() / ds
        assert np.abs(dec).max() == 448.0
        normal = np.abs(xs) >= 2.0 ** -6
        assert np.all(np.abs(dec[normal] - xs[normal]) <= 2.0 ** -4 * np.abs(xs[normal]))
        assert np.all(np.abs(dec[~normal] - xs[~normal]) <= 2.0 ** -10)

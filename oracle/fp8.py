"""Attention with FP8 (E4M3) queries and keys: plain fp64 reference.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): slow, obvious, CPU.

[L] "Key ideas": FlashAttention-3 adds FP8 (on Hopper); the pages give no
format, scaling or placement.  Readings:

* The format is the 8-bit "E4M3" floating point of the OCP FP8 specification
  (the variant without infinities): 1 sign bit, 4 exponent bits with bias 7,
  3 mantissa bits; exponent 0 encodes subnormals m/8 * 2^-6; the codes
  S.1111.111 are NaN; the largest finite magnitude is 448.
* Q and K arrive as E4M3 codes, each tensor with one positive descale factor
  (the real value of an element is its decoded code times the factor).  V
  stays bf16, as do P and O.
* S = scale * q_descale * k_descale * (Q K^T) on the decoded values; the rest
  is the plain forward (three-pass softmax, lse of the scaled scores).

Because both sides consume the same codes, the FP8 rounding of the inputs is
not part of the comparison: the products of two E4M3 values are exact in
fp32, so the plain forward's tolerances apply unchanged.
"""

from __future__ import annotations

import numpy as np

from oracle.attention import attention_forward

__all__ = ["e4m3_decode", "attention_forward_fp8"]


def e4m3_decode(codes):
    """E4M3 codes (uint8 array) -> float64 values (NaN for the NaN codes)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = (c & 0x7).astype(np.float64)
    normal = (1.0 + man / 8.0) * np.exp2(exp.astype(np.float64) - 7.0)
    subnormal = (man / 8.0) * 2.0 ** -6
    val = sign * np.where(exp == 0, subnormal, normal)
    return np.where((c & 0x7F) == 0x7F, np.nan, val)


def attention_forward_fp8(q8, k8, q_descale, k_descale, v, scale, causal):
    """O and lse for E4M3 codes q8, k8 [B, H, N, d] (uint8), descale factors and V."""
    q = e4m3_decode(q8) * float(q_descale)
    k = e4m3_decode(k8) * float(k_descale)
    return attention_forward(q, k, np.asarray(v, dtype=np.float64), scale, causal)

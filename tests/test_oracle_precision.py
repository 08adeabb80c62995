"""Pins of the bf16 precision model (oracle/precision.py) and what it says about the tolerances (CPU only).

* ``round_bf16`` equals PyTorch's own bf16 conversion on values exact in
  fp32 (where that conversion rounds once), ties to even included.
* With every rounding switched off the model is the plain oracle: the lazy
  running maximum changes nothing in exact arithmetic (forward to 1e-12), and
  the backward equals the analytic one.
* On inputs whose rows are dominated by single keys, the roundings alone move
  O past the plain 1e-2 bound while staying inside 1e-2 + 2^-8 |O|: the
  stress allowance the GPU tests use is what bf16 costs (one rounding of the
  output, one of the dominant probability).
"""

import math

import numpy as np
import pytest
import torch

from oracle import attention_backward_head, attention_forward_head_rows
from oracle.precision import attention_backward_bf16, attention_forward_bf16, round_bf16
from workloads import make_inputs


def _torch_bf16(x32):
    return torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()


def test_round_bf16_matches_torch_on_fp32_values():
    rng = np.random.default_rng(7)
    for scale in (1e-30, 1e-3, 1.0, 37.0, 1e20):
        x = (rng.standard_normal(20000) * scale).astype(np.float32)
        assert np.array_equal(round_bf16(x.astype(np.float64)), _torch_bf16(x))
    sub = (rng.standard_normal(5000) * 2.0 ** -130).astype(np.float32)   # bf16 / fp32 subnormals
    assert np.array_equal(round_bf16(sub.astype(np.float64)), _torch_bf16(sub))


def test_round_bf16_ties_to_even_and_is_idempotent():
    one_ulp = 2.0 ** -7                                   # bf16 spacing in [1, 2)
    assert round_bf16(1.0 + one_ulp / 2) == 1.0           # tie, 1.0 is even
    assert round_bf16(1.0 + 3 * one_ulp / 2) == 1.0 + 2 * one_ulp
    assert round_bf16(-(1.0 + one_ulp / 2)) == -1.0
    x = np.random.default_rng(8).standard_normal(1000)
    r = round_bf16(x)
    assert np.array_equal(round_bf16(r), r)
    assert np.all(np.abs(r - x) <= 2.0 ** -8 * np.abs(x))   # unit roundoff of 8 significant bits


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("stress", [None, "wide", "sorted"])
def test_without_rounding_the_model_is_the_plain_oracle(causal, stress):
    n, d = 300, 64
    q, k, v, do = (t[0, 0].double().numpy() for t in make_inputs(1, 1, n, d, 5000 + n, stress=stress))
    scale = 1.0 / math.sqrt(d)
    o, o_b, lse = attention_forward_bf16(q, k, v, scale, causal, tile=64, rounding=False)
    o_ref, lse_ref = attention_forward_head_rows(q, k, v, np.arange(n), scale, causal)
    assert np.max(np.abs(o - o_ref)) < 1e-12 and np.array_equal(o, o_b)
    assert np.max(np.abs(lse - lse_ref)) < 1e-12
    grads = attention_backward_bf16(q, k, v, do, scale, causal, o_ref, lse_ref, rounding=False)
    refs = attention_backward_head(q, k, v, do, scale, causal)[:3]
    for g, r in zip(grads, refs):
        assert np.max(np.abs(g - r)) < 1e-11


STRESS = [("wide", 512, 64, False), ("wide", 512, 128, True), ("spike", 640, 128, False), ("sorted", 700, 128, True)]


@pytest.mark.parametrize("stress,n,d,causal", STRESS)
def test_rounding_alone_costs_the_stress_allowance(stress, n, d, causal):
    q, k, v, _ = (t[0, 0].double().numpy() for t in make_inputs(1, 1, n, d, 3000 + n, stress=stress))
    scale = 1.0 / math.sqrt(d)
    _, o_b, lse = attention_forward_bf16(q, k, v, scale, causal)
    o_ref, lse_ref = attention_forward_head_rows(q, k, v, np.arange(n), scale, causal)
    err = np.abs(o_b - o_ref)
    assert np.max(err - (1e-2 + 2.0 ** -8 * np.abs(o_ref))) <= 0.0   # inside the allowance
    assert np.max(np.abs(lse - lse_ref)) < 1e-6                     # lse carries no bf16 rounding
    assert np.max(np.abs(o_ref)) > 2.0                              # rows reach |O| where one ulp > 1e-2


def test_rounding_alone_can_exceed_the_plain_bound():
    """The plain 1e-2 on O is not met by bf16 rounding alone on single-key-dominated rows."""
    q, k, v, _ = (t[0, 0].double().numpy() for t in make_inputs(1, 1, 513, 64, 3513, stress="wide"))
    _, o_b, _ = attention_forward_bf16(q, k, v, 0.125, False)
    o_ref, _ = attention_forward_head_rows(q, k, v, np.arange(513), 0.125, False)
    assert np.max(np.abs(o_b - o_ref)) > 1e-2

"""The stress inputs' extra error is bf16 rounding and nothing else (needs a GB300).

On inputs whose rows are dominated by single keys (queries x8, a spiked key,
sorted keys) the GPU's O exceeds the plain 1e-2 bound against the exact
oracle, and its dQ, dK need the allowance for D formed from the stored bf16
O (tests/test_gpu_parity.py).  Here the same GPU results are compared with
the oracle's precision model (oracle/precision.py: exact arithmetic except
P rounded to bf16 before P V under the lazy running maximum, the output
rounded to bf16, and in the backward bf16 P, bf16 dS and D from that stored
output):

* O: within two bf16 units in the last place of the model's stored O (or
  1e-3 where O is small enough for that to be more), and bit-identical in
  most elements: one rounding on each side plus the odd probability that
  fp32 and fp64 round to neighbouring bf16 values;
* lse: the plain 1e-3;
* dQ, dK, dV: the plain 2e-2 of each gradient's max-abs, with no allowance.
"""

import math

import numpy as np
import pytest

from oracle.precision import attention_backward_bf16, attention_forward_bf16
from tests.gpu_util import TOL_GRAD_REL, TOL_LSE, f64, require_gpu, run_bwd, run_fwd
from workloads import make_inputs

pytestmark = pytest.mark.gpu

# the stress cases of tests/test_gpu_parity.py (same seeds)
STRESS = [("wide", 512, 64, False), ("wide", 512, 128, True), ("spike", 384, 64, True),
          ("spike", 640, 128, False), ("sorted", 512, 64, False), ("sorted", 700, 128, True)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _bf16_ulp(b):
    """The spacing of bf16 values at b (8 significant bits)."""
    _, e = np.frexp(b)
    return np.ldexp(1.0, np.maximum(e, -125) - 8)


@pytest.mark.parametrize("stress,N,d,causal", STRESS, ids=[f"{s}-n{n}d{d}{'c' if c else ''}" for s, n, d, c in STRESS])
def test_stress_residual_is_bf16_rounding(stress, N, d, causal):
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = make_inputs(1, 2, N, d, seed=3000 + N, stress=stress)
    qg, kg, vg, o, lse = run_fwd(q, k, v, scale, causal)
    dq, dk, dv = run_bwd(qg, kg, vg, o, lse, do, scale, causal)
    o_g, lse_g = f64(o), f64(lse)
    identical, worst = 0, 0.0
    for h in range(2):
        qd, kd, vd, dod = (t[0, h].double().numpy() for t in (q, k, v, do))
        _, o_b, lse_m = attention_forward_bf16(qd, kd, vd, scale, causal)
        diff = np.abs(o_g[0, h] - o_b)
        worst = max(worst, float((diff - np.maximum(2.0 * _bf16_ulp(o_b), 1e-3)).max()))
        identical += int((diff == 0).sum())
        assert float(np.abs(lse_g[0, h] - lse_m).max()) <= TOL_LSE
        grads = attention_backward_bf16(qd, kd, vd, dod, scale, causal, o_b, lse_m)
        for name, g, r in zip(("dq", "dk", "dv"), (dq[0, h], dk[0, h], dv[0, h]), grads):
            err = float(np.abs(f64(g) - r).max())
            assert err <= TOL_GRAD_REL * float(np.abs(r).max()), f"{stress} head {h} {name}: {err}"
    assert worst <= 0.0, f"{stress}: O beyond two bf16 ulps (and 1e-3) of the model by {worst}"
    assert identical >= 0.8 * o_g.size, f"{stress}: only {identical} of {o_g.size} O elements equal the model's"

"""FP8 (E4M3) query/key forward vs the oracle through the C ABI (needs a GB300).

The kernel and the oracle consume the same E4M3 codes and descale factors
(``workloads.make_fp8_inputs``), so the comparison measures the kernel's
arithmetic, not the quantisation of the inputs, and the plain forward's
tolerances apply (O max-abs 1e-2, lse max-abs 1e-3).

* Small shapes compared element by element with the full oracle: several
  tiles, ragged tails (N = 1, 129, 777, 1000), both masks, batched heads,
  causal N = 4096 (the block-major unit order), wide-score stress inputs.
* The long-sequence shape B1 H16 N16384 d128 at full size, both masks: every
  row of the first head and every fifth row (plus the last) of the last head
  against the oracle, finiteness everywhere.
* Descale factors: moving a factor between scale and a descale leaves the
  output unchanged up to rounding; k_descale = 0 gives uniform attention.
"""

import math

import numpy as np
import pytest
import torch

import exact_io_aware_31_gb300 as fa
import oracle
from oracle import fp8 as ofp8
from tests.gpu_util import TOL_LSE, TOL_O, assert_fwd_close, f64, require_gpu
from workloads import make_fp8_inputs

pytestmark = pytest.mark.gpu

D = 128
SMALL = [
    (1, 2, 256, False, None), (1, 2, 256, True, None), (1, 1, 1, True, None), (1, 1, 129, False, None),
    (2, 3, 777, True, None), (1, 2, 1000, False, None), (1, 2, 4096, True, None), (1, 2, 640, True, "wide"),
    (1, 1, 900, False, "spike"),
]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _run(q8, k8, qs, ks, v, scale, causal):
    o, lse = fa.forward_fp8(q8.cuda(), k8.cuda(), v.cuda(), qs, ks, scale, causal)
    assert fa.fa_get_device_status(torch.cuda.current_stream().cuda_stream) == fa.FA_OK
    return o, lse


@pytest.mark.parametrize("B,H,N,causal,stress", SMALL,
                         ids=[f"b{b}h{h}n{n}{'c' if c else ''}{s or ''}" for b, h, n, c, s in SMALL])
def test_fp8_small(B, H, N, causal, stress):
    scale = 1.0 / math.sqrt(D)
    q8, k8, qs, ks, v = make_fp8_inputs(B, H, N, D, seed=5000 + N + causal, stress=stress)
    o, lse = _run(q8, k8, qs, ks, v, scale, causal)
    o_ref, lse_ref = ofp8.attention_forward_fp8(q8.numpy(), k8.numpy(), qs, ks, v.double().numpy(), scale, causal)
    o_rel = 2.0 ** -8 if stress else 0.0
    assert_fwd_close(o, lse, o_ref, lse_ref, f"fp8 {(B, H, N, causal, stress)}", o_rel=o_rel)


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_long_sequence_full_size(causal):
    B, H, N = 1, 16, 16384
    scale = 1.0 / math.sqrt(D)
    q8, k8, qs, ks, v = make_fp8_inputs(B, H, N, D, seed=1004 + causal)
    o, lse = _run(q8, k8, qs, ks, v, scale, causal)
    assert bool(torch.isfinite(o.float()).all()) and bool(torch.isfinite(lse).all())
    for h, rows in ((0, np.arange(N)), (H - 1, np.r_[np.arange(0, N, 5), N - 1])):
        qd = ofp8.e4m3_decode(q8[0, h].numpy()) * qs
        kd = ofp8.e4m3_decode(k8[0, h].numpy()) * ks
        o_ref, lse_ref = oracle.attention_forward_head_rows(qd, kd, v[0, h].double().numpy(), rows, scale, causal)
        assert_fwd_close(o[0, h][rows], lse[0, h][rows], o_ref, lse_ref, f"fp8 long head {h}")


def test_fp8_descale_moves_into_scale():
    q8, k8, qs, ks, v = make_fp8_inputs(1, 2, 500, D, seed=77)
    o1, l1 = _run(q8, k8, qs, ks, v, 0.1, True)
    o2, l2 = _run(q8, k8, 1.0, 1.0, v, 0.1 * qs * ks, True)
    assert float((o1.float() - o2.float()).abs().max()) <= TOL_O
    assert float((l1 - l2).abs().max()) <= TOL_LSE


def test_fp8_zero_key_descale_is_uniform_attention():
    N = 300
    q8, k8, qs, _, v = make_fp8_inputs(1, 1, N, D, seed=78)
    o, lse = _run(q8, k8, qs, 0.0, v, 0.1, True)
    vd = v[0, 0].double().numpy()
    o_ref = np.cumsum(vd, axis=0) / np.arange(1, N + 1)[:, None]
    lse_ref = np.log(np.arange(1, N + 1, dtype=np.float64))
    assert float(np.abs(f64(o[0, 0]) - o_ref).max()) <= TOL_O
    assert float(np.abs(f64(lse[0, 0]) - lse_ref).max()) <= TOL_LSE

"""Split-KV decode forward vs the oracle through the C ABI (needs a GB300).

Cases span: one and several queries (Nq = 1..8, rounded up inside to 1, 2, 4
or 8), ragged caches (Nk not a multiple of 128, Nk < 128, Nk = 1), Nq = Nk,
both masks, one split, the automatic choice, more splits than tiles (clamped),
both merge paths (a head's splits as one cluster merging in shared memory;
more than 16 splits through the workspace and the merge kernel), a split whose
keys some queries cannot see (empty partial), and wide score rows (Q x 8) so
the running maximum moves between tiles and splits.
Tolerances are the forward's: O max-abs 1e-2, lse max-abs 1e-3.
"""

import math

import numpy as np
import pytest
import torch

import exact_io_aware_31_gb300 as fa
from oracle.decode import attention_forward_rect
from tests.gpu_util import TOL_LSE, TOL_O, f64, require_gpu
from workloads import DECODE_ALL, make_decode_inputs

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, Nq, Nk, d, causal, splits, stress
    (1, 2, 1, 1, 64, True, 0, None),
    (1, 2, 1, 300, 64, True, 0, None),
    (2, 3, 4, 777, 128, True, 0, None),
    (1, 4, 8, 1000, 128, True, 3, None),
    (1, 2, 3, 129, 64, False, 2, None),
    (2, 2, 8, 8, 64, True, 1, None),
    (1, 1, 5, 4096, 128, False, 0, None),
    (4, 8, 2, 2048, 64, True, 40, None),
    (1, 1, 8, 130, 64, True, 2, None),
    (1, 3, 7, 3000, 128, True, 0, "wide"),
    (2, 2, 1, 5000, 64, False, 7, "wide"),
    (1, 2, 6, 100, 128, True, 5, None),
    (1, 2, 2, 4000, 128, True, 20, None),     # more than 16 splits: workspace + merge kernel
    (3, 2, 1, 2000, 128, True, 12, "wide"),   # 12 splits: one cluster per head where launchable
]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _run(q, k, v, scale, causal, splits):
    o, lse = fa.decode_forward(q.cuda(), k.cuda(), v.cuda(), scale, causal, splits)
    assert fa.fa_get_device_status(torch.cuda.current_stream().cuda_stream) == fa.FA_OK
    return o, lse


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,splits,stress", CASES,
                         ids=[f"b{c[0]}h{c[1]}q{c[2]}k{c[3]}d{c[4]}{'c' if c[5] else ''}s{c[6]}{c[7] or ''}"
                              for c in CASES])
def test_decode_matches_oracle(B, H, Nq, Nk, d, causal, splits, stress):
    scale = 1.0 / math.sqrt(d)
    q, k, v = make_decode_inputs(B, H, Nq, Nk, d, seed=5000 + Nq * 7 + Nk + d, stress=stress)
    o, lse = _run(q, k, v, scale, causal, splits)
    o_ref, lse_ref = attention_forward_rect(*(t.double().numpy() for t in (q, k, v)), scale, causal)
    o_rel = 2.0 ** -8 if stress else 0.0   # rows dominated by one key: one bf16 ulp of |O|
    diff = np.abs(f64(o) - o_ref)
    assert np.all(np.isfinite(f64(o)))
    assert float((diff - (TOL_O + o_rel * np.abs(o_ref))).max()) <= 0.0, float(diff.max())
    assert float(np.abs(f64(lse) - lse_ref).max()) <= TOL_LSE


def test_split_count_does_not_change_the_result_beyond_rounding():
    q, k, v = make_decode_inputs(1, 4, 2, 3000, 128, seed=77)
    outs = [_run(q, k, v, 0.1, True, s) for s in (1, 2, 5, 0, 24)]
    for o, lse in outs[1:]:
        assert float((o.float() - outs[0][0].float()).abs().max()) <= 2 * 2.0 ** -8
        assert float((lse - outs[0][1]).abs().max()) <= 1e-4


@pytest.mark.parametrize("w", DECODE_ALL, ids=[w.name for w in DECODE_ALL])
def test_decode_workloads_sampled_heads(w):
    """The measured decode workloads at full size; the oracle checks sampled heads."""
    q, k, v = make_decode_inputs(w.B, w.H, w.Nq, w.Nk, w.d, w.seed)
    o, lse = _run(q, k, v, w.scale, w.causal, 0)
    rng = np.random.default_rng(w.seed)
    picks = [(int(rng.integers(w.B)), int(rng.integers(w.H))) for _ in range(3)]
    for b, h in picks:
        o_ref, lse_ref = attention_forward_rect(*(t[b:b + 1, h:h + 1].double().numpy() for t in (q, k, v)),
                                                w.scale, w.causal)
        assert float(np.abs(f64(o[b:b + 1, h:h + 1]) - o_ref).max()) <= TOL_O
        assert float(np.abs(f64(lse[b:b + 1, h:h + 1]) - lse_ref).max()) <= TOL_LSE


def test_workspace_rules():
    # 20 splits (more than a cluster takes) of a 4000-key cache (32 tiles): the workspace path
    q, k, v = (t.cuda() for t in make_decode_inputs(1, 2, 1, 4000, 64, seed=3))
    o = torch.empty_like(q)
    lse = torch.empty((1, 2, 1), device="cuda", dtype=torch.float32)
    s = torch.cuda.current_stream().cuda_stream
    need = fa.fa_fwd_splitkv_workspace_size(1, 2, 1, 4000, 64, 20)
    assert need > 0
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 2, 1, 4000, 64, 0.125, 1, 20)
    assert fa.fa_fwd_splitkv(*args, None, 0, s) == fa.FA_ERR_WORKSPACE
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    assert fa.fa_fwd_splitkv(*args, ws.data_ptr(), need - 256, s) == fa.FA_ERR_WORKSPACE
    assert fa.fa_fwd_splitkv(*args, ws.data_ptr(), need, s) == fa.FA_OK
    assert fa.fa_fwd_splitkv_workspace_size(1, 2, 1, 1000, 64, 1) == 0   # one split: none needed
    assert fa.fa_get_device_status(s) == fa.FA_OK


@pytest.mark.parametrize("Nq,Nk,d,splits", [(1, 2000, 128, 0), (4, 777, 64, 3)])
def test_decode_negative_scale(Nq, Nk, d, splits):
    scale = -1.0 / math.sqrt(d)
    q, k, v = make_decode_inputs(1, 2, Nq, Nk, d, seed=5900 + Nq + Nk)
    o, lse = _run(q, k, v, scale, True, splits)
    o_ref, lse_ref = attention_forward_rect(*(t.double().numpy() for t in (q, k, v)), scale, True)
    assert float(np.abs(f64(o) - o_ref).max()) <= TOL_O
    assert float(np.abs(f64(lse) - lse_ref).max()) <= TOL_LSE

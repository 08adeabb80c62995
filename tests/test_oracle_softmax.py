"""Pins of the oracle's softmax pieces (CPU only).

* The worked example of lensaml.com "FlashAttention" Step 4 "Online Softmax"
  (values printed on the page, tests/golden/online_softmax_worked_example.txt).
* The running (m, l) after every chunk against the direct prefix normaliser
  sum_{j <= t} exp(x_j - max_{j <= t} x_j), which the recurrence must equal.
* SciPy's softmax / logsumexp as an independent library routine.
"""

import math

import numpy as np
import pytest
import scipy.special

from oracle import online_softmax_trace, softmax_three_pass


def test_worked_example_printed_softmax(golden):
    g = golden("online_softmax_worked_example.txt")
    x = np.array(g["scores"])
    y, m, l = softmax_three_pass(x)
    assert np.allclose(np.round(y, 2), g["softmax_2dp"], atol=0, rtol=0)
    _, y_online = online_softmax_trace(x, int(g["chunk"]))
    assert np.allclose(np.round(y_online, 2), g["softmax_2dp"], atol=0, rtol=0)
    assert abs(y.sum() - 1.0) < 1e-15


def test_worked_example_running_statistics(golden):
    g = golden("online_softmax_worked_example.txt")
    x = [float(v) for v in g["scores"]]
    chunk = int(g["chunk"])
    trace, _ = online_softmax_trace(np.array(x), chunk)
    assert len(trace) == 4
    for t, (m, l) in enumerate(trace):
        seen = x[:chunk * (t + 1)]
        m_direct = max(seen)
        l_direct = sum(math.exp(v - m_direct) for v in seen)
        assert m == m_direct
        assert abs(l - l_direct) < 1e-14
    # the page's running max after chunks (1.2, 3.0), (0.4, 2.1), (4.5, 1.8), (3.6, 0.9)
    assert [m for m, _ in trace] == [3.0, 3.0, 4.5, 4.5]


@pytest.mark.parametrize("chunk", [1, 2, 3, 5, 8, 64])
def test_online_equals_three_pass_random(chunk):
    rng = np.random.default_rng(7 + chunk)
    x = rng.normal(scale=6.0, size=200)
    _, y_online = online_softmax_trace(x, chunk)
    y, m, l = softmax_three_pass(x)
    assert np.max(np.abs(y_online - y)) < 1e-15
    assert np.max(np.abs(y - scipy.special.softmax(x))) < 1e-15
    assert abs((m + math.log(l)) - scipy.special.logsumexp(x)) < 1e-12


def test_three_pass_survives_large_scores():
    # fp16 overflows above 65504 = e^11.1 (lensaml.com Step 4); max subtraction keeps
    # exponents <= 0 so even scores of 1e3 give a finite, exact softmax in fp64.
    x = np.array([1000.0, 999.0, 998.0])
    y, _, _ = softmax_three_pass(x)
    e = np.exp([0.0, -1.0, -2.0])
    assert np.allclose(y, e / e.sum(), rtol=1e-15, atol=0)
    assert abs(math.log(65504.0) - 11.09) < 0.01

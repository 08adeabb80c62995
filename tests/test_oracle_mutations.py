"""Planted mistakes in a copy of the oracle must be caught by its pins (CPU only).

Each case rewrites one line of ``oracle/attention.py`` in memory (a dropped
term, a wrong index or sign, a transposed operand), loads the result as a
throwaway module and runs the independent checks used by the pin tests:
PyTorch fp64 SDPA and autograd, SciPy logsumexp, and tiled-vs-three-pass.
The real oracle is never modified.
"""

import importlib.util
import math
import os
import sys
import types

import numpy as np
import pytest
import scipy.special
import torch

ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                          "oracle", "attention.py")

MUTATIONS = [
    ("causal off by one", "s = np.where(j > i, -np.inf, s)", "s = np.where(j >= i + 1 + (i % 2), -np.inf, s)"),
    ("lse drops the log", "lse[r0:r1] = m + np.log(l)", "lse[r0:r1] = m + l"),
    ("forward uses unnormalised P", "o[r0:r1] = p @ v", "o[r0:r1] = np.exp(s - m[:, None]) @ v"),
    ("dK loses the scale", "dk += scale * (ds.T @ q[r0:r1])", "dk += ds.T @ q[r0:r1]"),
    ("dS drops D", "ds = p * (dp - D[r0:r1, None])", "ds = p * dp"),
    ("dQ transposed dS", "dq[r0:r1] = scale * (ds @ k)", "dq[r0:r1] = scale * (ds.T[:r1 - r0, :] @ k)"),
    ("dK transposed dS", "dk += scale * (ds.T @ q[r0:r1])", "dk += scale * (ds @ q[r0:r1])"),
    ("P rebuilt without lse", "p = np.exp(s - lse[r0:r1, None])", "p = np.exp(s - np.max(s, axis=1, keepdims=True))"),
    ("dP wrong operand", "dp = do[r0:r1] @ v.T", "dp = do[r0:r1] @ k.T"),
    ("tiled forgets to rescale l", "l = a_old * l + a_new * l_b", "l = l + l_b"),
    ("tiled forgets to rescale O", "acc = a_old[:, None] * acc + a_new[:, None] * (p_b @ vh[j0:j1])",
     "acc = acc + a_new[:, None] * (p_b @ vh[j0:j1])"),
    ("softmax pass 3 wrong sign", "y = np.exp(x - m) / l                                  # pass 3",
     "y = np.exp(m - x) / l"),
]


def _load_mutant(old, new):
    with open(ORACLE_SRC) as f:
        src = f.read()
    assert src.count(old) == 1, old
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src.replace(old, new), "oracle_mutant", "exec"), mod.__dict__)
    return mod


def _pins_pass(mod):
    rng = np.random.default_rng(5)
    n, d = 40, 8
    q, k, v, do = (rng.normal(scale=2.0, size=(1, 2, n, d)) for _ in range(4))
    scale = 1 / math.sqrt(d)
    try:
        for causal in (False, True):
            o, lse = mod.attention_forward(q, k, v, scale, causal)
            tq, tk, tv = (torch.from_numpy(a.copy()).requires_grad_(True) for a in (q, k, v))
            out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
            if np.max(np.abs(o - out.detach().numpy())) > 1e-12:
                return False
            s = scale * (q @ np.swapaxes(k, -1, -2))
            if causal:
                s = np.where(np.triu(np.ones((n, n), bool), 1), -np.inf, s)
            if np.max(np.abs(lse - scipy.special.logsumexp(s, axis=-1))) > 1e-12:
                return False
            out.backward(torch.from_numpy(do))
            dq, dk, dv, _ = mod.attention_backward(q, k, v, do, scale, causal)
            for g, t in ((dq, tq), (dk, tk), (dv, tv)):
                if np.max(np.abs(g - t.grad.numpy())) > 1e-11:
                    return False
            ot, lset = mod.attention_forward_tiled(q, k, v, scale, causal, 7)
            if np.max(np.abs(ot - o)) > 1e-12 or np.max(np.abs(lset - lse)) > 1e-12:
                return False
        y, _, _ = mod.softmax_three_pass(np.array([1.2, 3.0, 0.4]))
        if abs(y.sum() - 1) > 1e-15 or not y[1] > y[0] > y[2]:
            return False
    except Exception:
        return False
    return True


def test_unmodified_oracle_passes_the_checks():
    spec = importlib.util.spec_from_file_location("oracle_copy", ORACLE_SRC)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    assert _pins_pass(mod)


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new):
    assert not _pins_pass(_load_mutant(old, new)), name

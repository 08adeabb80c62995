"""Attention with the bf16 roundings of the fused method made explicit, fp64 otherwise.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): slow, obvious, CPU.

The pages fix no precision.  The readings this library takes (bf16 operands
and outputs, fp32 accumulation) put exactly three bf16 roundings between the
plain definition and what a bf16 kernel can return:

* the probabilities enter the second contraction as bf16: P V in the forward,
  P^T dO and the dS product in the backward;
* dS enters dK = scale dS^T Q and dQ = scale dS K as bf16;
* O is stored as bf16, and the backward's D = rowsum(dO * O) is formed from
  that stored O (the method keeps only O and the row statistics: [T] "The
  backward pass: recompute instead of read").

The forward's probabilities are relative to the running maximum of the
online softmax ([T] "FlashAttention's move: rescale the output, too"), kept
lazily: the maximum used for the exponentials moves only when a key tile's
maximum exceeds it by more than ``threshold`` in log2 units.  In exact
arithmetic that changes nothing (the common factor cancels in the final
division); with P rounded it decides which values are rounded, so the model
follows it tile by tile.  Everything else is fp64.

This module shows what those roundings cost on inputs whose rows are
dominated by single keys, where the plain tolerances on O and on dQ, dK are
not met by rounding alone.
"""

from __future__ import annotations

import numpy as np

__all__ = ["round_bf16", "attention_forward_bf16", "attention_backward_bf16"]

_LOG2E = 1.0 / np.log(2.0)


def round_bf16(x):
    """Round to the nearest bf16 value, ties to even (8 significant bits, fp32's exponent range).

    Written from the format: a finite x with 2^(e-1) <= |x| < 2^e is a
    multiple of 2^(e-8) once rounded; below 2^-126 the spacing stays 2^-133
    (subnormals).  Magnitudes past the largest finite bf16 are not handled
    (they do not occur here).
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    ulp = np.ldexp(1.0, np.maximum(e, -125) - 8)
    return np.where(x == 0, x, np.rint(x / ulp) * ulp)


def _identity(x):
    return np.asarray(x, dtype=np.float64)


def _lazy_row_softmax(s2_rows, tile, threshold, group, rnd):
    """Online softmax of score rows given in log2 units, tile by tile with the lazy maximum.

    Rows move their reference maximum together in groups of ``group``
    consecutive rows: when any row of a group sees a key tile whose maximum
    exceeds its reference by more than ``threshold``, every row of the group
    takes max(reference, tile maximum).  Returns ``(P, m, l)``: the bf16
    probabilities each tile feeds its P V product, brought to the final
    reference maximum by the rescale factors (which the method applies to O,
    the same products), the final reference maximum m (log2 units) and the
    sum l of the unrounded probabilities relative to m.
    """
    n_rows, n_keys = s2_rows.shape
    m = np.full(n_rows, -np.inf)
    l = np.zeros(n_rows)
    pr = np.zeros_like(s2_rows)
    gid = np.arange(n_rows) // group
    for j0 in range(0, n_keys, tile):
        j1 = min(n_keys, j0 + tile)
        blk = s2_rows[:, j0:j1]
        mb = blk.max(axis=1)
        first = m == -np.inf
        need = first | (mb > m + threshold)
        move = np.bincount(gid, weights=need.astype(np.float64))[gid] > 0
        m_new = np.where(move, np.where(first, mb, np.maximum(m, mb)), m)
        seen = ~first
        alpha = np.where(seen, np.exp2(np.where(seen, m, 0.0) - np.where(seen, m_new, 0.0)), 0.0)
        l = alpha * l
        pr[:, :j0] *= alpha[:, None]
        live = m_new > -np.inf
        p = np.where(live[:, None], np.exp2(blk - np.where(live, m_new, 0.0)[:, None]), 0.0)
        l = l + p.sum(axis=1)
        pr[:, j0:j1] = rnd(p)
        m = m_new
    return pr, m, l


def attention_forward_bf16(q, k, v, scale, causal, tile=128, threshold=8.0, group=32, rounding=True):
    """One head ``q, k, v [N, d]``: the forward with P rounded to bf16 before P V (lazy running max).

    Returns ``(o, o_bf16, lse)``: the output before its own rounding, the
    stored bf16 output, and the natural-log logsumexp.  ``rounding=False``
    makes every rounding the identity, which leaves the plain result.
    """
    rnd = round_bf16 if rounding else _identity
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    n = q.shape[0]
    s2 = (scale * (q @ k.T)) * _LOG2E
    if causal:
        s2[np.triu_indices(n, 1, m=k.shape[0])] = -np.inf
    pr, m, l = _lazy_row_softmax(s2, tile, threshold, group, rnd)
    o = (pr @ v) / l[:, None]
    lse = (m + np.log2(l)) / _LOG2E
    return o, rnd(o), lse


def attention_backward_bf16(q, k, v, do, scale, causal, o_stored, lse, rounding=True):
    """One head: gradients with bf16 P (for dV and dS), bf16 dS (for dK, dQ) and D from the stored O.

    ``o_stored`` and ``lse`` are the forward's stored output and logsumexp
    (from :func:`attention_forward_bf16`); P is rebuilt from lse as the
    backward recomputes it.  Returns ``(dq, dk, dv)`` before their own bf16
    rounding.
    """
    rnd = round_bf16 if rounding else _identity
    q, k, v, do, o_stored = (np.asarray(t, dtype=np.float64) for t in (q, k, v, do, o_stored))
    n = q.shape[0]
    s = scale * (q @ k.T)
    if causal:
        s[np.triu_indices(n, 1, m=k.shape[0])] = -np.inf
    p = rnd(np.exp(s - np.asarray(lse)[:, None]))
    D = np.sum(do * o_stored, axis=1)
    dv = p.T @ do
    dp = do @ v.T
    ds = rnd(p * (dp - D[:, None]))
    return scale * (ds @ k), scale * (ds.T @ q), dv

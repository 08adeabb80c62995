"""Plain fp64 attention: three-pass forward, tiled online-softmax forward, analytic backward.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): slow, obvious, CPU.

Conventions
-----------
* Arrays are numpy float64 of shape ``[B, H, N, d]`` (q, k, v, o, do) and
  ``[B, H, N]`` (lse, D).  Callers upcast the bf16-rounded inputs the GPU
  consumes, so both sides see identical operands.
* ``scale`` multiplies ``Q K^T`` before the mask (reading: the pages apply the
  1/sqrt(d) factor to the scores, [V] "The Quadratic IO Bottleneck" and [L]
  FAQ "What is FlashAttention?"; the mask then overwrites entries).
* ``causal`` is the square, top-left aligned mask: key j is visible to query i
  iff j <= i.  No other mask exists in this library.
* ``lse`` is the natural-log logsumexp of the scaled, masked score row,
  ``m + ln(l)``: the per-row statistics (m, l) that [T] "The backward pass:
  recompute instead of read" says the forward keeps, folded into one number.

Row blocking (``row_block``) only batches independent rows to bound memory;
every row is still computed by the unmodified three-pass definition.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "scores",
    "softmax_three_pass",
    "online_softmax_trace",
    "attention_forward",
    "attention_forward_head_rows",
    "attention_forward_tiled",
    "attention_backward",
    "attention_backward_head",
    "attention_backward_head_rows",
]

_DEFAULT_ROW_BLOCK = 1024


def scores(q_rows, k, scale, causal, row_offset=0):
    """Scaled, masked score rows ``S[i, j] = scale * q_i . k_j`` (-inf where masked).

    [T] "The hierarchy attention keeps ignoring": standard attention first forms
    ``S = Q K^T``; [L] Step 2 draws the same first kernel.  ``q_rows`` holds
    queries ``row_offset .. row_offset + len(q_rows) - 1`` of one head.
    """
    s = scale * (q_rows @ k.T)
    if causal:
        i = np.arange(q_rows.shape[0])[:, None] + row_offset
        j = np.arange(k.shape[0])[None, :]
        s = np.where(j > i, -np.inf, s)
    return s


def softmax_three_pass(x):
    """Numerically safe softmax of each row of ``x`` in three passes.

    [T] "Softmax is the anti-tiling operation": pass 1 takes the row maximum
    m, pass 2 the normaliser l = sum exp(x - m), pass 3 divides
    exp(x - m) by l.  Returns ``(y, m, l)``.
    """
    x = np.asarray(x, dtype=np.float64)
    m = np.max(x, axis=-1, keepdims=True)                  # pass 1
    l = np.sum(np.exp(x - m), axis=-1, keepdims=True)      # pass 2
    y = np.exp(x - m) / l                                  # pass 3
    return y, m[..., 0], l[..., 0]


def online_softmax_trace(x, chunk):
    """Single-pass running (m, l) over ``x`` in chunks; returns the trace and softmax.

    [T] "Softmax is the anti-tiling operation" (the Milakov-Gimelshein update)
    and [L] Step 4 "Online Softmax": start from m = -inf, l = 0; for each chunk
    take its max m_b and its own sum l_b = sum exp(x - m_b), then
    m_new = max(m, m_b) and l_new = exp(m - m_new) * l + exp(m_b - m_new) * l_b.
    A factor exp(-inf - m_new) is 0 (nothing seen yet).  The final softmax is
    exp(x - m) / l with the final statistics.
    Returns ``(trace, y)`` where ``trace`` is a list of ``(m, l)`` after each chunk.
    """
    x = np.asarray(x, dtype=np.float64)
    m, l = -np.inf, 0.0
    trace = []
    for start in range(0, x.shape[0], chunk):
        xb = x[start:start + chunk]
        m_b = float(np.max(xb))
        l_b = float(np.sum(np.exp(xb - m_b)))
        m_new = max(m, m_b)
        old = 0.0 if m == -np.inf else float(np.exp(m - m_new))
        l = old * l + float(np.exp(m_b - m_new)) * l_b
        m = m_new
        trace.append((m, l))
    y = np.exp(x - m) / l
    return trace, y


def _forward_head(q, k, v, scale, causal, row_block):
    """Three-pass forward for one head: returns ``(o [N, d], lse [N])``."""
    n = q.shape[0]
    o = np.empty((n, v.shape[1]), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    for r0 in range(0, n, row_block):
        r1 = min(n, r0 + row_block)
        s = scores(q[r0:r1], k, scale, causal, row_offset=r0)
        p, m, l = softmax_three_pass(s)
        o[r0:r1] = p @ v                                   # O = P V
        lse[r0:r1] = m + np.log(l)
    return o, lse


def attention_forward(q, k, v, scale, causal, row_block=_DEFAULT_ROW_BLOCK):
    """Exact attention ``O = softmax(scale * Q K^T + mask) V`` and the row logsumexp.

    The plain definition the method must reproduce up to rounding: [T] "The
    hierarchy attention keeps ignoring" (S = QK^T, P = softmax(S), O = PV) with
    the safe softmax of "Softmax is the anti-tiling operation"; [L] Step 2 and
    the FAQ state that the fused method returns this same result.
    Inputs ``[B, H, N, d]`` float64; returns ``o [B, H, N, d]``, ``lse [B, H, N]``.
    """
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    b, h, n, _ = q.shape
    o = np.empty(q.shape[:3] + (v.shape[3],), dtype=np.float64)
    lse = np.empty((b, h, n), dtype=np.float64)
    for bi in range(b):
        for hi in range(h):
            o[bi, hi], lse[bi, hi] = _forward_head(q[bi, hi], k[bi, hi], v[bi, hi],
                                                   scale, causal, row_block)
    return o, lse


def attention_forward_head_rows(q, k, v, rows, scale, causal):
    """Forward outputs of selected query ``rows`` of ONE head ``q, k, v [N, d]``.

    Same three-pass definition as :func:`attention_forward`, evaluated only
    for the rows asked for (each row depends only on its own query and on all
    keys/values), so full-size workloads can be checked on samples.
    Returns ``(o [len(rows), d], lse [len(rows)])``.
    """
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    rows = np.asarray(rows)
    s = scale * (q[rows] @ k.T)
    if causal:
        j = np.arange(k.shape[0])[None, :]
        s = np.where(j > rows[:, None], -np.inf, s)
    p, m, l = softmax_three_pass(s)
    return p @ v, m + np.log(l)


def attention_forward_tiled(q, k, v, scale, causal, block):
    """Tiled forward with online softmax and a rescaled output accumulator.

    [T] "FlashAttention's move: rescale the output, too" and [L] Step 3/4: keep,
    per query row, the running max m, the running normaliser l and an
    unnormalised output O~.  For each key/value block b: compute its scores
    S_b, its row max m_b, P~_b = exp(S_b - m_b), l_b = rowsum(P~_b); then
        m_new = max(m, m_b)
        l     = exp(m - m_new) * l + exp(m_b - m_new) * l_b
        O~    = exp(m - m_new) * O~ + exp(m_b - m_new) * (P~_b V_b)
    and divide O~ by l after the last block ([L] Step 4).  A block whose row
    is fully masked (m_b = -inf) leaves that row's state unchanged; a factor
    exp(-inf - m_new) is 0.  Returns ``(o, lse)`` like :func:`attention_forward`.
    """
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    bsz, heads, n, _ = q.shape
    o = np.empty(q.shape[:3] + (v.shape[3],), dtype=np.float64)
    lse = np.empty((bsz, heads, n), dtype=np.float64)
    for bi in range(bsz):
        for hi in range(heads):
            qh, kh, vh = q[bi, hi], k[bi, hi], v[bi, hi]
            m = np.full((n,), -np.inf)
            l = np.zeros((n,))
            acc = np.zeros((n, vh.shape[1]))
            for j0 in range(0, kh.shape[0], block):
                j1 = min(kh.shape[0], j0 + block)
                s_b = scale * (qh @ kh[j0:j1].T)
                if causal:
                    i = np.arange(n)[:, None]
                    j = np.arange(j0, j1)[None, :]
                    s_b = np.where(j > i, -np.inf, s_b)
                m_b = np.max(s_b, axis=1)
                live = m_b > -np.inf                      # rows with a visible key here
                m_b_safe = np.where(live, m_b, 0.0)
                p_b = np.where(live[:, None], np.exp(s_b - m_b_safe[:, None]), 0.0)
                l_b = np.sum(p_b, axis=1)
                m_new = np.maximum(m, m_b)
                seen = m > -np.inf
                a_old = np.where(seen, np.exp(np.where(seen, m, 0.0) - np.where(seen, m_new, 0.0)), 0.0)
                a_new = np.where(live, np.exp(m_b_safe - np.where(live, m_new, 0.0)), 0.0)
                l = a_old * l + a_new * l_b
                acc = a_old[:, None] * acc + a_new[:, None] * (p_b @ vh[j0:j1])
                m = m_new
            o[bi, hi] = acc / l[:, None]
            lse[bi, hi] = m + np.log(l)
    return o, lse


def attention_backward_head(q, k, v, do, scale, causal, row_block=_DEFAULT_ROW_BLOCK):
    """Gradients of one head ``q, k, v, do [N, d]``; returns ``(dq, dk, dv, D, o, lse)``.

    [T] "The backward pass: recompute instead of read": the backward rebuilds S
    and P from Q, K, V and the saved row statistics instead of reading a stored
    P.  The pages give no gradient formulas; these follow from the forward by
    the chain rule (with P = softmax(S), S = scale * Q K^T):
        dV = P^T dO,   dP = dO V^T,   D_i = sum_k dO_ik O_ik (= sum_j P_ij dP_ij),
        dS = P * (dP - D),   dQ = scale * dS K,   dK = scale * dS^T Q.
    P is rebuilt row-block by row-block from the saved logsumexp:
    P_ij = exp(S_ij - lse_i).  ``D`` is returned for both of its forms to agree
    in tests (the second form is checked there).
    """
    q, k, v, do = (np.asarray(t, dtype=np.float64) for t in (q, k, v, do))
    o, lse = _forward_head(q, k, v, scale, causal, row_block)
    D = np.sum(do * o, axis=1)
    dq = np.empty_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    n = q.shape[0]
    for r0 in range(0, n, row_block):
        r1 = min(n, r0 + row_block)
        s = scores(q[r0:r1], k, scale, causal, row_offset=r0)
        p = np.exp(s - lse[r0:r1, None])                   # recomputed P rows
        dv += p.T @ do[r0:r1]
        dp = do[r0:r1] @ v.T
        ds = p * (dp - D[r0:r1, None])
        dq[r0:r1] = scale * (ds @ k)
        dk += scale * (ds.T @ q[r0:r1])
    return dq, dk, dv, D, o, lse


def attention_backward(q, k, v, do, scale, causal, row_block=_DEFAULT_ROW_BLOCK):
    """Gradients of ``L = sum(O * dO)`` w.r.t. q, k, v for ``[B, H, N, d]`` inputs.

    Per head as in :func:`attention_backward_head`.
    Returns ``(dq, dk, dv, D [B, H, N])``.
    """
    q, k, v, do = (np.asarray(t, dtype=np.float64) for t in (q, k, v, do))
    bsz, heads, n, _ = q.shape
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    D = np.empty((bsz, heads, n))
    for bi in range(bsz):
        for hi in range(heads):
            dq[bi, hi], dk[bi, hi], dv[bi, hi], D[bi, hi], _, _ = attention_backward_head(
                q[bi, hi], k[bi, hi], v[bi, hi], do[bi, hi], scale, causal, row_block)
    return dq, dk, dv, D


def attention_backward_head_rows(q, k, v, do, rows, scale, causal):
    """What query ``rows`` of ONE head contribute to the gradients: ``(dq_rows, dk_part, dv_part)``.

    The formulas of :func:`attention_backward_head` evaluated for the asked
    rows only.  Row i's forward output, logsumexp, D_i and dS row depend on
    row i alone (and on every key and value), so ``dq_rows`` is exactly those
    rows of dQ, while dK and dV are sums over query rows: ``dk_part`` and
    ``dv_part`` are the asked rows' terms, and summing them over a partition of
    all rows gives dK and dV.  Lets a bounded sample of a large workload be
    timed or checked without the whole head.
    """
    q, k, v, do = (np.asarray(t, dtype=np.float64) for t in (q, k, v, do))
    rows = np.asarray(rows)
    o_r, lse_r = attention_forward_head_rows(q, k, v, rows, scale, causal)
    D = np.sum(do[rows] * o_r, axis=1)
    s = scale * (q[rows] @ k.T)
    if causal:
        j = np.arange(k.shape[0])[None, :]
        s = np.where(j > rows[:, None], -np.inf, s)
    p = np.exp(s - lse_r[:, None])                         # recomputed P rows
    dv_part = p.T @ do[rows]
    dp = do[rows] @ v.T
    ds = p * (dp - D[:, None])
    dq_rows = scale * (ds @ k)
    dk_part = scale * (ds.T @ q[rows])
    return dq_rows, dk_part, dv_part

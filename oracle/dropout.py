"""Plain fp64 attention with dropout on the probabilities, and its counter-based mask.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): slow, obvious, CPU.

[T] "The backward pass: recompute instead of read": the forward saves only O,
the row statistics and the dropout PRNG state, and the backward regenerates
the dropout mask from that state.  Readings (the pages fix none of the
details):

* The random numbers come from Philox4x32-10 (Salmon, Moraes, Dror, Shaw,
  "Parallel random numbers: as easy as 1, 2, 3", SC'11), a counter-based
  generator: every element's bits are a pure function of (key, counter), so
  the backward regenerates exactly the forward's mask.  One call maps a
  128-bit counter and a 64-bit key to four 32-bit words.
* Element (b, h, query i, key j) uses word ``j mod 4`` of the call with
  counter ``(j div 4, i, b * H + h, offset)`` and key ``(seed mod 2^32,
  seed div 2^32)``; it is kept iff that word is >= ``threshold(p)`` =
  ``round(p * 2^32)`` (clamped to 2^32 - 1), so it survives with probability
  1 - p up to 2^-32.
* Dropout acts on the softmax probabilities after normalisation, with the
  usual 1 / (1 - p) scaling of the kept ones: O = (P o M / (1 - p)) V.  lse is
  the undropped softmax's.  Backward (chain rule through the mask):
  dV = (P o M / (1 - p))^T dO,  dP = (dO V^T) o M / (1 - p),
  D_i = sum_j P_ij dP_ij = dO_i . O_i,  dS = P o (dP - D),
  dQ = scale dS K,  dK = scale dS^T Q.
"""

from __future__ import annotations

import numpy as np

from oracle.attention import scores, softmax_three_pass

__all__ = ["philox4x32", "keep_threshold", "dropout_keep_mask", "attention_forward_dropout",
           "attention_backward_dropout"]

_M0 = 0xD2511F53   # Philox4x32 multipliers (Salmon et al., Table 3)
_M1 = 0xCD9E8D57
_W0 = 0x9E3779B9   # Weyl key increments (golden ratio and sqrt(3) - 1, scaled to 32 bits)
_W1 = 0xBB67AE85
_MASK32 = 0xFFFFFFFF


def philox4x32(c0, c1, c2, c3, k0, k1, rounds=10):
    """Philox4x32 with ``rounds`` rounds on arrays of 32-bit counters (one call per element).

    Each round multiplies the first and third counter words by M0 and M1,
    splits the 64-bit products into high and low halves and permutes:
        (c0, c1, c2, c3) <- (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0))
    then bumps the key by the Weyl constants.  Returns the four output words.
    """
    c = [np.asarray(x, dtype=np.uint64) & _MASK32 for x in (c0, c1, c2, c3)]
    k0 = np.asarray(k0, dtype=np.uint64) & _MASK32
    k1 = np.asarray(k1, dtype=np.uint64) & _MASK32
    for _ in range(rounds):
        p0 = c[0] * np.uint64(_M0)
        p1 = c[2] * np.uint64(_M1)
        hi0, lo0 = p0 >> np.uint64(32), p0 & np.uint64(_MASK32)
        hi1, lo1 = p1 >> np.uint64(32), p1 & np.uint64(_MASK32)
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
        k0 = (k0 + np.uint64(_W0)) & np.uint64(_MASK32)
        k1 = (k1 + np.uint64(_W1)) & np.uint64(_MASK32)
    return [x.astype(np.uint32) for x in c]


def keep_threshold(p):
    """Words >= this are kept: round(p * 2^32), clamped to 2^32 - 1."""
    t = int(round(float(p) * 4294967296.0))
    return min(max(t, 0), _MASK32)


def dropout_keep_mask(B, H, Nq, Nk, p, seed, offset):
    """Boolean keep mask [B, H, Nq, Nk] of the reading above."""
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    k0, k1 = seed & _MASK32, seed >> 32
    i = np.arange(Nq, dtype=np.uint64)[:, None]
    j = np.arange(Nk, dtype=np.uint64)[None, :]
    thr = np.uint64(keep_threshold(p))
    mask = np.empty((B, H, Nq, Nk), dtype=bool)
    for b in range(B):
        for h in range(H):
            bh = np.uint64(b * H + h)
            words = philox4x32(np.broadcast_to(j >> np.uint64(2), (Nq, Nk)), np.broadcast_to(i, (Nq, Nk)),
                               np.full((Nq, Nk), bh, dtype=np.uint64), np.full((Nq, Nk), offset, dtype=np.uint64),
                               k0, k1)
            sel = (j & np.uint64(3)).astype(np.int64)
            w = np.choose(np.broadcast_to(sel, (Nq, Nk)), words)
            mask[b, h] = w.astype(np.uint64) >= thr
    return mask


def attention_forward_dropout(q, k, v, scale, causal, p, seed, offset):
    """``O = (P o M / (1 - p)) V`` with P the exact softmax; lse of the undropped rows.

    Returns ``o [B, H, N, d]``, ``lse [B, H, N]`` and the keep mask.
    """
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    B, H, N, d = q.shape
    m = dropout_keep_mask(B, H, N, k.shape[2], p, seed, offset)
    o = np.empty_like(v)
    lse = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            s = scores(q[b, h], k[b, h], scale, causal)
            pr, mx, l = softmax_three_pass(s)
            o[b, h] = (pr * m[b, h] / (1.0 - p)) @ v[b, h]
            lse[b, h] = mx + np.log(l)
    return o, lse, m


def attention_backward_dropout(q, k, v, do, scale, causal, p, seed, offset):
    """Gradients of ``L = sum(O * dO)`` for the dropout forward; returns ``(dq, dk, dv)``."""
    q, k, v, do = (np.asarray(t, dtype=np.float64) for t in (q, k, v, do))
    B, H, N, d = q.shape
    m = dropout_keep_mask(B, H, N, k.shape[2], p, seed, offset)
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    keep = 1.0 / (1.0 - p)
    for b in range(B):
        for h in range(H):
            s = scores(q[b, h], k[b, h], scale, causal)
            pr, _, _ = softmax_three_pass(s)
            pd = pr * m[b, h] * keep
            o = pd @ v[b, h]
            dv[b, h] = pd.T @ do[b, h]
            dp = (do[b, h] @ v[b, h].T) * m[b, h] * keep
            dsum = np.sum(do[b, h] * o, axis=1, keepdims=True)
            ds = pr * (dp - dsum)
            dq[b, h] = scale * ds @ k[b, h]
            dk[b, h] = scale * ds.T @ q[b, h]
    return dq, dk, dv

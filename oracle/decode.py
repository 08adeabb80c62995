"""Plain fp64 split-KV attention (decode): rectangular forward, per-split partials, merge.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): slow, obvious, CPU.

[L] FAQ "Does FlashAttention help during LLM decoding?": at decode time each
step brings only a few new queries per sequence, so the score matrix is a
single row (or a few) against a long key/value cache and the cost is reading
that cache; Flash-Decoding splits the read over many thread blocks.  Each
block's partial result is a softmax over its own keys, and the partials are
merged with the same rescale rule the pages give for the online softmax ([T]
"Softmax is the anti-tiling operation" and "FlashAttention's move: rescale
the output, too": m_new = max(m_a, m_b), each side's sum and output scaled by
exp(m_side - m_new)).

Conventions (readings, the pages fix none of them for decode):
* ``q`` is ``[B, H, Nq, d]``, ``k``/``v`` are ``[B, H, Nk, d]``; the Nq queries are
  the LAST Nq positions of the Nk-long sequence.  Under ``causal`` key j is
  visible to query i iff ``j <= i + (Nk - Nq)`` (bottom-right aligned); with
  Nq == Nk this is the square top-left mask of ``oracle.attention``.
  Causal requires Nq <= Nk, so every query sees at least one key.
* ``lse`` is the natural-log logsumexp of the scaled, masked score row.
* A split with no visible key for a query contributes lse = -inf and a zero
  output row (weight exp(-inf) = 0 in the merge).
"""

from __future__ import annotations

import numpy as np

from oracle.attention import scores, softmax_three_pass

__all__ = ["attention_forward_rect", "split_partials", "merge_partials", "split_bounds"]


def attention_forward_rect(q, k, v, scale, causal):
    """Exact ``O = softmax(scale * Q K^T + mask) V`` with Nq queries against Nk keys.

    The three-pass definition ([T] "Softmax is the anti-tiling operation") on
    every row; the bottom-right causal mask is the square mask shifted by
    Nk - Nq (``scores`` with ``row_offset = Nk - Nq``).
    Returns ``o [B, H, Nq, d]``, ``lse [B, H, Nq]``.
    """
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    B, H, nq, d = q.shape
    nk = k.shape[2]
    if causal and nq > nk:
        raise ValueError("causal decode needs Nq <= Nk")
    o = np.empty((B, H, nq, v.shape[3]), dtype=np.float64)
    lse = np.empty((B, H, nq), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            s = scores(q[b, h], k[b, h], scale, causal, row_offset=nk - nq)
            p, m, l = softmax_three_pass(s)
            o[b, h] = p @ v[b, h]
            lse[b, h] = m + np.log(l)
    return o, lse


def split_bounds(nk, num_splits, tile=128):
    """Key ranges of the splits: whole ``tile``-key tiles, spread as evenly as possible.

    Split s covers tiles [s * T // S, (s + 1) * T // S) of the T = ceil(Nk / tile)
    tiles (the last one clipped at Nk); a split may be empty when S > T.
    """
    tiles = (nk + tile - 1) // tile
    out = []
    for s in range(num_splits):
        a = (s * tiles) // num_splits * tile
        b = min(nk, ((s + 1) * tiles) // num_splits * tile)
        out.append((a, max(a, b)))
    return out


def split_partials(q, k, v, scale, causal, bounds):
    """Each split's own softmax attention over keys [a, b) only.

    Returns ``o_s [S, B, H, Nq, d]`` (normalised within the split) and
    ``lse_s [S, B, H, Nq]``; a (split, query) with no visible key gets lse -inf
    and a zero row.
    """
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    B, H, nq, d = q.shape
    nk = k.shape[2]
    S = len(bounds)
    o_s = np.zeros((S, B, H, nq, v.shape[3]), dtype=np.float64)
    lse_s = np.full((S, B, H, nq), -np.inf, dtype=np.float64)
    for si, (a, b) in enumerate(bounds):
        if b <= a:
            continue
        for bb in range(B):
            for h in range(H):
                # scores of the split's keys, masked as in the full row
                s = scores(q[bb, h], k[bb, h], scale, causal, row_offset=nk - nq)[:, a:b]
                for i in range(nq):
                    row = s[i]
                    if np.all(row == -np.inf):
                        continue
                    p, m, l = softmax_three_pass(row[None, :])
                    o_s[si, bb, h, i] = p[0] @ v[bb, h, a:b]
                    lse_s[si, bb, h, i] = m[0] + np.log(l[0])
    return o_s, lse_s


def merge_partials(o_s, lse_s):
    """Merge per-split (O_s, lse_s) into the full (O, lse).

    The online-softmax rescale applied across splits: with m = max_s lse_s,
    weights w_s = exp(lse_s - m) (0 for an empty split), l = sum_s w_s,
    O = sum_s w_s O_s / l and lse = m + ln l.  (lse_s = m_s + ln l_s, so
    w_s = l_s exp(m_s - m) / exp(0): the [T] update with each split's sum and
    output rescaled to the common maximum.)
    """
    o_s = np.asarray(o_s, dtype=np.float64)
    lse_s = np.asarray(lse_s, dtype=np.float64)
    m = np.max(lse_s, axis=0)
    w = np.where(np.isneginf(lse_s), 0.0, np.exp(lse_s - m[None]))
    l = np.sum(w, axis=0)
    o = np.sum(w[..., None] * o_s, axis=0) / l[..., None]
    return o, m + np.log(l)

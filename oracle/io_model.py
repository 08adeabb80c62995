"""The pages' analytic memory and IO model of standard vs tiled attention.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  These are the closed
forms the pages print; tests pin them to the pages' own worked numbers, and
``bench.py`` quotes them as context beside measured traffic.

Units: "accesses" and "elements" count matrix elements; "bytes" multiply by
the element size given.
"""

from __future__ import annotations

import math


def standard_hbm_accesses(n, d):
    """Theta(N d + N^2) HBM accesses of standard attention.

    [T] "FlashAttention's move: rescale the output, too" and [L] Step 5
    "IO Savings" (Theorem 2 of the original paper as the page quotes it).
    """
    return n * d + n * n


def flash_hbm_accesses(n, d, m_sram):
    """Theta(N^2 d^2 / M) HBM accesses of the tiled method, M = on-chip size in elements.

    [T] "FlashAttention's move: rescale the output, too"; [L] Step 5.
    """
    return n * n * d * d / m_sram


def kv_tile_rows(m_sram, d):
    """K/V tile height ceil(M / 4d) that [L] Step 3 "Tiling" attributes to the paper."""
    return math.ceil(m_sram / (4 * d))


def q_block_rows(m_sram, d):
    """Q block height min(ceil(M / 4d), d), [L] Step 3 "Tiling"."""
    return min(kv_tile_rows(m_sram, d), d)


def score_matrix_bytes(n, elem_bytes=2):
    """Size of one head's N x N score (or probability) matrix.

    [T] "The hierarchy attention keeps ignoring" (N = 4096 in fp16) and [L]
    Step 1/Step 2 (one head's S at N = 4096).
    """
    return n * n * elem_bytes


def standard_traffic_elements_per_head(n, d):
    """About 4 N^2 + 4 N d elements moved per head by the three-kernel path, [L] Step 2.

    S written and read, P written and read (4 N^2); Q, K, V read and O
    written (4 N d).
    """
    return 4 * n * n + 4 * n * d


def standard_sp_share(n, d):
    """Fraction of the per-head traffic that is S and P round trips, [L] Step 2."""
    return 4 * n * n / standard_traffic_elements_per_head(n, d)


def layer_memory_time_s(n, d, heads, bandwidth_bytes_per_s, elem_bytes=2):
    """Time one layer's standard-attention traffic takes at a given bandwidth, [L] Step 2."""
    return heads * standard_traffic_elements_per_head(n, d) * elem_bytes / bandwidth_bytes_per_s


def extra_memory_bytes_standard(n, elem_bytes=2):
    """Extra memory per head kept by standard attention: the N^2 scores, [L] Step 5."""
    return n * n * elem_bytes


def extra_memory_bytes_flash(n, stat_bytes=4):
    """Extra memory per head kept by the tiled method: m and l per row (O(N)), [L] Step 5."""
    return 2 * n * stat_bytes


def tile_step_sram_bytes(block_rows, d, elem_bytes=2):
    """On-chip bytes of one tile step: Q block, K tile, V tile, S tile, O block.

    [L] Step 3 "Tiling" (fp16 tiles; fp32 accumulators and statistics not counted).
    """
    qkvo = 4 * block_rows * d * elem_bytes
    s_tile = block_rows * block_rows * elem_bytes
    return qkvo + s_tile


def attention_flops(b, h, n, d, causal, backward=False):
    """FLOPs by the formula this library reports throughput with.

    4 B H N^2 d for the forward (two N x N x d contractions, [L] Step 2 counts
    about 4 N^2 d per head), halved under the causal mask; the backward counts
    2.5 times the forward (five contractions instead of two).
    """
    f = 4.0 * b * h * n * n * d
    if causal:
        f /= 2.0
    if backward:
        f *= 2.5
    return f

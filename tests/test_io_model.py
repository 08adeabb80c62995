"""Pins of the IO-model helpers against the numbers the pages print (CPU only).

Fixture: tests/golden/io_model_numbers.txt (each block cites its passage).
"""

from oracle import io_model as io

MB = 1e6
MiB = 2 ** 20
KiB = 1024


def _close(value, printed, digits):
    """``value`` rounds to the printed figure at the printed number of digits."""
    return round(value, digits) == round(printed, digits)


def test_step5_io_savings(golden):
    g = golden("io_model_numbers.txt")
    n, d, m = int(g["step5.n"]), int(g["step5.d"]), int(g["step5.m_elements"])
    std = io.standard_hbm_accesses(n, d)
    fl = io.flash_hbm_accesses(n, d, m)
    assert _close(std / 1e6, g["step5.standard_accesses_millions"], 1)
    assert _close(fl / 1e6, g["step5.flash_accesses_millions"], 1)
    assert _close(std / fl, g["step5.ratio"], 1)
    assert io.kv_tile_rows(m, d) == g["step5.kv_tile_rows"]
    assert io.q_block_rows(m, d) == min(192, d)
    assert _close(io.extra_memory_bytes_standard(n) / MB, g["step5.extra_standard_mb"], 0)
    assert _close(io.extra_memory_bytes_flash(n) / 1e3, g["step5.extra_flash_kb"], 0)


def test_step2_standard_attention_traffic(golden):
    g = golden("io_model_numbers.txt")
    n, d, heads = int(g["step2.n"]), int(g["step2.d"]), int(g["step2.heads"])
    assert _close(io.score_matrix_bytes(n) / MB, g["step2.s_per_head_mb"], 0)
    assert _close(io.standard_traffic_elements_per_head(n, d) * 2 / MB, g["step2.traffic_per_head_mb"], 0)
    assert _close(100 * io.standard_sp_share(n, d), g["step2.sp_share_percent"], 0)
    t = io.layer_memory_time_s(n, d, heads, g["step2.bandwidth_tb_s"] * 1e12)
    assert _close(t * 1e3, g["step2.layer_time_ms"], 2)
    assert _close(heads * io.score_matrix_bytes(n) / 1e9, g["step2.s_layer_gb"], 1)
    assert _close(io.score_matrix_bytes(n) / MB, g["step1.s_4096_mb"], 1)


def test_step3_tiling_footprint(golden):
    g = golden("io_model_numbers.txt")
    rows, d = int(g["step3.block_rows"]), int(g["step3.d"])
    assert io.tile_step_sram_bytes(rows, d) / KiB == g["step3.sram_kib"]
    assert rows * d * 2 / KiB == g["step3.q_tile_kib"]
    assert rows * rows * 2 / KiB == g["step3.s_tile_kib"]


def test_teqners_score_matrix_size(golden):
    g = golden("io_model_numbers.txt")
    assert io.score_matrix_bytes(int(g["teqners.n"])) / MiB == g["teqners.s_mib"]


def test_flop_formula():
    # 4 B H N^2 d forward, halved for causal, backward 2.5x the forward
    assert io.attention_flops(1, 1, 10, 2, False) == 800
    assert io.attention_flops(1, 1, 10, 2, True) == 400
    assert io.attention_flops(1, 1, 10, 2, True, backward=True) == 1000
    gpt2 = io.attention_flops(64, 16, 1024, 64, True)
    assert round(gpt2 / 1e9, 1) == 137.4

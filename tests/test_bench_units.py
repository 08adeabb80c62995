"""The CPU baseline's accounting in bench.py (no GPU needed).

The oracle is timed on sample units (one block of up to 1024 query rows of one
(b, h) slice) and credited with the metric's FLOPs for the rows it ran.  Under
the causal mask row i covers keys 0 .. i, so blocks late in a slice carry more
work than early ones; the credit follows the (query, key) pairs, counted here
by brute force, and the units of a workload add up to its whole step.
"""

import workloads

import bench


def _w(B, H, N, causal, backward=True):
    return workloads.Workload(f"t_b{B}_h{H}_n{N}", 99, B, H, N, 64, causal, backward)


CASES = [_w(1, 2, 4096, True), _w(2, 3, 3000, True), _w(1, 2, 4096, False), _w(3, 1, 2500, False),
         _w(1, 4, 1000, True, backward=False), _w(2, 2, 5000, True)]


def test_units_add_up_to_the_step():
    for w in CASES:
        fwd, bwd = bench.flops_per_step(w)
        total = sum(bench.oracle_unit_flops(w, r0, rows) for _, _, r0, rows in bench.oracle_units(w))
        assert abs(total - (fwd + bwd)) <= 1e-9 * (fwd + bwd), w.name


def test_causal_credit_follows_the_attended_pairs():
    w = _w(1, 1, 2500, True)
    fwd, bwd = bench.flops_per_step(w)
    slice_pairs = sum(i + 1 for i in range(w.N))  # brute force
    for _, _, r0, rows in bench.oracle_units(w):
        pairs = sum(i + 1 for i in range(r0, r0 + rows))
        expect = (fwd + bwd) * pairs / slice_pairs
        assert abs(bench.oracle_unit_flops(w, r0, rows) - expect) <= 1e-9 * expect
    first, last = bench.oracle_unit_flops(w, 0, 1024), bench.oracle_unit_flops(w, 2048, 452)
    assert last > first  # 452 late rows outweigh 1024 early ones


def test_noncausal_credit_is_per_row():
    w = _w(2, 3, 3000, False)
    fwd, bwd = bench.flops_per_step(w)
    for _, _, r0, rows in bench.oracle_units(w):
        expect = (fwd + bwd) * rows / (w.B * w.H * w.N)
        assert abs(bench.oracle_unit_flops(w, r0, rows) - expect) <= 1e-9 * expect

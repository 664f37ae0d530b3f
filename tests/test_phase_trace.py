"""The phase-trace summariser of the profiling build (host logic, CPU): a synthetic timeline
with known phase lengths comes back as those lengths, per layer, median and max over blocks."""

import numpy as np

from moe_decode_weight_gb300 import phase_trace as PT


def test_summarise_recovers_phase_lengths():
    layers, blocks = 3, 5
    tr = np.zeros((layers, PT.TRACE_POINTS, blocks), dtype=np.uint64)
    t = np.full(blocks, 1_000_000, dtype=np.int64)
    lengths = {}
    for l in range(layers):
        tr[l, 0] = t
        for k, (point, name) in enumerate(PT.PHASES):
            ns = 100 * (k + 1) + 1000 * l + np.arange(blocks) * 10   # block b is 10 ns slower
            t = t + ns
            tr[l, point] = t
            lengths[(l, name)] = ns
    rows = PT.summarise(tr)
    assert len(rows) == layers
    for l, row in enumerate(rows):
        for _, name in PT.PHASES:
            med, mx = row[name]
            assert med == np.median(lengths[(l, name)]) / 1000.0
            assert mx == lengths[(l, name)].max() / 1000.0
        assert row["total_us"] == (tr[l, 9].max() - tr[l, 0].min()) / 1000.0
    assert "L2: total" in PT.format_rows(rows)


def test_phase_points_cover_the_layer_once():
    points = [p for p, _ in PT.PHASES]
    assert len(set(points)) == len(points) and points[-1] == 9 and 0 not in points
    assert all(0 < p < PT.TRACE_POINTS for p in points)

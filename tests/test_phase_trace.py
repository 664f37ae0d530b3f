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


def test_summarise_head_phases_and_timeline():
    blocks = 20
    tr = np.zeros((blocks, PT.HEAD_SLOTS), dtype=np.uint64)
    t0 = 5_000_000
    b = np.arange(blocks, dtype=np.int64)
    tr[:, 0] = t0 + b                                   # block starts (first at t0)
    tr[:, 1] = tr[:, 0] + 1000
    for w in range(PT.HEAD_WARPS):                      # warp w of block b ends at 60 us + 100 w + b
        tr[:, 8 + w] = t0 + 60_000 + 100 * w + b
    tr[:, 2] = tr[:, 8 + PT.HEAD_WARPS - 1] + 10
    tr[:, 20] = tr[:, 2] + 2000
    tr[:, 21] = tr[:, 20] + 1500
    tr[:, 22] = tr[:, 21] + 2500
    tr[:, 3] = tr[:, 22] + 300
    tr[:, 4] = 1                                        # stale from an older launch
    tr[[15, 19], 4] = tr[[15, 19], 3] + 700             # this launch's two group mergers
    tr[:, 5] = 1
    tr[19, 5] = tr[19, 4] + 4000
    tr[19, 6] = tr[19, 5] + 2000
    s = PT.summarise_head(tr)
    assert s["hidden states"] == (1.0, 1.0, 1.0)
    assert s["cut tiles"] == (2.0, 2.0, 2.0) and s["block tree"] == (2.5, 2.5, 2.5)
    assert s["warp spread"] == (1.1, 1.1, 1.1)
    assert s["tiles done (from start)"][2] == (60_000 + 1100 + 19 + 10) / 1000.0
    assert s["group mergers"] == 2
    assert s["final merge start"] == (float(tr[19, 5]) - t0) / 1000.0
    assert s["end"] == s["final merge start"] + 2.0
    assert "group mergers: 2" in PT.format_head(s)

"""The timeline summary on a synthetic stamp array (host logic, no GPU)."""
import numpy as np

from weight_streaming_q4_gb300 import timeline, _lib


def _fake(n_layers=2, grid=4, phase_us=(3.0, 2.0, 12.0, 6.0), gap_us=2.0):
    """Every CTA: phase p reached/staged/last unit/stored at fixed offsets."""
    tl = np.zeros((_lib.TIMELINE_CTAS, _lib.TIMELINE_PHASES, _lib.TIMELINE_EVENTS), np.uint64)
    t = 1_000_000.0
    n_phases = 4 * n_layers + 1
    for p in range(n_phases):
        dur = phase_us[p % 4] if p < n_phases - 1 else 0.0
        for c in range(grid):
            skew = 0.1 * c
            tl[c, p, 0] = t * 1e3
            tl[c, p, 1] = (t + 0.1) * 1e3
            tl[c, p, 2] = (t + gap_us) * 1e3
            if dur:
                tl[c, p, 3] = (t + gap_us + dur + skew) * 1e3
                tl[c, p, 4] = (t + gap_us + dur + skew + 0.2) * 1e3
                tl[c, p, 5] = (t + 0.5) * 1e3
        t += gap_us + dur + 0.1 * (grid - 1) + 0.2
    return tl, n_phases, grid


def test_summary_splits_a_layer():
    tl, n_phases, grid = _fake()
    r = timeline.summarise(tl, n_phases, grid)
    assert len(r["phases"]) == n_phases and r["phases"][-1]["kind"] == "closing"
    lay = r["layers"][0]
    # per phase: loop (median CTA) = dur + median skew; spread = max - median skew; the
    # boundary from the slowest store to the next median staging = gap_us
    assert abs(lay["unit_loops_us"] - (3 + 2 + 12 + 6 + 4 * 0.15)) < 0.05
    assert abs(lay["spread_us"] - 4 * 0.15) < 0.05
    assert abs(lay["boundaries_us"] - 4 * 2.0) < 0.05
    assert 0 < lay["unit_loop_frac"] < 1


def test_batched_summary_splits_a_layer():
    """The batched engine's layout: phase 0 an RMSNorm, then q|k|v, o, norm,
    gate|up, down, norm per layer; a layer spans the previous layer's last
    RMSNorm (slowest CTA published) to its own, and its product loops are the
    median CTA's first stage landed -> last unit of the four product phases."""
    n_layers, grid = 3, 4
    loop_us = {1: 2.0, 2: 2.0, 4: 18.0, 5: 10.0}   # by position in the layer
    tl = np.zeros((_lib.TIMELINE_CTAS, _lib.TIMELINE_PHASES, _lib.TIMELINE_EVENTS), np.uint64)
    t = 1_000_000.0
    for p in range(6 * n_layers + 1):
        pos = 0 if p == 0 else (p - 1) % 6 + 1
        dur = loop_us.get(pos, 0.0)
        for c in range(grid):
            tl[c, p, 0] = t * 1e3
            tl[c, p, 1] = (t + 0.5) * 1e3
            tl[c, p, 2] = (t + 1.0) * 1e3
            if dur:
                tl[c, p, 3] = (t + 1.0 + dur) * 1e3
                tl[c, p, 5] = (t + 0.8) * 1e3
            tl[c, p, 4] = (t + 1.0 + dur + 1.5 + 0.1 * c) * 1e3
        t += 1.0 + dur + 1.5 + 0.1 * (grid - 1) + 2.0
    r = timeline.summarise_batched(tl, n_layers, grid)
    assert [p["kind"] for p in r["phases"][:7]] == ["norm", "q|k|v", "o", "norm", "gate|up", "down", "norm"]
    assert len(r["layers"]) == n_layers - 1
    for lay in r["layers"]:
        assert abs(lay["unit_loops_us"] - sum(loop_us.values())) < 1e-6
        per_phase = 1.0 + 1.5 + 0.1 * (grid - 1) + 2.0
        assert abs(lay["us"] - (sum(loop_us.values()) + 6 * per_phase)) < 1e-6
        assert abs(lay["rest_us"] - 6 * per_phase) < 1e-6

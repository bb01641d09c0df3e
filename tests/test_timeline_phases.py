"""The phase summary of `bench.py --timeline` on hand-made stamps (CPU)."""
import numpy as np

import bench


def stamps(release, stream_end, end, ctas=4):
    a = np.zeros((ctas, 8, 3), np.int64)
    for c in range(ctas):
        for w in range(8):
            a[c, w] = [release + c * 100, stream_end[c] + w, end[c] + w]
    return a


def test_phases_of_hand_made_launches():
    t = 1_000_000
    a = stamps(t, [t + 30_000, t + 35_000, t + 40_000, t + 38_000],
               [t + 33_000, t + 36_000, t + 45_000, t + 39_000])
    b = stamps(t + 48_000, [0] * 4, [0] * 4)
    ph = bench.timeline_phases(a, b)
    assert ph["ctas"] == 4
    assert ph["release_spread_us"] == 0.3
    assert ph["stream_end_us"]["max"] == 40.01                # latest warp of the slowest CTA
    assert ph["cta_end_us"]["max"] == 45.01
    assert ph["end_phase_us"]["max"] == 5.0
    assert ph["next_release_us"] == 48.0
    assert ph["gap_after_last_end_us"] == 2.99


def test_a_cta_without_work_is_left_out():
    t = 5_000
    a = stamps(t, [t + 9000] * 3, [t + 9500] * 3, ctas=3)
    a[1] = 0                                                  # no work: wrote nothing
    ph = bench.timeline_phases(a, np.zeros_like(a))
    assert ph["ctas"] == 2
    assert ph["next_release_us"] is None and ph["gap_after_last_end_us"] is None

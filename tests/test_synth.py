"""The seeded input generators (shared by both sides; no method arithmetic)."""
import numpy as np

import synth
from conftest import golden_lines


def test_splitmix64_published_vector():
    want = [int(r[0]) for r in golden_lines("splitmix64_seed1234567.txt")]
    got = [int(v) for v in synth.draws(1234567, np.arange(5))]
    assert got == want


def test_q_range_and_uniformity():
    q = synth.q_full(synth.seed_of(0, 0, 0, synth.T_Q), 256, 1024)
    assert q.min() == -8 and q.max() == 7
    h = np.bincount((q.astype(np.int64) + 8).ravel(), minlength=16)
    assert np.all(np.abs(h / q.size - 1 / 16) < 0.002)


def test_scale_range():
    s = synth.scale_full(synth.seed_of(0, 0, 0, synth.T_SCALE), 512, 28).view(np.float16)
    v = s.astype(np.float64)
    assert v.min() >= 0.005 - 1e-5 and v.max() <= 0.02 + 1e-5
    assert abs(v.mean() - 0.0125) < 2e-4


def test_x_standard_normal():
    x = synth.x_full(synth.seed_of(0, 0, 0, synth.T_X), 16, 4096).view(np.float16).astype(np.float64)
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1) < 0.02


def test_row_sampling_equals_slicing():
    sq = synth.seed_of(1, 2, 3, synth.T_Q)
    full = synth.q_full(sq, 40, 256)
    rows = np.array([0, 7, 39, 13])
    assert np.array_equal(synth.q_rows(sq, 256, rows), full[rows])
    ss = synth.seed_of(1, 2, 3, synth.T_SCALE)
    assert np.array_equal(synth.scale_rows(ss, 2, rows), synth.scale_full(ss, 40, 2)[rows])


def test_seeds_are_distinct():
    seeds = {synth.seed_of(c, l, p, t) for c in range(5) for l in range(28)
             for p in range(4) for t in range(3)}
    assert len(seeds) == 5 * 28 * 4 * 3

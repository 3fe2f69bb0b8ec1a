"""Pins of the oracle's non-uniform level-table fit (KVQuant summary,
"technical approach": per-layer non-uniform datatypes computed offline; here
the unweighted version -- Lloyd's algorithm on calibration vectors -- since
the sensitivity weights need a model's gradients).

What fixes the fit without retyping it: Lloyd's fixed point (every free
level is the mean of the values it is nearest to), exact recovery of a
planted 8-point distribution, the closed form for uniform data (equally
spaced levels), a distortion that never grows from one update to the next,
and hand-computed grid positions that drop exactly the encoder's outliers."""
import numpy as np
import pytest

from oracle import kvq_oracle as O

D = 128
GRID = 65536


def _cells(pos, levels):
    """Index of the nearest level of every position (ties go down)."""
    t = (levels[:-1] + levels[1:]) / 2.0
    return (pos[:, None].astype(np.float64) > t[None, :]).sum(1)


def test_positions_by_hand():
    """mn = -1, mx = 3 on the dense part, two outliers (+-40) removed:
    position = rint((x + 1) / 4 * 2^16)."""
    x = np.zeros(D, np.float16)
    x[:] = 0.5
    x[3], x[9] = -1.0, 3.0
    x[5], x[70] = 40.0, -40.0
    x[11] = 0.25
    pos = O.nuq_fit_positions(x[None, :], k=2)
    assert pos.size == D - 2
    want = np.rint((x.astype(np.float64) + 1.0) / 4.0 * GRID).astype(np.int64)
    keep = np.ones(D, bool)
    keep[[5, 70]] = False
    assert np.array_equal(pos, want[keep])
    assert pos.min() == 0 and pos.max() == GRID
    # the dropped channels are the encoder's outliers
    _, _, _, cols, _ = O.nuq_encode(x, 2, [-1.5, -0.9, -0.5, -0.2, 0.2, 0.5, 0.9, 1.5])
    assert sorted(cols.tolist()) == [5, 70]
    # a constant dense part contributes no position
    assert O.nuq_fit_positions(np.full((1, D), 0.75, np.float16), k=0).size == 0


def test_planted_levels_are_recovered_exactly():
    rng = np.random.default_rng(3)
    planted = np.array([0.0, 0.125, 0.3125, 0.4375, 0.5625, 0.6875, 0.875, 1.0])
    x = planted[rng.integers(0, 8, (500, D))].astype(np.float16)
    x[:, 0], x[:, 1] = 0.0, 1.0              # every dense part spans [0, 1]: positions are exact
    x[:, 2] = 30.0 * rng.choice([-1, 1], 500)  # one outlier per vector, removed
    lut, it, lv = O.nuq_fit_lut(x, k=1, levels=True)
    assert it >= 1
    assert np.array_equal(lv, planted * GRID)
    assert lut == planted.tolist()


def test_fixed_point_property():
    """At convergence each interior level equals the mean of its cell's
    positions; the end levels stay at 0 and 1."""
    x = np.random.default_rng(5).standard_normal((1500, D)).astype(np.float16)
    lut, it, lv = O.nuq_fit_lut(x, k=2, max_iters=500, levels=True)
    assert 0 < it < 500
    assert lv[0] == 0.0 and lv[7] == GRID and lut[0] == 0.0 and lut[7] == 1.0
    pos = O.nuq_fit_positions(x, k=2)
    c = _cells(pos, lv)
    for i in range(1, 7):
        sel = pos[c == i].astype(np.int64)
        assert sel.size > 0
        assert float(sel.sum()) / float(sel.size) == lv[i]
    assert all(b > a for a, b in zip(lut, lut[1:]))


def test_uniform_data_gives_equally_spaced_levels():
    """For a uniform density on [0, 1] with the ends held, the Lloyd fixed
    point is l_i = i / 7 (each cell's mean is its level); the sample gives it
    to within sampling noise."""
    rng = np.random.default_rng(9)
    x = rng.uniform(0.0, 1.0, (2000, D)).astype(np.float16)
    x[:, 0], x[:, 1] = 0.0, 1.0
    lut, it, lv = O.nuq_fit_lut(x, k=0, max_iters=500, levels=True)
    assert np.allclose(lv / GRID, np.arange(8) / 7.0, atol=3e-3)


def test_distortion_never_grows():
    """Lloyd: every update lowers (or keeps) the squared distance of the
    positions to their nearest level."""
    x = np.random.default_rng(13).laplace(size=(800, D)).astype(np.float16)
    pos = O.nuq_fit_positions(x, k=2).astype(np.float64)
    prev = np.inf
    for n in range(1, 12):
        _, _, lv = O.nuq_fit_lut(x, k=2, max_iters=n, levels=True)
        dist = float(((pos - lv[_cells(pos, lv)]) ** 2).sum())
        assert dist <= prev * (1 + 1e-12)
        prev = dist


def test_hadamard_option_fits_the_rotated_vectors():
    x = np.random.default_rng(17).standard_t(3, (300, D)).astype(np.float16)
    rot = np.stack([O.hadamard_rotate(v) for v in x]).view(np.float16)
    assert O.nuq_fit_lut(x, k=2, hadamard=1) == O.nuq_fit_lut(rot, k=2, hadamard=0)
    assert not np.array_equal(O.nuq_fit_positions(x, 2, 1), O.nuq_fit_positions(x, 2, 0))


def test_fitted_table_beats_the_quantile_table_on_its_data():
    """The fitted levels lower the encoder's reconstruction error on the data
    they were fitted to, against the seeded N(0, 1) quantile table."""
    rng = np.random.default_rng(21)
    x = rng.laplace(size=(400, D)).astype(np.float16)
    fitted, _ = O.nuq_fit_lut(x, k=2)
    xs = np.sort(np.random.default_rng(0).standard_normal(65536))
    quant = [float(v) for v in xs[((np.arange(8) + 0.5) * 65536 / 8).astype(int)].astype(np.float16)]

    def mse(lut):
        e = 0.0
        for v in x:
            codes, mn, s, cols, vals = O.nuq_encode(v, 2, lut)
            e += float(((O.nuq_decode(codes, mn, s, lut, cols, vals) - v.astype(np.float64)) ** 2).sum())
        return e

    assert mse(fitted) < mse(quant)

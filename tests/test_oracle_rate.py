"""Pins of the oracle's per-head bit allocation (RateQuant summary,
"Methodology" 1, 3 and 4): the measured distortion of the cache's quantizer,
the fit D(b) = alpha beta^-b, reverse water-filling and the greedy
marginal-gain allocation over the bit widths the cache supports.

Fixed by: zero distortion on on-grid data and the step^2 / 12 law on
uniform data; the same error as the stored cache's reconstruction; exact
recovery of model-generated curves and numpy's least squares; the page's
closed form for a common beta and stationarity for per-component beta; the
budget, monotonicity and no improving exchange for the greedy result, and
brute force where all steps cost the same."""
import itertools

import numpy as np
import pytest

from oracle import kvq_oracle as O

D = 128


def cfg(**kw):
    c = dict(head_dim=D, k_bits=4, v_bits=4, k_group_tokens=32, v_group_channels=64, v_hadamard=0,
             hybrid_groups=0, k_group_channels=0, k_channel_norm=0)
    c.update(kw)
    return c


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_distortion_zero_on_grid_and_uniform_law(bits):
    rng = np.random.default_rng(bits)
    q = (1 << bits) - 1
    T = 64
    # on the grid of every K channel group and every V token group: zero error
    codes = rng.integers(0, q + 1, (T, D))
    codes[0], codes[1] = 0, q
    codes[32], codes[33] = 0, q
    K = (codes * 2.0 ** -4 - 1.0).astype(np.float16)
    vc = rng.integers(0, q + 1, (T, D))
    vc[:, 0], vc[:, 1], vc[:, 64], vc[:, 65] = 0, q, 0, q
    V = (vc * 2.0 ** -5).astype(np.float16)
    assert O.quant_distortion(cfg(), K, V, bits) == (0.0, 0.0)
    # uniform values: MSE close to step^2 / 12 with step = range / (2^b - 1)
    if bits <= 4:
        X = rng.uniform(-1, 1, (4096, D)).astype(np.float16)
        X[:, 0], X[:, 1], X[:, 64], X[:, 65] = -1, 1, -1, 1  # both 64-channel groups span [-1, 1]
        dk, dv = O.quant_distortion(cfg(), X, X, bits)
        law = (2.0 / q) ** 2 / 12
        assert abs(dv / law - 1) < 0.05


def test_distortion_matches_the_stored_cache():
    """The K and V error of a cache the oracle builds (no sinks or window,
    T a multiple of 32) equals the measured distortion at the same bits."""
    rng = np.random.default_rng(4)
    T = 256
    K = rng.standard_normal((T, D)).astype(np.float16)
    V = rng.laplace(size=(T, D)).astype(np.float16)
    for kb, vb in [(4, 4), (2, 8)]:
        c = cfg(k_bits=kb, v_bits=vb, n_sink=0, n_recent=0, rope_theta=1e4, outliers_per_vector=0,
                softmax_scale=0.0, k_pre_rope=0)
        st = O.build_stream(c, K, V)
        kcodes = np.stack([O.unpack_bits(r, D, kb) for r in st["kc"]]).astype(np.float64)
        ks = st["ks"].view(np.float16).astype(np.float64)  # [groups, d, 2]
        kh = ks[np.arange(T) // 32, :, 0] + kcodes * ks[np.arange(T) // 32, :, 1]
        vcodes = np.stack([O.unpack_bits(r, D, vb) for r in st["vc"]]).astype(np.float64)
        vs = st["vs"].view(np.float16).astype(np.float64)  # [T, 2, 2]
        vh = vs[:, np.arange(D) // 64, 0] + vcodes * vs[:, np.arange(D) // 64, 1]
        dk_cache = np.mean((kh - K.astype(np.float64)) ** 2)
        dv_cache = np.mean((vh - V.astype(np.float64)) ** 2)
        dk, _ = O.quant_distortion(c, K, V, kb)
        _, dv = O.quant_distortion(c, K, V, vb)
        assert abs(dk - dk_cache) <= 1e-12 * dk_cache and abs(dv - dv_cache) <= 1e-12 * dv_cache


def test_distortion_falls_about_fourfold_per_bit():
    rng = np.random.default_rng(6)
    K = rng.standard_normal((512, D)).astype(np.float16)
    V = rng.laplace(size=(512, D)).astype(np.float16)
    d = [O.quant_distortion(cfg(), K, V, b) for b in (2, 4, 8)]
    for side in (0, 1):
        a, beta = O.fit_rd([2, 4, 8], [x[side] for x in d])
        assert d[0][side] > d[1][side] > d[2][side] > 0
        assert 3.0 < beta < 5.5  # ~4 per bit for a uniform grid


def test_fit_recovers_the_model_and_matches_least_squares():
    for a0, b0 in [(2.5, 4.2), (0.03, 3.6), (11.0, 5.3)]:
        b = np.array([2.0, 4.0, 8.0])
        a, be = O.fit_rd(b, a0 * b0 ** -b)
        assert abs(a / a0 - 1) < 1e-12 and abs(be / b0 - 1) < 1e-12
    rng = np.random.default_rng(1)
    b = np.array([2.0, 3.0, 4.0, 6.0, 8.0])
    Dv = 3.0 * 4.0 ** -b * np.exp(rng.normal(0, 0.1, b.size))
    a, be = O.fit_rd(b, Dv)
    slope, icpt = np.polyfit(b, np.log(Dv), 1)
    assert abs(np.log(a) - icpt) < 1e-10 and abs(np.log(be) + slope) < 1e-10


def test_waterfill_closed_form_and_stationarity():
    rng = np.random.default_rng(2)
    n, B = 9, 9 * 4.0
    alpha = rng.uniform(0.1, 3, n)
    w = rng.uniform(0.2, 5, n)
    beta = np.full(n, 4.3)
    b = O.rate_waterfill(alpha, beta, B, w)
    wa = w * alpha
    closed = B / n + (np.log(wa) - np.log(wa).mean()) / np.log(4.3)  # the page's formula, w -> w alpha
    assert np.allclose(b, closed, atol=1e-9)
    beta2 = rng.uniform(3.6, 5.3, n)
    b2 = O.rate_waterfill(alpha, beta2, B, w)
    assert abs(b2.sum() - B) < 1e-9
    lam = w * alpha * np.log(beta2) * beta2 ** -b2
    assert np.allclose(lam, lam[0], rtol=1e-9)


def _objective(alpha, beta, w, bits):
    return float(np.sum(w * alpha * beta ** -np.asarray(bits, float)))


def test_greedy_budget_monotone_and_no_improving_exchange():
    rng = np.random.default_rng(3)
    for trial in range(40):
        n = int(rng.integers(2, 12))
        alpha = rng.uniform(0.05, 5, n)
        beta = rng.uniform(3.6, 5.3, n) if trial % 2 else np.full(n, 4.4)
        w = rng.uniform(0.2, 5, n)
        total = int(rng.integers(2 * n, 8 * n + 1))
        bits, used = O.rate_greedy(alpha, beta, total, w)
        assert used == bits.sum() <= total and set(bits.tolist()) <= {2, 4, 8}
        f = _objective(alpha, beta, w, bits)
        # no upgrade fits and improves, no (down, up) exchange within budget improves
        steps_up = {2: 4, 4: 8}
        steps_dn = {4: 2, 8: 4}
        for i in range(n):
            if bits[i] in steps_up and used + steps_up[bits[i]] - bits[i] <= total:
                raise AssertionError("an upgrade still fits")
        for i, j in itertools.permutations(range(n), 2):
            if bits[i] in steps_dn and bits[j] in steps_up:
                nb = bits.copy()
                nb[i], nb[j] = steps_dn[bits[i]], steps_up[bits[j]]
                if nb.sum() <= total:
                    assert _objective(alpha, beta, w, nb) >= f * (1 - 1e-12) or bits[j] == 4
        if trial % 2 == 0:  # common beta: larger w alpha never gets fewer bits
            order = np.argsort(w * alpha)
            assert np.all(np.diff(bits[order]) >= 0)


def test_greedy_equals_brute_force_when_steps_cost_the_same():
    """With a budget that admits only 2 -> 4 steps (each 2 bits), the greedy
    picks the k largest gains: the brute-force optimum."""
    rng = np.random.default_rng(8)
    for _ in range(30):
        n = int(rng.integers(2, 7))
        alpha = rng.uniform(0.05, 5, n)
        beta = rng.uniform(3.6, 5.3, n)
        k = int(rng.integers(0, n + 1))
        total = 2 * n + 2 * k + 1  # one spare bit: never enough for a 4 -> 8 step
        bits, _ = O.rate_greedy(alpha, beta, total)
        best = min((b for b in itertools.product([2, 4], repeat=n) if sum(b) <= total),
                   key=lambda b: _objective(alpha, beta, 1.0, b))
        assert _objective(alpha, beta, 1.0, bits) == pytest.approx(_objective(alpha, beta, 1.0, best), rel=1e-12)


def test_greedy_rejects_a_budget_below_two_bits_each():
    bits, used = O.rate_greedy([1.0, 1.0], [4.0, 4.0], 3)
    assert used == -1

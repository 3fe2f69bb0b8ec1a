"""The append kernel's uniform code without a division per element.

The kernel computes code = clamp(rint(RN((x - mn) / scale)), 0, 2^b - 1) as
rint(RN(d * RN(1 / scale))) and falls back to the IEEE division only when
that product lies within 1e-4 of a half-integer (|qa - rint(qa)| > 0.4999);
it drops the clamp, which never binds for x in [mn, mx].  This checks, in float32
arithmetic on the host (the same correctly rounded operations the kernel
uses), that the shortcut and the division give the same code everywhere
outside the guard band, over random groups and over quotients placed right
next to half-integers.  The non-uniform encoder's comparisons of
u = RN(d / s) with the level midpoints use the same product and fall back to
the division within 2^-21 relative of a midpoint; checked the same way."""
import numpy as np
import pytest


def codes_both(x, mn, scale, qmax):
    f = np.float32
    d = (x - mn).astype(f)
    rs = (f(1.0) / scale).astype(f)
    qa = (d * rs).astype(f)
    exact = np.clip(np.rint((d / scale).astype(f)), 0, qmax)  # the definition, clamped
    fast = np.rint(qa)
    guard = np.abs((qa - fast).astype(f)) > f(0.4999)        # within 1e-4 of a half-integer
    fast = np.where(guard, np.rint((d / scale).astype(f)), fast)  # the kernel: no clamp
    return fast, exact, guard


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_shortcut_equals_division_on_random_groups(bits):
    rng = np.random.default_rng(bits)
    qmax = np.float32(2 ** bits - 1)
    for _ in range(200):
        scale_mag = 10.0 ** rng.uniform(-4, 2)
        x = (rng.standard_normal(4096) * scale_mag).astype(np.float16).astype(np.float32)
        mn, mx = x.min(), x.max()
        scale = ((mx - mn) / qmax).astype(np.float32)
        if scale == 0:
            continue
        fast, exact, _ = codes_both(x, mn, scale, qmax)
        assert np.array_equal(fast, exact)


def test_shortcut_near_half_integers():
    # quotients pinned within a few ulps of k + 1/2 for every k: the guard
    # must catch all of them
    rng = np.random.default_rng(7)
    f = np.float32
    for bits in (2, 4, 8):
        qmax = f(2 ** bits - 1)
        for _ in range(2000):
            scale = f(10.0 ** rng.uniform(-3, 1))
            k = rng.integers(0, int(qmax))
            target = (f(k) + f(0.5)) * scale
            d = np.nextafter(target, np.inf if rng.random() < 0.5 else -np.inf).astype(f)
            for step in range(rng.integers(0, 4)):
                d = np.nextafter(d, f(np.inf)).astype(f)
            x = np.array([d], dtype=f)
            fast, exact, guard = codes_both(x, f(0.0), scale, qmax)
            assert fast[0] == exact[0]


def nuq_codes_both(x, mn, s, tau):
    """Code = #{i : u > tau_i}, u = RN(d / s): the kernel's product with the
    shared reciprocal and a relative guard band of 2^-21, against the
    division."""
    f = np.float32
    d = (x - mn).astype(f)
    rs = (f(1.0) / s).astype(f)
    uf = (d * rs).astype(f)
    ue = (d / s).astype(f)
    band = (uf * f(2.0 ** -21)).astype(f)
    near = (np.abs((uf[:, None] - tau[None, :]).astype(f)) <= band[:, None]).any(axis=1)
    u = np.where(near, ue, uf)
    fast = (u[:, None] > tau[None, :]).sum(axis=1)
    exact = (ue[:, None] > tau[None, :]).sum(axis=1)
    return fast, exact


def test_nuq_shortcut_equals_division():
    f = np.float32
    rng = np.random.default_rng(11)
    for trial in range(300):
        lut = np.sort(rng.standard_normal(8) * rng.uniform(0.5, 20)).astype(np.float16).astype(f)
        if np.any(np.diff(lut) <= 0):
            continue
        tau = ((lut[:-1] + lut[1:]).astype(f) * f(0.5) - lut[0]).astype(f)
        x = (rng.standard_normal(2048) * 10.0 ** rng.uniform(-3, 2)).astype(np.float16).astype(f)
        mn, mx = x.min(), x.max()
        s = ((mx - mn) / (lut[7] - lut[0])).astype(f)
        if s == 0:
            continue
        # also quotients placed within a few ulps of every midpoint
        near = []
        for t in tau:
            d0 = (t * s).astype(f)
            for k in range(-3, 4):
                near.append(mn + np.nextafter(d0, f(np.inf) if k > 0 else f(-np.inf)) if k else mn + d0)
        xs = np.concatenate([x, np.array(near, dtype=f)]).astype(f)
        fast, exact = nuq_codes_both(xs, mn, s, tau)
        assert np.array_equal(fast, exact), trial

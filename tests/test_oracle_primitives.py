"""Pins of the CPU oracle's primitives against things other than itself:
numpy's binary16 conversion, hand-computed golden values, brute force over
all quantization levels, scipy's Sylvester Hadamard matrix, and RoPE written
as complex multiplication."""
import json
import os

import numpy as np
import pytest
import scipy.linalg

from oracle import kvq_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------- fp16

def test_half_to_float_exhaustive_vs_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([O.half_to_float(int(b)) for b in bits], np.float32)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite].view(np.uint32), ref[finite].view(np.uint32))
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got) & (got > 0), np.isinf(ref) & (ref > 0))


def test_float_to_half_vs_numpy():
    rng = np.random.default_rng(1)
    halves = np.arange(0, 0x7c00, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float32)
    mids = (halves[:-1].astype(np.float64) + halves[1:]) / 2  # exact ties between neighbours
    mids = mids.astype(np.float32)
    near = np.concatenate([np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(0))])
    rand = np.concatenate([rng.standard_normal(20000) * s for s in (1e-7, 1e-5, 1e-2, 1, 100, 7e4)])
    xs = np.concatenate([halves, mids, near, rand.astype(np.float32)])
    xs = np.concatenate([xs, -xs]).astype(np.float32)
    with np.errstate(over="ignore"):
        ref = xs.astype(np.float16).view(np.uint16)
    got = np.array([O.float_to_half(float(x)) for x in xs], np.uint16)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(xs[i]), hex(got[i]), hex(ref[i])) for i in bad[:5]]


# ------------------------------------------------------------ quantizer

def test_uniform_quantizer_golden():
    cases = json.load(open(os.path.join(GOLD, "quant_examples.json")))["cases"]
    for c in cases:
        codes, mn, sc = O.quantize_uniform(np.array(c["x"], np.float16), c["bits"])
        assert list(codes) == c["codes"], c
        assert O.half_to_float(mn) == c["min"], c
        assert O.half_to_float(sc) == c["scale"], c


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_uniform_on_grid_roundtrip(bits):
    """x = min + code * scale with a power-of-two scale, an fp16 min and codes
    that reach 0 and 2^b - 1 must come back with the same codes, min, scale."""
    rng = np.random.default_rng(bits)
    qmax = (1 << bits) - 1
    for trial in range(200):
        n = int(rng.integers(2, 70))
        scale = 2.0 ** int(rng.integers(-8, 0))
        mn = float(np.float16(rng.uniform(-4, 4)))
        mn = np.round(mn / scale) * scale  # keep every grid point fp16-exact
        codes = rng.integers(0, qmax + 1, n)
        codes[:2] = [0, qmax]
        rng.shuffle(codes)
        x = (mn + codes * scale).astype(np.float16)
        assert np.array_equal(x.astype(np.float64), mn + codes * scale)
        got, gmn, gsc = O.quantize_uniform(x, bits)
        assert np.array_equal(got, codes)
        assert O.half_to_float(gmn) == mn and O.half_to_float(gsc) == scale


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_uniform_brute_force_nearest_level(bits):
    """The code is the nearest of the 2^b grid levels min + k*scale32 (found by
    exhaustive search in fp64), except within fp32 rounding of an exact tie;
    and |x - (min + code*scale32)| <= scale32/2 up to that rounding."""
    rng = np.random.default_rng(10 + bits)
    qmax = (1 << bits) - 1
    checked = 0
    for trial in range(300):
        n = int(rng.integers(2, 65))
        x = (rng.standard_normal(n) * rng.uniform(0.01, 20)).astype(np.float16)
        codes, mn_h, sc_h = O.quantize_uniform(x, bits)
        xf = x.astype(np.float32)
        mn, mx = xf.min(), xf.max()
        scale32 = np.float32(mx - mn) / np.float32(qmax)
        if scale32 == 0:
            assert not codes.any()
            continue
        assert O.half_to_float(mn_h) == mn
        assert sc_h == np.float32(scale32).astype(np.float16).view(np.uint16)
        levels = float(mn) + np.arange(qmax + 1) * float(scale32)
        dist = np.abs(xf.astype(np.float64)[:, None] - levels[None, :])
        best = dist.argmin(1)
        srt = np.sort(dist, 1)
        clear = (srt[:, 1] - srt[:, 0]) > 1e-5 * float(scale32)
        assert np.array_equal(codes[clear], best[clear])
        err = np.abs(xf.astype(np.float64) - (float(mn) + codes * float(scale32)))
        assert np.all(err <= float(scale32) * (0.5 + 1e-5))
        checked += int(clear.sum())
    assert checked > 1000


def test_uniform_error_falls_with_bits():
    """b = 8 error well under b = 4 (D(b) = alpha * beta^-b, RateQuant
    problem formulation: each extra bit divides the MSE by beta > 1)."""
    rng = np.random.default_rng(5)
    mse = {}
    for bits in (2, 4, 8):
        e = []
        for _ in range(200):
            x = rng.standard_normal(64).astype(np.float16)
            c, mn, sc = O.quantize_uniform(x, bits)
            xh = O.half_to_float(mn) + c * O.half_to_float(sc)
            e.append(np.mean((xh - x.astype(np.float64)) ** 2))
        mse[bits] = np.mean(e)
    assert mse[2] > 8 * mse[4] and mse[4] > 64 * mse[8]


# ---------------------------------------------------------------- packing

def test_pack_golden():
    for c in json.load(open(os.path.join(GOLD, "pack_examples.json")))["cases"]:
        got = O.pack_bits(c["codes"], c["bits"])
        assert list(got) == c["bytes"], c
        assert list(O.unpack_bits(got, len(c["codes"]), c["bits"])) == c["codes"]


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_pack_vs_numpy_bitstream(bits):
    """numpy.unpackbits(bitorder='little') of the packed row, read b bits at a
    time LSB-first, gives the codes back; pack o unpack is the identity."""
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, 1 << bits, 128).astype(np.uint8)
    packed = O.pack_bits(codes, bits)
    assert packed.size == 128 * bits // 8
    stream = np.unpackbits(packed, bitorder="little").reshape(128, bits)
    back = (stream * (1 << np.arange(bits))).sum(1)
    assert np.array_equal(back, codes)
    assert np.array_equal(O.unpack_bits(packed, 128, bits), codes)


# --------------------------------------------------------------- Hadamard

def test_hadamard_matrix_matches_scipy_and_squares_to_nI():
    n = 128
    H = scipy.linalg.hadamard(n)
    assert np.array_equal(H @ H, n * np.eye(n, dtype=H.dtype))
    # the oracle's dense fp64 map is Hn = H / sqrt(n): apply it to the unit vectors
    cols = np.stack([O.hadamard_apply(np.eye(n)[j]) for j in range(n)], 1)
    assert np.allclose(cols * np.sqrt(n), H, atol=1e-12)


def test_hadamard_apply_is_involution():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(128)
    assert np.allclose(O.hadamard_apply(O.hadamard_apply(x)), x, atol=1e-12)
    assert np.allclose(O.hadamard_apply(x), scipy.linalg.hadamard(128) @ x / np.sqrt(128), atol=1e-12)


def test_fwht_rotation_vs_dense():
    """fp32 butterflies then fp16 rounding agree with the dense fp64 product
    to within one fp16 rounding step (plus fp32 accumulation)."""
    rng = np.random.default_rng(4)
    H = scipy.linalg.hadamard(128) / np.sqrt(128)
    for _ in range(50):
        v = (rng.standard_t(3, 128)).astype(np.float16)
        got = O.hadamard_rotate(v).view(np.float16).astype(np.float64)
        ref = H @ v.astype(np.float64)
        ulp = np.spacing(np.abs(ref).astype(np.float16)).astype(np.float64)
        assert np.all(np.abs(got - ref) <= ulp * 0.5 + 1e-5 * np.abs(ref) + 1e-7)


# -------------------------------------------------------------------- NUQ

def _lut(seed=0):
    x = np.sort(np.random.default_rng(seed).standard_normal(65536))
    return x[((np.arange(8) + 0.5) * 65536 / 8).astype(int)].astype(np.float16).astype(np.float32)


def test_nuq_lut_shape():
    lut = _lut()
    assert np.all(np.diff(lut) > 0)
    assert np.allclose(lut, -lut[::-1], atol=0.05)  # N(0,1) quantiles are near-symmetric
    assert 1.3 < lut[-1] < 1.8


def test_nuq_outliers_match_sort_topk():
    rng = np.random.default_rng(7)
    lut = _lut()
    for _ in range(300):
        x = rng.standard_normal(128).astype(np.float16)
        if rng.random() < 0.3:  # force magnitude ties
            x[rng.integers(128)] = x[rng.integers(128)]
            x[rng.integers(128)] = -x[rng.integers(128)]
        k = int(rng.integers(0, 5))
        codes, mn, s, cols, vals = O.nuq_encode(x, k, lut)
        mag = np.abs(x.astype(np.float32))
        order = np.lexsort((np.arange(128), -mag))  # |x| descending, ties -> lower index
        want = np.sort(order[:k])
        assert np.array_equal(cols, want)
        assert np.array_equal(vals, x.view(np.uint16)[want])
        dense = np.setdiff1d(np.arange(128), want)
        assert O.half_to_float(mn) == x[dense].astype(np.float32).min()
        assert not codes[want].any()


def test_nuq_code_is_nearest_level():
    """Dense codes pick the nearest of the 8 affinely mapped LUT levels
    (brute force over the levels in fp64), except within rounding of a tie;
    the decode puts the outliers back exactly."""
    rng = np.random.default_rng(8)
    lut = _lut(1)
    checked = 0
    for _ in range(300):
        x = rng.laplace(size=128).astype(np.float16)
        codes, mn_h, s_h, cols, vals = O.nuq_encode(x, 2, lut)
        dense = np.setdiff1d(np.arange(128), cols)
        xd = x[dense].astype(np.float32)
        mn, mx = xd.min(), xd.max()
        s32 = np.float32(mx - mn) / np.float32(np.float32(lut[7]) - np.float32(lut[0]))
        u = (xd.astype(np.float64) - float(mn)) / float(s32)
        lev = lut.astype(np.float64) - float(lut[0])
        dist = np.abs(u[:, None] - lev[None, :])
        best = dist.argmin(1)
        srt = np.sort(dist, 1)
        clear = (srt[:, 1] - srt[:, 0]) > 1e-5
        assert np.array_equal(codes[dense][clear], best[clear])
        checked += int(clear.sum())
        rec = O.nuq_decode(codes, mn_h, s_h, lut, cols, vals)
        assert np.array_equal(rec[cols], x[cols].astype(np.float64))
        gap = np.max(np.diff(lut)) * O.half_to_float(s_h)
        assert np.all(np.abs(rec[dense] - xd) <= gap / 2 + 1e-3 * np.abs(xd) + 1e-6)
    assert checked > 30000


def test_nuq_on_grid_roundtrip():
    """Dense values exactly on the mapped levels s*L_c (s a power of two,
    levels L0 and L7 present) decode back exactly."""
    rng = np.random.default_rng(9)
    lut = _lut(2)
    for _ in range(100):
        s = 2.0 ** int(rng.integers(-4, 2))
        c = rng.integers(0, 8, 128)
        c[:2] = [0, 7]
        rng.shuffle(c)
        x = (s * lut[c].astype(np.float64)).astype(np.float16)
        assert np.array_equal(x.astype(np.float64), s * lut[c])
        codes, mn_h, s_h, cols, vals = O.nuq_encode(x, 0, lut)
        assert np.array_equal(codes, c)
        rec = O.nuq_decode(codes, mn_h, s_h, lut, cols, vals)
        assert np.array_equal(rec, x.astype(np.float64))


# ------------------------------------------------------------------- RoPE

def test_rope_vs_complex_rotation():
    """Rotate-half RoPE equals multiplying z_i = x_i + j x_{i+d/2} by
    exp(j * t * theta_i), theta_i = base^(-2i/d)."""
    rng = np.random.default_rng(11)
    d, base = 128, 10000.0
    th = base ** (-2.0 * np.arange(d // 2) / d)
    for t in [0, 1, 7, 1000, 123457, 1048575]:
        x = rng.standard_normal(d)
        z = (x[: d // 2] + 1j * x[d // 2:]) * np.exp(1j * t * th)
        got = O.rope_apply(x, t, base)
        assert np.allclose(got[: d // 2], z.real, atol=1e-9)
        assert np.allclose(got[d // 2:], z.imag, atol=1e-9)


def test_rope_invariants():
    rng = np.random.default_rng(12)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    assert np.array_equal(O.rope_apply(q, 0, 1e4), q)
    assert np.isclose(np.linalg.norm(O.rope_apply(q, 777, 1e4)), np.linalg.norm(q))
    for m, n in [(3, 10), (1000, 5000), (65536, 70000)]:
        a = O.rope_apply(q, m, 1e4) @ O.rope_apply(k, n, 1e4)
        b = q @ O.rope_apply(k, n - m, 1e4)
        assert np.isclose(a, b, rtol=1e-9, atol=1e-9)
    # at the million-token positions of the long-context layer the fp64
    # angles still keep the relative-position property (rounding of
    # pos * theta_i is ~1e-10 rad there)
    for m, n in [(1_000_000, 1_048_575), (1_048_575, 1_048_575)]:
        a = O.rope_apply(q, m, 1e4) @ O.rope_apply(k, n, 1e4)
        b = q @ O.rope_apply(k, n - m, 1e4)
        assert np.isclose(a, b, rtol=1e-8, atol=1e-8)
        assert np.isclose(np.linalg.norm(O.rope_apply(k, n, 1e4)), np.linalg.norm(k))


def test_nuq_golden():
    for c in json.load(open(os.path.join(GOLD, "nuq_examples.json")))["cases"]:
        x = np.array(c["x"], np.float16)
        codes, mn, s, cols, vals = O.nuq_encode(x, c["k"], c["lut"])
        assert list(codes) == c["codes"], c
        assert O.half_to_float(mn) == c["min"] and O.half_to_float(s) == c["s"]
        assert list(cols) == c["cols"]
        assert [O.half_to_float(v) for v in vals] == c["vals"]
        assert list(O.nuq_decode(codes, mn, s, c["lut"], cols, vals)) == c["decoded"]

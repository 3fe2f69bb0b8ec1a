"""Pins of the oracle's InnerQ pieces (InnerQ summary, "Methodology" 1-4):
keys grouped along the hidden dimension (per token, 64-channel groups), a
per-group choice between a symmetric and an asymmetric grid from the group's
statistics, and a per-channel key normalisation fixed at prefill and folded
into the query.

Fixed by: the asymmetric branch equal byte for byte to the pinned uniform
quantizer; hand-worked symmetric groups; on-grid caches that must reproduce
dense attention exactly; the normalisation's power-of-two rule; and the
invariance that makes folding it into q legitimate (scaling a key channel by
2^s and the query channel by 2^-s changes no stored byte and no output)."""
import numpy as np
import pytest

from oracle import kvq_oracle as O
from test_oracle_attention import dense_attention

D = 128


def icfg(kb, vb, S=0, R=0, gkc=64, hybrid=0, norm=0, **kw):
    c = dict(head_dim=D, k_bits=kb, v_bits=vb, k_group_tokens=32, v_group_channels=64, n_sink=S, n_recent=R,
             v_hadamard=0, k_pre_rope=0, rope_theta=10000.0, outliers_per_vector=0, softmax_scale=0.0,
             k_group_channels=gkc, hybrid_groups=hybrid, k_channel_norm=norm)
    c.update(kw)
    return c


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_asymmetric_branch_equals_the_uniform_quantizer(bits):
    rng = np.random.default_rng(bits)
    for trial in range(300):
        x = (rng.standard_normal(64) * rng.uniform(0.01, 30) + rng.uniform(-5, 5)).astype(np.float16)
        if trial % 50 == 0:
            x[:] = x[0]  # a constant group
        a = O.quantize_group(x.astype(np.float32), bits, hybrid=0)
        b = O.quantize_uniform(x, bits)
        assert np.array_equal(a[0], b[0]) and a[1:] == b[1:]


def test_symmetric_group_by_hand():
    """Mean 0 (centred): symmetric, 4 bits: a = 1, scale = fp32(1/7), codes
    rint(x * 7) + 8 (ties to even), stored min = -8 * fp16(scale)."""
    x = np.zeros(64, np.float32)
    x[:8] = [-1.0, 1.0, -0.5, 0.5, 0.25, -0.25, 0.0, 0.0]
    codes, mn, sc = O.quantize_group(x, 4, hybrid=1)
    scale32 = np.float32(1.0) / np.float32(7.0)
    want = np.rint(x / scale32).astype(int) + 8
    assert np.array_equal(codes, want)
    # fp32(1/7) lies just above 1/7, so 0.5 / scale = 3.4999998 rounds to 3
    assert codes[0] == 1 and codes[1] == 15 and codes[2] == 5 and codes[3] == 11
    assert sc == np.float16(scale32).view(np.uint16)
    assert mn == np.float16(-8.0 * np.float32(np.float16(scale32))).view(np.uint16)
    # the same group shifted off centre is asymmetric: codes span 0 .. 15
    codes2, mn2, _ = O.quantize_group(x + np.float32(0.75), 4, hybrid=1)
    assert codes2.min() == 0 and codes2.max() == 15
    assert mn2 == np.float16(-0.25).view(np.uint16)


def test_symmetric_threshold_is_half_an_asymmetric_step():
    """|mean| * 2^(b+1) <= max - min picks the symmetric grid; just above it
    the asymmetric one (2 bits, span 2: the bound is |mean| <= 0.25)."""
    x = np.zeros(64, np.float32)
    x[0], x[1] = -1.0, 1.0
    x[2:34] = 0.5                         # sum 16: mean exactly 0.25 (the bound, inclusive)
    c1, _, _ = O.quantize_group(x, 2, hybrid=1)
    assert c1.min() >= 1                  # symmetric codes never use 0
    x[34] = np.float32(2.0 ** -10)        # mean just above the bound
    c2, _, _ = O.quantize_group(x, 2, hybrid=1)
    assert c2.min() == 0
    c3, _, _ = O.quantize_group(-x, 2, hybrid=1)  # the sign of the mean does not matter
    assert c3.min() == 0


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_symmetric_on_grid_round_trip_and_bound(bits):
    rng = np.random.default_rng(100 + bits)
    qs = (1 << (bits - 1)) - 1
    for _ in range(100):
        scale = 2.0 ** int(rng.integers(-6, 0))
        c = rng.integers(-qs, qs + 1, 64)
        c[0], c[1] = -qs, qs
        c[2:] -= int(np.round(c[2:].mean()))  # centred
        c = np.clip(c, -qs, qs)
        c[0], c[1] = -qs, qs
        x = (c * scale).astype(np.float32)
        codes, mn, sc = O.quantize_group(x, bits, hybrid=1)
        if codes.min() == 0:
            continue  # mean drifted past the bound: asymmetric (covered elsewhere)
        assert np.array_equal(codes.astype(int) - (1 << (bits - 1)), c)
        xhat = np.float64(O.half_to_float(mn)) + codes * np.float64(O.half_to_float(sc))
        assert np.array_equal(xhat, x.astype(np.float64))
    # error bound on random centred groups
    for _ in range(200):
        x = rng.standard_normal(64).astype(np.float32)
        x -= np.float32(x.mean())
        codes, mn, sc = O.quantize_group(x, bits, hybrid=1)
        s = np.float64(O.half_to_float(sc))
        xhat = np.float64(O.half_to_float(mn)) + codes * s
        a = np.abs(x).max()
        s32 = np.float64(np.float32(a) / np.float32(qs))
        assert np.all(np.abs(xhat - x) <= s32 / 2 + (1 << (bits - 1)) * abs(s - s32) * 2 + 1e-7)


def test_key_norm_powers_of_two():
    K = np.zeros((5, D), np.float16)
    K[:, 0] = [0.3, -0.7, 0.1, 0.2, 0.0]     # max 0.7 -> 1
    K[:, 1] = [4.0, -2.0, 1.0, 0.0, 0.0]     # max exactly 4 -> 4
    K[:, 2] = [-9.0, 3.0, 0.0, 0.0, 0.0]     # 9 -> 16
    K[2, 3] = 1e-3                            # tiny -> 2^-9
    n = O.key_norm(K)
    assert n[0] == 1.0 and n[1] == 4.0 and n[2] == 16.0 and n[3] == 2.0 ** -9
    assert n[4] == 1.0                        # an all-zero channel
    m = np.abs(K.astype(np.float32)).max(0)
    nz = m > 0
    assert np.all(m[nz] <= n[nz]) and np.all(n[nz] < 2 * m[nz])
    assert np.all(np.log2(n) == np.round(np.log2(n)))


def _on_grid_innerq_stream(cfg, T, rng):
    """fp16 K, V whose quantized tokens' 64-channel groups sit on their grid
    (asymmetric, or symmetric and centred when the config is hybrid)."""
    K = rng.standard_normal((T, D)).astype(np.float16)
    V = rng.standard_normal((T, D)).astype(np.float16)
    S, Nq, W = O.layout_counts(cfg, T)
    kb, vb = cfg["k_bits"], cfg["v_bits"]

    def grid(bits):
        scale = 2.0 ** int(rng.integers(-5, -2))
        if cfg["hybrid_groups"]:
            qs = (1 << (bits - 1)) - 1
            c = rng.integers(-qs, qs + 1, 64)
            c[:32] = -c[32:]          # mean exactly 0
            c[0], c[32] = qs, -qs
            return (c * scale).astype(np.float16)
        q = (1 << bits) - 1
        mn = np.round(rng.uniform(-2, 0) / scale) * scale
        c = rng.integers(0, q + 1, 64)
        c[:2] = [0, q]
        rng.shuffle(c)
        return (mn + c * scale).astype(np.float16)

    for i in range(Nq):
        for j in (0, 64):
            K[S + i, j:j + 64] = grid(kb)
            V[S + i, j:j + 64] = grid(vb)
    return K, V


@pytest.mark.parametrize("kb,vb", [(8, 8), (4, 4), (4, 2), (2, 2), (8, 4)])
@pytest.mark.parametrize("hybrid", [0, 1])
def test_innerq_on_grid_equals_dense(kb, vb, hybrid):
    rng = np.random.default_rng(10 * kb + vb + hybrid)
    cfg = icfg(kb, vb, S=4, R=40, hybrid=hybrid)
    T = 300
    K, V = _on_grid_innerq_stream(cfg, T, rng)
    q = rng.standard_normal((1, 4, D)).astype(np.float16)
    st = O.build_stream(cfg, K, V)
    out, lse = O.decode_stream(cfg, T, st, q[0])
    ref, rlse = dense_attention(cfg, q.astype(np.float64), K[None, None].astype(np.float64),
                                V[None, None].astype(np.float64))
    assert np.allclose(out, ref[0], rtol=0, atol=1e-10)
    assert np.allclose(lse, rlse[0], rtol=0, atol=1e-10)
    if hybrid:  # every quantized group took the symmetric grid: codes never 0
        S, Nq, _ = O.layout_counts(cfg, T)
        kcodes = np.stack([O.unpack_bits(r, D, kb) for r in st["kc"]])
        assert kcodes.min() >= 1


def test_key_normalisation_folds_into_the_query():
    """Scaling key channel c by 2^s_c (and query channel c by 2^-s_c) leaves
    every logit unchanged; with the normalisation the stored codes and
    scales are unchanged too (only n_c moves), so the output is the same."""
    rng = np.random.default_rng(77)
    T = 400
    cfg = icfg(4, 4, S=4, R=32, hybrid=1, norm=1)
    K = rng.standard_normal((T, D)).astype(np.float16)
    K[:, [3, 50, 99]] *= 8
    V = rng.laplace(size=(T, D)).astype(np.float16)
    q = rng.standard_normal((2, D))
    q = (np.sign(q) * (0.1 + np.abs(q))).astype(np.float16)  # no fp16 subnormal after / 2^s
    s = rng.integers(0, 4, D)  # keys scaled up: exact in fp16
    Ks = (K.astype(np.float32) * 2.0 ** s).astype(np.float16)
    qs = (q.astype(np.float32) * 2.0 ** -s).astype(np.float16)
    assert np.array_equal(Ks.astype(np.float32) * 2.0 ** -s, K.astype(np.float32))
    assert np.array_equal(qs.astype(np.float32) * 2.0 ** s, q.astype(np.float32))
    a, b = O.build_stream(cfg, K, V), O.build_stream(cfg, Ks, V)
    for name in ("kc", "ks", "vc", "vs"):
        assert np.array_equal(a[name], b[name]), name
    assert np.array_equal(b["kn"], a["kn"] * 2.0 ** s)
    oa, la = O.decode_stream(cfg, T, a, q)
    ob, lb = O.decode_stream(cfg, T, b, qs)
    assert np.allclose(oa, ob, rtol=0, atol=1e-12) and np.allclose(la, lb, rtol=0, atol=1e-12)


def test_normalisation_uses_the_prefill_tokens_only():
    rng = np.random.default_rng(5)
    T = 300
    K = rng.standard_normal((T, D)).astype(np.float16)
    K[250, 7] = 100.0  # after the prefill
    V = rng.standard_normal((T, D)).astype(np.float16)
    st = O.build_stream(icfg(4, 4, norm=1, norm_tokens=200), K, V)
    assert np.array_equal(st["kn"], O.key_norm(K[:200]))
    assert st["kn"][7] < 100.0


def test_normalisation_lowers_the_key_error_on_outlier_channels():
    """Per-token groups span all channels, so a few large channels set the
    whole group's step; dividing them down first shrinks the error of the
    other channels (the reason for the normalisation)."""
    rng = np.random.default_rng(8)
    T = 260
    K = rng.standard_normal((T, D)).astype(np.float16)
    K[:, [1, 40, 90]] *= 10
    V = rng.standard_normal((T, D)).astype(np.float16)
    q = rng.standard_normal((8, D)).astype(np.float16)

    def err(norm):
        cfg = icfg(4, 8, norm=norm)
        st = O.build_stream(cfg, K, V)
        out, _ = O.decode_stream(cfg, T, st, q)
        ref, _ = dense_attention(cfg, q[None].astype(np.float64), K[None, None].astype(np.float64),
                                 V[None, None].astype(np.float64))
        return np.abs(out - ref[0]).max()

    assert err(1) < 0.5 * err(0)

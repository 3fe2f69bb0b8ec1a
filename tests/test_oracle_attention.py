"""Pins of the oracle's cache build + fp64 decode attention.

The main pin builds caches whose quantized values sit exactly on the
quantization grid, so the stored cache reconstructs the inputs exactly; the
oracle's decode must then equal a dense numpy softmax attention on the raw
inputs (with GQA by numpy.repeat and RoPE as complex multiplication).  A
dropped, duplicated or misrouted token, a wrong GQA mapping, a transposed
operand or a sign error in RoPE all break that equality."""
import numpy as np
import pytest

from oracle import kvq_oracle as O

D = 128


def dense_attention(cfg, q, K, V):
    """q [B,Hq,d], K,V [B,Hkv,T,d] (fp64) -> out [B,Hq,d], lse [B,Hq].
    Token t sits at position position_offset + t."""
    B, Hq, d = q.shape
    Hkv, T = K.shape[1], K.shape[2]
    K = K.copy()
    if cfg.get("k_pre_rope"):
        th = cfg["rope_theta"] ** (-2.0 * np.arange(d // 2) / d)
        pos = cfg.get("position_offset", 0) + np.arange(T)
        z = (K[..., : d // 2] + 1j * K[..., d // 2:]) * np.exp(1j * pos[:, None] * th)
        K = np.concatenate([z.real, z.imag], -1)
    Kx = np.repeat(K, Hq // Hkv, axis=1)
    Vx = np.repeat(V, Hq // Hkv, axis=1)
    sm = cfg.get("softmax_scale") or 1.0 / np.sqrt(d)
    z = np.einsum("bhd,bhtd->bht", q, Kx) * sm
    m = z.max(-1, keepdims=True)
    p = np.exp(z - m)
    out = np.einsum("bht,bhtd->bhd", p, Vx) / p.sum(-1)[..., None]
    return out, (m[..., 0] + np.log(p.sum(-1)))


def make_cfg(kb, vb, S=0, R=0, gk=32, gv=64, **kw):
    c = dict(head_dim=D, k_bits=kb, v_bits=vb, k_group_tokens=gk, v_group_channels=gv,
             n_sink=S, n_recent=R, v_hadamard=0, k_pre_rope=0, rope_theta=10000.0,
             outliers_per_vector=0, softmax_scale=0.0)
    c.update(kw)
    return c


def _lut(seed):
    x = np.sort(np.random.default_rng(seed).standard_normal(65536))
    return x[((np.arange(8) + 0.5) * 65536 / 8).astype(int)].astype(np.float16).astype(np.float32)


def on_grid_stream(cfg, T, rng):
    """fp16 K, V [T, d] whose quantized part lies exactly on the grid."""
    K = (rng.standard_normal((T, D))).astype(np.float16)
    V = (rng.standard_normal((T, D))).astype(np.float16)
    S, Nq, W = O.layout_counts(cfg, T)
    kb, vb = cfg["k_bits"], cfg["v_bits"]

    def grid(n, bits):
        q = (1 << bits) - 1
        scale = 2.0 ** int(rng.integers(-5, -2))
        mn = np.round(rng.uniform(-2, 0) / scale) * scale
        c = rng.integers(0, q + 1, n)
        c[:2] = [0, q]
        rng.shuffle(c)
        return (mn + c * scale).astype(np.float16)

    def nuq(lut):
        s = 2.0 ** int(rng.integers(-3, 0))
        c = rng.integers(0, 8, D)
        c[:2] = [0, 7]
        rng.shuffle(c)
        x = (s * lut[c].astype(np.float64)).astype(np.float16)
        k = cfg["outliers_per_vector"]
        big = np.abs(x.astype(np.float32)).max()
        cols = rng.choice(D, k, replace=False)
        x[cols] = (np.sign(rng.standard_normal(k)) * big * rng.uniform(2, 4, k)).astype(np.float16)
        return x

    if kb == 3:
        for i in range(Nq):
            K[S + i] = nuq(np.array(cfg["k_lut"], np.float32))
    elif kb != 16:
        for g0 in range(0, Nq, cfg["k_group_tokens"]):
            for ch in range(D):
                K[S + g0:S + g0 + cfg["k_group_tokens"], ch] = grid(cfg["k_group_tokens"], kb)
    if vb == 3:
        for i in range(Nq):
            V[S + i] = nuq(np.array(cfg["v_lut"], np.float32))
    elif vb != 16:
        gv = cfg["v_group_channels"]
        for i in range(Nq):
            for j in range(0, D, gv):
                V[S + i, j:j + gv] = grid(gv, vb)
    return K, V


def run_layer(cfg, B, Hq, Hkv, T, seed, on_grid=True):
    rng = np.random.default_rng(seed)
    K = np.zeros((B, Hkv, T, D), np.float16)
    V = np.zeros_like(K)
    for b in range(B):
        for h in range(Hkv):
            if on_grid:
                K[b, h], V[b, h] = on_grid_stream(cfg, T, rng)
            else:
                K[b, h] = rng.standard_normal((T, D)).astype(np.float16)
                V[b, h] = rng.standard_normal((T, D)).astype(np.float16)
    q = rng.standard_normal((B, Hq, D)).astype(np.float16)
    stores = O.build_layer(cfg, K, V)
    out, lse = O.decode_layer(cfg, T, stores, q)
    ref, rlse = dense_attention(cfg, q.astype(np.float64), K.astype(np.float64), V.astype(np.float64))
    return out, lse, ref, rlse


PAIRS = [(8, 8), (8, 4), (4, 4), (4, 2), (2, 2)]


@pytest.mark.parametrize("kb,vb", PAIRS)
@pytest.mark.parametrize("S,R,T", [(0, 32, 100), (4, 64, 300), (4, 0, 68), (0, 0, 64), (3, 5, 140)])
def test_on_grid_uniform_equals_dense(kb, vb, S, R, T):
    cfg = make_cfg(kb, vb, S=S, R=R)
    out, lse, ref, rlse = run_layer(cfg, 2, 4, 2, T, seed=kb * 100 + vb + T)
    assert np.allclose(out, ref, rtol=0, atol=1e-12)
    assert np.allclose(lse, rlse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("gv", [32, 64, 128])
def test_on_grid_v_groups(gv):
    cfg = make_cfg(4, 2, S=2, R=8, gv=gv)
    out, lse, ref, rlse = run_layer(cfg, 1, 2, 1, 150, seed=gv)
    assert np.allclose(out, ref, atol=1e-12)


@pytest.mark.parametrize("T", [1, 3, 4, 5, 36, 67, 68, 69, 100])
def test_window_edges(T):
    """Contexts shorter than the sinks, than sinks + recent, and exactly at a
    flush boundary (S=4, R=32, G_K=32: first group at T=68)."""
    cfg = make_cfg(4, 4, S=4, R=32)
    out, lse, ref, rlse = run_layer(cfg, 1, 3, 1, T, seed=T)
    assert np.allclose(out, ref, atol=1e-12)


def test_fp16_mode_equals_dense():
    cfg = make_cfg(16, 16)
    out, lse, ref, rlse = run_layer(cfg, 2, 8, 2, 77, seed=1, on_grid=False)
    assert np.allclose(out, ref, atol=1e-12) and np.allclose(lse, rlse, atol=1e-12)


def test_all_recent_equals_dense():
    """With R >= T nothing is quantized: plain attention on the inputs."""
    cfg = make_cfg(2, 2, S=4, R=500)
    out, lse, ref, rlse = run_layer(cfg, 1, 4, 4, 300, seed=2, on_grid=False)
    assert np.allclose(out, ref, atol=1e-12)


@pytest.mark.parametrize("rope", [0, 1])
def test_on_grid_nuq_with_outliers_equals_dense(rope):
    cfg = make_cfg(3, 3, S=0, R=0, outliers_per_vector=2, k_pre_rope=rope,
                   k_lut=list(_lut(1)), v_lut=list(_lut(2)))
    out, lse, ref, rlse = run_layer(cfg, 1, 2, 2, 200, seed=3 + rope)
    assert np.allclose(out, ref, atol=1e-10)
    assert np.allclose(lse, rlse, atol=1e-10)


def test_pre_rope_uniform_on_grid_equals_dense():
    cfg = make_cfg(8, 4, S=4, R=16, k_pre_rope=1)
    out, lse, ref, rlse = run_layer(cfg, 1, 4, 1, 180, seed=5)
    assert np.allclose(out, ref, atol=1e-10)


def test_softmax_scale_override():
    cfg = make_cfg(4, 4, S=0, R=32, softmax_scale=0.05)
    out, lse, ref, rlse = run_layer(cfg, 1, 1, 1, 100, seed=6)
    assert np.allclose(out, ref, atol=1e-12)


def _normwise(a, b):
    return np.max(np.abs(a - b), -1) / np.max(np.abs(b), -1)


def test_hadamard_8bit_close_to_dense_and_inverse_applied():
    """Rotated 8-bit V is close to unquantized attention; without the inverse
    rotation after the sum the result would be far off."""
    cfg = make_cfg(8, 8, S=4, R=16, v_hadamard=1)
    out, lse, ref, rlse = run_layer(cfg, 2, 4, 2, 300, seed=7, on_grid=False)
    assert np.max(_normwise(out, ref)) < 2e-2
    assert np.allclose(lse, rlse, atol=5e-2)


def test_quantization_error_ordering():
    """8-bit attention stays within 1e-2 of unquantized attention, and the
    error drops by >= 8x from 4 to 8 bits."""
    errs = {}
    for b in (4, 8):
        cfg = make_cfg(b, b, S=0, R=32)
        out, lse, ref, rlse = run_layer(cfg, 2, 2, 2, 600, seed=8, on_grid=False)
        errs[b] = np.max(_normwise(out, ref))
    assert errs[8] < 1e-2
    assert errs[4] > 8 * errs[8]


def _fp16_stream(T, rng, V=None):
    K = rng.standard_normal((T, D)).astype(np.float16)
    if V is None:
        V = rng.standard_normal((T, D)).astype(np.float16)
    return K, V


def test_softmax_weights_sum_to_one():
    """A V that is the same vector for every token must come back exactly:
    the weights sum to 1 (fp16 cache, and a quantized cache whose V rows
    sit on the grid)."""
    rng = np.random.default_rng(41)
    # on the 4-bit grid of every 64-channel group: min -1, scale 1/8, codes 0 and 15 present
    codes = rng.integers(0, 16, D)
    codes[0], codes[1], codes[64], codes[65] = 0, 15, 0, 15
    c = (-1.0 + codes / 8.0).astype(np.float16)
    for cfg, T in [(make_cfg(16, 16), 300), (make_cfg(4, 4, S=4, R=32), 300)]:
        K, _ = _fp16_stream(T, rng)
        V = np.tile(c, (T, 1))
        store = O.build_stream(cfg, K, V)
        q = rng.standard_normal((2, D)).astype(np.float16)
        out, _ = O.decode_stream(cfg, T, store, q)
        assert np.allclose(out, c.astype(np.float64)[None, :], rtol=0, atol=1e-12)


def test_split_lse_merge_equals_single_pass():
    """Attention over a prefix and over the rest, merged by log-sum-exp with
    the returned lse, equals the single pass over all tokens -- the merge the
    split kernels perform, and the meaning of lse (natural log of the sum of
    exp of the scaled logits)."""
    rng = np.random.default_rng(43)
    cfg = make_cfg(16, 16)
    T, T1 = 500, 173
    K, V = _fp16_stream(T, rng)
    q = rng.standard_normal((3, D)).astype(np.float16)
    full, lse = O.decode_stream(cfg, T, O.build_stream(cfg, K, V), q)
    oa, la = O.decode_stream(cfg, T1, O.build_stream(cfg, K[:T1], V[:T1]), q)
    ob, lb = O.decode_stream(cfg, T - T1, O.build_stream(cfg, K[T1:], V[T1:]), q)
    m = np.maximum(la, lb)
    wa, wb = np.exp(la - m), np.exp(lb - m)
    merged = (wa[:, None] * oa + wb[:, None] * ob) / (wa + wb)[:, None]
    assert np.allclose(merged, full, rtol=0, atol=1e-12)
    assert np.allclose(m + np.log(wa + wb), lse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("kb", [3, 4])
def test_pre_rope_position_offset_equals_dense(kb):
    """A stream whose first token sits at absolute position 1_000_003 (a
    later context shard): RoPE after dequantization uses that position."""
    kw = dict(k_pre_rope=1, position_offset=1_000_003)
    if kb == 3:
        kw.update(outliers_per_vector=2, k_lut=list(_lut(5)), v_lut=list(_lut(6)))
        cfg = make_cfg(3, 3, **kw)
    else:
        cfg = make_cfg(4, 4, S=2, R=16, **kw)
    out, lse, ref, rlse = run_layer(cfg, 1, 4, 2, 200, seed=51)
    assert np.allclose(out, ref, rtol=0, atol=1e-10)
    assert np.allclose(lse, rlse, rtol=0, atol=1e-10)
    cfg0 = dict(cfg, position_offset=0)
    out0, _, _, _ = run_layer(cfg0, 1, 4, 2, 200, seed=51)
    assert np.abs(out0 - out).max() > 1e-3  # the offset changes the result


def _parts_by_hand(cfg, T, cuts):
    """Context parts at the quantized-group boundaries S + 32 * c for c in
    cuts: part 0 keeps the sinks, the last part the fp16 window; every other
    part is quantized groups only.  Returns [(first token, tokens, part cfg)]."""
    S, R = cfg["n_sink"], cfg["n_recent"]
    bounds = [0] + [S + 32 * c for c in cuts] + [T]
    parts = []
    for r in range(len(bounds) - 1):
        a, b = bounds[r], bounds[r + 1]
        pc = dict(cfg, position_offset=a, n_sink=S if r == 0 else 0,
                  n_recent=R if r == len(bounds) - 2 else 0)
        parts.append((a, b - a, pc))
    return parts


@pytest.mark.parametrize("kind", ["kv4_sinks_window", "nuq_rope", "hadamard_k4v2", "fp16"])
def test_merge_parts_equals_single_pass(kind):
    """The context cut into parts at group boundaries, each part stored and
    decoded on its own (sinks in the first, the window in the last, RoPE at
    absolute positions), then merged by log-sum-exp, equals the decode of
    the whole context: same quantized groups, same softmax.  An empty part
    (lse = -inf) contributes nothing."""
    rng = np.random.default_rng(61)
    T = 900
    if kind == "kv4_sinks_window":
        cfg = make_cfg(4, 4, S=4, R=64)
    elif kind == "nuq_rope":
        cfg = make_cfg(3, 3, k_pre_rope=1, outliers_per_vector=2, k_lut=list(_lut(7)), v_lut=list(_lut(8)))
    elif kind == "hadamard_k4v2":
        cfg = make_cfg(4, 2, S=2, R=32, v_hadamard=1)
    else:
        cfg = make_cfg(16, 16)
    K = rng.standard_normal((T, D)).astype(np.float16)
    V = rng.laplace(size=(T, D)).astype(np.float16)
    q = rng.standard_normal((4, D)).astype(np.float16)
    full, flse = O.decode_stream(cfg, T, O.build_stream(cfg, K, V), q)
    _, Nq, _ = O.layout_counts(cfg, T)
    ng = Nq // 32 if cfg["k_bits"] != 16 else T // 32
    cuts = [ng // 3, ng // 3, (2 * ng) // 3]  # the second part is empty
    outs, lses = [], []
    for a, n, pc in _parts_by_hand(cfg, T, cuts):
        if n == 0:
            outs.append(np.zeros((4, D)))
            lses.append(np.full(4, -np.inf))
            continue
        o, l = O.decode_stream(pc, n, O.build_stream(pc, K[a:a + n], V[a:a + n]), q)
        outs.append(o)
        lses.append(l)
    merged, mlse = O.merge_parts(np.stack(outs), np.stack(lses))
    assert np.allclose(merged, full, rtol=0, atol=1e-12)
    assert np.allclose(mlse, flse, rtol=0, atol=1e-12)


def test_merge_parts_closed_form():
    """Two parts with known lse: weights e^lse_r / sum; all parts empty gives
    lse -inf and a zero output."""
    o = np.array([[[1.0, 0.0]], [[0.0, 1.0]]])
    out, lse = O.merge_parts(o, np.array([[np.log(3.0)], [np.log(1.0)]]))
    assert np.allclose(out, [[0.75, 0.25]], rtol=0, atol=1e-15)
    assert np.allclose(lse, [np.log(4.0)], rtol=0, atol=1e-15)
    out, lse = O.merge_parts(o, np.full((2, 1), -np.inf))
    assert lse[0] == -np.inf and not out.any()

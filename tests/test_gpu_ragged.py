"""GPU parity of sequences of different lengths in one call
(kvq_append_ragged, kvq_decode_attn_ragged) against the CPU oracle run row
by row: every stream's stored bytes must equal the oracle's store built from
that row's tokens alone, and every row's attention must match the oracle's
fp64 attention over that row's own length (2e-3 normwise).  Lengths cross
the sink, window and flush boundaries; rows that append nothing stay as
they are."""
import numpy as np
import pytest
import torch

from _kvq_testutil import TOL, assert_store_equal, gpu_store, normwise_err
from oracle import kvq_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from bit_kv_cache_07_gb300 import build
    build.build_library()
    from bit_kv_cache_07_gb300 import binding
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    return binding


def cfg_of(kb, vb, Bt, Hq, Hkv, max_tokens, **kw):
    c = dict(batch=Bt, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=128, max_tokens=max_tokens, k_bits=kb, v_bits=vb,
             k_group_tokens=32, v_group_channels=64, n_sink=4, n_recent=32, v_hadamard=0, k_pre_rope=0,
             rope_theta=10000.0, outliers_per_vector=0, softmax_scale=0.0, split_tokens=0,
             k_lut=[0.0] * 8, v_lut=[0.0] * 8)
    c.update(kw)
    if kb == 3:
        from bit_kv_cache_07_gb300 import synth
        c["k_lut"] = synth.lut_from_seed(1000)
        c["v_lut"] = synth.lut_from_seed(2000)
    return c


def check_rows(layer, cfg, lengths, Kh, Vh, norm_tokens=None):
    """Every stream's store equals the oracle's for its row's tokens."""
    Hkv = cfg["n_kv_heads"]
    refs = []
    for s in range(cfg["batch"] * Hkv):
        b, h = divmod(s, Hkv)
        T = lengths[b]
        c = dict(cfg) if norm_tokens is None else dict(cfg, norm_tokens=norm_tokens[b])
        ref = O.build_stream(c, Kh[b, h, :T], Vh[b, h, :T])
        assert_store_equal(gpu_store(layer, s, T, O.layout_counts(cfg, T)), ref, where=f"stream {s} (T={T})")
        refs.append(ref)
    return refs


def check_ragged_decode(B, layer, cfg, lengths, refs, seed):
    from bit_kv_cache_07_gb300 import synth
    q = synth.random_q(cfg["batch"], cfg["n_q_heads"], seed=seed, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    ws = B.new_workspace(cfg)
    layer.decode_ragged(lengths, q, out, lse, ws)
    torch.cuda.synchronize()
    qh = q.cpu().numpy()
    Hkv = cfg["n_kv_heads"]
    g = cfg["n_q_heads"] // Hkv
    for s in range(cfg["batch"] * Hkv):
        b, h = divmod(s, Hkv)
        ref, rlse = O.decode_stream(cfg, lengths[b], refs[s], qh[b, h * g:(h + 1) * g])
        o = out[b, h * g:(h + 1) * g].cpu().numpy()
        err = normwise_err(o, ref)
        assert err.max() < TOL, f"row {b} (T={lengths[b]}) head group {h}: normwise error {err.max():.3g}"
        assert np.allclose(lse[b, h * g:(h + 1) * g].cpu().numpy(), rlse, rtol=1e-4, atol=1e-3)
    ns = cfg["batch"] * Hkv
    assert not ws[:4 * ns].any(), "split counters must be back at zero"
    return out


# (kb, vb, batch rows, Hq, Hkv, extra config); row lengths are LENGTHS[:rows].
# Uniform codes with 64-channel V groups and the fp16 cache run on the
# persistent kernel (1, 4 and 7 query heads per KV head), the others on the
# split kernel.
CASES = {
    "kv4_gqa4": (4, 4, 4, 8, 2, {}),
    "k4v2_hadamard_g7": (4, 2, 3, 14, 2, dict(v_hadamard=1)),
    "k2v8_mha": (2, 8, 4, 3, 3, {}),
    "kv8_gv32": (8, 8, 3, 4, 1, dict(v_group_channels=32)),
    "k8v4_rope": (8, 4, 3, 4, 2, dict(k_pre_rope=1)),
    "nuq_rope_outliers": (3, 3, 4, 2, 2, dict(k_pre_rope=1, outliers_per_vector=2)),
    "fp16": (16, 16, 4, 4, 2, dict(n_sink=0, n_recent=0)),
}
LENGTHS = [700, 1, 133, 417]


@pytest.mark.parametrize("name", list(CASES))
def test_ragged_prefill_and_decode(B, name):
    from bit_kv_cache_07_gb300 import synth
    kb, vb, rows, Hq, Hkv, ex = CASES[name]
    lengths = LENGTHS[:rows]
    cfg = cfg_of(kb, vb, rows, Hq, Hkv, max(lengths) + 40, **ex)
    K, V = synth.random_kv(rows, Hkv, max(lengths), seed=sum(map(ord, name)), device="cuda")
    layer = B.Layer(cfg)
    layer.append_ragged([0] * rows, lengths, K, V)
    torch.cuda.synchronize()
    Kh, Vh = K.cpu().numpy(), V.cpu().numpy()
    refs = check_rows(layer, cfg, lengths, Kh, Vh)
    check_ragged_decode(B, layer, cfg, lengths, refs, seed=7)


def test_ragged_steps_cross_flushes_at_different_times(B):
    """Rows at different positions append one token per step (one row
    pauses every other step); flushes happen in different steps for
    different rows.  After every step the stored bytes and the ragged decode
    match the oracle built from each row's tokens so far."""
    from bit_kv_cache_07_gb300 import synth
    rows, Hkv, Hq = 3, 2, 8
    start = [60, 95, 5]
    steps = 40
    cfg = cfg_of(4, 2, rows, Hq, Hkv, 200, n_sink=4, n_recent=32)
    total = [s + steps for s in start]
    K, V = synth.random_kv(rows, Hkv, max(total), seed=11, device="cuda")
    layer = B.Layer(cfg)
    layer.append_ragged([0] * rows, start, K, V)
    have = list(start)
    Kh, Vh = K.cpu().numpy(), V.cpu().numpy()
    for step in range(steps):
        n = [1, 1 if step % 2 == 0 else 0, 1]
        k1 = torch.stack([K[b, :, have[b]:have[b] + 1] if n[b] else K[b, :, :1] for b in range(rows)]).contiguous()
        v1 = torch.stack([V[b, :, have[b]:have[b] + 1] if n[b] else V[b, :, :1] for b in range(rows)]).contiguous()
        layer.append_ragged(have, n, k1, v1)
        have = [h + x for h, x in zip(have, n)]
        if step % 13 == 12 or step == steps - 1:
            torch.cuda.synchronize()
            refs = check_rows(layer, cfg, have, Kh, Vh)
            check_ragged_decode(B, layer, cfg, have, refs, seed=step)


def test_ragged_equal_lengths_match_the_uniform_calls(B):
    """All rows at one length: the ragged append writes the same bytes as
    kvq_append, and the ragged decode (the persistent kernel's row-by-row
    schedule) agrees with kvq_decode_attn (its uniform schedule) and the
    oracle."""
    from bit_kv_cache_07_gb300 import synth
    rows, Hkv, Hq, T = 3, 2, 8, 450
    cfg = cfg_of(4, 4, rows, Hq, Hkv, T + 40)
    K, V = synth.random_kv(rows, Hkv, T, seed=5, device="cuda")
    a, b = B.Layer(cfg), B.Layer(cfg)
    a.append(0, K, V)
    b.append_ragged([0] * rows, [T] * rows, K, V)
    torch.cuda.synchronize()
    for r in B.REGIONS:  # every cache region (the ragged call also leaves its row counts in `rows`)
        if r != "rows":
            assert torch.equal(a.region(r), b.region(r)), r
    q = synth.random_q(rows, Hq, seed=3, device="cuda")
    out_u, out_r = torch.empty_like(q), torch.empty_like(q)
    a.decode(T, q, out_u, None, B.new_workspace(cfg))
    refs = check_rows(b, cfg, [T] * rows, K.cpu().numpy(), V.cpu().numpy())
    out_r = check_ragged_decode(B, b, cfg, [T] * rows, refs, seed=3)
    torch.cuda.synchronize()
    assert normwise_err(out_u.cpu().numpy(), out_r.cpu().numpy().astype(np.float64)).max() < TOL


def test_ragged_innerq_row_starts_later(B):
    """InnerQ key normalisation with rows that start at different calls: a
    row still empty after the first ragged append gets its normalisation
    from its own first append, while the other rows keep theirs."""
    from bit_kv_cache_07_gb300 import synth
    rows, Hkv, Hq = 3, 2, 8
    cfg = cfg_of(4, 4, rows, Hq, Hkv, 400, k_group_channels=64, hybrid_groups=1, k_channel_norm=1)
    K, V = synth.random_kv(rows, Hkv, 300, seed=23, device="cuda")
    layer = B.Layer(cfg)
    first = [200, 0, 150]   # row 1 stays empty
    layer.append_ragged([0, 0, 0], first, K, V)
    more = [40, 260, 0]     # row 1 starts now; row 2 appends nothing
    k2 = torch.stack([K[b, :, first[b]:first[b] + 260] if first[b] + 260 <= 300 else
                      torch.cat([K[b, :, first[b]:], K[b, :, :first[b] + 260 - 300]], 1) for b in range(rows)]).contiguous()
    v2 = torch.stack([V[b, :, first[b]:first[b] + 260] if first[b] + 260 <= 300 else
                      torch.cat([V[b, :, first[b]:], V[b, :, :first[b] + 260 - 300]], 1) for b in range(rows)]).contiguous()
    layer.append_ragged(first, more, k2, v2)
    torch.cuda.synchronize()
    lengths = [f + m for f, m in zip(first, more)]
    Kh, Vh = K.cpu().numpy(), V.cpu().numpy()
    # each row's tokens in order: its first slice, then the first `more` rows of its second input
    k2h, v2h = k2.cpu().numpy(), v2.cpu().numpy()
    refs = []
    for s in range(rows * Hkv):
        b, h = divmod(s, Hkv)
        kt = np.concatenate([Kh[b, h, :first[b]], k2h[b, h, :more[b]]], 0)
        vt = np.concatenate([Vh[b, h, :first[b]], v2h[b, h, :more[b]]], 0)
        norm_from = first[b] if first[b] > 0 else more[b]
        c = dict(cfg, norm_tokens=norm_from)
        ref = O.build_stream(c, kt, vt)
        assert_store_equal(gpu_store(layer, s, lengths[b], O.layout_counts(cfg, lengths[b])), ref,
                           where=f"stream {s} (T={lengths[b]})")
        refs.append(ref)
    check_ragged_decode(B, layer, cfg, lengths, refs, seed=4)


def test_ragged_innerq_append_and_decode(B):
    """InnerQ keys with key normalisation: each row's normalisation comes
    from its own first append, and the ragged decode (persistent kernel,
    InnerQ key path) matches the oracle row by row."""
    from bit_kv_cache_07_gb300 import synth
    rows, Hkv, Hq = 3, 2, 8
    lengths = [300, 64, 161]
    cfg = cfg_of(4, 4, rows, Hq, Hkv, 400, k_group_channels=64, hybrid_groups=1, k_channel_norm=1)
    K, V = synth.random_kv(rows, Hkv, max(lengths), seed=21, device="cuda")
    layer = B.Layer(cfg)
    layer.append_ragged([0] * rows, lengths, K, V)
    torch.cuda.synchronize()
    refs = check_rows(layer, cfg, lengths, K.cpu().numpy(), V.cpu().numpy(), norm_tokens=lengths)
    check_ragged_decode(B, layer, cfg, lengths, refs, seed=1)


@pytest.mark.parametrize("rows,hi", [(70, 300), (256, 80)])
def test_ragged_many_rows(B, rows, hi):
    """More batch rows than a warp has lanes (the decode finds a warp's rows
    by a ballot over 32 rows at a time), up to the 256-row limit; rows from
    one token to a few groups, many with no quantized group at all."""
    from bit_kv_cache_07_gb300 import synth
    rng = np.random.default_rng(rows)
    lengths = [int(x) for x in rng.integers(1, hi + 1, rows)]
    cfg = cfg_of(4, 4, rows, 2, 1, hi + 8, n_sink=4, n_recent=16)
    K, V = synth.random_kv(rows, 1, hi, seed=rows, device="cuda")
    layer = B.Layer(cfg)
    layer.append_ragged([0] * rows, lengths, K, V)
    torch.cuda.synchronize()
    refs = check_rows(layer, cfg, lengths, K.cpu().numpy(), V.cpu().numpy())
    check_ragged_decode(B, layer, cfg, lengths, refs, seed=rows + 1)

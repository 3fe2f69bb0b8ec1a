"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Every case goes append -> packed layer buffer -> decode (the cache is really
filled and read back, as the Hadamard write-up's "measurement trap" section
insists).  Packed codes, scales, CSR outliers and fp16 sink / window bytes
must be identical to the oracle's; attention must agree with the oracle's
fp64 result on the same stored cache within 2e-3 (normwise per output
vector)."""
import zlib

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


def cfg_dict(kb, vb, Bt, Hq, Hkv, T, S=0, R=0, gv=64, had=0, rope=0, nout=0, max_tokens=None, split=0,
             lut_seed=None, offset=0):
    c = dict(batch=Bt, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=128,
             max_tokens=T + 40 if max_tokens is None else max_tokens, k_bits=kb, v_bits=vb,
             k_group_tokens=32, v_group_channels=gv, n_sink=S, n_recent=R, v_hadamard=had,
             k_pre_rope=rope, rope_theta=10000.0, outliers_per_vector=nout, softmax_scale=0.0,
             split_tokens=split, position_offset=offset, k_lut=[0.0] * 8, v_lut=[0.0] * 8)
    if kb == 3:
        from bit_kv_cache_07_gb300 import synth
        c["k_lut"] = synth.lut_from_seed(1000 + (lut_seed or 0))
        c["v_lut"] = synth.lut_from_seed(2000 + (lut_seed or 0))
    return c


def fill(binding, cfg, T, seed, chunks=None, v_dist="laplace"):
    from bit_kv_cache_07_gb300 import synth
    K, V = synth.random_kv(cfg["batch"], cfg["n_kv_heads"], T, seed=seed, device="cuda", v_dist=v_dist)
    assert torch.isfinite(K).all() and torch.isfinite(V).all()
    layer = binding.Layer(cfg)
    if chunks is None:
        chunks = [T]
    t = 0
    for n in chunks:
        layer.append(t, K[:, :, t:t + n].contiguous(), V[:, :, t:t + n].contiguous())
        t += n
    assert t == T
    torch.cuda.synchronize()
    return layer, K.cpu().numpy(), V.cpu().numpy()


def check_store(layer, cfg, T, Kh, Vh):
    refs = O.build_layer(cfg, Kh, Vh)
    counts = O.layout_counts(cfg, T)
    for s in range(cfg["batch"] * cfg["n_kv_heads"]):
        assert_store_equal(gpu_store(layer, s, T, counts), refs[s], where=f"stream {s}")
    return refs


def check_decode(binding, layer, cfg, T, refs, seed=0, tol=TOL):
    from bit_kv_cache_07_gb300 import synth
    q = synth.random_q(cfg["batch"], cfg["n_q_heads"], seed=seed, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    ws = binding.new_workspace(cfg)
    layer.decode(T, q, out, lse, ws)
    torch.cuda.synchronize()
    ref, rlse = O.decode_layer(cfg, T, refs, q.cpu().numpy())
    err = normwise_err(out.cpu().numpy(), ref)
    assert err.max() < tol, f"max normwise error {err.max():.3g}"
    assert np.allclose(lse.cpu().numpy(), rlse, rtol=1e-4, atol=1e-3)
    ns = cfg["batch"] * cfg["n_kv_heads"]
    assert not ws[:4 * ns].any(), "split counters must be back at zero"
    return out, lse


CASES = {
    # name: (kb, vb, B, Hq, Hkv, T, extra)
    "toy_k4v2": (4, 2, 1, 1, 1, 1024, dict(R=32)),
    "kv4_mha_ragged": (4, 4, 2, 4, 4, 700, dict(S=4, R=64)),
    "kv8_gqa4": (8, 8, 2, 8, 2, 1000, dict(S=4, R=128)),
    "k8v4_gqa4": (8, 4, 2, 8, 2, 1000, dict(S=4, R=128)),
    "kv4_gqa4": (4, 4, 2, 8, 2, 1000, dict(S=4, R=128)),
    "k4v2_gqa4": (4, 2, 2, 8, 2, 1000, dict(S=4, R=128)),
    "kv2_gqa4": (2, 2, 2, 8, 2, 1000, dict(S=4, R=128)),
    "k2v8_g2": (2, 8, 1, 4, 2, 513, dict(S=1, R=5)),
    "hadamard_g7": (4, 2, 2, 14, 2, 600, dict(S=4, R=32, had=1)),
    # 5 to 8 heads per KV head run head-major on the tensor cores
    "kv8_g8": (8, 8, 1, 8, 1, 700, dict(S=4, R=32)),
    "kv4_g5": (4, 4, 2, 10, 2, 650, dict(S=2, R=40)),
    "k2v8_g6_hadamard": (2, 8, 1, 6, 1, 500, dict(S=4, R=16, had=1)),
    "k8v2_g8": (8, 2, 1, 16, 2, 400, dict(S=0, R=0)),
    "hadamard_kv8": (8, 8, 1, 4, 1, 400, dict(S=4, R=32, had=1)),
    "gv32": (4, 4, 1, 2, 1, 300, dict(S=2, R=16, gv=32)),
    "gv128": (4, 2, 1, 2, 1, 300, dict(S=2, R=16, gv=128)),
    "nuq_rope": (3, 3, 1, 4, 4, 1000, dict(rope=1, nout=2)),
    "nuq_norope_sinks": (3, 3, 1, 8, 2, 777, dict(S=4, R=32, nout=2)),
    "nuq_no_outliers": (3, 3, 1, 2, 2, 300, dict(nout=0)),
    "nuq_hadamard_k4": (3, 3, 1, 1, 1, 333, dict(nout=4, had=1)),
    # one query head with pre-RoPE keys (the query-folded 16-offset table,
    # two anchor sets) at 1, 3, 4 and 8 outliers per vector (from 3 on: 3 CTAs
    # per SM)
    "nuq_rope_k1": (3, 3, 2, 2, 2, 611, dict(rope=1, nout=1, S=4, R=16)),
    "nuq_rope_k3": (3, 3, 1, 3, 3, 450, dict(rope=1, nout=3)),
    "nuq_rope_k4_hadamard": (3, 3, 1, 2, 2, 389, dict(rope=1, nout=4, had=1)),
    "nuq_rope_k8": (3, 3, 1, 1, 1, 300, dict(rope=1, nout=8)),
    "k8v4_rope": (8, 4, 1, 4, 1, 500, dict(S=4, R=16, rope=1)),
    "k2v2_rope_g8": (2, 2, 1, 8, 1, 300, dict(S=0, R=8, rope=1)),
    "fp16": (16, 16, 2, 8, 2, 777, dict()),
    "fp16_mha": (16, 16, 1, 3, 3, 100, dict()),
    "fp16_g7": (16, 16, 1, 14, 2, 300, dict(S=4, R=16)),
    "fp16_rope": (16, 16, 1, 2, 1, 200, dict(rope=1)),
    # 3 query heads per KV head fill 3 of the 4 head slots (one padded slot)
    # in both kernels
    "kv4_g3": (4, 4, 1, 6, 2, 500, dict(S=4, R=32)),
    "k2v4_g3_hadamard": (2, 4, 2, 3, 1, 333, dict(S=2, R=16, had=1)),
    "fp16_g3": (16, 16, 1, 3, 1, 150, dict()),
    "nuq_rope_g3": (3, 3, 1, 3, 1, 300, dict(rope=1, nout=2)),
    "k4v2_gv32_g3": (4, 2, 1, 6, 2, 300, dict(S=2, R=16, gv=32)),
    # RoPE at absolute positions that start far from 0 (a later context shard):
    # the group anchors, the fp64 fallback past 2^16 groups and the fp16 tokens
    "nuq_rope_offset": (3, 3, 1, 2, 2, 700, dict(rope=1, nout=2, offset=2_000_003)),
    "k4v4_rope_offset_sinks": (4, 4, 1, 4, 1, 500, dict(S=4, R=16, rope=1, offset=123_456)),
    "fp16_rope_offset": (16, 16, 1, 2, 1, 200, dict(rope=1, offset=999_999)),
    # the cache filled to its capacity
    "kv8_full_capacity": (8, 8, 1, 4, 2, 417, dict(S=4, R=64, max_tokens=417)),
}


@pytest.mark.parametrize("name", list(CASES))
def test_bulk_append_and_decode(B, name):
    kb, vb, Bt, Hq, Hkv, T, ex = CASES[name]
    cfg = cfg_dict(kb, vb, Bt, Hq, Hkv, T, **ex)
    layer, Kh, Vh = fill(B, cfg, T, seed=zlib.crc32(name.encode()) % 1000)
    refs = check_store(layer, cfg, T, Kh, Vh)
    check_decode(B, layer, cfg, T, refs, seed=1)


@pytest.mark.parametrize("T", [1, 3, 4, 67, 68, 69, 99, 100, 101, 131, 132, 133])
def test_context_edges(B, T):
    """Contexts inside the sinks, inside sinks + recent, and around flush
    boundaries (S=4, R=64, G_K=32: first group at T=100, second at T=132)."""
    cfg = cfg_dict(4, 4, 1, 4, 2, T, S=4, R=64, max_tokens=200)
    layer, Kh, Vh = fill(B, cfg, T, seed=T)
    refs = check_store(layer, cfg, T, Kh, Vh)
    check_decode(B, layer, cfg, T, refs, seed=T)


@pytest.mark.parametrize("kind", ["kv4", "nuq", "hadamard", "fp16"])
def test_token_by_token_append_equals_bulk(B, kind):
    """Appending one token at a time (flushing a group whenever the window
    reaches R + G_K) leaves the same bytes as the oracle's bulk build."""
    if kind == "kv4":
        cfg = cfg_dict(4, 4, 2, 4, 2, 230, S=4, R=32)
    elif kind == "nuq":
        cfg = cfg_dict(3, 3, 1, 2, 2, 230, S=0, R=0, nout=2, rope=1)
    elif kind == "hadamard":
        cfg = cfg_dict(4, 2, 1, 7, 1, 230, S=3, R=10, had=1)
    else:
        cfg = cfg_dict(16, 16, 1, 2, 1, 230)
    T = 230
    layer, Kh, Vh = fill(B, cfg, T, seed=7, chunks=[1] * T)
    refs = check_store(layer, cfg, T, Kh, Vh)
    check_decode(B, layer, cfg, T, refs, seed=3)


def test_chunked_append_equals_bulk(B):
    rng = np.random.default_rng(0)
    T = 1500
    cuts = np.sort(rng.choice(np.arange(1, T), 12, replace=False))
    chunks = list(np.diff(np.concatenate([[0], cuts, [T]])))
    cfg = cfg_dict(8, 4, 2, 8, 2, T, S=4, R=64)
    layer, Kh, Vh = fill(B, cfg, T, seed=11, chunks=chunks)
    refs = check_store(layer, cfg, T, Kh, Vh)
    check_decode(B, layer, cfg, T, refs)


@pytest.mark.parametrize("split", [0, 32, 64, 96, 4096])
def test_split_k_counts_agree(B, split):
    """Any split-K partition (1 group per split up to one split) merges to
    the same attention."""
    T = 2100
    cfg = cfg_dict(4, 2, 1, 4, 1, T, S=4, R=32, had=1, split=split)
    layer, Kh, Vh = fill(B, cfg, T, seed=5)
    refs = check_store(layer, cfg, T, Kh, Vh)
    check_decode(B, layer, cfg, T, refs, seed=2)


def test_repeated_decode_reuses_workspace(B):
    """Counters are left at zero, so back-to-back calls on one workspace agree."""
    T = 900
    cfg = cfg_dict(4, 4, 2, 8, 2, T, S=4, R=64)
    layer, Kh, Vh = fill(B, cfg, T, seed=9)
    from bit_kv_cache_07_gb300 import synth
    q = synth.random_q(2, 8, seed=4, device="cuda")
    ws = B.new_workspace(cfg)
    outs = []
    for _ in range(3):
        out = torch.empty_like(q)
        layer.decode(T, q, out, None, ws)
        outs.append(out)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


def test_decode_after_incremental_steps(B):
    """Decode interleaved with single-token appends (the serving loop): each
    step's output matches the oracle at that step's length."""
    T0, steps = 160, 40
    cfg = cfg_dict(4, 2, 1, 4, 1, T0 + steps, S=4, R=32, had=1)
    from bit_kv_cache_07_gb300 import synth
    K, V = synth.random_kv(1, 1, T0 + steps, seed=21, device="cuda", v_dist="student_t3")
    layer = B.Layer(cfg)
    layer.append(0, K[:, :, :T0].contiguous(), V[:, :, :T0].contiguous())
    ws = B.new_workspace(cfg)
    Kh, Vh = K.cpu().numpy(), V.cpu().numpy()
    for i in range(steps):
        T = T0 + i + 1
        layer.append(T - 1, K[:, :, T - 1:T].contiguous(), V[:, :, T - 1:T].contiguous())
        if i % 7 == 0 or i == steps - 1:
            q = synth.random_q(1, 4, seed=100 + i, device="cuda")
            out = torch.empty_like(q)
            layer.decode(T, q, out, None, ws)
            torch.cuda.synchronize()
            refs = O.build_layer(cfg, Kh[:, :, :T], Vh[:, :, :T])
            ref, _ = O.decode_layer(cfg, T, refs, q.cpu().numpy())
            assert normwise_err(out.cpu().numpy(), ref).max() < TOL


def test_negative_control_corrupted_byte_is_detected(B):
    """Flipping one packed code byte must break the byte comparison and move
    the attention output (the checks above are not vacuous)."""
    T = 500
    cfg = cfg_dict(4, 2, 1, 1, 1, T, R=32)
    layer, Kh, Vh = fill(B, cfg, T, seed=13)
    refs = O.build_layer(cfg, Kh, Vh)
    counts = O.layout_counts(cfg, T)
    from bit_kv_cache_07_gb300 import synth
    q = synth.random_q(1, 1, seed=1, device="cuda")
    clean = torch.empty_like(q)
    layer.decode(T, q, clean, None, B.new_workspace(cfg))
    kc = layer.region("k_codes")
    kc[100] ^= 0xFF
    torch.cuda.synchronize()
    with pytest.raises(AssertionError):
        assert_store_equal(gpu_store(layer, 0, T, counts), refs[0])
    bad = torch.empty_like(q)
    layer.decode(T, q, bad, None, B.new_workspace(cfg))
    torch.cuda.synchronize()
    assert not torch.equal(bad, clean)


def _tie_values(rng, shape, qmax):
    """fp16 values on a grid of step 2^-4 from an offset of 1: the group's
    extremes 1 and 1 + qmax/16 are planted at the first two positions of
    every group, every other value is 1 + (k + 0.5)/16 (an exact tie of the
    quantizer's quotient, which must round half to even) or 1 + k/16."""
    k = rng.integers(0, qmax, shape)
    half = rng.integers(0, 2, shape)
    return 1.0 + (k + 0.5 * half) / 16.0


@pytest.mark.parametrize("kb,vb,iq", [(2, 2, 0), (4, 4, 0), (8, 8, 0), (4, 2, 0), (4, 4, 1), (8, 2, 1)])
def test_exact_ties_round_half_even(B, kb, vb, iq):
    """Groups whose quotients (x - min) / scale sit exactly on half-integers:
    the kernel's reciprocal shortcut flags them and the IEEE division rounds
    them half to even, byte for byte as the oracle."""
    rng = np.random.default_rng(kb * 10 + vb + 100 * iq)
    Bt, Hkv, T = 1, 2, 96
    cfg = cfg_dict(kb, vb, Bt, 2 * Hkv, Hkv, T)
    if iq:
        cfg.update(k_group_channels=64)
    qk, qv = (1 << kb) - 1, (1 << vb) - 1
    K = _tie_values(rng, (Bt, Hkv, T, 128), qk)
    V = _tie_values(rng, (Bt, Hkv, T, 128), qv)
    if iq:  # per token, channel groups of 64: extremes at channels 0, 1 and 64, 65
        K[..., 0], K[..., 1], K[..., 64], K[..., 65] = 1.0, 1.0 + qk / 16, 1.0, 1.0 + qk / 16
    else:  # per channel over 32-token groups: extremes at tokens 32 g and 32 g + 1
        K[:, :, 0::32, :], K[:, :, 1::32, :] = 1.0, 1.0 + qk / 16
    V[..., 0], V[..., 1], V[..., 64], V[..., 65] = 1.0, 1.0 + qv / 16, 1.0, 1.0 + qv / 16
    K, V = K.astype(np.float16), V.astype(np.float16)
    assert np.all(K.astype(np.float64) == 1.0 + np.round((K.astype(np.float64) - 1.0) * 32) / 32)
    layer = B.Layer(cfg)
    layer.append(0, torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda())
    torch.cuda.synchronize()
    refs = check_store(layer, cfg, T, K, V)
    check_decode(B, layer, cfg, T, refs, seed=3)

"""GPU parity of the InnerQ cache (InnerQ summary, "Key Contributions" and
"Methodology" 1-4) through the C ABI: keys grouped per token along the
hidden dimension (64-channel groups), hybrid symmetric / asymmetric groups,
and the per-channel key normalisation fixed by the first append.  Packed
codes, scales and the normalisation must equal the oracle's byte for byte;
attention within 2e-3 of the oracle's fp64 result on the same stored cache."""
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
    assert torch.cuda.is_available()
    return binding


def cfg_iq(kb, vb, Bt, Hq, Hkv, T, S=4, R=32, hybrid=1, norm=1, had=0, gkc=64):
    return dict(batch=Bt, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=128, max_tokens=T + 40, k_bits=kb, v_bits=vb,
                k_group_tokens=32, v_group_channels=64, n_sink=S, n_recent=R, v_hadamard=had, k_pre_rope=0,
                rope_theta=10000.0, outliers_per_vector=0, softmax_scale=0.0, split_tokens=0, position_offset=0,
                k_group_channels=gkc, hybrid_groups=hybrid, k_channel_norm=norm, k_lut=[0.0] * 8, v_lut=[0.0] * 8)


def run_case(B, cfg, T, seed, chunks=None, v_dist="laplace", centred_k=False):
    from bit_kv_cache_07_gb300 import synth
    K, V = synth.random_kv(cfg["batch"], cfg["n_kv_heads"], T, seed=seed, device="cuda", v_dist=v_dist)
    if centred_k:  # every 64-channel group's mean exactly 0 (channel c + 32 = -channel c): symmetric groups
        K = K.clone()
        K[..., 32:64] = -K[..., 0:32]
        K[..., 96:128] = -K[..., 64:96]
    layer = B.Layer(cfg)
    chunks = chunks or [T]
    t = 0
    for n in chunks:
        layer.append(t, K[:, :, t:t + n].contiguous(), V[:, :, t:t + n].contiguous())
        t += n
    torch.cuda.synchronize()
    Kh, Vh = K.cpu().numpy(), V.cpu().numpy()
    ocfg = dict(cfg, norm_tokens=chunks[0])  # the first append fixes the normalisation
    refs = O.build_layer(ocfg, Kh, Vh)
    counts = O.layout_counts(cfg, T)
    for s in range(cfg["batch"] * cfg["n_kv_heads"]):
        assert_store_equal(gpu_store(layer, s, T, counts), refs[s], where=f"stream {s}")
    q = synth.random_q(cfg["batch"], cfg["n_q_heads"], seed=seed + 1, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    ws = B.new_workspace(cfg)
    persistent, _ = B.kvq_decode_path(cfg, T)
    assert persistent
    layer.decode(T, q, out, lse, ws)
    torch.cuda.synchronize()
    ref, rlse = O.decode_layer(ocfg, T, refs, q.cpu().numpy())
    err = normwise_err(out.float().cpu().numpy(), ref)
    assert err.max() < TOL, err.max()
    assert np.allclose(lse.cpu().numpy(), rlse, rtol=1e-4, atol=1e-3)
    assert not ws[:4 * cfg["batch"] * cfg["n_kv_heads"]].any()
    return refs


CASES = {
    # name: (kb, vb, B, Hq, Hkv, T, extra)
    "kv4_g4": (4, 4, 2, 8, 2, 1000, dict()),
    "kv8_g4": (8, 8, 2, 8, 2, 1000, dict()),
    "k8v4_g4": (8, 4, 2, 8, 2, 1000, dict()),
    "k4v2_g4": (4, 2, 2, 8, 2, 1000, dict()),
    "kv2_g4": (2, 2, 2, 8, 2, 1000, dict()),
    "kv4_mha": (4, 4, 2, 4, 4, 700, dict(S=0, R=64)),
    "kv2_g2": (2, 2, 1, 4, 2, 600, dict()),
    "kv4_g7_hadamard": (4, 2, 1, 14, 2, 600, dict(had=1)),
    "kv8_g8": (8, 8, 1, 8, 1, 500, dict()),
    "k2v8_g3": (2, 8, 1, 6, 2, 500, dict(S=2, R=16)),
    "kv4_no_hybrid": (4, 4, 1, 8, 2, 800, dict(hybrid=0)),
    "kv4_no_norm": (4, 4, 1, 8, 2, 800, dict(norm=0)),
    "kv4_plain": (4, 4, 1, 8, 2, 800, dict(hybrid=0, norm=0)),
}


@pytest.mark.parametrize("name", list(CASES))
def test_innerq_bulk_append_and_decode(B, name):
    kb, vb, Bt, Hq, Hkv, T, ex = CASES[name]
    run_case(B, cfg_iq(kb, vb, Bt, Hq, Hkv, T, **ex), T, seed=zlib.crc32(name.encode()) % 1000)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_innerq_centred_keys_take_symmetric_groups(B, bits):
    """Keys centred per token: most groups pick the symmetric grid (codes
    never 0 there); bytes and attention still match the oracle."""
    T = 600
    refs = run_case(B, cfg_iq(bits, 4, 1, 4, 2, T), T, seed=17, centred_k=True)
    kc = np.stack([O.unpack_bits(r, 128, bits) for r in refs[0]["kc"]])
    ks = refs[0]["ks"].reshape(-1, 2, 2)
    sym = 0
    for i in range(kc.shape[0]):
        for j in range(2):
            if kc[i, 64 * j:64 * j + 64].min() >= 1 and \
                    O.half_to_float(int(ks[i, j, 0])) == -(1 << (bits - 1)) * O.half_to_float(int(ks[i, j, 1])):
                sym += 1
    assert sym == 2 * kc.shape[0]  # every group of every quantized token


def test_innerq_chunked_append_normalisation_from_first_chunk(B):
    """The first append fixes the normalisation; later chunks and single
    tokens are coded with it (the oracle builds with norm_tokens = the first
    chunk)."""
    T = 900
    run_case(B, cfg_iq(4, 2, 2, 8, 2, T), T, seed=23, chunks=[300, 1, 1, 150, 448])


def test_innerq_token_by_token(B):
    T = 200
    run_case(B, cfg_iq(8, 4, 1, 4, 1, T, S=2, R=16), T, seed=29, chunks=[1] * T)


def test_innerq_rejects_unsupported_combinations(B):
    with pytest.raises(B.KvqError):
        B.kvq_layout_query(cfg_iq(4, 4, 1, 4, 1, 100, gkc=32))
    c = cfg_iq(4, 4, 1, 4, 1, 100)
    c["k_pre_rope"] = 1
    with pytest.raises(B.KvqError):
        B.kvq_layout_query(c)
    c = cfg_iq(4, 4, 1, 4, 1, 100, gkc=0)  # normalisation needs the InnerQ key layout
    with pytest.raises(B.KvqError):
        B.kvq_layout_query(c)


@pytest.mark.parametrize("kind", ["per_channel_k", "nuq"])
def test_hybrid_groups_with_the_other_layouts(B, kind):
    """Hybrid groups with per-channel keys (the decision on 32-token channel
    groups) match the oracle; non-uniform codes reject it."""
    if kind == "per_channel_k":
        T = 700
        run_case(B, cfg_iq(4, 2, 1, 8, 2, T, gkc=0, norm=0), T, seed=31, centred_k=True)
    else:
        c = cfg_iq(3, 3, 1, 4, 1, 100, gkc=0, norm=0)
        c.update(k_lut=[-1.5, -0.9, -0.5, -0.2, 0.2, 0.5, 0.9, 1.5], v_lut=[-1.5, -0.9, -0.5, -0.2, 0.2, 0.5, 0.9, 1.5])
        with pytest.raises(B.KvqError):
            B.kvq_layout_query(c)


def test_innerq_full_size_sampled(B):
    """The bench's InnerQ workload layer at full size (B=16, 32 / 8 heads,
    T=32768), sampled streams against the oracle."""
    from _kvq_testutil import gpu_store as gs
    from bit_kv_cache_07_gb300 import synth, workloads
    name = "llama3_8b_innerq_kv4_t32k"
    w = workloads.WORKLOADS[name]
    T = w["tokens"]
    cfg = workloads.layer_config(name, 0)
    K, V = synth.layer_kv(name, 0, tokens=T, device="cuda")
    layer = B.Layer(cfg)
    layer.append(0, K[:, :, :T - 1].contiguous(), V[:, :, :T - 1].contiguous())
    layer.append(T - 1, K[:, :, T - 1:].contiguous(), V[:, :, T - 1:].contiguous())
    q = synth.query(name, 0, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    layer.decode(T, q, out, lse, B.new_workspace(cfg))
    torch.cuda.synchronize()
    ocfg = dict(cfg, norm_tokens=T - 1)
    counts = O.layout_counts(cfg, T)
    g = w["n_q_heads"] // w["n_kv_heads"]
    for s in (0, 127):
        b, h = divmod(s, w["n_kv_heads"])
        st = O.build_stream(ocfg, K[b, h].cpu().numpy(), V[b, h].cpu().numpy())
        assert_store_equal(gs(layer, s, T, counts), st, where=f"stream {s}")
        ref, rlse = O.decode_stream(ocfg, T, st, q[b, h * g:(h + 1) * g].cpu().numpy())
        assert normwise_err(out[b, h * g:(h + 1) * g].float().cpu().numpy(), ref).max() < TOL

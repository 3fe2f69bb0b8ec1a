"""GPU parity of per-head (K, V) bits (RateQuant summary, "Methodology" 1-4)
through the C ABI: a layer held as one cache per distinct pair over its KV
heads (the config's head map), the per-head distortion measurement against
the oracle's, and the allocation it feeds against the oracle's fit and
greedy rule."""
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


def base_cfg(Bt, Hq, Hkv, T, **kw):
    c = dict(batch=Bt, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=128, max_tokens=T + 40, k_bits=4, v_bits=4,
             k_group_tokens=32, v_group_channels=64, n_sink=4, n_recent=32, v_hadamard=0, k_pre_rope=0,
             rope_theta=10000.0, outliers_per_vector=0, softmax_scale=0.0, split_tokens=0, position_offset=0,
             k_group_channels=0, hybrid_groups=0, k_channel_norm=0, k_lut=[0.0] * 8, v_lut=[0.0] * 8)
    c.update(kw)
    return c


@pytest.mark.parametrize("kind", ["gqa4", "mha_hadamard", "innerq", "split_gv32", "g8"])
def test_mixed_pairs_match_the_oracle(B, kind):
    from bit_kv_cache_07_gb300 import mixed, synth
    T = 900
    if kind == "gqa4":
        cfg, pairs = base_cfg(2, 16, 4, T), [(8, 8), (4, 2), (2, 2), (4, 2)]
    elif kind == "mha_hadamard":
        cfg, pairs = base_cfg(1, 5, 5, T, v_hadamard=1), [(2, 4), (8, 4), (4, 4), (2, 4), (8, 8)]
    elif kind == "innerq":
        cfg, pairs = base_cfg(2, 8, 4, T, k_group_channels=64, hybrid_groups=1, k_channel_norm=1), \
            [(4, 4), (8, 2), (4, 4), (2, 8)]
    elif kind == "split_gv32":  # 32-channel V groups: the split kernel
        cfg, pairs = base_cfg(1, 4, 2, T, v_group_channels=32), [(8, 2), (2, 4)]
    else:
        cfg, pairs = base_cfg(1, 16, 2, T), [(4, 2), (8, 4)]
    K, V = synth.random_kv(cfg["batch"], cfg["n_kv_heads"], T, seed=31, device="cuda")
    layer = mixed.MixedLayer(cfg, pairs)
    layer.append(0, K[:, :, :T - 5].contiguous(), V[:, :, :T - 5].contiguous())
    for t in range(T - 5, T):
        layer.append(t, K[:, :, t:t + 1].contiguous(), V[:, :, t:t + 1].contiguous())
    q = synth.random_q(cfg["batch"], cfg["n_q_heads"], seed=32, device="cuda")
    out = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.zeros(max(16, layer.workspace_bytes()), dtype=torch.uint8, device="cuda")
    layer.decode(T, q, out, lse, ws)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()  # every head written
    Kh, Vh, qh = K.cpu().numpy(), V.cpu().numpy(), q.cpu().numpy()
    Hkv, g = cfg["n_kv_heads"], cfg["n_q_heads"] // cfg["n_kv_heads"]
    for pair, heads, sub in layer.parts:
        pc = dict(cfg, k_bits=pair[0], v_bits=pair[1], norm_tokens=T - 5)
        counts = O.layout_counts(pc, T)
        for b in range(cfg["batch"]):
            for i, h in enumerate(heads):
                st = O.build_stream(pc, Kh[b, h], Vh[b, h])
                assert_store_equal(gpu_store(sub, b * len(heads) + i, T, counts), st, where=f"{pair} b{b} h{h}")
                ref, rlse = O.decode_stream(pc, T, st, qh[b, h * g:(h + 1) * g])
                err = normwise_err(out[b, h * g:(h + 1) * g].float().cpu().numpy(), ref).max()
                assert err < TOL, (pair, b, h, err)
                assert np.allclose(lse[b, h * g:(h + 1) * g].cpu().numpy(), rlse, rtol=1e-4, atol=1e-3)


def test_mixed_pairs_with_ragged_rows(B):
    """Per-head pairs and rows of different lengths together: every part
    takes the ragged calls over its heads; each (row, head) matches the
    oracle built from that row's tokens at that head's pair."""
    from bit_kv_cache_07_gb300 import mixed, synth
    lengths = [700, 133, 2]
    cfg, pairs = base_cfg(3, 8, 4, max(lengths)), [(8, 4), (2, 2), (4, 4), (2, 2)]
    K, V = synth.random_kv(3, 4, max(lengths), seed=51, device="cuda")
    layer = mixed.MixedLayer(cfg, pairs)
    layer.append_ragged([0, 0, 0], lengths, K, V)
    q = synth.random_q(3, 8, seed=52, device="cuda")
    out = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    layer.decode_ragged(lengths, q, out, lse)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    Kh, Vh, qh = K.cpu().numpy(), V.cpu().numpy(), q.cpu().numpy()
    g = 2
    for pair, heads, sub in layer.parts:
        pc = dict(cfg, k_bits=pair[0], v_bits=pair[1])
        for b, T in enumerate(lengths):
            for i, h in enumerate(heads):
                st = O.build_stream(pc, Kh[b, h, :T], Vh[b, h, :T])
                assert_store_equal(gpu_store(sub, b * len(heads) + i, T, O.layout_counts(pc, T)), st,
                                   where=f"{pair} b{b} h{h}")
                ref, rlse = O.decode_stream(pc, T, st, qh[b, h * g:(h + 1) * g])
                err = normwise_err(out[b, h * g:(h + 1) * g].float().cpu().numpy(), ref).max()
                assert err < TOL, (pair, b, h, err)
                assert np.allclose(lse[b, h * g:(h + 1) * g].cpu().numpy(), rlse, rtol=1e-4, atol=1e-3)


@pytest.mark.parametrize("kind", ["per_channel", "hadamard_hybrid", "innerq_norm"])
def test_distortion_matches_the_oracle(B, kind):
    from bit_kv_cache_07_gb300 import synth
    T = 333
    if kind == "per_channel":
        cfg = base_cfg(2, 8, 4, T)
    elif kind == "hadamard_hybrid":
        cfg = base_cfg(2, 8, 4, T, v_hadamard=1, hybrid_groups=1)
    else:
        cfg = base_cfg(2, 8, 4, T, k_group_channels=64, hybrid_groups=1, k_channel_norm=1)
    K, V = synth.random_kv(2, 4, T, seed=41, device="cuda", v_dist="student_t3")
    Kh, Vh = K.cpu().numpy(), V.cpu().numpy()
    for bits in (2, 4, 8):
        got = B.kvq_measure_distortion(cfg, K, V, bits).cpu().numpy()
        for h in range(4):
            ref = np.mean([O.quant_distortion(cfg, Kh[b, h], Vh[b, h], bits) for b in range(2)], 0)
            assert np.allclose(got[h], ref, rtol=1e-9, atol=0), (bits, h, got[h], ref)


def test_allocation_pipeline_matches_the_oracle(B):
    """GPU distortions -> library fit + greedy, against oracle distortions ->
    oracle fit + greedy: the same per-head pairs."""
    from bit_kv_cache_07_gb300 import mixed, synth, workloads
    name = "llama3_8b_rateq_t32k"  # heads of different spread: the allocation mixes pairs
    cfg = workloads.layer_config(name, 0)
    K, V = synth.layer_kv(name, 0, tokens=512, batch=1, device="cuda")
    pairs, rep = mixed.allocate_pairs(cfg, K, V, 4.0)
    Kh, Vh = K.cpu().numpy(), V.cpu().numpy()
    base = dict(cfg, k_bits=4, v_bits=4)
    comps = []
    for h in range(cfg["n_kv_heads"]):
        d = [O.quant_distortion(base, Kh[0, h], Vh[0, h], b) for b in (2, 4, 8)]
        comps.append([x[0] for x in d])
        comps.append([x[1] for x in d])
    fits = [O.fit_rd([2, 4, 8], c) for c in comps]
    bits, used = O.rate_greedy([f[0] for f in fits], [f[1] for f in fits], rep["total_bits"])
    assert np.allclose(rep["distortion"], comps, rtol=1e-9)
    assert rep["bits"] == bits.tolist()
    assert pairs == [(int(bits[2 * h]), int(bits[2 * h + 1])) for h in range(cfg["n_kv_heads"])]
    assert sum(rep["bits"]) <= rep["total_bits"]
    assert len(set(pairs)) > 1

"""GPU parity of context-parallel decode (KVQuant summary: a 10M-token
context on an 8-GPU system), through the C ABI on one GPU: the context cut
into shards by kvq_context_shard, every shard stored in its own cache and
decoded with kvq_decode_attn, the parts merged by kvq_merge_attn.  The shard
caches' bytes must equal the oracle's for the shard configs, the merged
attention must be within 2e-3 of the oracle's decode of the whole context,
and the merge kernel must agree with the oracle's merge of the same parts.

(On one GPU the shards are decoded one after another; the all-gather
between GPUs is covered on CPU with gloo ranks in
test_context_parallel_host.py.)"""
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


def _cfg(kb, vb, Bt=2, Hq=8, Hkv=2, T=1500, **kw):
    c = dict(batch=Bt, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=128, max_tokens=T + 64, k_bits=kb, v_bits=vb,
             k_group_tokens=32, v_group_channels=64, n_sink=0, n_recent=0, v_hadamard=0, k_pre_rope=0,
             rope_theta=10000.0, outliers_per_vector=0, softmax_scale=0.0, split_tokens=0, position_offset=0,
             k_lut=[0.0] * 8, v_lut=[0.0] * 8)
    c.update(kw)
    if kb == 3:
        from bit_kv_cache_07_gb300 import synth
        c["k_lut"], c["v_lut"] = synth.lut_from_seed(31), synth.lut_from_seed(32)
    return c


CASES = {
    "kv4_sinks_window": _cfg(4, 4, n_sink=4, n_recent=64),
    "k4v2_hadamard_g7": _cfg(4, 2, Hq=14, n_sink=4, n_recent=32, v_hadamard=1),
    "nuq3_rope": _cfg(3, 3, Hq=4, Hkv=4, k_pre_rope=1, outliers_per_vector=2),
    "k8v4_rope_offset": _cfg(8, 4, Hq=4, Hkv=1, n_sink=4, n_recent=16, k_pre_rope=1, position_offset=70000),
    "fp16": _cfg(16, 16),
}


def _decode_shards(B, cfg, T, n, K, V, q):
    outs = torch.zeros((n,) + tuple(q.shape), dtype=torch.float16, device="cuda")
    lses = torch.full((n,) + tuple(q.shape[:2]), float("-inf"), dtype=torch.float32, device="cuda")
    shards = []
    for r in range(n):
        sc, a, m = B.kvq_context_shard(cfg, T, n, r)
        shards.append((sc, a, m))
        if m == 0:
            continue
        layer = B.Layer(sc)
        layer.append(0, K[:, :, a:a + m].contiguous(), V[:, :, a:a + m].contiguous())
        layer.decode(m, q, outs[r], lses[r], B.new_workspace(sc))
        shards[-1] = (sc, a, m, layer)
    torch.cuda.synchronize()
    return outs, lses, shards


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("n", [2, 3, 5])
def test_sharded_decode_merged_matches_whole_context(B, name, n):
    from bit_kv_cache_07_gb300 import synth
    cfg = CASES[name]
    T = 1500
    K, V = synth.random_kv(cfg["batch"], cfg["n_kv_heads"], T, seed=90 + n, device="cuda")
    q = synth.random_q(cfg["batch"], cfg["n_q_heads"], seed=91, device="cuda")
    outs, lses, shards = _decode_shards(B, cfg, T, n, K, V, q)
    Kh, Vh = K.cpu().numpy(), V.cpu().numpy()
    # every shard's cache holds the oracle's bytes for the shard config
    for sh in shards:
        if sh[2] == 0:
            continue
        sc, a, m, layer = sh
        refs = O.build_layer(sc, Kh[:, :, a:a + m], Vh[:, :, a:a + m])
        counts = O.layout_counts(sc, m)
        for s in range(cfg["batch"] * cfg["n_kv_heads"]):
            assert_store_equal(gpu_store(layer, s, m, counts), refs[s], where=f"shard at {a}, stream {s}")
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    B.kvq_merge_attn(outs, lses, out, lse)
    torch.cuda.synchronize()
    # against the oracle's decode of the whole context
    refs = O.build_layer(cfg, Kh, Vh)
    ref, rlse = O.decode_layer(cfg, T, refs, q.cpu().numpy())
    err = normwise_err(out.float().cpu().numpy(), ref)
    assert err.max() < TOL, err.max()
    assert np.allclose(lse.cpu().numpy(), rlse, rtol=1e-4, atol=1e-3)
    # the merge kernel against the oracle's merge of the same fp16 parts
    mo, ml = O.merge_parts(outs.float().cpu().numpy().astype(np.float64), lses.cpu().numpy().astype(np.float64))
    assert normwise_err(out.float().cpu().numpy(), mo).max() < 1e-3
    assert np.allclose(lse.cpu().numpy(), ml, rtol=1e-6, atol=1e-5)


def test_merge_kernel_edges(B):
    """One part passes through; an empty part (lse = -inf) is ignored; all
    parts empty gives a zero output and lse = -inf."""
    g = torch.Generator(device="cuda").manual_seed(5)
    outs = torch.randn((3, 7, 128), generator=g, device="cuda").half()
    lses = torch.randn((3, 7), generator=g, device="cuda")
    out = torch.empty((7, 128), dtype=torch.float16, device="cuda")
    lse = torch.empty(7, device="cuda")
    B.kvq_merge_attn(outs[:1], lses[:1], out, lse)
    torch.cuda.synchronize()
    assert torch.equal(out, outs[0]) and torch.allclose(lse, lses[0])
    lses2 = lses.clone()
    lses2[1] = float("-inf")
    B.kvq_merge_attn(outs, lses2, out, lse)
    mo, ml = O.merge_parts(outs.float().cpu().numpy().astype(np.float64), lses2.cpu().numpy().astype(np.float64))
    torch.cuda.synchronize()
    assert normwise_err(out.float().cpu().numpy(), mo).max() < 1e-3
    B.kvq_merge_attn(outs, torch.full_like(lses, float("-inf")), out, lse)
    torch.cuda.synchronize()
    assert not out.float().abs().sum().item() and torch.isinf(lse).all() and (lse < 0).all()


def test_serving_loop_appends_to_the_last_shard(B):
    """Prefill 3 shards, then append tokens one at a time to the last shard
    (its window flushes groups as a single cache's would) and decode."""
    from bit_kv_cache_07_gb300 import synth
    cfg = _cfg(4, 2, Bt=1, Hq=4, Hkv=1, T=900, n_sink=4, n_recent=32, v_hadamard=1)
    T0, steps = 700, 70
    K, V = synth.random_kv(1, 1, T0 + steps, seed=95, device="cuda", v_dist="student_t3")
    q = synth.random_q(1, 4, seed=96, device="cuda")
    n = 3
    layers = []
    for r in range(n):
        sc, a, m = B.kvq_context_shard(cfg, T0, n, r)
        layer = B.Layer(sc)
        layer.append(0, K[:, :, a:a + m].contiguous(), V[:, :, a:a + m].contiguous())
        layers.append((sc, a, m, layer))
    sc_last, a_last, _, last = layers[-1]
    Kh, Vh = K.cpu().numpy(), V.cpu().numpy()
    for i in range(steps):
        T = T0 + i + 1
        last.append(T - 1 - a_last, K[:, :, T - 1:T].contiguous(), V[:, :, T - 1:T].contiguous())
        if i % 23 == 0 or i == steps - 1:
            outs = torch.zeros((n, 1, 4, 128), dtype=torch.float16, device="cuda")
            lses = torch.full((n, 1, 4), float("-inf"), device="cuda")
            for r, (sc, a, m, layer) in enumerate(layers):
                tl = T - a if r == n - 1 else m
                layer.decode(tl, q, outs[r], lses[r], B.new_workspace(sc))
            out = torch.empty_like(q)
            B.kvq_merge_attn(outs, lses, out)
            torch.cuda.synchronize()
            refs = O.build_layer(cfg, Kh[:, :, :T], Vh[:, :, :T])
            ref, _ = O.decode_layer(cfg, T, refs, q.cpu().numpy())
            assert normwise_err(out.float().cpu().numpy(), ref).max() < TOL

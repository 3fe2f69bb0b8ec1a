"""GPU parity at the workloads' full sizes, with the automatic split-K plan
the benchmark uses.  The oracle recomputes a sample of streams one by one:
their packed bytes must be identical and their heads' attention within 2e-3.
Every layer is filled the way the benchmark fills it (bulk append of T - 1
tokens, then a single-token append), then decoded at T."""
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


def run_layer(binding, name, layer_idx, sample_streams):
    from bit_kv_cache_07_gb300 import synth, workloads
    w = workloads.WORKLOADS[name]
    T = w["tokens"]
    cfg = workloads.layer_config(name, layer_idx)
    if cfg["k_bits"] == 3:
        from bit_kv_cache_07_gb300 import calibrate
        cfg["k_lut"], cfg["v_lut"] = calibrate.nuq_tables(name, layer_idx)
        if w.get("lut") == "fitted":
            # the library's fit against the oracle's on the same calibration tokens
            Kc, Vc = calibrate.calibration_kv(name, layer_idx)
            k = w["outliers_per_vector"]
            assert O.nuq_fit_lut(Kc.cpu().numpy(), k)[0] == cfg["k_lut"]
            assert O.nuq_fit_lut(Vc.cpu().numpy(), k, w["v_hadamard"])[0] == cfg["v_lut"]
    K, V = synth.layer_kv(name, layer_idx, tokens=T, device="cuda")
    assert torch.isfinite(K).all() and torch.isfinite(V).all()
    layer = binding.Layer(cfg)
    layer.append(0, K[:, :, :T - 1].contiguous(), V[:, :, :T - 1].contiguous())
    layer.append(T - 1, K[:, :, T - 1:].contiguous(), V[:, :, T - 1:].contiguous())
    q = synth.query(name, layer_idx, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    ws = binding.new_workspace(cfg)
    layer.decode(T, q, out, lse, ws)
    torch.cuda.synchronize()
    Hkv, g = w["n_kv_heads"], w["n_q_heads"] // w["n_kv_heads"]
    counts = O.layout_counts(cfg, T)
    worst = 0.0
    for s in sample_streams:
        b, h = divmod(s, Hkv)
        Kh, Vh = K[b, h].cpu().numpy(), V[b, h].cpu().numpy()
        ref_store = O.build_stream(cfg, Kh, Vh)
        assert_store_equal(gpu_store(layer, s, T, counts), ref_store, where=f"{name} layer {layer_idx} stream {s}")
        ref, rlse = O.decode_stream(cfg, T, ref_store, q[b, h * g:(h + 1) * g].cpu().numpy())
        got = out[b, h * g:(h + 1) * g].float().cpu().numpy()
        err = normwise_err(got, ref).max()
        assert err < TOL, f"{name} layer {layer_idx} stream {s}: {err:.3g}"
        assert np.allclose(lse[b, h * g:(h + 1) * g].cpu().numpy(), rlse, rtol=1e-4, atol=1e-3)
        worst = max(worst, err)
    assert np.isfinite(out.float().cpu().numpy()).all()
    ns = w["batch"] * Hkv
    assert not ws[:4 * ns].any()
    del K, V, layer
    torch.cuda.empty_cache()
    return worst


def test_full_toy_k4v2_t1k(B):
    run_layer(B, "toy_k4v2_t1k", 0, [0])


def test_full_llama2_kv4_t4k(B):
    run_layer(B, "llama2_7b_kv4_t4k", 0, [0, 137, 255])


def test_full_llama3_mixed_pairs_t32k(B):
    """One layer of each of the five (K, V) pairs the seeded per-layer draw uses."""
    from bit_kv_cache_07_gb300 import workloads
    pairs = workloads.layer_pairs("llama3_8b_mixed_t32k")
    seen = {}
    for i, p in enumerate(pairs):
        seen.setdefault(p, i)
    assert len(seen) == 5
    for p, i in seen.items():
        run_layer(B, "llama3_8b_mixed_t32k", i, [0, 127])


def test_full_qwen_hadamard_t8k(B):
    run_layer(B, "qwen_gqa_hadamard_t8k", 0, [0, 131, 255])


@pytest.mark.timeout(1200)
def test_full_llama7b_nuq3_t1m(B):
    run_layer(B, "llama7b_nuq3_t1m", 0, [19])

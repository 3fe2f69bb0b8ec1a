"""The seeded generators give finite fp16 data of the stated distributions."""
import numpy as np
import torch

from bit_kv_cache_07_gb300 import synth, workloads


def test_distributions_finite_and_shaped():
    g = torch.Generator().manual_seed(0)
    for dist in ("normal", "laplace", "student_t3"):
        x = synth._draw(dist, (1 << 20,), g, "cpu")
        assert torch.isfinite(x).all()
        if dist == "laplace":  # Laplace(0,1): mean |x| = 1, var 2
            assert abs(x.abs().mean().item() - 1.0) < 0.01 and abs(x.var().item() - 2.0) < 0.03
        if dist == "normal":
            assert abs(x.std().item() - 1.0) < 0.01
        if dist == "student_t3":  # heavy tails: kurtosis well above normal
            assert (x.abs() > 5).float().mean().item() > 1e-3


def test_layer_kv_outlier_channels_and_determinism():
    K1, V1 = synth.layer_kv("llama2_7b_kv4_t4k", 3, tokens=100, batch=1)
    K2, V2 = synth.layer_kv("llama2_7b_kv4_t4k", 3, tokens=100, batch=1)
    assert torch.equal(K1, K2) and torch.equal(V1, V2)
    och = synth.k_outlier_channels("llama2_7b_kv4_t4k", 3, 32, 128)
    assert och.shape == (32, 3)
    std = K1.float().std(dim=2)[0]  # [H, d]
    for h in range(4):
        big = std[h, och[h]]
        assert (big > 4).all() and (std[h].median() < 1.5)


def test_toy_fixed_outlier_channels():
    och = synth.k_outlier_channels("toy_k4v2_t1k", 0, 1, 128)
    assert sorted(och[0].tolist()) == sorted(np.random.default_rng(0).permutation(128)[:4].tolist())


def test_seeded_pairs_and_mean_bits():
    pairs = workloads.layer_pairs("llama3_8b_mixed_t32k")
    assert pairs[0] == pairs[1] == pairs[31] == "KV8"
    from collections import Counter
    assert Counter(pairs) == {"KV8": 9, "K8V4": 4, "KV4": 5, "K4V2": 7, "KV2": 7}
    assert abs(workloads.mean_bits("llama3_8b_mixed_t32k") - 4.71875) < 1e-9


def test_nuq_lut_levels():
    lut = synth.nuq_lut("llama7b_nuq3_t1m", 0, "k")
    assert np.all(np.diff(lut) > 0) and np.allclose(np.float16(lut), lut)
    assert 1.4 < lut[-1] < 1.7 and -1.7 < lut[0] < -1.4

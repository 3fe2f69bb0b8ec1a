"""The five decode workloads, as plain parameter dicts.

Each workload fixes the model shape (layers, heads, head dim, batch,
context), the cache scheme per layer (K/V bits, groups, sink / recent fp16
windows, Hadamard V, pre-RoPE K, NUQ outliers) and the value distributions
that ``synth`` draws from.  Nothing here computes any part of the method.

Shapes follow the pages' workloads: a toy single head at 1k context, a
Llama-2-7B MHA decode at 4k, a Llama-3-8B GQA decode at 32k with per-layer
(K, V) bit pairs, a Qwen-like GQA decode with Hadamard-rotated 2-bit V, and
a LLaMA-7B layer at 1M context with pre-RoPE 3-bit non-uniform codes whose
level tables are fitted per layer on the layer's first 2048 tokens
(``lut="fitted"``; see calibrate.py).
"""
from __future__ import annotations

import numpy as np

# (K bits, V bits) of the five pairs kept after intra-layer pruning
# ("KVTuner" review, Intra-Layer KV Cache Quantization Precision Pair Pruning)
PAIRS = {"KV8": (8, 8), "K8V4": (8, 4), "KV4": (4, 4), "K4V2": (4, 2), "KV2": (2, 2)}
PAIR_ORDER = ["KV8", "K8V4", "KV4", "K4V2", "KV2"]

_BASE = dict(head_dim=128, k_group_tokens=32, v_group_channels=64, n_sink=0, n_recent=0,
             v_hadamard=0, k_pre_rope=0, rope_theta=10000.0, outliers_per_vector=0,
             softmax_scale=0.0, split_tokens=0, position_offset=0, k_group_channels=0, hybrid_groups=0,
             k_channel_norm=0)

WORKLOADS = {
    "toy_k4v2_t1k": dict(
        _BASE, layers=1, batch=1, n_q_heads=1, n_kv_heads=1, tokens=1024,
        pairs="K4V2", n_recent=32,
        k_dist="normal", k_outlier_channels="fixed4", k_outlier_scale=10.0, v_dist="normal"),
    "llama2_7b_kv4_t4k": dict(
        _BASE, layers=32, batch=8, n_q_heads=32, n_kv_heads=32, tokens=4096,
        pairs="KV4", n_sink=4, n_recent=64,
        k_dist="normal", k_outlier_channels="random3", k_outlier_scale=8.0, v_dist="laplace"),
    "llama3_8b_mixed_t32k": dict(
        _BASE, layers=32, batch=16, n_q_heads=32, n_kv_heads=8, tokens=32768,
        pairs="seeded", n_sink=4, n_recent=128,
        k_dist="normal", k_outlier_channels="random3", k_outlier_scale=8.0, v_dist="laplace"),
    "qwen_gqa_hadamard_t8k": dict(
        _BASE, layers=28, batch=64, n_q_heads=28, n_kv_heads=4, tokens=8192,
        pairs="K4V2", v_hadamard=1, n_sink=4, n_recent=32,
        k_dist="normal", k_outlier_channels="random3", k_outlier_scale=8.0, v_dist="student_t3"),
    # InnerQ: keys grouped per token along the hidden dimension (64 channels),
    # hybrid symmetric / asymmetric groups, per-channel key normalisation, at
    # the Llama-3-8B shape with the pages' 4-bit example and 32 recent tokens
    "llama3_8b_innerq_kv4_t32k": dict(
        _BASE, layers=32, batch=16, n_q_heads=32, n_kv_heads=8, tokens=32768,
        pairs="KV4", n_sink=4, n_recent=32, k_group_channels=64, hybrid_groups=1, k_channel_norm=1,
        k_dist="normal", k_outlier_channels="random3", k_outlier_scale=8.0, v_dist="laplace"),
    # the Llama-3-8B per-layer pairs of the mixed workload with InnerQ keys
    # (per-token 64-channel groups, hybrid groups, key normalisation)
    "llama3_8b_mixed_innerq_t32k": dict(
        _BASE, layers=32, batch=16, n_q_heads=32, n_kv_heads=8, tokens=32768,
        pairs="seeded", n_sink=4, n_recent=128, k_group_channels=64, hybrid_groups=1, k_channel_norm=1,
        k_dist="normal", k_outlier_channels="random3", k_outlier_scale=8.0, v_dist="laplace"),
    # RateQuant: per-head (K, V) bits allocated per layer from the measured
    # distortion of the cache's quantizer on the layer's first 2048 tokens, an
    # average of 4 bits per K or V component, at the Llama-3-8B shape, with
    # heads of different spread (K and V scales per head in [1/4, 4])
    "llama3_8b_rateq_t32k": dict(
        _BASE, layers=32, batch=16, n_q_heads=32, n_kv_heads=8, tokens=32768,
        pairs="rateq", rateq_avg_bits=4.0, rateq_calib_tokens=2048, n_sink=4, n_recent=128, head_spread=4.0,
        k_dist="normal", k_outlier_channels="random3", k_outlier_scale=8.0, v_dist="laplace"),
    # sequences of different lengths in one batch (a serving batch of
    # requests at different positions): KV4 at the Llama-3-8B shape, batch
    # row b at its own length drawn uniformly from [8192, 32768]
    "llama3_8b_kv4_ragged_t32k": dict(
        _BASE, layers=32, batch=16, n_q_heads=32, n_kv_heads=8, tokens=32768,
        pairs="KV4", n_sink=4, n_recent=128, ragged_min_tokens=8192,
        k_dist="normal", k_outlier_channels="random3", k_outlier_scale=8.0, v_dist="laplace"),
    "llama7b_nuq3_t1m": dict(
        _BASE, layers=1, batch=1, n_q_heads=32, n_kv_heads=32, tokens=1048576,
        pairs="NUQ3", k_pre_rope=1, outliers_per_vector=2, lut="fitted", lut_calib_tokens=2048,
        k_dist="normal", k_outlier_channels="random3", k_outlier_scale=8.0, v_dist="laplace"),
}

# order of the workloads as listed with the method's benchmark
WORKLOAD_ORDER = ["toy_k4v2_t1k", "llama2_7b_kv4_t4k", "llama3_8b_mixed_t32k",
                  "qwen_gqa_hadamard_t8k", "llama7b_nuq3_t1m", "llama3_8b_innerq_kv4_t32k",
                  "llama3_8b_rateq_t32k", "llama3_8b_mixed_innerq_t32k", "llama3_8b_kv4_ragged_t32k"]


def layer_pairs(name: str) -> list[str]:
    """Per-layer (K, V) pair names.  The seeded workload draws each layer's
    pair index from numpy default_rng(0).integers(0, 5, layers) over
    PAIR_ORDER and forces layers 0, 1 and the last to KV8."""
    w = WORKLOADS[name]
    if w["pairs"] == "rateq":  # per-head pairs are allocated at run time (mixed.py); KV4 is the layer's base
        return ["KV4"] * w["layers"]
    if w["pairs"] != "seeded":
        return [w["pairs"]] * w["layers"]
    idx = np.random.default_rng(0).integers(0, 5, w["layers"])
    idx[[0, 1, w["layers"] - 1]] = 0
    return [PAIR_ORDER[i] for i in idx]


def layer_config(name: str, layer: int, max_tokens: int | None = None,
                 tokens: int | None = None, batch: int | None = None,
                 k_lut=None, v_lut=None) -> dict:
    """kvq_config fields (as a dict) of one layer of a workload.  ``tokens``
    and ``batch`` shrink the workload for small parity cases; ``max_tokens``
    defaults to the context plus 64 tokens of headroom for appends."""
    w = WORKLOADS[name]
    T = w["tokens"] if tokens is None else tokens
    pair = layer_pairs(name)[layer]
    if pair == "NUQ3":
        kb = vb = 3
    elif pair == "FP16":
        kb = vb = 16
    else:
        kb, vb = PAIRS[pair]
    cfg = {k: w[k] for k in _BASE}
    cfg.update(batch=w["batch"] if batch is None else batch, n_q_heads=w["n_q_heads"],
               n_kv_heads=w["n_kv_heads"], max_tokens=(T + 64) if max_tokens is None else max_tokens,
               k_bits=kb, v_bits=vb)
    cfg["k_lut"] = list(k_lut) if k_lut is not None else [0.0] * 8
    cfg["v_lut"] = list(v_lut) if v_lut is not None else [0.0] * 8
    return cfg


def row_tokens(name: str, tokens: int | None = None) -> list[int] | None:
    """Per batch row lengths of a ragged workload at its decode step (the
    longest row has `tokens`, default the workload's context; the others are
    drawn uniformly from [ragged_min_tokens scaled alike, tokens] by
    numpy default_rng(1)), or None for a uniform workload."""
    w = WORKLOADS[name]
    if "ragged_min_tokens" not in w:
        return None
    T = w["tokens"] if tokens is None else tokens
    lo = max(1, w["ragged_min_tokens"] * T // w["tokens"])
    rows = np.random.default_rng(1).integers(lo, T + 1, w["batch"])
    rows[0] = T
    return [int(r) for r in rows]


def fp16_baseline_config(cfg: dict) -> dict:
    """The same shape as an all-fp16 cache (the baseline decode)."""
    c = dict(cfg)
    c.update(k_bits=16, v_bits=16, n_sink=0, n_recent=0, v_hadamard=0, k_pre_rope=0,
             outliers_per_vector=0, k_group_channels=0, hybrid_groups=0, k_channel_norm=0)
    return c


def mean_bits(name: str) -> float:
    """f_m: mean bits over the 2L K/V tensors ("KVTuner" review, problem formulation)."""
    ps = layer_pairs(name)
    if ps[0] == "NUQ3":
        return 3.0
    return sum(sum(PAIRS[p]) for p in ps) / (2 * len(ps))

"""The benchmark's algorithmic bytes per decode launch against the library's
own layout (host only, no GPU): at a context whose quantized part fills the
layer exactly (Nq = q_cap, fp16 window = n_recent), the bytes the roofline
divides by must equal the layout regions one decode reads -- packed codes,
their scales, CSR outlier columns and values (the row pointers are not
read), the key normalisation, the fp16 sinks and window -- plus q and out.
A region counted twice or missed (the InnerQ key scales once were charged
per channel instead of per token) fails here."""
import pytest

import bench
from bit_kv_cache_07_gb300 import binding, workloads

D = 128
NAMES = ["llama2_7b_kv4_t4k", "llama3_8b_mixed_t32k", "qwen_gqa_hadamard_t8k", "llama3_8b_innerq_kv4_t32k",
         "llama3_8b_mixed_innerq_t32k", "llama7b_nuq3_t1m"]


def _cases():
    for name in NAMES:
        seen = set()
        for layer, pair in enumerate(workloads.layer_pairs(name)):
            if pair not in seen:
                seen.add(pair)
                yield name, layer


@pytest.mark.parametrize("name,layer", list(_cases()))
def test_algorithmic_bytes_equal_the_regions_a_decode_reads(name, layer):
    lut = [i / 7.0 for i in range(8)]  # any increasing table (non-uniform layers need one)
    probe = workloads.layer_config(name, layer, tokens=1024, batch=2, max_tokens=4096, k_lut=lut, v_lut=lut)
    S, R = probe["n_sink"], probe["n_recent"]
    T = S + R + 32 * ((2048 - S - R) // 32)  # quantized part a whole number of groups
    cfg = dict(probe, max_tokens=T)
    L = binding.kvq_layout_query(cfg)
    s, nq, w = bench.window_counts(cfg, T)
    assert (s, nq, w) == (S, L.q_cap, R)
    NS = cfg["batch"] * cfg["n_kv_heads"]
    read = ["k_codes", "k_scales", "v_codes", "v_scales", "k_csr_col", "k_csr_val", "v_csr_col", "v_csr_val",
            "k_norm", "k_sink", "v_sink"]
    cache = sum(getattr(L, r).bytes for r in read) + 2 * NS * R * D * 2  # ring: only the R live window tokens
    qo = cfg["batch"] * cfg["n_q_heads"] * D * 2 * 2
    assert bench.algorithmic_bytes(cfg, T) == cache + qo


def test_fp16_cache_bytes():
    cfg = workloads.fp16_baseline_config(workloads.layer_config("llama3_8b_mixed_t32k", 0, batch=2,
                                                                max_tokens=2048))
    NS = cfg["batch"] * cfg["n_kv_heads"]
    qo = cfg["batch"] * cfg["n_q_heads"] * D * 2 * 2
    assert bench.algorithmic_bytes(cfg, 1000) == NS * 1000 * D * 2 * 2 + qo


def test_ragged_bytes_sum_the_rows():
    """A ragged batch's bytes are its rows' bytes at their own lengths: equal
    rows give the uniform count, and each row adds what a one-row batch at
    its length reads."""
    cfg = workloads.layer_config("llama3_8b_kv4_ragged_t32k", 0, batch=3, max_tokens=4096)
    assert bench.algorithmic_bytes(cfg, 2000, [2000] * 3) == bench.algorithmic_bytes(cfg, 2000)
    one = dict(cfg, batch=1)
    rows = [2000, 37, 1500]
    assert bench.algorithmic_bytes(cfg, 2000, rows) == sum(bench.algorithmic_bytes(one, t) for t in rows)
    lengths = workloads.row_tokens("llama3_8b_kv4_ragged_t32k")
    w = workloads.WORKLOADS["llama3_8b_kv4_ragged_t32k"]
    assert len(lengths) == w["batch"] and max(lengths) == w["tokens"]
    assert min(lengths) >= w["ragged_min_tokens"]

"""Per-layer non-uniform level tables for a workload (KVQuant summary,
"technical approach": non-uniform per-layer datatypes computed offline from
calibration activations).

A workload whose ``lut`` is ``"fitted"`` takes each layer's K and V tables
from ``kvq_fit_nuq_lut`` (unweighted Lloyd, run on the GPU by libkvq) over
the layer's first ``lut_calib_tokens`` tokens of batch row 0, all KV heads:
K as cached (before RoPE), V as the encoder sees it (rotated first when the
cache rotates V).  Otherwise the tables are the seeded N(0, 1) quantiles of
``synth.nuq_lut``.  This module only draws the calibration tokens and calls
the library.
"""
from __future__ import annotations

from . import binding, synth
from .workloads import WORKLOADS


def calibration_kv(name: str, layer: int, device="cuda"):
    """fp16 K, V [1, Hkv, n, d] the tables of a fitted workload are fitted to."""
    w = WORKLOADS[name]
    return synth.layer_kv(name, layer, tokens=w["lut_calib_tokens"], batch=1, device=device)


def nuq_tables(name: str, layer: int, device="cuda"):
    """(k_lut, v_lut) of one layer of a 3-bit non-uniform workload."""
    w = WORKLOADS[name]
    if w.get("lut") != "fitted":
        return synth.nuq_lut(name, layer, "k"), synth.nuq_lut(name, layer, "v")
    K, V = calibration_kv(name, layer, device=device)
    k = w["outliers_per_vector"]
    klut, kit = binding.kvq_fit_nuq_lut(K, k, 0)
    vlut, vit = binding.kvq_fit_nuq_lut(V, k, w["v_hadamard"])
    if kit < 0 or vit < 0:
        raise RuntimeError(f"{name} layer {layer}: the fitted level table is not strictly increasing")
    return klut, vlut

"""Shared helpers of the GPU parity tests: read a stream's stored cache out of
a GPU layer buffer in the oracle's array shapes, and compare attention
outputs the way the method's tolerance is stated (normwise per output
vector: max |o_gpu - o_ref| / max |o_ref| over the head dimension)."""
from __future__ import annotations

import numpy as np

TOL = 2e-3  # attention: max relative (normwise) error against the fp64 oracle


def gpu_store(layer, s: int, T: int, counts) -> dict:
    """Stream s of a binding.Layer after T tokens, as the oracle's store dict."""
    cfg = layer.cfg
    lay = layer.layout
    S, Nq, W = counts
    d = cfg.head_dim
    NS = cfg.batch * cfg.n_kv_heads
    kb, vb = cfg.k_bits, cfg.v_bits
    host = {}

    import torch
    tdt = {np.uint8: torch.uint8, np.uint16: torch.int16, np.int32: torch.int32, np.float32: torch.float32}

    class _Reg:
        """Region viewed as [NS, ...] on the device; only stream s is copied."""

        def __init__(self, name, dtype):
            self.r = layer.region(name)
            self.dtype = dtype

        def reshape(self, *shape):
            self.shape = shape
            return self

        def __getitem__(self, idx):
            s_, rest = idx[0], idx[1:]
            if self.r.numel() == 0:
                return np.zeros(tuple(self.shape[1:]), self.dtype)[rest]
            t = self.r.view(tdt[self.dtype]).view(*self.shape)[s_].cpu().numpy().view(self.dtype)
            return t[rest] if rest else t

    def reg(name, dtype):
        return _Reg(name, dtype)

    qcap = lay.q_cap
    if kb == 16:
        ring = reg("k_ring", np.uint16).reshape(NS, lay.ring_slots, d)
        vring = reg("v_ring", np.uint16).reshape(NS, lay.ring_slots, d)
        host["kwin"] = ring[s, :T].copy()
        host["vwin"] = vring[s, :T].copy()
        return host
    krow, vrow = d * kb // 8, d * vb // 8
    host["kc"] = reg("k_codes", np.uint8).reshape(NS, qcap, krow)[s, :Nq]
    if kb == 3:
        host["ks"] = reg("k_scales", np.uint16).reshape(NS, qcap, 2)[s, :Nq]
        host["vs"] = reg("v_scales", np.uint16).reshape(NS, qcap, 2)[s, :Nq]
        k = cfg.outliers_per_vector
        for side in ("k", "v"):
            host[f"{side}_rowptr"] = reg(f"{side}_csr_rowptr", np.int32).reshape(NS, qcap + 1)[s, :Nq + 1]
            host[f"{side}_cols"] = reg(f"{side}_csr_col", np.uint8).reshape(NS, qcap * k)[s, :Nq * k]
            host[f"{side}_vals"] = reg(f"{side}_csr_val", np.uint16).reshape(NS, qcap * k)[s, :Nq * k]
    else:
        gcap = qcap // 32
        nvg = d // cfg.v_group_channels
        if cfg.k_group_channels:  # InnerQ keys: per token, per 64-channel group
            nkg = d // cfg.k_group_channels
            host["ks"] = reg("k_scales", np.uint16).reshape(NS, qcap, nkg, 2)[s, :Nq]
        else:
            host["ks"] = reg("k_scales", np.uint16).reshape(NS, gcap, d, 2)[s, :Nq // 32]
        host["vs"] = reg("v_scales", np.uint16).reshape(NS, qcap, nvg, 2)[s, :Nq]
        if cfg.k_channel_norm:
            host["kn"] = reg("k_norm", np.float32).reshape(NS, d)[s, :]
    host["vc"] = reg("v_codes", np.uint8).reshape(NS, qcap, vrow)[s, :Nq]
    Sc = cfg.n_sink
    host["ksink"] = reg("k_sink", np.uint16).reshape(NS, Sc, d)[s, :S] if Sc else np.zeros((0, d), np.uint16)
    host["vsink"] = reg("v_sink", np.uint16).reshape(NS, Sc, d)[s, :S] if Sc else np.zeros((0, d), np.uint16)
    R = lay.ring_slots
    slots = [(cfg.n_sink + Nq + w - cfg.n_sink) % R for w in range(W)]
    host["kwin"] = reg("k_ring", np.uint16).reshape(NS, R, d)[s,][slots]
    host["vwin"] = reg("v_ring", np.uint16).reshape(NS, R, d)[s,][slots]
    return host


def assert_store_equal(gpu: dict, ref: dict, where=""):
    for name, a in gpu.items():
        b = ref[name]
        assert a.shape == b.shape, (where, name, a.shape, b.shape)
        if not np.array_equal(a, b):
            bad = np.argwhere(a != b)
            raise AssertionError(f"{where}: region {name} differs at {len(bad)} places, first {bad[:3].tolist()}")


def normwise_err(out, ref):
    out = np.asarray(out, np.float64)
    ref = np.asarray(ref, np.float64)
    return np.max(np.abs(out - ref), -1) / np.maximum(np.max(np.abs(ref), -1), 1e-30)

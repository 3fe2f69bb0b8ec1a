"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module only draws random numbers in the shapes and distributions of the
workloads (``workloads.py``); it holds none of the method's arithmetic.  The
same call gives the same tensor on every machine and device type for a
given torch version: every tensor gets its own ``torch.Generator`` seeded
from a CRC of (workload, layer, tensor name, chunk).

Recipe (per layer):
  K  ~ N(0, 1), with a few outlier channels multiplied by a constant
       (4 fixed channels x10 for the toy workload; 3 channels per KV head,
       drawn per layer, x8 for the others) -- K outliers are channel-wise
       ("KVTuner" review, observation 2; KVQuant per-channel keys);
  V  ~ N(0, 1), Laplace(0, 1) or Student-t(nu=3) per workload;
  per-head spread (the per-head bit workload): K and V of each KV head
       scaled by factors log-uniform in [1/4, 4], drawn per layer;
  q  ~ N(0, 1);
  NUQ level tables: 8 quantiles of 65,536 seeded N(0, 1) samples, rounded
  to fp16 (a stand-in for the per-layer offline datatype of KVQuant).
All tensors are rounded to fp16 before use.
"""
from __future__ import annotations

import zlib

import numpy as np
import torch

from .workloads import WORKLOADS

CHUNK = 4096  # tokens drawn per generator call (keeps temporaries small)


def seed_of(*parts) -> int:
    return zlib.crc32("/".join(str(p) for p in parts).encode()) & 0x7FFFFFFF


def _gen(device, *parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed_of(*parts))
    return g


def k_outlier_channels(name: str, layer: int, n_kv_heads: int, d: int) -> np.ndarray:
    """[n_kv_heads, n] channel indices whose K values are scaled up."""
    w = WORKLOADS[name]
    if w["k_outlier_channels"] == "fixed4":
        ch = np.random.default_rng(0).permutation(d)[:4]
        return np.tile(ch, (n_kv_heads, 1))
    n = int(round(0.02 * d))
    rng = np.random.default_rng(seed_of(name, layer, "k_outlier_channels"))
    return np.stack([rng.permutation(d)[:n] for _ in range(n_kv_heads)])


def _draw(dist: str, shape, g: torch.Generator, device) -> torch.Tensor:
    if dist == "normal":
        return torch.randn(shape, generator=g, device=device)
    if dist == "laplace":
        # difference of two Exp(1) draws; -log1p(-r) is finite for r in [0, 1)
        e1 = -torch.log1p(-torch.rand(shape, generator=g, device=device))
        e2 = -torch.log1p(-torch.rand(shape, generator=g, device=device))
        return e1 - e2
    if dist == "student_t3":
        z = torch.randn(shape, generator=g, device=device)
        chi2 = torch.randn((3,) + tuple(shape), generator=g, device=device).pow(2).sum(0)
        return z / torch.sqrt(chi2 / 3.0)
    raise ValueError(dist)


def head_scales(name: str, layer: int, n_kv_heads: int, spread: float):
    """Per-KV-head K and V scale factors, log-uniform in [1/spread, spread]
    (seeded per layer): heads whose values differ in spread."""
    rng = np.random.default_rng(seed_of(name, layer, "head_scales"))
    return (spread ** rng.uniform(-1, 1, n_kv_heads), spread ** rng.uniform(-1, 1, n_kv_heads))


def layer_kv(name: str, layer: int, tokens: int | None = None, batch: int | None = None,
             device="cpu", t0: int = 0):
    """fp16 K, V of one layer: [B, Hkv, tokens, d], token positions [t0, t0 + tokens)."""
    w = WORKLOADS[name]
    B = w["batch"] if batch is None else batch
    H, d = w["n_kv_heads"], w["head_dim"]
    T = w["tokens"] if tokens is None else tokens
    K = torch.empty((B, H, T, d), dtype=torch.float16, device=device)
    V = torch.empty((B, H, T, d), dtype=torch.float16, device=device)
    och = torch.as_tensor(k_outlier_channels(name, layer, H, d), device=device)
    kscale = torch.ones((H, d), device=device)
    kscale.scatter_(1, och, float(w["k_outlier_scale"]))
    vscale = torch.ones((H, 1), device=device)
    if w.get("head_spread"):  # heads of different spread: K and V scales per head, log-uniform in [1/s, s]
        hk, hv = head_scales(name, layer, H, w["head_spread"])
        kscale = kscale * torch.as_tensor(hk, dtype=torch.float32, device=device)[:, None]
        vscale = torch.as_tensor(hv, dtype=torch.float32, device=device)[:, None]
    first, last = t0 // CHUNK, (t0 + T - 1) // CHUNK
    for c in range(first, last + 1):
        a, b = max(t0, c * CHUNK), min(t0 + T, (c + 1) * CHUNK)
        shape = (B, H, CHUNK, d)
        kc = _draw(w["k_dist"], shape, _gen(device, name, layer, "K", c), device)
        vc = _draw(w["v_dist"], shape, _gen(device, name, layer, "V", c), device)
        kc = kc * kscale[None, :, None, :]
        vc = vc * vscale[None, :, :, None]
        lo, hi = a - c * CHUNK, b - c * CHUNK
        K[:, :, a - t0:b - t0] = kc[:, :, lo:hi].to(torch.float16)
        V[:, :, a - t0:b - t0] = vc[:, :, lo:hi].to(torch.float16)
    return K, V


def query(name: str, layer: int, batch: int | None = None, device="cpu", step: int = 0):
    """fp16 query [B, Hq, d] for one decode step (already position-encoded)."""
    w = WORKLOADS[name]
    B = w["batch"] if batch is None else batch
    g = _gen(device, name, layer, "q", step)
    return torch.randn((B, w["n_q_heads"], w["head_dim"]), generator=g,
                       device=device).to(torch.float16)


def new_token_kv(name: str, layer: int, step: int, batch: int | None = None, device="cpu"):
    """fp16 K, V of one appended decode token: [B, Hkv, 1, d]."""
    w = WORKLOADS[name]
    B = w["batch"] if batch is None else batch
    shape = (B, w["n_kv_heads"], 1, w["head_dim"])
    k = _draw(w["k_dist"], shape, _gen(device, name, layer, "k_new", step), device)
    v = _draw(w["v_dist"], shape, _gen(device, name, layer, "v_new", step), device)
    return k.to(torch.float16), v.to(torch.float16)


def nuq_lut(name: str, layer: int, which: str) -> list[float]:
    """8 increasing fp16-representable levels: the samples at ranks
    floor((i + 0.5) * 65536 / 8) of 65,536 sorted seeded N(0, 1) draws."""
    rng = np.random.default_rng(seed_of(name, layer, which + "_lut"))
    x = np.sort(rng.standard_normal(65536))
    idx = ((np.arange(8) + 0.5) * 65536 / 8).astype(np.int64)
    return [float(v) for v in x[idx].astype(np.float16).astype(np.float32)]


def random_halves(shape, seed: int, scale: float = 1.0) -> np.ndarray:
    """Plain N(0, scale^2) fp16 array for small oracle-only tests."""
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(shape) * scale).astype(np.float16)


def random_kv(B: int, Hkv: int, T: int, d: int = 128, seed: int = 0, device="cpu",
              k_outlier_channels: int = 3, k_outlier_scale: float = 8.0, v_dist: str = "laplace"):
    """Generic fp16 K, V [B, Hkv, T, d] for parity cases of any shape:
    K ~ N(0,1) with a few per-head outlier channels scaled up, V from v_dist."""
    g = _gen(device, "random_kv", seed)
    K = torch.randn((B, Hkv, T, d), generator=g, device=device)
    if k_outlier_channels:
        idx = torch.stack([torch.randperm(d, generator=g, device=device)[:k_outlier_channels]
                           for _ in range(Hkv)])
        sc = torch.ones((Hkv, d), device=device)
        sc.scatter_(1, idx, float(k_outlier_scale))
        K = K * sc[None, :, None, :]
    V = _draw(v_dist, (B, Hkv, T, d), g, device)
    return K.to(torch.float16), V.to(torch.float16)


def random_q(B: int, Hq: int, d: int = 128, seed: int = 0, device="cpu"):
    g = _gen(device, "random_q", seed)
    return torch.randn((B, Hq, d), generator=g, device=device).to(torch.float16)


def lut_from_seed(seed: int) -> list[float]:
    """8 fp16 N(0,1) sample quantiles (see nuq_lut) from a plain seed."""
    rng = np.random.default_rng(seed)
    x = np.sort(rng.standard_normal(65536))
    idx = ((np.arange(8) + 0.5) * 65536 / 8).astype(np.int64)
    return [float(v) for v in x[idx].astype(np.float16).astype(np.float32)]

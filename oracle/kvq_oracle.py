"""Python wrapper around the plain-C CPU oracle (``kvq_oracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the
benchmark's CPU-baseline leg are the only callers.  Nothing here imports the
product package, and the product package never imports this module.

A configuration is a plain ``dict`` with the field names of the library's
``kvq_config`` (``head_dim``, ``k_bits``, ``v_bits``, ``k_group_tokens``,
``v_group_channels``, ``n_sink``, ``n_recent``, ``v_hadamard``,
``k_pre_rope``, ``rope_theta``, ``outliers_per_vector``, ``k_lut``,
``v_lut``, ``softmax_scale``; plus ``batch``, ``n_q_heads``, ``n_kv_heads``
for the layer-level helpers).  fp16 data travels as ``numpy.float16`` or its
``uint16`` bit pattern.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_LIB = os.environ.get("KVQ_ORACLE_LIB") or os.path.join(_HERE, "libkvq_oracle.so")
_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]

_lib = None


def build_library(force: bool = False) -> str:
    """Compile kvq_oracle.c into oracle/libkvq_oracle.so with gcc."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *_CFLAGS, "-o", tmp, os.environ.get("KVQ_ORACLE_SRC", _SRC), "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Cfg(C.Structure):
    _fields_ = [
        ("d", C.c_int32), ("k_bits", C.c_int32), ("v_bits", C.c_int32),
        ("gk", C.c_int32), ("gv", C.c_int32), ("n_sink", C.c_int32),
        ("n_recent", C.c_int32), ("v_hadamard", C.c_int32), ("k_pre_rope", C.c_int32),
        ("outliers", C.c_int32), ("rope_theta", C.c_double), ("sm_scale", C.c_double),
        ("k_lut", C.c_float * 8), ("v_lut", C.c_float * 8), ("pos_offset", C.c_int32),
        ("gkc", C.c_int32), ("hybrid", C.c_int32), ("k_norm", C.c_int32), ("norm_tokens", C.c_int32),
    ]


def _P(a, ct):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(C.POINTER(ct))


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(build_library())
        u8, u16, i32, f64 = (C.POINTER(t) for t in (C.c_uint8, C.c_uint16, C.c_int32, C.c_double))
        L = _lib
        L.orc_half_to_float.argtypes = [C.c_uint16]
        L.orc_half_to_float.restype = C.c_float
        L.orc_float_to_half.argtypes = [C.c_float]
        L.orc_float_to_half.restype = C.c_uint16
        L.orc_quantize_uniform.argtypes = [u16, C.c_int, C.c_int, C.c_int, u8, C.c_int, u16, u16]
        L.orc_pack_bits.argtypes = [u8, C.c_int, C.c_int, u8]
        L.orc_unpack_bits.argtypes = [u8, C.c_int, C.c_int, u8]
        L.orc_hadamard_rotate.argtypes = [u16, C.c_int, u16]
        L.orc_hadamard_apply_f64.argtypes = [f64, C.c_int, f64]
        L.orc_nuq_encode.argtypes = [u16, C.c_int, C.c_int, C.POINTER(C.c_float), u8, u16, u16, u8, u16]
        L.orc_nuq_decode.argtypes = [u8, C.c_int, C.c_uint16, C.c_uint16, C.POINTER(C.c_float),
                                     C.c_int, u8, u16, f64]
        L.orc_rope_apply.argtypes = [f64, C.c_int, C.c_double, C.c_double]
        L.orc_layout_counts.argtypes = [C.POINTER(_Cfg), C.c_int, C.POINTER(C.c_int),
                                        C.POINTER(C.c_int), C.POINTER(C.c_int)]
        f32 = C.POINTER(C.c_float)
        L.orc_build_stream.argtypes = [C.POINTER(_Cfg), C.c_int, u16, u16,
                                       u8, u16, u8, u16, u16, u16, u16, u16,
                                       i32, u8, u16, i32, u8, u16, f32]
        L.orc_quantize_group.argtypes = [f32, C.c_int, C.c_int, C.c_int, C.c_int, u8, C.c_int, u16, u16]
        L.orc_key_norm.argtypes = [u16, C.c_int, C.c_int, f32]
        L.orc_nuq_fit_lut.argtypes = [u16, C.c_long, C.c_int, C.c_int, C.c_int, C.c_int, C.POINTER(C.c_float),
                                      f64]
        L.orc_nuq_fit_lut.restype = C.c_int
        L.orc_nuq_fit_positions.argtypes = [u16, C.c_long, C.c_int, C.c_int, C.c_int, i32, C.c_long]
        L.orc_nuq_fit_positions.restype = C.c_long
        L.orc_quant_distortion.argtypes = [C.POINTER(_Cfg), C.c_int, u16, u16, C.c_int, f64, f64]
        L.orc_fit_rd.argtypes = [C.c_int, f64, f64, f64, f64]
        L.orc_rate_waterfill.argtypes = [C.c_int, f64, f64, f64, C.c_double, f64]
        L.orc_rate_greedy.argtypes = [C.c_int, f64, f64, f64, C.c_int, i32]
        L.orc_rate_greedy.restype = C.c_int
        L.orc_merge_parts.argtypes = [C.c_int, C.c_int, C.c_int, f64, f64, f64, f64]
        L.orc_decode_stream.argtypes = [C.POINTER(_Cfg), C.c_int, C.c_int, u16,
                                        u8, u16, u8, u16, u16, u16, u16, u16,
                                        i32, u8, u16, i32, u8, u16, f32, f64, f64]
    return _lib


# ---------------------------------------------------------------- primitives

def _u16(x) -> np.ndarray:
    x = np.asarray(x)
    if x.dtype == np.float16:
        x = x.view(np.uint16)
    return np.ascontiguousarray(x, dtype=np.uint16)


def half_to_float(h: int) -> float:
    return lib().orc_half_to_float(int(h))


def float_to_half(x: float) -> int:
    return lib().orc_float_to_half(float(x))


def quantize_uniform(x, bits: int):
    """Uniform asymmetric quantization of one group -> (codes u8, min_h u16, scale_h u16)."""
    x = _u16(x).ravel()
    codes = np.zeros(x.size, np.uint8)
    mn, sc = C.c_uint16(), C.c_uint16()
    lib().orc_quantize_uniform(_P(x, C.c_uint16), x.size, 1, bits, _P(codes, C.c_uint8), 1,
                               C.byref(mn), C.byref(sc))
    return codes, mn.value, sc.value


def pack_bits(codes, bits: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, np.uint8).ravel()
    out = np.zeros((codes.size * bits + 7) // 8, np.uint8)
    lib().orc_pack_bits(_P(codes, C.c_uint8), codes.size, bits, _P(out, C.c_uint8))
    return out


def unpack_bits(packed, n: int, bits: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, np.uint8).ravel()
    out = np.zeros(n, np.uint8)
    lib().orc_unpack_bits(_P(packed, C.c_uint8), n, bits, _P(out, C.c_uint8))
    return out


def hadamard_rotate(v) -> np.ndarray:
    """fp16 v -> fp16 bits of fp32(1/sqrt(n)) * (H v), H Sylvester."""
    v = _u16(v).ravel()
    out = np.zeros_like(v)
    lib().orc_hadamard_rotate(_P(v, C.c_uint16), v.size, _P(out, C.c_uint16))
    return out


def hadamard_apply(x) -> np.ndarray:
    """fp64 Hn x, Hn = H / sqrt(n)."""
    x = np.ascontiguousarray(x, np.float64).ravel()
    out = np.zeros_like(x)
    lib().orc_hadamard_apply_f64(_P(x, C.c_double), x.size, _P(out, C.c_double))
    return out


def nuq_encode(x, k: int, lut):
    x = _u16(x).ravel()
    n = x.size
    lut_a = (C.c_float * 8)(*[float(v) for v in lut])
    codes = np.zeros(n, np.uint8)
    cols = np.zeros(max(k, 1), np.uint8)
    vals = np.zeros(max(k, 1), np.uint16)
    mn, s = C.c_uint16(), C.c_uint16()
    lib().orc_nuq_encode(_P(x, C.c_uint16), n, k, lut_a, _P(codes, C.c_uint8), C.byref(mn),
                         C.byref(s), _P(cols, C.c_uint8), _P(vals, C.c_uint16))
    return codes, mn.value, s.value, cols[:k].copy(), vals[:k].copy()


def nuq_decode(codes, min_h: int, s_h: int, lut, cols, vals) -> np.ndarray:
    codes = np.ascontiguousarray(codes, np.uint8).ravel()
    cols = np.ascontiguousarray(cols, np.uint8).ravel()
    vals = _u16(vals).ravel()
    lut_a = (C.c_float * 8)(*[float(v) for v in lut])
    out = np.zeros(codes.size, np.float64)
    lib().orc_nuq_decode(_P(codes, C.c_uint8), codes.size, min_h, s_h, lut_a, cols.size,
                         _P(cols, C.c_uint8) if cols.size else None,
                         _P(vals, C.c_uint16) if vals.size else None, _P(out, C.c_double))
    return out


def rope_apply(x, pos: float, base: float) -> np.ndarray:
    x = np.array(x, np.float64).ravel()
    lib().orc_rope_apply(_P(x, C.c_double), x.size, float(pos), float(base))
    return x


# ------------------------------------------------------------------ streams

def _cfg(cfg: dict) -> _Cfg:
    c = _Cfg()
    c.d = cfg["head_dim"]
    c.k_bits = cfg["k_bits"]
    c.v_bits = cfg["v_bits"]
    c.gk = cfg.get("k_group_tokens", 32)
    c.gv = cfg.get("v_group_channels", 64)
    c.n_sink = cfg.get("n_sink", 0)
    c.n_recent = cfg.get("n_recent", 0)
    c.v_hadamard = cfg.get("v_hadamard", 0)
    c.k_pre_rope = cfg.get("k_pre_rope", 0)
    c.outliers = cfg.get("outliers_per_vector", 0)
    c.rope_theta = cfg.get("rope_theta", 10000.0)
    c.sm_scale = cfg.get("softmax_scale", 0.0)
    c.pos_offset = cfg.get("position_offset", 0)
    c.gkc = cfg.get("k_group_channels", 0)
    c.hybrid = cfg.get("hybrid_groups", 0)
    c.k_norm = cfg.get("k_channel_norm", 0)
    c.norm_tokens = cfg.get("norm_tokens", 0)
    for i, v in enumerate(cfg.get("k_lut", [0.0] * 8)):
        c.k_lut[i] = v
    for i, v in enumerate(cfg.get("v_lut", [0.0] * 8)):
        c.v_lut[i] = v
    return c


def layout_counts(cfg: dict, T: int):
    """(S_eff, Nq, W): sink tokens, quantized tokens, fp16 window tokens."""
    s, nq, w = C.c_int(), C.c_int(), C.c_int()
    c = _cfg(cfg)
    lib().orc_layout_counts(C.byref(c), T, C.byref(s), C.byref(nq), C.byref(w))
    return s.value, nq.value, w.value


def _store_shapes(cfg: dict, T: int):
    d = cfg["head_dim"]
    kb, vb = cfg["k_bits"], cfg["v_bits"]
    S, Nq, W = layout_counts(cfg, T)
    k = cfg.get("outliers_per_vector", 0)
    gk = cfg.get("k_group_tokens", 32)
    gv = cfg.get("v_group_channels", 64)
    gkc = cfg.get("k_group_channels", 0)
    shapes = {
        "kc": ((Nq, d * kb // 8 if kb != 16 else 0), np.uint8),
        "ks": (((Nq, 2) if kb == 3 else (Nq, d // gkc, 2) if gkc else (Nq // gk if kb != 16 else 0, d, 2)),
               np.uint16),
        "vc": ((Nq, d * vb // 8 if vb != 16 else 0), np.uint8),
        "vs": (((Nq, 2) if vb == 3 else (Nq, d // gv if vb != 16 else 0, 2)), np.uint16),
        "ksink": ((S, d), np.uint16), "vsink": ((S, d), np.uint16),
        "kwin": ((W, d), np.uint16), "vwin": ((W, d), np.uint16),
        "k_rowptr": ((Nq + 1 if kb == 3 else 0,), np.int32),
        "k_cols": ((Nq * k if kb == 3 else 0,), np.uint8),
        "k_vals": ((Nq * k if kb == 3 else 0,), np.uint16),
        "v_rowptr": ((Nq + 1 if vb == 3 else 0,), np.int32),
        "v_cols": ((Nq * k if vb == 3 else 0,), np.uint8),
        "v_vals": ((Nq * k if vb == 3 else 0,), np.uint16),
        "kn": ((d if cfg.get("k_channel_norm", 0) else 0,), np.float32),
    }
    return shapes


_ORDER = ["kc", "ks", "vc", "vs", "ksink", "vsink", "kwin", "vwin",
          "k_rowptr", "k_cols", "k_vals", "v_rowptr", "v_cols", "v_vals", "kn"]
_CT = {np.uint8: C.c_uint8, np.uint16: C.c_uint16, np.int32: C.c_int32, np.float32: C.c_float}


def _ptrs(store):
    out = []
    for name in _ORDER:
        a = store[name]
        ct = _CT[a.dtype.type]
        # an empty array still needs a valid (never dereferenced) pointer
        out.append(_P(a if a.size else np.zeros(1, a.dtype), ct))
    return out


def build_stream(cfg: dict, K, V) -> dict:
    """Stored representation of one stream from its fp16 K, V ([T, d])."""
    K, V = _u16(K), _u16(V)
    T, d = K.shape
    assert d == cfg["head_dim"] and V.shape == K.shape
    store = {n: np.zeros(shp, dt) for n, (shp, dt) in _store_shapes(cfg, T).items()}
    c = _cfg(cfg)
    lib().orc_build_stream(C.byref(c), T, _P(K, C.c_uint16), _P(V, C.c_uint16), *_ptrs(store))
    return store


def decode_stream(cfg: dict, T: int, store: dict, q):
    """fp64 attention output [g, d] and lse [g] of one stream's g query heads."""
    q = _u16(q)
    g, d = q.shape
    out = np.zeros((g, d), np.float64)
    lse = np.zeros(g, np.float64)
    c = _cfg(cfg)
    lib().orc_decode_stream(C.byref(c), T, g, _P(q, C.c_uint16), *_ptrs(store),
                            _P(out, C.c_double), _P(lse, C.c_double))
    return out, lse


# ------------------------------------------------------------------- layers

def build_layer(cfg: dict, K, V, streams=None) -> list:
    """Per-stream stores for K, V of shape [B, Hkv, T, d]; stream s = b*Hkv + h.
    ``streams`` restricts the work to a subset (others are None)."""
    K, V = _u16(K), _u16(V)
    B, H, T, d = K.shape
    out = [None] * (B * H)
    for s in (range(B * H) if streams is None else streams):
        b, h = divmod(s, H)
        out[s] = build_stream(cfg, K[b, h], V[b, h])
    return out


def decode_layer(cfg: dict, T: int, stores: list, q, streams=None):
    """fp64 attention [B, Hq, d] and lse [B, Hq]; q is [B, Hq, d] fp16.
    Query head h reads KV head h // (Hq / Hkv)."""
    q = _u16(q)
    B, Hq, d = q.shape
    Hkv = len(stores) // B
    g = Hq // Hkv
    out = np.full((B, Hq, d), np.nan)
    lse = np.full((B, Hq), np.nan)
    for s in (range(B * Hkv) if streams is None else streams):
        b, h = divmod(s, Hkv)
        o, l = decode_stream(cfg, T, stores[s], q[b, h * g:(h + 1) * g])
        out[b, h * g:(h + 1) * g] = o
        lse[b, h * g:(h + 1) * g] = l
    return out, lse


def merge_parts(outs, lses):
    """Attention over the union of n disjoint context parts from each part's
    normalised output and log-sum-exp: outs [n, ..., d], lses [n, ...]
    (fp64; -inf marks an empty part) -> (out [..., d], lse [...])."""
    outs = np.ascontiguousarray(outs, np.float64)
    lses = np.ascontiguousarray(lses, np.float64)
    n, d = outs.shape[0], outs.shape[-1]
    rows = int(np.prod(outs.shape[1:-1])) if outs.ndim > 2 else 1
    assert lses.shape == outs.shape[:-1]
    out = np.zeros(outs.shape[1:], np.float64)
    lse = np.zeros(lses.shape[1:], np.float64)
    lib().orc_merge_parts(n, rows, d, _P(outs, C.c_double), _P(lses, C.c_double),
                          _P(out, C.c_double), _P(lse, C.c_double))
    return out, lse


def nuq_fit_lut(x, k: int, hadamard: int = 0, max_iters: int = 100, levels: bool = False):
    """Fit 8 non-uniform levels to the vectors x [..., d] (fp16): unweighted
    Lloyd on the dense values' positions in their vector's [min, max] range,
    end levels held at 0 and 1.  Returns (lut list of 8 floats, updates made
    or -1 if the fp16-rounded levels are not strictly increasing), plus the
    unrounded levels in grid units (fp64 array) when levels=True."""
    x = _u16(x)
    d = x.shape[-1]
    nvec = x.size // d
    lut = (C.c_float * 8)()
    lv = np.zeros(8, np.float64)
    it = lib().orc_nuq_fit_lut(_P(np.ascontiguousarray(x.reshape(nvec, d)), C.c_uint16), nvec, d, k,
                               hadamard, max_iters, lut, _P(lv, C.c_double))
    if levels:
        return [float(v) for v in lut], it, lv
    return [float(v) for v in lut], it


def nuq_fit_positions(x, k: int, hadamard: int = 0) -> np.ndarray:
    """The grid positions (0 .. 2^16) of the dense values the fit sees."""
    x = _u16(x)
    d = x.shape[-1]
    nvec = x.size // d
    xs = np.ascontiguousarray(x.reshape(nvec, d))
    cap = nvec * d
    pos = np.zeros(max(cap, 1), np.int32)
    n = lib().orc_nuq_fit_positions(_P(xs, C.c_uint16), nvec, d, k, hadamard, _P(pos, C.c_int32), cap)
    return pos[:n]


def quantize_group(x, bits: int, hybrid: int):
    """InnerQ group quantizer on fp32 values -> (codes u8, min_h u16, scale_h u16)."""
    x = np.ascontiguousarray(x, np.float32).ravel()
    codes = np.zeros(x.size, np.uint8)
    mn, sc = C.c_uint16(), C.c_uint16()
    lib().orc_quantize_group(_P(x, C.c_float), x.size, 1, bits, hybrid, _P(codes, C.c_uint8), 1,
                             C.byref(mn), C.byref(sc))
    return codes, mn.value, sc.value


def key_norm(K) -> np.ndarray:
    """Per-channel key normalisation (powers of two) of fp16 K [T, d]."""
    K = _u16(K)
    T, d = K.shape
    out = np.zeros(d, np.float32)
    lib().orc_key_norm(_P(K, C.c_uint16), T, d, _P(out, C.c_float))
    return out


def quant_distortion(cfg: dict, K, V, bits: int):
    """(D_K, D_V): mean squared error of the cache's quantizers on one
    stream's calibration tokens K, V [T, d] at `bits`."""
    K, V = _u16(K), _u16(V)
    dk, dv = C.c_double(), C.c_double()
    c = _cfg(cfg)
    lib().orc_quant_distortion(C.byref(c), K.shape[0], _P(K, C.c_uint16), _P(V, C.c_uint16), bits,
                               C.byref(dk), C.byref(dv))
    return dk.value, dv.value


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, np.float64)


def fit_rd(bits, D):
    """(alpha, beta) of D(b) = alpha beta^-b, least squares in ln D."""
    b, D = _f64(bits), _f64(D)
    a, be = C.c_double(), C.c_double()
    lib().orc_fit_rd(b.size, _P(b, C.c_double), _P(D, C.c_double), C.byref(a), C.byref(be))
    return a.value, be.value


def rate_waterfill(alpha, beta, B: float, w=None):
    alpha, beta, w = _f64(alpha), _f64(beta), _f64(w)
    out = np.zeros(alpha.size)
    lib().orc_rate_waterfill(alpha.size, _P(alpha, C.c_double), _P(beta, C.c_double),
                             _P(w, C.c_double) if w is not None else None, float(B), _P(out, C.c_double))
    return out


def rate_greedy(alpha, beta, total: int, w=None):
    """Greedy bits in {2, 4, 8} per component under a total budget; (bits, used)."""
    alpha, beta, w = _f64(alpha), _f64(beta), _f64(w)
    out = np.zeros(alpha.size, np.int32)
    used = lib().orc_rate_greedy(alpha.size, _P(alpha, C.c_double), _P(beta, C.c_double),
                                 _P(w, C.c_double) if w is not None else None, int(total), _P(out, C.c_int32))
    return out, used

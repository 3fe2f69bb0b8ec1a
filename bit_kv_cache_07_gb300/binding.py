"""Thin ctypes binding of libkvq's C ABI (include/kvq.h).

Argument marshalling only: every step of the method runs in the CUDA
kernels of libkvq.so.  There is no fallback: if the library is missing the
import of any entry point raises.

Tensors are torch CUDA tensors (or raw device addresses as ints); the
binding checks device, dtype, contiguity and size before calling so that a
wrong pointer becomes a Python exception rather than a GPU fault.
"""
from __future__ import annotations

import ctypes as C
import os

from . import build as _build

KVQ_OK = 0
STATUS = {0: "KVQ_OK", -1: "KVQ_ERR_INVALID_ARG", -2: "KVQ_ERR_UNSUPPORTED",
          -3: "KVQ_ERR_CAPACITY", -4: "KVQ_ERR_WORKSPACE", -5: "KVQ_ERR_CUDA"}


class KvqError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS.get(status, status)} ({kvq_status_string(status)})")


class kvq_config(C.Structure):
    _fields_ = [
        ("batch", C.c_int32), ("n_q_heads", C.c_int32), ("n_kv_heads", C.c_int32),
        ("head_dim", C.c_int32), ("max_tokens", C.c_int32), ("k_bits", C.c_int32),
        ("v_bits", C.c_int32), ("k_group_tokens", C.c_int32), ("v_group_channels", C.c_int32),
        ("n_sink", C.c_int32), ("n_recent", C.c_int32), ("v_hadamard", C.c_int32),
        ("k_pre_rope", C.c_int32), ("rope_theta", C.c_float), ("outliers_per_vector", C.c_int32),
        ("k_lut", C.c_float * 8), ("v_lut", C.c_float * 8), ("softmax_scale", C.c_float),
        ("split_tokens", C.c_int32), ("position_offset", C.c_int32),
        ("k_group_channels", C.c_int32), ("hybrid_groups", C.c_int32), ("k_channel_norm", C.c_int32),
        ("kv_heads_total", C.c_int32), ("kv_head_index", C.c_void_p), ("sm_budget", C.c_int32),
    ]


class kvq_region(C.Structure):
    _fields_ = [("offset", C.c_uint64), ("bytes", C.c_uint64)]


_REGIONS_HEAD = ["k_codes", "k_scales", "v_codes", "v_scales", "k_sink", "v_sink", "k_ring", "v_ring",
                 "k_csr_rowptr", "k_csr_col", "k_csr_val", "v_csr_rowptr", "v_csr_col", "v_csr_val"]
REGIONS = _REGIONS_HEAD + ["k_norm", "rows"]


class kvq_layout(C.Structure):
    _fields_ = [(n, kvq_region) for n in _REGIONS_HEAD] + [
        ("layer_bytes", C.c_uint64), ("workspace_bytes", C.c_uint64), ("max_splits", C.c_int32),
        ("ring_slots", C.c_int32), ("q_cap", C.c_int32), ("k_norm", kvq_region), ("rows", kvq_region)]


EXPORTS = ["kvq_layout_query", "kvq_append", "kvq_decode_attn", "kvq_decode_plan",
           "kvq_decode_path", "kvq_status_string", "kvq_decode_attn_noalloc", "kvq_context_shard",
           "kvq_merge_attn", "kvq_fit_nuq_lut", "kvq_measure_distortion", "kvq_rate_allocate",
           "kvq_append_ragged", "kvq_decode_attn_ragged"]
NUQ_FIT_WORKSPACE_BYTES = 3 * 65538 * 8

_lib = None


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded libkvq.so.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it first (python -m bit_kv_cache_07_gb300.build)")
        L = C.CDLL(path)
        vp, u16p = C.c_void_p, C.c_void_p
        L.kvq_layout_query.argtypes = [C.POINTER(kvq_config), C.POINTER(kvq_layout)]
        L.kvq_layout_query.restype = C.c_int
        L.kvq_append.argtypes = [C.POINTER(kvq_config), vp, C.c_int32, u16p, u16p, C.c_int32, vp]
        L.kvq_append.restype = C.c_int
        L.kvq_decode_attn.argtypes = [C.POINTER(kvq_config), vp, C.c_int32, u16p, u16p, vp, vp,
                                      C.c_uint64, vp]
        L.kvq_decode_attn.restype = C.c_int
        L.kvq_decode_plan.argtypes = [C.POINTER(kvq_config), C.c_int32, C.POINTER(C.c_int32),
                                      C.POINTER(C.c_int32)]
        L.kvq_decode_plan.restype = C.c_int
        L.kvq_decode_path.argtypes = [C.POINTER(kvq_config), C.c_int32, C.POINTER(C.c_int32),
                                      C.POINTER(C.c_int32)]
        L.kvq_decode_path.restype = C.c_int
        L.kvq_context_shard.argtypes = [C.POINTER(kvq_config), C.c_int32, C.c_int32, C.c_int32,
                                        C.POINTER(kvq_config), C.POINTER(C.c_int32), C.POINTER(C.c_int32)]
        L.kvq_context_shard.restype = C.c_int
        L.kvq_merge_attn.argtypes = [C.c_int32, C.c_int64, C.c_int32, vp, vp, vp, vp, vp]
        L.kvq_merge_attn.restype = C.c_int
        L.kvq_fit_nuq_lut.argtypes = [vp, C.c_int64, C.c_int32, C.c_int32, C.c_int32, C.c_int32, vp, C.c_uint64,
                                      vp, vp, vp]
        L.kvq_fit_nuq_lut.restype = C.c_int
        L.kvq_measure_distortion.argtypes = [C.POINTER(kvq_config), vp, vp, C.c_int32, C.c_int32, vp, C.c_uint64,
                                             vp, vp]
        L.kvq_measure_distortion.restype = C.c_int
        f64p = C.POINTER(C.c_double)
        L.kvq_rate_allocate.argtypes = [C.c_int32, f64p, f64p, C.c_int32, C.POINTER(C.c_int32), f64p, f64p, f64p]
        L.kvq_rate_allocate.restype = C.c_int
        L.kvq_decode_attn_noalloc.argtypes = [C.POINTER(kvq_config), vp, C.c_int32, u16p, u16p, vp, vp]
        L.kvq_decode_attn_noalloc.restype = C.c_int
        i32p = C.POINTER(C.c_int32)
        L.kvq_append_ragged.argtypes = [C.POINTER(kvq_config), vp, i32p, i32p, u16p, u16p, C.c_int32, vp]
        L.kvq_append_ragged.restype = C.c_int
        L.kvq_decode_attn_ragged.argtypes = [C.POINTER(kvq_config), vp, i32p, u16p, u16p, vp, vp, C.c_uint64, vp]
        L.kvq_decode_attn_ragged.restype = C.c_int
        L.kvq_status_string.argtypes = [C.c_int]
        L.kvq_status_string.restype = C.c_char_p
        _lib = L
    return _lib


def kvq_status_string(status: int) -> str:
    return lib().kvq_status_string(int(status)).decode()


def make_config(d: dict) -> kvq_config:
    """kvq_config from a dict with the same field names (missing -> 0).  A
    kv_head_index given as a list of ints becomes a host array kept alive by
    the returned struct."""
    c = kvq_config()
    for name, ctype in kvq_config._fields_:
        if name in ("k_lut", "v_lut"):
            for i, v in enumerate(d.get(name, [0.0] * 8)):
                getattr(c, name)[i] = float(v)
        elif name == "kv_head_index":
            idx = d.get(name)
            if isinstance(idx, (list, tuple)):
                arr = (C.c_int32 * len(idx))(*[int(v) for v in idx])
                c._kv_head_index_keep = arr
                c.kv_head_index = C.cast(arr, C.c_void_p)
            elif idx:
                c.kv_head_index = int(idx)
        elif name in d:
            setattr(c, name, float(d[name]) if ctype is C.c_float else int(d[name]))
    return c


def _totals(c: kvq_config):
    """(KV heads, query heads) of the whole layer the cache belongs to."""
    hkv = c.kv_heads_total or c.n_kv_heads
    return hkv, hkv * (c.n_q_heads // c.n_kv_heads)


def _cfg(cfg) -> kvq_config:
    return cfg if isinstance(cfg, kvq_config) else make_config(cfg)


def _check(fn: str, st: int):
    if st != KVQ_OK:
        raise KvqError(fn, st)


def kvq_layout_query(cfg) -> kvq_layout:
    out = kvq_layout()
    _check("kvq_layout_query", lib().kvq_layout_query(C.byref(_cfg(cfg)), C.byref(out)))
    return out


def kvq_decode_plan(cfg, tokens: int):
    a, b = C.c_int32(), C.c_int32()
    _check("kvq_decode_plan", lib().kvq_decode_plan(C.byref(_cfg(cfg)), int(tokens), C.byref(a), C.byref(b)))
    return a.value, b.value


def kvq_decode_path(cfg, tokens: int):
    """(persistent, gq_slots): whether the decode of `tokens` runs the persistent
    tensor-core kernel (else the split-K kernel), and its head-slot count."""
    a, b = C.c_int32(), C.c_int32()
    _check("kvq_decode_path", lib().kvq_decode_path(C.byref(_cfg(cfg)), int(tokens), C.byref(a), C.byref(b)))
    return bool(a.value), b.value


def decode_kernel_name(cfg, tokens: int) -> str:
    """Name of the kernel instantiation a decode launches (as ncu lists it)."""
    c = _cfg(cfg)
    persistent, gt = kvq_decode_path(c, tokens)
    if persistent:
        nt = 1 if gt <= 4 else 2
        return f"decode_persist_kernel<{c.k_bits}, {c.v_bits}, {nt}, {gt}>"
    return f"decode_kernel<{c.k_bits}, {c.v_bits}, {gt}>"


def _ptr(t, what: str, dtype=None, numel: int | None = None, allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{what} is required")
    if isinstance(t, int):
        return t
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{what}: expected a torch tensor or a device address")
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{what} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() * t.element_size() < numel:
        raise ValueError(f"{what} too small: {t.numel() * t.element_size()} < {numel} bytes")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def kvq_append(cfg, layer_buf, tokens_before: int, k_new, v_new, n_new: int, stream=None):
    import torch
    c = _cfg(cfg)
    lay = kvq_layout_query(c)
    row = c.batch * _totals(c)[0] * int(n_new) * c.head_dim * 2
    st = lib().kvq_append(C.byref(c), _ptr(layer_buf, "layer_buf", numel=lay.layer_bytes), int(tokens_before),
                          _ptr(k_new, "k_new", torch.float16, row), _ptr(v_new, "v_new", torch.float16, row),
                          int(n_new), _stream(stream))
    _check("kvq_append", st)


def kvq_decode_attn(cfg, layer_buf, tokens: int, q, out, lse=None, workspace=None, ws_bytes=None,
                    stream=None):
    import torch
    c = _cfg(cfg)
    lay = kvq_layout_query(c)
    hq = _totals(c)[1]
    nq = c.batch * hq * c.head_dim * 2
    if ws_bytes is None:
        ws_bytes = 0 if workspace is None else (
            workspace if isinstance(workspace, int) else workspace.numel() * workspace.element_size())
        if isinstance(workspace, int):
            raise ValueError("ws_bytes is required with a raw workspace address")
    st = lib().kvq_decode_attn(
        C.byref(c), _ptr(layer_buf, "layer_buf", numel=lay.layer_bytes), int(tokens),
        _ptr(q, "q", torch.float16, nq), _ptr(out, "out", torch.float16, nq),
        _ptr(lse, "lse", torch.float32, c.batch * hq * 4, allow_none=True),
        _ptr(workspace, "workspace", allow_none=True), int(ws_bytes), _stream(stream))
    _check("kvq_decode_attn", st)


def _rows(values, batch: int, what: str):
    """A host int32 array of one value per batch row."""
    vals = [int(v) for v in values]
    if len(vals) != batch:
        raise ValueError(f"{what}: one value per batch row ({batch}), got {len(vals)}")
    return (C.c_int32 * batch)(*vals)


def kvq_append_ragged(cfg, layer_buf, tokens_before, n_new, k_new, v_new, stream=None):
    """Row b appends n_new[b] tokens (the first of its k_new / v_new rows,
    [B, Hkv, n_stride, d]) after tokens_before[b]."""
    import torch
    c = _cfg(cfg)
    lay = kvq_layout_query(c)
    n_stride = int(k_new.shape[2])
    row = c.batch * _totals(c)[0] * n_stride * c.head_dim * 2
    st = lib().kvq_append_ragged(C.byref(c), _ptr(layer_buf, "layer_buf", numel=lay.layer_bytes),
                                 _rows(tokens_before, c.batch, "tokens_before"), _rows(n_new, c.batch, "n_new"),
                                 _ptr(k_new, "k_new", torch.float16, row), _ptr(v_new, "v_new", torch.float16, row),
                                 n_stride, _stream(stream))
    _check("kvq_append_ragged", st)


def kvq_decode_attn_ragged(cfg, layer_buf, tokens, q, out, lse=None, workspace=None, ws_bytes=None, stream=None):
    """Attention of batch row b over its own tokens[b] tokens."""
    import torch
    c = _cfg(cfg)
    lay = kvq_layout_query(c)
    hq = _totals(c)[1]
    nq = c.batch * hq * c.head_dim * 2
    if ws_bytes is None:
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().kvq_decode_attn_ragged(
        C.byref(c), _ptr(layer_buf, "layer_buf", numel=lay.layer_bytes), _rows(tokens, c.batch, "tokens"),
        _ptr(q, "q", torch.float16, nq), _ptr(out, "out", torch.float16, nq),
        _ptr(lse, "lse", torch.float32, c.batch * hq * 4, allow_none=True),
        _ptr(workspace, "workspace", allow_none=True), int(ws_bytes), _stream(stream))
    _check("kvq_decode_attn_ragged", st)


def kvq_decode_attn_noalloc(cfg, layer_buf, tokens: int, q, out, lse=None, stream=None):
    """kvq_decode_attn for callers that cannot allocate: the split-K scratch
    is the library's own fixed 8 MiB device array (see include/kvq.h)."""
    import torch
    c = _cfg(cfg)
    lay = kvq_layout_query(c)
    hq = _totals(c)[1]
    nq = c.batch * hq * c.head_dim * 2
    st = lib().kvq_decode_attn_noalloc(
        C.byref(c), _ptr(layer_buf, "layer_buf", numel=lay.layer_bytes), int(tokens),
        _ptr(q, "q", torch.float16, nq), _ptr(out, "out", torch.float16, nq),
        _ptr(lse, "lse", torch.float32, c.batch * hq * 4, allow_none=True), _stream(stream))
    _check("kvq_decode_attn_noalloc", st)


def config_dict(c: kvq_config) -> dict:
    """The fields of a kvq_config as a dict (the inverse of make_config)."""
    d = {}
    for name, _ in kvq_config._fields_:
        v = getattr(c, name)
        d[name] = [float(x) for x in v] if name in ("k_lut", "v_lut") else v
    return d


def kvq_context_shard(cfg, tokens: int, n_shards: int, shard: int):
    """(shard config dict, first token, tokens) of one shard of a context of
    `tokens` tokens cut into n_shards (host only; see include/kvq.h)."""
    out = kvq_config()
    a, n = C.c_int32(), C.c_int32()
    _check("kvq_context_shard", lib().kvq_context_shard(C.byref(_cfg(cfg)), int(tokens), int(n_shards), int(shard),
                                                        C.byref(out), C.byref(a), C.byref(n)))
    return config_dict(out), a.value, n.value


def kvq_fit_nuq_lut(x, outliers: int, hadamard: int = 0, max_iters: int = 100, workspace=None, stream=None):
    """Fit a non-uniform level table to the vectors x [..., 128] (fp16, on
    the GPU).  Returns (lut as a list of 8 floats, updates made or -1); the
    call synchronises `stream` to read the result."""
    import torch
    d = x.shape[-1]
    n = x.numel() // d
    if workspace is None:
        workspace = torch.empty(NUQ_FIT_WORKSPACE_BYTES, dtype=torch.uint8, device=x.device)
    lut = torch.empty(8, dtype=torch.float32, device=x.device)
    info = torch.empty(1, dtype=torch.int32, device=x.device)
    st = lib().kvq_fit_nuq_lut(_ptr(x, "x", torch.float16, n * d * 2), n, d, int(outliers), int(hadamard),
                               int(max_iters), _ptr(workspace, "workspace", numel=NUQ_FIT_WORKSPACE_BYTES),
                               NUQ_FIT_WORKSPACE_BYTES, lut.data_ptr(), info.data_ptr(), _stream(stream))
    _check("kvq_fit_nuq_lut", st)
    if stream is not None and not isinstance(stream, int):
        stream.synchronize()
    else:
        torch.cuda.synchronize(x.device)
    return [float(v) for v in lut.cpu()], int(info.item())


def kvq_measure_distortion(cfg, k, v, bits: int, stream=None):
    """{D_K, D_V} per layer KV head ([Hkv_total, 2] float64 tensor on the GPU)
    of this cache's quantizers at `bits` on calibration tokens k, v
    [B, Hkv_total, n, 128] fp16."""
    import torch
    c = _cfg(cfg)
    hkv = _totals(c)[0]
    n = k.shape[2]
    ws = torch.empty(max(16, c.batch * c.n_kv_heads * 128 * 4), dtype=torch.uint8, device=k.device)
    out = torch.empty((hkv, 2), dtype=torch.float64, device=k.device)
    nb = c.batch * hkv * n * 256
    st = lib().kvq_measure_distortion(C.byref(c), _ptr(k, "k", torch.float16, nb), _ptr(v, "v", torch.float16, nb),
                                      int(n), int(bits), ws.data_ptr(), ws.numel(), out.data_ptr(), _stream(stream))
    _check("kvq_measure_distortion", st)
    return out


def kvq_rate_allocate(distortion, total_bits: int, weights=None):
    """Greedy per-component bits (2/4/8) from distortions [n, 3] at 2, 4, 8
    bits; returns (bits, alpha, beta, continuous water-filling bits)."""
    import numpy as np
    D = np.ascontiguousarray(distortion, np.float64)
    n = D.shape[0]
    w = None if weights is None else np.ascontiguousarray(weights, np.float64)
    bits = np.zeros(n, np.int32)
    a, b, wf = np.zeros(n), np.zeros(n), np.zeros(n)
    f64p = C.POINTER(C.c_double)
    st = lib().kvq_rate_allocate(n, D.ctypes.data_as(f64p), None if w is None else w.ctypes.data_as(f64p),
                                 int(total_bits), bits.ctypes.data_as(C.POINTER(C.c_int32)), a.ctypes.data_as(f64p),
                                 b.ctypes.data_as(f64p), wf.ctypes.data_as(f64p))
    _check("kvq_rate_allocate", st)
    return bits, a, b, wf


def kvq_merge_attn(outs, lses, out, lse_out=None, stream=None):
    """Merge n parts' outputs [n, rows.., 128] fp16 and lse [n, rows..] f32
    into out [rows.., 128] fp16 (and lse_out), by log-sum-exp."""
    import torch
    n = outs.shape[0]
    rows = outs[0].numel() // outs.shape[-1]
    if lses.shape[0] != n or lses[0].numel() != rows:
        raise ValueError("lses must be [n_parts, rows]")
    st = lib().kvq_merge_attn(
        n, rows, int(outs.shape[-1]), _ptr(outs, "outs", torch.float16, n * rows * 256),
        _ptr(lses, "lses", torch.float32, n * rows * 4), _ptr(out, "out", torch.float16, rows * 256),
        _ptr(lse_out, "lse_out", torch.float32, rows * 4, allow_none=True), _stream(stream))
    _check("kvq_merge_attn", st)


# ------------------------------------------------------------ conveniences

class Layer:
    """One layer's cache: a zeroed device buffer of layer_bytes plus its
    config.  ``append`` / ``decode`` call the C ABI."""

    def __init__(self, cfg: dict, device="cuda"):
        import torch
        self.cfg_dict = dict(cfg)
        self.cfg = make_config(cfg)
        self.layout = kvq_layout_query(self.cfg)
        self.buf = torch.zeros(self.layout.layer_bytes, dtype=torch.uint8, device=device)

    def region(self, name: str):
        r = getattr(self.layout, name)
        return self.buf[r.offset:r.offset + r.bytes]

    def append(self, tokens_before: int, k_new, v_new, stream=None):
        kvq_append(self.cfg, self.buf, tokens_before, k_new, v_new, k_new.shape[2], stream)

    def decode(self, tokens: int, q, out, lse=None, workspace=None, stream=None):
        kvq_decode_attn(self.cfg, self.buf, tokens, q, out, lse, workspace, None, stream)

    def append_ragged(self, tokens_before, n_new, k_new, v_new, stream=None):
        kvq_append_ragged(self.cfg, self.buf, tokens_before, n_new, k_new, v_new, stream)

    def decode_ragged(self, tokens, q, out, lse=None, workspace=None, stream=None):
        kvq_decode_attn_ragged(self.cfg, self.buf, tokens, q, out, lse, workspace, None, stream)


def new_workspace(cfg, device="cuda"):
    """A zeroed decode workspace of layout.workspace_bytes (counters at zero)."""
    import torch
    lay = kvq_layout_query(_cfg(cfg))
    return torch.zeros(max(int(lay.workspace_bytes), 16), dtype=torch.uint8, device=device)

"""Decode-attention benchmark of libkvq on one GB300 (or N replicas).

One step = one decode step of the whole model: for every layer, append the
new token's K/V (kvq_append) and attend over the cache (kvq_decode_attn).
Default workload: Llama-3-8B-shaped GQA decode, 32 layers x 32 query heads /
8 KV heads, head dim 128, batch 16, context 32768, with a per-layer (K, V)
bit pair drawn by seed from KV8, K8V4, KV4, K4V2, KV2 (layers 0, 1 and 31
KV8); K per channel over 32-token groups, V per token over 64-channel
groups, 4 sink + 128 recent fp16 tokens.  The same step on a plain fp16
cache is timed beside it.

The step time is the median of several timed rounds of exactly --steps
CUDA-graph replays (the rounds repeat until at least 1.5 s has been timed,
so that the clock sampler sees the timed region).  Each layer's decode
kernel time comes from decode-only CUDA graphs (one per (K, V) pair, its
layers' decode launches back to back, replayed between two events); the
roofline fraction comes from those in-graph durations.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle
instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import signal
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "llama3_8b_mixed_t32k"
HBM_NOMINAL_GBS = 8000.0  # the 8 TB/s HBM figure the metric names
METRIC = "decode-attention µs/step and effective cache GB/s (fraction of 8 TB/s HBM) at 1 GB300"
UNIT = "us/step"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--min-timed-seconds", type=float, default=1.5,
                    help="repeat rounds of exactly --steps graph replays until this much was timed")
    ap.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-fp16-baseline", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling only: build just the first N layers (the bench line needs all)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="profiling only: a shorter context than the workload's")
    return ap.parse_args()


# ------------------------------------------------------------------ bytes

def window_counts(cfg: dict, T: int):
    """(sinks present, quantized tokens, fp16 window tokens) at T tokens: the
    cache's window rule (sinks [0,S), Nq = 32*floor((T-S-R)/32) quantized
    tokens, the rest fp16; an fp16 cache quantizes nothing)."""
    if cfg["k_bits"] == 16:
        return 0, 0, T
    S, R = cfg["n_sink"], cfg["n_recent"]
    rest = T - S - R
    nq = 32 * (rest // 32) if rest > 0 else 0
    s = min(S, T)
    return s, nq, T - s - nq


def algorithmic_bytes(cfg: dict, T: int, rows=None) -> int:
    """Bytes one decode launch must move: packed codes, scales, CSR outlier
    entries and fp16 sink/window tokens of every stream (each read once per
    KV head), plus q in and out.  With per-row lengths `rows` (a ragged
    batch) every row's streams count at their own length."""
    if rows is not None:
        one = dict(cfg, batch=1)
        qo1 = cfg["n_q_heads"] * cfg["head_dim"] * 2 * 2
        return sum(algorithmic_bytes(one, t) - qo1 for t in rows) + cfg["batch"] * qo1
    S, Nq, W = window_counts(cfg, T)
    d = cfg["head_dim"]
    NS = cfg["batch"] * cfg["n_kv_heads"]
    kb, vb = cfg["k_bits"], cfg["v_bits"]
    per = 0
    if kb != 16:
        per += Nq * (d * kb // 8 + d * vb // 8)
        if kb == 3:
            # per-token {min, s} for K and V, and k CSR entries (1-byte column + fp16 value)
            # per token vector; every row holds exactly k entries, so the decode does not
            # need the row pointers
            k = cfg["outliers_per_vector"]
            per += Nq * 4 * 2 + 2 * (Nq * k * 3)
        else:
            gkc = cfg.get("k_group_channels", 0)
            if gkc:  # InnerQ keys: {scale, min} per token and 64-channel group
                per += Nq * (d // gkc) * 4
            else:  # per-channel keys: {scale, min} per channel and 32-token group
                per += (Nq // 32) * d * 4
            per += Nq * (d // cfg["v_group_channels"]) * 4
        if cfg.get("k_channel_norm", 0):
            per += d * 4  # the stream's per-channel key normalisation (fp32)
    per += (S + W) * d * 2 * 2
    qo = cfg["batch"] * cfg["n_q_heads"] * d * 2 * 2
    return NS * per + qo


# ----------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"kvq_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.send_signal(signal.SIGTERM)
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = [r.split(",") for r in open(self.path).read().strip().splitlines() if r.count(",") >= 8]
        os.unlink(self.path)
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if "Active" in r[5 + i]
                          and "Not" not in r[5 + i]})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "samples": len(rows), "reasons": reasons}


# ------------------------------------------------------------------- peaks

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def ncu_traffic(tag: str):
    """DRAM bytes per decode launch (dram__bytes_read.sum + dram__bytes_write.sum)
    from the committed ncu record for `tag` (decode:<workload>:<pair>), if it
    was taken on the current decode kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.txt")
    if not os.path.exists(path):
        return None
    h = source_hash()
    for line in open(path):
        m = re.match(r"\s*(\S+)\s+src=(\w+)\s+traffic_per_launch=(\d+)", line)
        if m and m.group(1) == tag and m.group(2) == h:
            return int(m.group(3))
    return None


def source_hash() -> str:
    hs = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_kv_cache_07_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.startswith("kvq_decode"):
            hs.update(open(os.path.join(csrc, f), "rb").read())
    return hs.hexdigest()[:12]


# --------------------------------------------------------------- the model

class Model:
    """All layers of one workload: caches filled to T-1 tokens, plus the
    per-layer inputs of one decode step.  A layer is one or more decode
    units: one cache per layer, or with per-head (K, V) bits one cache per
    distinct pair over its KV heads (their head maps address the layer's
    whole K/V, q and out)."""

    def __init__(self, name: str, device, fp16: bool, layers: int = 0, tokens: int = 0):
        import torch
        from bit_kv_cache_07_gb300 import binding, mixed, synth, workloads
        w = workloads.WORKLOADS[name]
        self.name, self.T = name, (tokens if tokens > 0 else w["tokens"])
        self.rows = workloads.row_tokens(name, self.T)  # per batch row lengths (ragged), or None
        self.L = layers if layers > 0 else w["layers"]
        self.cfgs, self.units, self.unit_layer = [], [], []
        self.q, self.k_new, self.v_new, self.out = [], [], [], []
        self.head_pairs, self.mixed = [], [None] * self.L
        for l in range(self.L):
            cfg = workloads.layer_config(name, l, tokens=self.T)
            if cfg["k_bits"] == 3:
                from bit_kv_cache_07_gb300 import calibrate
                cfg["k_lut"], cfg["v_lut"] = calibrate.nuq_tables(name, l, device=device)
            if fp16:
                cfg = workloads.fp16_baseline_config(cfg)
            K, V = synth.layer_kv(name, l, tokens=self.T - 1, device=device)
            if w["pairs"] == "rateq" and not fp16:
                Kc, Vc = synth.layer_kv(name, l, tokens=w["rateq_calib_tokens"], batch=1, device=device)
                pairs, _ = mixed.allocate_pairs(cfg, Kc, Vc, w["rateq_avg_bits"])
                del Kc, Vc
                ml = mixed.MixedLayer(cfg, pairs, device=device)
                ml.append(0, K, V)
                self.head_pairs.append(pairs)
                self.mixed[l] = ml
                parts = [sub for _, _, sub in ml.parts]
            else:
                layer = binding.Layer(cfg, device=device)
                if self.rows is not None:
                    layer.append_ragged([0] * cfg["batch"], [t - 1 for t in self.rows], K, V)
                else:
                    layer.append(0, K, V)
                parts = [layer]
            del K, V
            for sub in parts:
                self.cfgs.append(sub.cfg_dict)
                self.units.append(sub)
                self.unit_layer.append(l)
            self.q.append(synth.query(name, l, device=device))
            k, v = synth.new_token_kv(name, l, 0, device=device)
            self.k_new.append(k)
            self.v_new.append(v)
            self.out.append(torch.empty_like(self.q[-1]))
        # a step's inputs (every layer's q and new K/V) and outputs (every
        # layer's attention) each in one contiguous buffer, the per-layer
        # tensors views into it: a step moves them with one copy each way
        self.inputs = self._gather(self.q + self.k_new + self.v_new)
        self.outputs = self._gather(self.out)
        self.q = self._views(self.inputs, self.q)
        self.k_new = self._views(self.inputs[sum(t.numel() for t in self.q):], self.k_new)
        self.v_new = self._views(self.inputs[sum(t.numel() for t in self.q + self.k_new):], self.v_new)
        self.out = self._views(self.outputs, self.out)
        ws_bytes = max(u.layout.workspace_bytes for u in self.units)
        self.ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=device)
        torch.cuda.synchronize()
        self.binding = binding

    @staticmethod
    def _gather(ts):
        import torch
        return torch.cat([t.reshape(-1) for t in ts])

    @staticmethod
    def _views(flat, ts):
        out, o = [], 0
        for t in ts:
            out.append(flat[o:o + t.numel()].view(t.shape))
            o += t.numel()
        return out

    def step(self, stream):
        B = self.binding
        for i, u in enumerate(self.units):
            l = self.unit_layer[i]
            if self.rows is not None:
                B.kvq_append_ragged(u.cfg, u.buf, [t - 1 for t in self.rows], [1] * len(self.rows),
                                    self.k_new[l], self.v_new[l], stream)
            else:
                B.kvq_append(u.cfg, u.buf, self.T - 1, self.k_new[l], self.v_new[l], 1, stream)
        for l in range(self.L):
            self.decode_layer(l, stream)

    def decode(self, i: int, stream):
        u, l = self.units[i], self.unit_layer[i]
        if self.rows is not None:
            self.binding.kvq_decode_attn_ragged(u.cfg, u.buf, self.rows, self.q[l], self.out[l], None, self.ws,
                                                None, stream)
            return
        self.binding.kvq_decode_attn(u.cfg, u.buf, self.T, self.q[l], self.out[l], None, self.ws, None, stream)

    def unit_bytes(self, i: int) -> int:
        return algorithmic_bytes(self.cfgs[i], self.T, self.rows)

    def decode_layer(self, l: int, stream):
        if self.mixed[l] is not None:  # its pairs' caches side by side (fork / join on side streams)
            self.mixed[l].decode(self.T, self.q[l], self.out[l], None, None, stream)
            return
        for i, ul in enumerate(self.unit_layer):
            if ul == l:
                self.decode(i, stream)

    def decode_bytes(self):
        return sum(self.unit_bytes(i) for i in range(len(self.cfgs)))

    def launches_per_step(self):
        """Kernel launches of one step: per decode unit the 1-token append's
        window copy (plus a quantize launch when the append flushes a group)
        and the decode."""
        n = 0
        for c in self.cfgs:
            n += 1  # fp16 window copy of the appended token
            if any(window_counts(c, t)[1] > window_counts(c, t - 1)[1] for t in (self.rows or [self.T])):
                n += 1  # the append flushes one 32-token group (of some row)
            n += 1  # decode
        return n

    def kernel_names(self):
        return [self.binding.decode_kernel_name(c, self.T) for c in self.cfgs]


def time_steps(model, stream, steps: int, warmup: int):
    """Eager steps (host launches every call) timed with CUDA events: ms total."""
    import torch
    for _ in range(warmup):
        model.step(stream)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(steps):
        model.step(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    return t0.elapsed_time(t1)


def time_graph(model, stream, steps: int, warmup: int, min_seconds: float = 1.5, max_rounds: int = 200):
    """One step (every layer's append + decode) captured once in a CUDA graph
    and replayed: the per-step time without host launch gaps.  Rounds of
    exactly `steps` replays are timed back to back (CUDA events on the
    launching stream, one pair per round) until at least `min_seconds` of
    GPU time has been timed; returns (median ms per step over the rounds,
    rounds, None) or (None, 0, why) if the capture is not possible."""
    import torch
    try:
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
            model.step(stream)
        torch.cuda.synchronize()
    except Exception as e:  # pragma: no cover - reported in the JSON line
        return None, 0, f"graph capture failed: {type(e).__name__}: {e}"
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
    torch.cuda.synchronize()
    # size the rounds from one untimed probe round
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        p0.record(stream)
        for _ in range(steps):
            g.replay()
        p1.record(stream)
    torch.cuda.synchronize()
    round_s = max(p0.elapsed_time(p1) * 1e-3, 1e-6)
    rounds = max(1, min(max_rounds, int(min_seconds / round_s + 0.999)))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(rounds)]
    barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for e0, e1 in evs:
            e0.record(stream)
            for _ in range(steps):
                g.replay()
            e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    per_round = [e0.elapsed_time(e1) / steps for e0, e1 in evs]
    del g
    return statistics.median(per_round), rounds, None


def time_decode_only(model, stream, steps: int, warmup: int):
    """Each decode unit's kernel time, measured inside replayed CUDA graphs:
    for every (K, V) pair, the decode launches of that pair's units are
    captured back to back in one graph (no appends, nothing between them), the
    graph is replayed `steps` times between two CUDA events on the launching
    stream, and the time is divided by the launches.  Every unit gets the
    mean of its pair.  Returns (per-unit ms, None) or (None, why)."""
    import torch
    if any(m is not None for m in model.mixed):
        return _time_mixed_layers(model, stream, steps, warmup)
    groups = {}
    for l, c in enumerate(model.cfgs):
        groups.setdefault(_pair_name(c), []).append(l)
    per_layer = [0.0] * len(model.cfgs)
    for pair, layers in groups.items():
        try:
            g = torch.cuda.CUDAGraph()
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
                for l in layers:
                    model.decode(l, stream)
            torch.cuda.synchronize()
        except Exception as e:  # pragma: no cover - reported in the JSON line
            return None, f"decode-only graph capture failed: {type(e).__name__}: {e}"
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(steps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / (steps * len(layers))
        for l in layers:
            per_layer[l] = ms
        del g
    return per_layer, None


def _time_mixed_layers(model, stream, steps: int, warmup: int):
    """Per-head pairs: every layer's decode (its pairs' caches side by side)
    captured back to back in one graph, replayed between two events; each
    layer's time is split over its decode units by their bytes."""
    import torch
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
        for l in range(model.L):
            model.decode_layer(l, stream)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    layer_ms = e0.elapsed_time(e1) / (steps * model.L)
    b = [model.unit_bytes(i) for i in range(len(model.cfgs))]
    lb = [0] * model.L
    for i, l in enumerate(model.unit_layer):
        lb[l] += b[i]
    del g
    return [layer_ms * b[i] / lb[model.unit_layer[i]] for i in range(len(b))], None


def time_append(name: str, dev, T: int, stream, reps: int = 20):
    """Append through the C ABI on layer 0 of the workload (reported beside the
    decode step): a bulk prefill of T - 1 tokens into an empty cache, a 1-token
    append that only copies the token into the fp16 window, and a 1-token
    append that also flushes (quantizes) one 32-token group.  The 1-token
    calls are captured reps at a time in a CUDA graph (no host time in the
    number); CUDA events on the launching stream."""
    import torch
    from bit_kv_cache_07_gb300 import binding, synth, workloads
    cfg = workloads.layer_config(name, 0, tokens=T)
    if cfg["k_bits"] == 3:
        from bit_kv_cache_07_gb300 import calibrate
        cfg["k_lut"], cfg["v_lut"] = calibrate.nuq_tables(name, 0, device=dev)
    layer = binding.Layer(cfg, device=dev)
    K, V = synth.layer_kv(name, 0, tokens=T - 1, device=dev)
    k1, v1 = synth.new_token_kv(name, 0, 0, device=dev)

    def events_us(fn, n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / n

    def prefill():
        binding.kvq_append(cfg, layer.buf, 0, K, V, T - 1, stream)

    for _ in range(2):
        prefill()
    pre_us = events_us(prefill, 3)

    def one_token_us(t):
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
            for _ in range(reps):
                binding.kvq_append(cfg, layer.buf, t, k1, v1, 1, stream)
        with torch.cuda.stream(stream):
            g.replay()
            us = events_us(g.replay, 3) / reps
        del g
        return us

    def nq(t):
        return window_counts(cfg, t)[1]
    t_copy = next((t for t in range(T - 2, 0, -1) if nq(t + 1) == nq(t)), None)
    t_flush = next((t for t in range(T - 2, 0, -1) if nq(t + 1) > nq(t)), None)
    copy_us = one_token_us(t_copy) if t_copy is not None else None
    flush_us = one_token_us(t_flush) if t_flush is not None else None
    d, NS = cfg["head_dim"], cfg["batch"] * cfg["n_kv_heads"]
    qo = cfg["batch"] * cfg["n_q_heads"] * d * 2 * 2
    pre_bytes = 2 * NS * (T - 1) * d * 2 + (algorithmic_bytes(cfg, T - 1) - qo)
    amort = None
    if copy_us is not None and flush_us is not None:
        amort = (31 * copy_us + flush_us) / 32
    del layer, K, V
    torch.cuda.empty_cache()
    return {
        "layer": 0, "prefill_tokens": T - 1, "prefill_us": pre_us,
        "prefill_bytes": pre_bytes, "prefill_gbs": pre_bytes / (pre_us * 1e-6) / 1e9,
        "token_us": copy_us, "flush_token_us": flush_us, "amortised_token_us": amort,
        "note": "prefill bytes = fp16 K/V read + packed codes, scales and fp16 sink/window written; "
                "1-token appends: one flush (a 32-token group quantized) every 32 tokens",
    }


def time_e2e(model, stream, steps: int, warmup: int):
    """Same step through the public API with this step's inputs copied in from
    pinned host memory and the outputs copied back, inside the timed region."""
    import torch
    h_in = model.inputs.cpu().pin_memory()  # every layer's q and new K/V of the step
    h_out = torch.empty(model.outputs.shape, dtype=model.outputs.dtype).pin_memory()
    h2d = h_in.numel() * h_in.element_size()
    d2h = h_out.numel() * h_out.element_size()

    def one():
        with torch.cuda.stream(stream):
            model.inputs.copy_(h_in, non_blocking=True)
            model.step(stream)
            h_out.copy_(model.outputs, non_blocking=True)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    t0.record(stream)
    for _ in range(steps):
        one()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    return t0.elapsed_time(t1) / steps, h2d, d2h


# --------------------------------------------------------- distributed bits

_DIST = {"on": False}


def init_dist(n: int):
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        _DIST["on"] = True
    return rank, ws, local


def barrier():
    if _DIST["on"]:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float) -> float:
    if not _DIST["on"]:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float) -> float:
    if not _DIST["on"]:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# -------------------------------------------------------------- CPU oracle

_ORACLE_STREAMS = {}


def _oracle_tables(name: str, layer: int):
    """The CPU-baseline leg's level tables: a fitted workload's tables are
    fitted by the oracle on CPU-drawn calibration tokens (nothing here comes
    from the CUDA path); otherwise the seeded quantile tables."""
    from bit_kv_cache_07_gb300 import synth, workloads
    from oracle import kvq_oracle as O
    w = workloads.WORKLOADS[name]
    if w.get("lut") != "fitted":
        return synth.nuq_lut(name, layer, "k"), synth.nuq_lut(name, layer, "v")
    K, V = synth.layer_kv(name, layer, tokens=w["lut_calib_tokens"], batch=1, device="cpu")
    k = w["outliers_per_vector"]
    return O.nuq_fit_lut(K.numpy(), k)[0], O.nuq_fit_lut(V.numpy(), k, w["v_hadamard"])[0]


def _oracle_streams(name: str):
    """Up to 4 prebuilt oracle streams of layer 0 of a workload at its full
    context, with their queries (built once per process; not timed)."""
    if name not in _ORACLE_STREAMS:
        from bit_kv_cache_07_gb300 import synth, workloads
        from oracle import kvq_oracle as O
        w = workloads.WORKLOADS[name]
        T = w["tokens"]
        cfg = workloads.layer_config(name, 0)
        if cfg["k_bits"] == 3:
            cfg["k_lut"], cfg["v_lut"] = _oracle_tables(name, 0)
        g = w["n_q_heads"] // w["n_kv_heads"]
        K, V = synth.layer_kv(name, 0, tokens=T, batch=1, device="cpu")
        q = synth.query(name, 0, batch=1, device="cpu").numpy()
        Kh, Vh = K.numpy(), V.numpy()
        nstore = min(4, w["n_kv_heads"])
        stores = [O.build_stream(cfg, Kh[0, h], Vh[0, h]) for h in range(nstore)]
        _ORACLE_STREAMS[name] = (cfg, T, g, q, stores)
    return _ORACLE_STREAMS[name]


def _ragged_scale(name: str):
    """(factor, note) turning a full-context stream decode into the mean row's
    of a ragged workload (the oracle's decode time grows linearly with T)."""
    from bit_kv_cache_07_gb300 import workloads
    rows = workloads.row_tokens(name)
    if rows is None:
        return 1.0, ""
    T = workloads.WORKLOADS[name]["tokens"]
    f = statistics.mean(rows) / T
    return f, f"; rows of different lengths: the full-context stream time scaled by their mean length / T = {f:.3f}"


def oracle_sample(name: str, seconds: float, layer_count: int | None = None):
    """Time the CPU oracle (single thread, as written) decoding whole streams of
    layer 0 at the workload's context until ~seconds have passed; scale the
    per-stream time to one full decode step (all streams of all layers)."""
    from bit_kv_cache_07_gb300 import workloads
    from oracle import kvq_oracle as O
    w = workloads.WORKLOADS[name]
    cfg, T, g, q, stores = _oracle_streams(name)
    nstore = len(stores)
    n, spent = 0, 0.0
    while spent < seconds or n < 3:
        h = n % nstore
        t0 = time.perf_counter()
        O.decode_stream(cfg, T, stores[h], q[0, h * g:(h + 1) * g])
        spent += time.perf_counter() - t0
        n += 1
    streams_per_step = w["layers"] * w["batch"] * w["n_kv_heads"]
    rf, rnote = _ragged_scale(name)
    per_stream = spent / n
    return {
        "streams": n, "seconds": spent,
        "value": per_stream * rf * streams_per_step * 1e6, "unit": UNIT, "cores": 1, "kind": "oracle",
        "sample": f"fp64 oracle decode of {n} (batch row, KV head) streams of layer 0 at T={T} "
                  f"(cycling over {nstore} prebuilt streams), "
                  f"{per_stream * 1e3:.1f} ms each, scaled x{streams_per_step / n:.0f} to one "
                  f"{w['layers']}-layer step; cache build not timed" + rnote,
    }


def _oracle_worker(name: str, head: int, seconds: float):
    """One process of the all-cores oracle timing: build one stream of layer
    0 (not timed), then decode it repeatedly for ~seconds."""
    from bit_kv_cache_07_gb300 import synth, workloads
    from oracle import kvq_oracle as O
    w = workloads.WORKLOADS[name]
    T = w["tokens"]
    cfg = workloads.layer_config(name, 0)
    if cfg["k_bits"] == 3:
        cfg["k_lut"], cfg["v_lut"] = _oracle_tables(name, 0)
    g = w["n_q_heads"] // w["n_kv_heads"]
    K, V = synth.layer_kv(name, 0, tokens=T, batch=1, device="cpu")
    q = synth.query(name, 0, batch=1, device="cpu").numpy()
    store = O.build_stream(cfg, K.numpy()[0, head], V.numpy()[0, head])
    del K, V
    n, spent = 0, 0.0
    while spent < seconds or n < 2:
        t0 = time.perf_counter()
        O.decode_stream(cfg, T, store, q[0, head * g:(head + 1) * g])
        spent += time.perf_counter() - t0
        n += 1
    return n, spent


def oracle_sample_all_cores(name: str, seconds: float, procs: int | None = None):
    """The same oracle, one process per independent stream on every host core
    (spawned workers, same code and results): streams decoded per second of
    wall time, scaled to one full decode step.  None when the workload's
    per-process inputs would not fit comfortably in host memory."""
    import multiprocessing as mp
    from concurrent.futures import ProcessPoolExecutor
    from bit_kv_cache_07_gb300 import workloads
    w = workloads.WORKLOADS[name]
    procs = procs or os.cpu_count() or 1
    per_proc = w["tokens"] * w["n_kv_heads"] * w["head_dim"] * 2 * 4  # K and V of one batch row, fp32 copies
    if per_proc * procs > 32 * 2 ** 30:
        return None
    heads = [i % w["n_kv_heads"] for i in range(procs)]
    try:
        with ProcessPoolExecutor(max_workers=procs, mp_context=mp.get_context("spawn")) as ex:
            res = list(ex.map(_oracle_worker, [name] * procs, heads, [seconds] * procs))
    except Exception as e:  # a worker that cannot start ends the pool instead of hanging it
        return {"unavailable": f"{type(e).__name__}: {e}"}
    n = sum(r[0] for r in res)
    wall = max(r[1] for r in res)
    streams_per_step = w["layers"] * w["batch"] * w["n_kv_heads"]
    rf, rnote = _ragged_scale(name)
    return {
        "value": wall / n * rf * streams_per_step * 1e6, "unit": UNIT, "cores": procs, "kind": "oracle",
        "sample": f"{procs} spawned processes, each decoding one prebuilt stream of layer 0 at "
                  f"T={w['tokens']} for ~{seconds:.0f} s: {n} streams in {wall:.1f} s of wall time, "
                  f"scaled to one {w['layers']}-layer step; cache build not timed" + rnote,
    }


def run_reference(args):
    """The reference arm: the CPU oracle as written (one host core, fp64),
    on the same workload.  Each of the warmup + steps "steps" times whole
    single-stream decodes of layer 0 for a bounded wall-clock budget and
    scales them to one full model step (every stream of every layer); the
    line states how many stream decodes were timed and the scale factor."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from bit_kv_cache_07_gb300 import workloads
    w = workloads.WORKLOADS[args.workload]
    per_step, timed_streams, timed_s = [], 0, 0.0
    budget = max(2.0, 150.0 / max(1, args.steps + args.warmup))
    t_start = time.perf_counter()
    for i in range(args.warmup + args.steps):
        r = oracle_sample(args.workload, budget)
        if i >= args.warmup:
            per_step.append(r["value"])
            timed_streams += r["streams"]
            timed_s += r["seconds"]
    wall = time.perf_counter() - t_start
    v = statistics.median(per_step)
    streams_per_step = w["layers"] * w["batch"] * w["n_kv_heads"]
    cb = {k: r[k] for k in ("unit", "cores", "kind", "sample")}
    cb["value"] = v
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": v / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "layers": w["layers"], "batch": w["batch"],
                   "q_heads": w["n_q_heads"], "kv_heads": w["n_kv_heads"], "context": w["tokens"]},
        "sampled": {
            "what": "each step is a bounded sample, not a whole model step: single-stream oracle decodes "
                    "of layer 0 at the full context, scaled to the step's streams",
            "stream_decodes_timed": timed_streams, "seconds_timed": timed_s, "wall_seconds": wall,
            "streams_per_model_step": streams_per_step,
            "extrapolation_per_step": streams_per_step / max(1, timed_streams / max(1, args.steps)),
        },
        "cpu_baseline": cb, "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# -------------------------------------------------------------------- main

def _pair_name(c: dict) -> str:
    if c["k_bits"] == 16:
        return "FP16"
    if c["k_bits"] == 3:
        return "NUQ3"
    return f"K{c['k_bits']}V{c['v_bits']}"


def decode_roofline(model, per_layer_ms, peak, peak_kind, workload):
    """Roofline object of the decode launches of one step (in-graph times),
    plus a per-(K, V)-pair breakdown when the layers differ."""
    names = model.kernel_names()
    layer_bytes = [model.unit_bytes(i) for i in range(len(model.cfgs))]
    total_b, total_ms = sum(layer_bytes), sum(per_layer_ms)
    achieved = total_b / (total_ms * 1e-3) / 1e9
    traffic = [ncu_traffic(f"decode:{workload}:{_pair_name(c)}") for c in model.cfgs]
    by_pair = {}
    for l, c in enumerate(model.cfgs):
        e = by_pair.setdefault(_pair_name(c), {"kernel": names[l], "layers": 0, "ms": [], "bytes": layer_bytes[l],
                                               "traffic": traffic[l]})
        e["layers"] += 1
        e["ms"].append(per_layer_ms[l])
    pairs = {}
    for k, e in by_pair.items():
        us = statistics.mean(e["ms"]) * 1e3
        gbs = e["bytes"] / (us * 1e-6) / 1e9
        pairs[k] = {"kernel": e["kernel"], "layers": e["layers"], "decode_us": us, "bytes_per_launch": e["bytes"],
                    "achieved_gbs": gbs, "frac": gbs / peak, "frac_of_8tbs": gbs / HBM_NOMINAL_GBS,
                    "traffic": e["traffic"]}
    kinds = sorted(set(names))
    roof = {
        "bound": "hbm",
        "kernel": kinds[0] if len(kinds) == 1 else f"{len(kinds)} instantiations: " + "; ".join(kinds),
        "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
        "frac": achieved / peak, "frac_of_8tbs": achieved / HBM_NOMINAL_GBS,
        "traffic": (sum(traffic) / len(traffic)) if all(t is not None for t in traffic) else None,
        "bytes_per_launch": total_b / len(layer_bytes),
        "launch_us": total_ms * 1e3 / len(layer_bytes),
        "timing": "mean decode duration per layer: each (K, V) pair's decode launches captured back to "
                  "back in a CUDA graph, replayed between two CUDA events, divided by the launches",
    }
    return roof, (pairs if len(pairs) > 1 else None)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    import torch
    rank, world, local = init_dist(args.gpus)
    import __graft_entry__
    __graft_entry__.build()
    from bit_kv_cache_07_gb300 import workloads
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    w = workloads.WORKLOADS[args.workload]

    model = Model(args.workload, dev, fp16=False, layers=args.layers, tokens=args.tokens)
    clocks = ClockSampler(local)
    clocks.start()
    total_ms = time_steps(model, stream, args.steps, args.warmup)
    g_ms, rounds, g_err = time_graph(model, stream, args.steps, args.warmup, args.min_timed_seconds)
    layer_ms, t_err = time_decode_only(model, stream, args.steps, args.warmup)
    clk = clocks.stop()
    eager_ms = max_over_ranks(total_ms / args.steps)
    ms_step = max_over_ranks(g_ms) if g_ms is not None else eager_ms
    if layer_ms is None:
        raise RuntimeError(t_err)
    dec_bytes = model.decode_bytes()
    peak, peak_kind = measured_peaks()
    roof, pairs = decode_roofline(model, layer_ms, peak, peak_kind, args.workload)
    if any(m is not None for m in model.mixed):
        pairs = None  # the parts of a layer run side by side: only the layer's time is measured
        roof["launch_us"] = sum(layer_ms) * 1e3 / model.L
        roof["bytes_per_launch"] = model.decode_bytes() / model.L
        roof["timing"] = ("mean decode time per layer (its per-pair caches decoded side by side on forked "
                          "streams, each on a byte-proportional share of the SMs): every layer's decode captured "
                          "back to back in a CUDA graph, replayed between two CUDA events")
    e2e_ms, h2d, d2h = time_e2e(model, stream, max(3, args.steps), 2)
    e2e_ms = max_over_ranks(e2e_ms)
    launches = model.launches_per_step() * args.steps
    model_layers, model_T = model.L, model.T
    model_kernels, model_rows = sorted(set(model.kernel_names())), model.rows
    head_pairs = model.head_pairs or None
    del model
    torch.cuda.empty_cache()
    append = time_append(args.workload, dev, model_T, stream)

    fp16 = None
    if not args.no_fp16_baseline:
        fmodel = Model(args.workload, dev, fp16=True, layers=args.layers, tokens=args.tokens)
        fg_ms, _, _ = time_graph(fmodel, stream, args.steps, args.warmup, 0.0)
        if fg_ms is None:
            f_total = time_steps(fmodel, stream, args.steps, args.warmup)
            fg_ms = f_total / args.steps
        f_ms = max_over_ranks(fg_ms)
        f_layer_ms, _ = time_decode_only(fmodel, stream, args.steps, args.warmup)
        f_bytes = fmodel.decode_bytes()
        fp16 = {"us_per_step": f_ms * 1e3, "cache_gbs": f_bytes / (f_ms * 1e-3) / 1e9,
                "bytes_per_step": f_bytes, "kernel": fmodel.kernel_names()[0]}
        if f_layer_ms is not None:
            f_dec = statistics.mean(f_layer_ms)
            nu = len(fmodel.cfgs)
            fp16.update(decode_kernel_us=f_dec * 1e3,
                        decode_kernel_gbs=(f_bytes / nu) / (f_dec * 1e-3) / 1e9,
                        decode_frac=(f_bytes / nu) / (f_dec * 1e-3) / 1e9 / peak)
        del fmodel
        torch.cuda.empty_cache()

    cpu = cpu_all = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_sample(args.workload, args.cpu_seconds)
        cpu = {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample")}
        cpu_all = oracle_sample_all_cores(args.workload, args.cpu_seconds)

    value = ms_step * 1e3
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "data": "synthetic",
        "dtype": ("f32 (CUDA cores) on u8-packed codes" if all(k.startswith("decode_kernel<") for k in model_kernels)
                  else "f16xf16->f32 (tensor cores) on u8-packed codes"),
        "config": {"workload": args.workload, "layers": model_layers, "batch": w["batch"],
                   "q_heads": w["n_q_heads"], "kv_heads": w["n_kv_heads"], "head_dim": w["head_dim"],
                   "context": model_T, "cache": w["pairs"], "n_sink": w["n_sink"], "n_recent": w["n_recent"],
                   "l2": "inputs larger than L2: %.2f GB of cache read per step" % (dec_bytes / 1e9),
                   "step": ("per layer: kvq_append_ragged of 1 token per row + kvq_decode_attn_ragged"
                            if model_rows else "per layer: kvq_append of 1 token + kvq_decode_attn"),
                   "rows": ({"lengths": model_rows, "mean": statistics.mean(model_rows)} if model_rows else None),
                   "timing": (f"one step captured in a CUDA graph; median over {rounds} timed rounds of "
                              f"exactly {args.steps} replays" if g_ms is not None else
                              "eager launches (" + str(g_err) + ")")},
        "ms_per_step_eager": eager_ms,
        "cache_gbs": sum_over_ranks(dec_bytes / (ms_step * 1e-3) / 1e9),
        "cache_frac_of_8tbs": dec_bytes / (ms_step * 1e-3) / 1e9 / HBM_NOMINAL_GBS,
        "cache_bytes_per_step": dec_bytes,
        "roofline": roof,
        "decode_by_pair": pairs,
        "head_pairs": head_pairs,
        "append": append,
        "fp16_baseline": fp16,
        "speedup_vs_fp16": (fp16["us_per_step"] / value) if fp16 else None,
        "byte_ratio_vs_fp16": (fp16["bytes_per_step"] / dec_bytes) if fp16 else None,
        "cpu_baseline": cpu,
        "cpu_baseline_all_cores": cpu_all,
        "e2e": {"value": e2e_ms * 1e3, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "eager calls of the public C ABI per layer; this step's q and new K/V of every layer "
                       "copied in from pinned host memory (one copy) and every layer's output copied back "
                       "(one copy), inside the timed region"},
        "gpu_launches": launches,
        "clocks": clk,
    }
    if t_err:
        line["roofline"]["timing_note"] = t_err
    if rank == 0:
        print(json.dumps(line), flush=True)
    if _DIST["on"]:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

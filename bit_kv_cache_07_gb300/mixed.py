"""Per-head (K, V) bits (RateQuant summary, "Methodology" 1-4).

A layer whose KV heads use different (K bits, V bits) pairs is held as one
libkvq cache per distinct pair, each covering its subset of the layer's
heads through the config's head map (``kv_heads_total``,
``kv_head_index``): every append reads the layer's whole K/V tensors and
every decode the whole q and out, so no data is gathered or scattered.  A
decode step launches one decode kernel per distinct pair.

``allocate_pairs`` chooses the pairs: the distortion of the cache's
quantizer is measured per head on calibration tokens at 2, 4 and 8 bits
(``kvq_measure_distortion``, on the GPU), and ``kvq_rate_allocate`` fits
D(b) = alpha beta^-b per component (K and V of every head: the page's K/V
separation) and spends the bit budget greedily.  This module only groups,
calls and keeps the sub-caches.
"""
from __future__ import annotations

from . import binding

LADDER = (2, 4, 8)


def allocate_pairs(cfg: dict, K, V, avg_bits: float, weights=None):
    """Per-head (K bits, V bits) for a layer shaped like cfg, from calibration
    tokens K, V [B, Hkv, n, d] (fp16, GPU), with an average of avg_bits per
    component (total = round(avg_bits * 2 * Hkv)).  Returns (pairs, report)."""
    import numpy as np
    base = dict(cfg)
    base.update(k_bits=4, v_bits=4, batch=K.shape[0])
    hkv = cfg["n_kv_heads"]
    D = np.stack([binding.kvq_measure_distortion(base, K, V, b).cpu().numpy() for b in LADDER], -1)  # [Hkv, 2, 3]
    comps = D.reshape(2 * hkv, 3)  # component 2h = K of head h, 2h + 1 = V of head h
    total = int(round(avg_bits * 2 * hkv))
    bits, alpha, beta, wf = binding.kvq_rate_allocate(comps, total, weights)
    pairs = [(int(bits[2 * h]), int(bits[2 * h + 1])) for h in range(hkv)]
    return pairs, {"distortion": comps.tolist(), "alpha": alpha.tolist(), "beta": beta.tolist(),
                   "waterfill_bits": wf.tolist(), "bits": bits.tolist(), "total_bits": total}


class MixedLayer:
    """One layer's cache with per-KV-head (K bits, V bits) pairs: a
    binding.Layer per distinct pair over its heads.  A decode runs the parts
    side by side: each gets a share of the SMs proportional to its cache
    bytes (the config's sm_budget) and its own workspace, the first on the
    caller's stream and the others on side streams that fork from it and
    join back into it (CUDA-graph capturable)."""

    def __init__(self, cfg: dict, pairs, device="cuda"):
        import torch
        hkv = cfg["n_kv_heads"]
        if len(pairs) != hkv:
            raise ValueError("one (K bits, V bits) pair per KV head")
        g = cfg["n_q_heads"] // hkv
        self.cfg = dict(cfg)
        self.pairs = [tuple(p) for p in pairs]
        groups = [(pair, [h for h in range(hkv) if self.pairs[h] == pair]) for pair in sorted(set(self.pairs))]
        subs = [dict(cfg, k_bits=pair[0], v_bits=pair[1], n_kv_heads=len(heads), n_q_heads=g * len(heads),
                     kv_heads_total=hkv, kv_head_index=heads) for pair, heads in groups]
        sms = torch.cuda.get_device_properties(torch.device(device)).multi_processor_count
        # SM shares proportional to each part's expected decode time: the larger
        # of its bytes over the copy bandwidth and its 32-token groups times the
        # per-group arithmetic (the low-bit parts are bound by the latter:
        # about the same instructions per group whatever the bit width)
        est = []
        for c in subs:
            lay = binding.kvq_layout_query(c)
            n_groups = c["batch"] * c["n_kv_heads"] * (lay.q_cap // 32)
            est.append(max(lay.layer_bytes / 6.0e12, n_groups * 1.05e-9))
        share = [max(1, int(sms * e / sum(est))) for e in est] if len(subs) > 1 else [0]
        self.parts, self.ws, self.side = [], [], []
        for (pair, heads), sub, sm in zip(groups, subs, share):
            sub["sm_budget"] = sm
            layer = binding.Layer(sub, device=device)
            self.parts.append((pair, heads, layer))
            self.ws.append(torch.zeros(max(16, layer.layout.workspace_bytes), dtype=torch.uint8, device=device))
        self.side = [torch.cuda.Stream(device=device) for _ in self.parts[1:]]

    def append(self, tokens_before: int, k_new, v_new, stream=None):
        for _, _, layer in self.parts:
            layer.append(tokens_before, k_new, v_new, stream)

    def append_ragged(self, tokens_before, n_new, k_new, v_new, stream=None):
        """Batch row b appends n_new[b] tokens after tokens_before[b] (every part)."""
        for _, _, layer in self.parts:
            layer.append_ragged(tokens_before, n_new, k_new, v_new, stream)

    def decode(self, tokens: int, q, out, lse=None, workspace=None, stream=None):
        """Attention over the layer's cache into out (all heads); each part
        uses its own workspace (`workspace` is not used)."""
        self._side_by_side(lambda layer, ws, s: layer.decode(tokens, q, out, lse, ws, s), stream)

    def decode_ragged(self, tokens, q, out, lse=None, workspace=None, stream=None):
        """decode with batch row b attending over its own tokens[b] tokens."""
        self._side_by_side(lambda layer, ws, s: layer.decode_ragged(tokens, q, out, lse, ws, s), stream)

    def _side_by_side(self, call, stream):
        import torch
        main = stream if stream is not None else torch.cuda.current_stream()
        if len(self.parts) == 1:
            call(self.parts[0][2], self.ws[0], main)
            return
        fork = torch.cuda.Event()
        fork.record(main)
        joins = []
        for i, (_, _, layer) in enumerate(self.parts):
            s = main if i == 0 else self.side[i - 1]
            if i:
                s.wait_event(fork)
            call(layer, self.ws[i], s)
            if i:
                e = torch.cuda.Event()
                e.record(s)
                joins.append(e)
        for e in joins:
            main.wait_event(e)

    def workspace_bytes(self) -> int:
        return max(layer.layout.workspace_bytes for _, _, layer in self.parts)

    def layer_bytes(self) -> int:
        return sum(layer.layout.layer_bytes for _, _, layer in self.parts)

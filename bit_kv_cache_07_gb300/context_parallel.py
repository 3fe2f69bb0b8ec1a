"""Context-parallel decode: every sequence's context cut into one shard per
rank (KVQuant summary: a 10M-token context on an 8-GPU system).

Each rank holds its shard in an ordinary libkvq cache whose configuration
comes from ``kvq_context_shard`` (sinks on the first shard, the fp16 window
on the last, RoPE at absolute positions).  A decode step attends over the
local shard with ``kvq_decode_attn``, all-gathers every rank's normalised
output and log-sum-exp (B * Hq * (128 fp16 + 1 f32) per rank: the one
exchange of the path), and merges them with ``kvq_merge_attn``.  Appended
tokens go to the last shard.  The arithmetic runs in libkvq's kernels; this
module only plans, calls and gathers.
"""
from __future__ import annotations

from . import binding


def _rank_world(group=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        return dist.get_rank(group), dist.get_world_size(group)
    return 0, 1


def gather_parts(out_local, lse_local, group=None):
    """All-gather every rank's part: (outs [world, ...], lses [world, ...]) in
    rank order (the local tensors when there is no process group)."""
    import torch
    import torch.distributed as dist
    rank, world = _rank_world(group)
    if world == 1:
        return out_local.unsqueeze(0), lse_local.unsqueeze(0)
    outs = [torch.empty_like(out_local) for _ in range(world)]
    lses = [torch.empty_like(lse_local) for _ in range(world)]
    dist.all_gather(outs, out_local.contiguous(), group=group)
    dist.all_gather(lses, lse_local.contiguous(), group=group)
    return torch.stack(outs), torch.stack(lses)


class ShardedLayer:
    """This rank's shard of one layer's cache for a context of `tokens`
    tokens (the length at prefill)."""

    def __init__(self, cfg: dict, tokens: int, group=None, device="cuda"):
        self.group = group
        self.rank, self.world = _rank_world(group)
        self.cfg = dict(cfg)
        self.shard_cfg, self.first, self.n = binding.kvq_context_shard(cfg, tokens, self.world, self.rank)
        self.last = self.rank == self.world - 1
        self.layer = binding.Layer(self.shard_cfg, device=device)

    def prefill(self, K, V, stream=None):
        """K, V [B, Hkv, tokens, d] fp16 of the whole context (every rank
        passes the same tensors); this rank stores its shard."""
        if self.n > 0:
            a, b = self.first, self.first + self.n
            self.layer.append(0, K[:, :, a:b].contiguous(), V[:, :, a:b].contiguous(), stream)

    def local_tokens(self, tokens: int) -> int:
        """Tokens of this shard when the whole context holds `tokens`."""
        return tokens - self.first if self.last else self.n

    def append(self, tokens_before: int, k_new, v_new, stream=None):
        """New tokens of the whole context (positions tokens_before ...): the
        last shard stores them, the other ranks do nothing."""
        if self.last:
            self.layer.append(tokens_before - self.first, k_new, v_new, stream)

    def decode(self, tokens: int, q, out, lse=None, workspace=None, stream=None):
        """Attention of q over the whole context of `tokens` tokens into out
        (and lse): local decode, all-gather of (out, lse), log-sum-exp merge."""
        import torch
        B, Hq, d = q.shape
        out_local = torch.zeros_like(out)
        lse_local = torch.full((B, Hq), float("-inf"), dtype=torch.float32, device=q.device)
        n_local = self.local_tokens(tokens)
        if n_local > 0:
            self.layer.decode(n_local, q, out_local, lse_local, workspace, stream)
        outs, lses = gather_parts(out_local, lse_local, self.group)
        binding.kvq_merge_attn(outs, lses, out, lse, stream)

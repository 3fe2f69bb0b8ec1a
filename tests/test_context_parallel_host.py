"""Context-parallel decode, host side (no GPU): libkvq's shard planner
(kvq_context_shard) and the gather + merge plumbing.

The shards the library plans, each stored and decoded by the CPU oracle on
its own and merged by log-sum-exp, must give the oracle's decode of the whole
context (KVQuant summary: a 10M-token context on an 8-GPU system).  Two gloo
ranks run the same through context_parallel.gather_parts."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from oracle import kvq_oracle as O

D = 128


@pytest.fixture(scope="module")
def B():
    from bit_kv_cache_07_gb300 import build
    build.build_library()
    from bit_kv_cache_07_gb300 import binding
    return binding


def cfg_of(kb, vb, S=0, R=0, T=1000, **kw):
    c = dict(batch=1, n_q_heads=4, n_kv_heads=1, head_dim=D, max_tokens=T + 64, k_bits=kb, v_bits=vb,
             k_group_tokens=32, v_group_channels=64, n_sink=S, n_recent=R, v_hadamard=0, k_pre_rope=0,
             rope_theta=10000.0, outliers_per_vector=0, softmax_scale=0.0, split_tokens=0,
             position_offset=0, k_lut=[0.0] * 8, v_lut=[0.0] * 8)
    c.update(kw)
    return c


def _lut(seed):
    x = np.sort(np.random.default_rng(seed).standard_normal(65536))
    return [float(v) for v in x[((np.arange(8) + 0.5) * 65536 / 8).astype(int)].astype(np.float16)]


CFGS = {
    "kv4_sinks_window": cfg_of(4, 4, S=4, R=64),
    "k8v2_hadamard": cfg_of(8, 2, S=2, R=32, v_hadamard=1),
    "nuq_rope": cfg_of(3, 3, k_pre_rope=1, outliers_per_vector=2, k_lut=_lut(3), v_lut=_lut(4)),
    "k4v4_rope_sinks": cfg_of(4, 4, S=4, R=16, k_pre_rope=1, position_offset=5000),
    "fp16": cfg_of(16, 16),
}


@pytest.mark.parametrize("name", list(CFGS))
@pytest.mark.parametrize("T,n", [(1000, 1), (1000, 2), (1000, 3), (1000, 8), (70, 4), (3, 2), (1000, 64)])
def test_shards_partition_the_context(B, name, T, n):
    """Shards are contiguous and cover [0, T); sinks only on shard 0, the
    fp16 window only on the last; together they hold the whole context's
    quantized groups (each shard's quantized tokens are whole groups at the
    whole context's group boundaries)."""
    cfg = CFGS[name]
    S_all, Nq_all, W_all = O.layout_counts(cfg, T)
    nxt, nq_sum = 0, 0
    for r in range(n):
        sc, a, m = B.kvq_context_shard(cfg, T, n, r)
        assert a == nxt and m >= 0
        nxt = a + m
        assert sc["position_offset"] == cfg["position_offset"] + a
        assert sc["n_sink"] == (cfg["n_sink"] if r == 0 else 0)
        assert sc["n_recent"] == (cfg["n_recent"] if r == n - 1 else 0)
        if m > 0:
            S_r, Nq_r, W_r = O.layout_counts(sc, m)
            nq_sum += Nq_r
            if cfg["k_bits"] != 16:
                if r > 0:
                    assert (a - cfg["n_sink"]) % 32 == 0  # starts on a whole-context group boundary
                if r < n - 1:
                    assert W_r == 0
                else:
                    assert W_r == W_all
        if r == n - 1:
            assert sc["max_tokens"] == cfg["max_tokens"] - a
    assert nxt == T
    assert nq_sum == Nq_all


@pytest.mark.parametrize("name", list(CFGS))
@pytest.mark.parametrize("n", [2, 3, 5])
def test_shard_decodes_merged_equal_the_whole_context(B, name, n):
    rng = np.random.default_rng(7)
    cfg = CFGS[name]
    T = 1000
    K = rng.standard_normal((T, D)).astype(np.float16)
    V = rng.laplace(size=(T, D)).astype(np.float16)
    q = rng.standard_normal((4, D)).astype(np.float16)
    full, flse = O.decode_stream(cfg, T, O.build_stream(cfg, K, V), q)
    outs, lses = [], []
    for r in range(n):
        sc, a, m = B.kvq_context_shard(cfg, T, n, r)
        if m == 0:
            outs.append(np.zeros((4, D)))
            lses.append(np.full(4, -np.inf))
            continue
        o, l = O.decode_stream(sc, m, O.build_stream(sc, K[a:a + m], V[a:a + m]), q)
        outs.append(o)
        lses.append(l)
    merged, mlse = O.merge_parts(np.stack(outs), np.stack(lses))
    assert np.allclose(merged, full, rtol=0, atol=1e-12)
    assert np.allclose(mlse, flse, rtol=0, atol=1e-12)


def test_shard_arguments_are_checked(B):
    cfg = CFGS["kv4_sinks_window"]
    for args in [(1000, 0, 0), (1000, 2, 2), (1000, 2, -1), (0, 2, 0)]:
        with pytest.raises(B.KvqError):
            B.kvq_context_shard(cfg, *args)
    with pytest.raises(B.KvqError):
        B.kvq_context_shard(cfg, 2000, 2, 0)  # beyond max_tokens


# ------------------------------------------------------------ two gloo ranks

def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, name: str, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from bit_kv_cache_07_gb300 import binding, context_parallel
    cfg = CFGS[name]
    rng = np.random.default_rng(11)  # every rank draws the same context and query
    T = 777
    K = rng.standard_normal((T, D)).astype(np.float16)
    V = rng.laplace(size=(T, D)).astype(np.float16)
    q = rng.standard_normal((4, D)).astype(np.float16)
    sc, a, m = binding.kvq_context_shard(cfg, T, world, rank)
    if m > 0:
        o, l = O.decode_stream(sc, m, O.build_stream(sc, K[a:a + m], V[a:a + m]), q)
    else:
        o, l = np.zeros((4, D)), np.full(4, -np.inf)
    outs, lses = context_parallel.gather_parts(torch.from_numpy(o), torch.from_numpy(l))
    merged, mlse = O.merge_parts(outs.numpy(), lses.numpy())
    full, flse = O.decode_stream(cfg, T, O.build_stream(cfg, K, V), q)
    results[rank] = (float(np.abs(merged - full).max()), float(np.abs(mlse - flse).max()), a, m)
    dist.destroy_process_group()


@pytest.mark.parametrize("name", ["kv4_sinks_window", "nuq_rope"])
def test_two_gloo_ranks_gather_and_merge(B, name):
    port = _free_port()
    with mp.Manager() as man:
        results = man.dict()
        mp.spawn(_rank_main, args=(2, port, name, results), nprocs=2, join=True)
        got = dict(results)
    assert set(got) == {0, 1}
    assert got[0][2] == 0 and got[0][2] + got[0][3] == got[1][2]  # rank 0 then rank 1
    for r in (0, 1):
        assert got[r][0] < 1e-12 and got[r][1] < 1e-12

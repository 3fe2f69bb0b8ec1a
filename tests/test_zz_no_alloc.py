"""kvq_decode_attn_noalloc: the decode entry point for callers that cannot
allocate device memory (its split-K scratch is a fixed array inside the
library).  Called through the C ABI, it must match kvq_decode_attn with a
caller-provided workspace, on two calls in a row (the shared scratch keeps
the previous call's contents), and reject work whose scratch would not fit.

This file is collected last on purpose: a failure here does not hide the
results of the other GPU tests."""
import ctypes as C

import numpy as np
import pytest
import torch

from _kvq_testutil import TOL, normwise_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from bit_kv_cache_07_gb300 import build
    build.build_library()
    from bit_kv_cache_07_gb300 import binding
    assert torch.cuda.is_available()
    return binding


def _cfg(**kw):
    c = dict(batch=2, n_q_heads=8, n_kv_heads=2, head_dim=128, max_tokens=3000, k_bits=4, v_bits=4,
             k_group_tokens=32, v_group_channels=64, n_sink=4, n_recent=64, v_hadamard=0, k_pre_rope=0,
             rope_theta=10000.0, outliers_per_vector=0, softmax_scale=0.0, split_tokens=0)
    c.update(kw)
    return c


_LUT_K = [-1.53, -0.88, -0.49, -0.16, 0.16, 0.49, 0.88, 1.53]
_LUT_V = [-1.5, -0.9, -0.5, -0.15, 0.15, 0.5, 0.9, 1.5]

# (config changes, kernel expected: True = persistent, False = split-K)
CASES = {
    "persistent_kv4_g4": (dict(), True),
    "persistent_k4v2_hadamard_g7": (dict(k_bits=4, v_bits=2, v_hadamard=1, n_q_heads=14), True),
    # the split-K kernel: its partials live in the fixed scratch, sized by the
    # host plan (the fixed-scratch entry point does not widen the grid)
    "split_nuq3_rope": (dict(k_bits=3, v_bits=3, k_pre_rope=1, outliers_per_vector=2, n_sink=0, n_recent=0,
                             k_lut=_LUT_K, v_lut=_LUT_V), False),
    "split_k4v4_gv32": (dict(v_group_channels=32), False),
}


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_workspace_entry_point_twice(B, name):
    from bit_kv_cache_07_gb300 import synth
    kw, want_persistent = CASES[name]
    cfg = _cfg(**kw)
    T = 2900
    persistent, _ = B.kvq_decode_path(cfg, T)
    assert persistent == want_persistent, "the case must exercise the intended decode kernel"
    K, V = synth.random_kv(cfg["batch"], cfg["n_kv_heads"], T, seed=77, device="cuda")
    layer = B.Layer(cfg)
    layer.append(0, K, V)
    q = synth.random_q(cfg["batch"], cfg["n_q_heads"], seed=78, device="cuda")
    ref = torch.empty_like(q)
    ref_lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    layer.decode(T, q, ref, ref_lse, B.new_workspace(cfg))
    if not persistent:
        splits, _ = B.kvq_decode_plan(cfg, T)
        assert splits > 1, "the split-K case must use more than one split (scratch partials)"
    c = B.make_config(cfg)
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        st = B.lib().kvq_decode_attn_noalloc(C.byref(c), layer.buf.data_ptr(), T, q.data_ptr(),
                                             out.data_ptr(), lse.data_ptr(),
                                             torch.cuda.current_stream().cuda_stream)
        assert st == 0, B.kvq_status_string(st)
        torch.cuda.synchronize()
        err = normwise_err(out.float().cpu().numpy(), ref.float().cpu().numpy())
        assert err.max() < TOL, (call, err.max())
        assert np.allclose(lse.cpu().numpy(), ref_lse.cpu().numpy(), rtol=1e-5, atol=1e-5)


def test_noalloc_rejects_scratch_beyond_its_size(B):
    """2048 streams x 8 query heads: even one partial result per stream
    (2048 x 8 x (2 + 128) floats) exceeds 8 MiB, so the call must return
    KVQ_ERR_WORKSPACE before launching anything."""
    cfg = _cfg(batch=64, n_kv_heads=32, n_q_heads=256, max_tokens=5000)
    assert 2048 * 8 * (2 + 128) * 4 > (8 << 20)
    c = B.make_config(cfg)
    fake = 1 << 20  # never dereferenced: the size check comes first
    assert B.lib().kvq_decode_attn_noalloc(C.byref(c), fake, 4000, fake, fake, None, None) == -4

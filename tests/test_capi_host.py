"""Host-side checks of libkvq's C ABI that need no GPU: the library loads,
exports every entry point declared in include/kvq.h, computes consistent
layouts, and rejects bad arguments before launching anything."""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    from bit_kv_cache_07_gb300 import build
    build.build_library()
    from bit_kv_cache_07_gb300 import binding
    return binding


def declared_functions():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_\w+)\s*\(", src)))


def test_exports_match_header(B):
    out = subprocess.check_output(["nm", "-D", "--defined-only", B.library_path()]).decode()
    exported = set(re.findall(r" T (kvq_\w+)", out))
    declared = declared_functions()
    assert declared, "no declarations parsed"
    assert set(declared) <= exported, set(declared) - exported
    assert set(B.EXPORTS) == set(declared)
    B.lib()  # loads


def base(**kw):
    c = dict(batch=2, n_q_heads=8, n_kv_heads=2, head_dim=128, max_tokens=1000, k_bits=4, v_bits=2,
             k_group_tokens=32, v_group_channels=64, n_sink=4, n_recent=64, v_hadamard=0,
             k_pre_rope=0, rope_theta=10000.0, outliers_per_vector=0, softmax_scale=0.0, split_tokens=0)
    c.update(kw)
    return c


def test_layout_sizes_and_alignment(B):
    c = base()
    L = B.kvq_layout_query(c)
    NS, d = 4, 128
    qcap = 32 * ((1000 - 4 - 64) // 32)
    assert L.q_cap == qcap and L.ring_slots == 64 + 32
    assert L.k_codes.bytes == NS * qcap * 64
    assert L.k_scales.bytes == NS * (qcap // 32) * d * 4
    assert L.v_codes.bytes == NS * qcap * 32
    assert L.v_scales.bytes == NS * qcap * 2 * 4
    assert L.k_sink.bytes == NS * 4 * d * 2 and L.k_ring.bytes == NS * 96 * d * 2
    regs = sorted((getattr(L, n).offset, getattr(L, n).bytes) for n in B.REGIONS)
    for (o0, b0), (o1, b1) in zip(regs, regs[1:]):
        assert o0 % 256 == 0 and o0 + b0 <= o1
    assert regs[-1][0] + regs[-1][1] <= L.layer_bytes


def test_layout_nuq_and_fp16(B):
    lut = [-1.5, -0.9, -0.5, -0.16, 0.16, 0.5, 0.9, 1.5]
    L = B.kvq_layout_query(base(k_bits=3, v_bits=3, outliers_per_vector=2, k_lut=lut, v_lut=lut,
                                n_sink=0, n_recent=0))
    qcap = 32 * (1000 // 32)
    assert L.k_codes.bytes == 4 * qcap * 48 and L.k_scales.bytes == 4 * qcap * 4
    assert L.k_csr_rowptr.bytes == 4 * (qcap + 1) * 4 and L.k_csr_val.bytes == 4 * qcap * 2 * 2
    F = B.kvq_layout_query(base(k_bits=16, v_bits=16))
    assert F.k_codes.bytes == 0 and F.k_ring.bytes == 4 * 1000 * 128 * 2 and F.ring_slots == 1000


@pytest.mark.parametrize("kw,code", [
    (dict(batch=0), -1), (dict(n_q_heads=6, n_kv_heads=4), -1), (dict(head_dim=64), -2),
    (dict(k_bits=5), -2), (dict(k_bits=16), -2), (dict(k_bits=3, v_bits=4), -2),
    (dict(k_group_tokens=64), -2), (dict(v_group_channels=48), -2), (dict(n_q_heads=32, n_kv_heads=2), -2),
    (dict(n_sink=-1), -1), (dict(split_tokens=40), -1), (dict(k_pre_rope=1, rope_theta=0.0), -1),
    (dict(k_bits=3, v_bits=3, outliers_per_vector=2), -1),  # LUT not increasing
    (dict(softmax_scale=-1.0), -1), (dict(max_tokens=0), -1),
])
def test_invalid_configs(B, kw, code):
    with pytest.raises(B.KvqError) as e:
        B.kvq_layout_query(base(**kw))
    assert e.value.status == code


def test_entry_points_reject_before_launch(B):
    """Bad arguments return an error code and never reach a launch (these
    calls would need a GPU otherwise)."""
    c = B.make_config(base())
    L = B.lib()
    fake = 1 << 20  # never dereferenced: every call below fails validation first
    assert L.kvq_append(c, None, 0, fake, fake, 1, None) == -1
    assert L.kvq_append(c, fake, 0, fake, fake, 0, None) == -1
    assert L.kvq_append(c, fake, -1, fake, fake, 1, None) == -1
    assert L.kvq_append(c, fake, 999, fake, fake, 2, None) == -3
    assert L.kvq_append(c, fake + 8, 0, fake, fake, 1, None) == -1  # misaligned
    assert L.kvq_decode_attn(c, fake, 0, fake, fake, None, None, 0, None) == -1
    assert L.kvq_decode_attn(c, fake, 1001, fake, fake, None, None, 0, None) == -3
    assert L.kvq_decode_attn(c, fake, 900, None, fake, None, None, 0, None) == -1
    # 900 tokens need several splits -> a workspace
    assert L.kvq_decode_attn(c, fake, 900, fake, fake, None, None, 0, None) == -4
    assert L.kvq_decode_attn(c, fake, 900, fake, fake, None, fake, 16, None) == -4
    assert B.kvq_status_string(-4).startswith("workspace")


def test_decode_plan(B):
    c = base()
    spl, qs = B.kvq_decode_plan(c, 900)
    assert qs >= 1 and spl == qs + 1
    assert B.kvq_decode_plan(c, 50) == (1, 0)  # fp16 tokens only
    s32, q32 = B.kvq_decode_plan(base(split_tokens=32), 900)
    assert q32 == (900 - 4 - 64) // 32
    big = base(max_tokens=1 << 20, batch=1, n_q_heads=1, n_kv_heads=1, n_sink=0, n_recent=0)
    spl, qs = B.kvq_decode_plan(big, 1 << 20)
    assert qs == 64 and spl == 64
    L = B.kvq_layout_query(big)
    assert spl <= L.max_splits


def test_decode_path(B):
    """Which decode kernel a configuration takes (host only): the persistent
    tensor-core kernel for uniform 2/4/8-bit K and V with 64-channel V groups
    and no pre-RoPE K, or the fp16 cache; the split kernel otherwise."""
    assert B.kvq_decode_path(base(), 900) == (True, 4)
    assert B.kvq_decode_path(base(v_group_channels=32), 900) == (False, 4)
    assert B.kvq_decode_path(base(k_pre_rope=1), 900)[0] is False
    assert B.kvq_decode_path(base(k_bits=16, v_bits=16), 900) == (True, 4)
    assert B.kvq_decode_path(base(n_q_heads=14), 900) == (True, 8)
    assert B.decode_kernel_name(base(), 900) == "decode_persist_kernel<4, 2, 1, 4>"
    assert B.decode_kernel_name(base(n_q_heads=2), 900) == "decode_persist_kernel<4, 2, 1, 1>"
    assert B.decode_kernel_name(base(k_pre_rope=1), 900) == "decode_kernel<4, 2, 4>"
    with pytest.raises(B.KvqError):
        B.kvq_decode_path(base(), 1001)


def test_ragged_entry_points_reject_before_launch(B):
    """The ragged calls validate every row before any launch: lengths,
    capacity, stride, alignment, the workspace and the batch limit."""
    import ctypes as C
    c = B.make_config(base())
    L = B.lib()
    fake = 1 << 20
    rows = lambda *v: (C.c_int32 * len(v))(*v)
    # append: null arrays, negative counts, a row past its stride or capacity, misalignment
    assert L.kvq_append_ragged(c, fake, None, rows(1, 1), fake, fake, 4, None) == -1
    assert L.kvq_append_ragged(c, fake, rows(0, -1), rows(1, 1), fake, fake, 4, None) == -1
    assert L.kvq_append_ragged(c, fake, rows(0, 0), rows(5, 1), fake, fake, 4, None) == -1
    assert L.kvq_append_ragged(c, fake, rows(0, 0), rows(1, 1), fake, fake, 0, None) == -1
    assert L.kvq_append_ragged(c, fake, rows(0, 998), rows(1, 3), fake, fake, 4, None) == -3
    assert L.kvq_append_ragged(c, fake + 8, rows(0, 0), rows(1, 1), fake, fake, 4, None) == -1
    # nothing to append in any row: success without a launch
    assert L.kvq_append_ragged(c, fake, rows(10, 20), rows(0, 0), fake, fake, 4, None) == 0
    # decode: a row of zero tokens or past capacity, null q, null lengths
    assert L.kvq_decode_attn_ragged(c, fake, rows(5, 0), fake, fake, None, None, 0, None) == -1
    assert L.kvq_decode_attn_ragged(c, fake, rows(5, 1001), fake, fake, None, None, 0, None) == -3
    assert L.kvq_decode_attn_ragged(c, fake, rows(5, 7), None, fake, None, None, 0, None) == -1
    assert L.kvq_decode_attn_ragged(c, fake, None, fake, fake, None, None, 0, None) == -1
    # the persistent kernel needs its workspace; more than 256 rows
    assert L.kvq_decode_attn_ragged(c, fake, rows(500, 7), fake, fake, None, None, 0, None) == -4
    big = B.make_config(base(batch=257))
    many = (C.c_int32 * 257)(*([5] * 257))
    assert L.kvq_decode_attn_ragged(big, fake, many, fake, fake, None, None, 0, None) == -2
    assert L.kvq_append_ragged(big, fake, many, many, fake, fake, 8, None) == -2

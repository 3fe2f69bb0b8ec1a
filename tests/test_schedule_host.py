"""The persistent decode's schedule arithmetic (shared host/device code in
csrc/kvq_internal.cuh) checked on the host over many shapes."""
import os
import shutil
import subprocess
import tempfile

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_persistent_schedule_partition():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "sched_check")
        subprocess.check_call([nvcc, "-std=c++17", "-o", exe, os.path.join(HERE, "sched_check.cu")])
        out = subprocess.run([exe], capture_output=True, text=True)
        assert out.returncode == 0, out.stdout[-2000:]
        assert "bad 0" in out.stdout


def test_innerq_key_fragment_layout():
    """k_offset_of inverts k_slot_of; InnerQ key channels split between the
    two 64-channel groups by k-step; the stage swizzle is a bijection without
    bank conflicts on the fragment loads (tests/iq_layout_check.cu)."""
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "iq_layout_check")
        subprocess.check_call([nvcc, "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-o", exe,
                               os.path.join(HERE, "iq_layout_check.cu")])
        out = subprocess.run([exe], capture_output=True, text=True)
        assert out.returncode == 0 and "bad 0" in out.stdout, out.stdout[-2000:]

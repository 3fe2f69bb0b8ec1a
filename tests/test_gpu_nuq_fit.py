"""GPU parity of the non-uniform level-table fit (kvq_fit_nuq_lut, through the
C ABI) against the oracle's Lloyd fit: the tables and the number of updates
must be identical (every sum in the fit is an exact integer and every level
an fp64 quotient of two of them, so the order in which the GPU counts the
values cannot change a bit).  KVQuant summary, "technical approach":
per-layer non-uniform datatypes computed offline."""
import numpy as np
import pytest
import torch

from oracle import kvq_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from bit_kv_cache_07_gb300 import build
    build.build_library()
    from bit_kv_cache_07_gb300 import binding
    assert torch.cuda.is_available()
    return binding


def _data(kind, n, seed):
    rng = np.random.default_rng(seed)
    if kind == "normal_outlier_channels":
        x = rng.standard_normal((n, 128))
        x[:, [5, 77, 100]] *= 8.0
    elif kind == "laplace":
        x = rng.laplace(size=(n, 128))
    elif kind == "student_t3":
        x = rng.standard_t(3, (n, 128))
    else:  # few distinct values, constant and tied rows: exact ties at midpoints and level edges
        x = rng.integers(-3, 4, (n, 128)).astype(np.float64) / 4.0
        x[::7] = 0.5
        x[1::11, :64] = 2.0
    return x.astype(np.float16)


@pytest.mark.parametrize("kind", ["normal_outlier_channels", "laplace", "student_t3", "coarse_ties"])
@pytest.mark.parametrize("k,had", [(0, 0), (2, 0), (2, 1), (8, 0)])
@pytest.mark.parametrize("iters", [1, 4, 200])
def test_fit_equals_oracle(B, kind, k, had, iters):
    x = _data(kind, 3001, seed=len(kind) * 7 + k)
    lut, it = B.kvq_fit_nuq_lut(torch.from_numpy(x).cuda(), k, had, iters)
    rlut, rit = O.nuq_fit_lut(x, k, had, iters)
    assert it == rit
    assert lut == rlut


def test_planted_levels_on_the_gpu(B):
    rng = np.random.default_rng(3)
    planted = np.array([0.0, 0.125, 0.3125, 0.4375, 0.5625, 0.6875, 0.875, 1.0])
    x = planted[rng.integers(0, 8, (4000, 128))].astype(np.float16)
    x[:, 0], x[:, 1] = 0.0, 1.0
    x[:, 2] = 30.0
    lut, it = B.kvq_fit_nuq_lut(torch.from_numpy(x).cuda(), 1, 0, 100)
    assert lut == planted.tolist() and it == 2


def test_fit_rejects_bad_arguments(B):
    x = torch.zeros((4, 128), dtype=torch.float16, device="cuda")
    with pytest.raises(B.KvqError):
        B.kvq_fit_nuq_lut(x, 9)
    with pytest.raises(B.KvqError):
        B.kvq_fit_nuq_lut(x, 2, 2)
    with pytest.raises(B.KvqError):
        B.kvq_fit_nuq_lut(x, 2, 0, 0)


def test_workload_tables_fit_on_calibration_tokens(B):
    """The 1M-token workload's per-layer tables: the library's fit of layer
    0's 2048 calibration tokens (32 KV heads) equals the oracle's."""
    from bit_kv_cache_07_gb300 import calibrate, workloads
    name = "llama7b_nuq3_t1m"
    w = workloads.WORKLOADS[name]
    klut, vlut = calibrate.nuq_tables(name, 0)
    K, V = calibrate.calibration_kv(name, 0)
    assert O.nuq_fit_lut(K.cpu().numpy(), w["outliers_per_vector"])[0] == klut
    assert O.nuq_fit_lut(V.cpu().numpy(), w["outliers_per_vector"], w["v_hadamard"])[0] == vlut

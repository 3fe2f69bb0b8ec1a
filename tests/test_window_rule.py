"""The window rule (which tokens are sinks, quantized, or fp16 recent) pinned
against a brute-force simulation of appending tokens and flushing one
G_K-token group whenever the fp16 window reaches R + G_K tokens (InnerQ,
Methodology 4: recent and sink tokens stay fp16)."""
import numpy as np
import pytest

from oracle import kvq_oracle as O


def simulate(S, R, gk, T, chunks):
    nq, t = 0, 0
    for n in chunks:
        t += n
        while t - min(t, S) - nq >= R + gk:
            nq += gk
    assert t == T
    return nq


@pytest.mark.parametrize("S,R,gk", [(0, 0, 32), (4, 64, 32), (4, 128, 32), (0, 32, 32), (3, 5, 16), (4, 32, 32)])
def test_closed_form_matches_simulation(S, R, gk):
    rng = np.random.default_rng(S * 1000 + R)
    cfg = dict(head_dim=128, k_bits=4, v_bits=4, k_group_tokens=gk, n_sink=S, n_recent=R)
    for T in range(0, 400):
        one_by_one = simulate(S, R, gk, T, [1] * T)
        cuts = np.sort(rng.integers(0, T + 1, 3)) if T else np.zeros(3, int)
        chunks = np.diff(np.concatenate([[0], cuts, [T]]))
        bulk = simulate(S, R, gk, T, list(chunks))
        s, nq, w = O.layout_counts(cfg, T)
        assert nq == one_by_one == bulk, (T, nq, one_by_one, bulk)
        assert s == min(S, T) and s + nq + w == T
        if T >= S + R:
            assert R <= w < R + gk
        assert nq % gk == 0


def test_fp16_mode_has_no_quantized_tokens():
    cfg = dict(head_dim=128, k_bits=16, v_bits=16, k_group_tokens=32, n_sink=4, n_recent=8)
    assert O.layout_counts(cfg, 1000) == (0, 0, 1000)

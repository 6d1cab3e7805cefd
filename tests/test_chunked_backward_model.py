"""The chunked backward algorithm (tests/chunked_backward_model.py, the plan
of a tensor-core backward kernel) against the oracle's token-by-token
adjoint: the same y, final state and every gradient, for SISO and MIMO,
chunk lengths that divide the sequence and ones that leave a ragged last
chunk, a strong-decay case, and theta = 0 / lam = 1."""
import numpy as np
import pytest

import oracle
from chunked_backward_model import chunked_unit_backward

KEYS = ("x", "B", "C", "dt", "lam", "theta", "A", "D", "h0", "prev_B", "prev_x")


def _unit(R, T, P=4, N=8, seed=0, dt_hi=0.6, special=False):
    rng = np.random.default_rng(seed)
    K = N // 2
    args = dict(x=rng.normal(size=(T, R, P)), B=rng.normal(size=(T, R, N)), C=rng.normal(size=(T, R, N)),
                dt=rng.uniform(0.05, dt_hi, T), lam=np.ones(T) if special else rng.uniform(0.1, 0.9, T),
                theta=np.zeros((T, K)) if special else rng.uniform(0, np.pi, (T, K)),
                A=-rng.uniform(0.3, 1.5), D=rng.normal(),
                h0=rng.normal(size=(K, P)) + 1j * rng.normal(size=(K, P)),
                prev_B=rng.normal(size=(R, N)), prev_x=rng.normal(size=(R, P)))
    dy = rng.normal(size=(T, R, P))
    dhf = rng.normal(size=(K, P)) + 1j * rng.normal(size=(K, P))
    return args, dy, dhf


@pytest.mark.parametrize("R,T,Q", [(1, 24, 8), (1, 23, 8), (2, 19, 4), (4, 12, 4), (1, 7, 16)])
def test_chunked_backward_matches_oracle(R, T, Q):
    args, dy, dhf = _unit(R, T, seed=R * 100 + T)
    y0, h0, g0 = oracle.unit_backward(**args, dy=dy, dh_final=dhf)
    y1, h1, g1 = chunked_unit_backward(**args, dy=dy, dh_final=dhf, Q=Q)
    assert np.allclose(y1, y0, rtol=1e-10, atol=1e-10)
    assert np.allclose(h1, h0, rtol=1e-10, atol=1e-10)
    for k in KEYS:
        a, b = np.asarray(g1[k]), np.asarray(g0[k])
        assert np.allclose(a, b, rtol=1e-9, atol=1e-9 * max(1.0, np.max(np.abs(b)))), k


def test_strong_decay_and_special_values():
    for special, dt_hi in ((False, 6.0), (True, 0.6)):
        args, dy, dhf = _unit(2, 20, seed=5, dt_hi=dt_hi, special=special)
        _, _, g0 = oracle.unit_backward(**args, dy=dy, dh_final=dhf)
        _, _, g1 = chunked_unit_backward(**args, dy=dy, dh_final=dhf, Q=8)
        for k in KEYS:
            a, b = np.asarray(g1[k]), np.asarray(g0[k])
            assert np.allclose(a, b, rtol=1e-9, atol=1e-9 * max(1.0, np.max(np.abs(b)))), (special, k)

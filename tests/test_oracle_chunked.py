"""Pins for the oracle's chunked (WY/UT) form (CPU only).

The chunked form is an algebraic reorganisation of the recurrence, so the
two independently coded evaluations must agree to FP64 rounding; T must be
the inverse of I + A (checked with a library solve), and chunk sizes 1 and
>= n reduce to the token-by-token and the fully parallel evaluations.
"""
import numpy as np
import pytest

import gdnsynth as sy
import oracle

RNG = np.random.default_rng(99)


def _unit(n, dk, dv, s0_std=0.1):
    q = RNG.standard_normal((n, dk))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    k = RNG.standard_normal((n, dk))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = RNG.standard_normal((n, dv))
    g = np.log(1 / (1 + np.exp(-(RNG.standard_normal(n) + 2))))
    beta = 1 / (1 + np.exp(-RNG.standard_normal(n)))
    return oracle.Unit(q, k, v, g, beta, s0_std * RNG.standard_normal((dv, dk)))


def _rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


@pytest.mark.parametrize("n,C", [(1, 64), (5, 1), (17, 4), (64, 64), (100, 64), (130, 16), (33, 200)])
@pytest.mark.parametrize("s0", [0.0, 0.1])
def test_chunked_equals_recurrent(n, C, s0):
    u = _unit(n, 32, 16, s0)
    Sr, orr, _ = oracle.recurrent_units([u])
    Sc, oc = oracle.chunked_units([u], C)
    assert _rel(Sc[0], Sr[0]) < 1e-10
    assert np.max(np.abs(oc[0] - orr[0])) < 1e-10 * max(1.0, np.max(np.abs(orr[0])))


def test_chunked_equals_recurrent_full_head_size_ragged_batch():
    units = [_unit(n, 128, 128) for n in (70, 1, 129)]
    Sr, orr, _ = oracle.recurrent_units(units)
    Sc, oc = oracle.chunked_units(units, 64)
    for i in range(len(units)):
        assert _rel(Sc[i], Sr[i]) < 1e-10
        assert np.max(np.abs(oc[i] - orr[i])) < 1e-10


def test_prefill_workload_sample_chunked_equals_recurrent():
    r, cu, s0 = sy.prefill_inputs([80, 129], sy.Dims(2, 4, 32, 32), seed=5)
    for i in range(2):
        a, b = int(cu[i]), int(cu[i + 1])
        rr = r.slice(a, b)
        Sr, orr, _ = oracle.gdn_recurrent(rr.q, rr.k, rr.v, rr.g, rr.beta, s0[i])
        Sc, oc = oracle.gdn_chunked(rr.q, rr.k, rr.v, rr.g, rr.beta, s0[i], 64)
        for h in range(4):
            assert _rel(Sc[h], Sr[h]) < 1e-10


def test_T_is_inverse_of_I_plus_A():
    n, dk, dv = 24, 16, 8
    u = _unit(n, dk, dv)
    G, T, W, Ut = oracle.chunk_wy(u.k, u.v, u.g, u.beta)
    np.testing.assert_allclose(G, np.cumsum(u.g), rtol=1e-14)
    # Build A from its definition and invert it with a library solve.
    A = np.zeros((n, n))
    for t in range(n):
        for i in range(t):
            A[t, i] = u.beta[t] * np.exp(G[t] - G[i]) * (u.k[t] @ u.k[i])
    Tref = np.linalg.solve(np.eye(n) + A, np.eye(n))
    np.testing.assert_allclose(T, Tref, rtol=1e-10, atol=1e-12)
    assert np.allclose(np.triu(T, 1), 0.0)
    assert np.allclose(np.diag(T), 1.0)


def test_chunk_of_one_row_reduces_to_single_update():
    # C = 1: T = [1], W = beta e^g k, Ut = beta v; U = beta (v - e^g S0 k).
    u = _unit(1, 16, 8, 1.0)
    G, T, W, Ut = oracle.chunk_wy(u.k, u.v, u.g, u.beta)
    assert T.shape == (1, 1) and T[0, 0] == 1.0
    np.testing.assert_allclose(W[0], u.beta[0] * np.exp(u.g[0]) * u.k[0], rtol=1e-14)
    np.testing.assert_allclose(Ut[0], u.beta[0] * u.v[0], rtol=1e-14)

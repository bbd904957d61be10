"""Pins for the oracle's gated delta rule (CPU only).

Each test fixes the oracle to something other than itself: a closed form, an
invariant of the delta rule, or an independent dense-matrix evaluation.
A plausible slip in the oracle (dropped decay on the prediction, o taken
before the update, S transposed, wrong GQA head, missing beta) fails at least
one of them; ``test_pins_catch_planted_mistakes`` checks that directly on
mutated copies of the rule.
"""
import numpy as np
import pytest
import torch

import gdnsynth as sy
import oracle

RNG = np.random.default_rng(1234)


def _rand_unit(n, dk, dv, s0_std=0.1, unit_k=False, g=None, beta=None):
    q = RNG.standard_normal((n, dk))
    k = RNG.standard_normal((n, dk))
    if unit_k:
        k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = RNG.standard_normal((n, dv))
    g = np.log(1 / (1 + np.exp(-(RNG.standard_normal(n) + 2)))) if g is None else np.asarray(g, float)
    beta = 1 / (1 + np.exp(-RNG.standard_normal(n))) if beta is None else np.asarray(beta, float)
    S0 = s0_std * RNG.standard_normal((dv, dk))
    return oracle.Unit(q, k, v, g, beta, S0)


def _run(u, q_scale=1.0):
    S, os_, cks = oracle.recurrent_units([u], q_scale, want_ckpt=True)
    return S[0], os_[0], cks[0]


def dense_product_form(u, q_scale=1.0):
    """The benchmark spec's product form with explicit d_k x d_k matrices:
    S_t = S_{t-1} . alpha_t (I - beta_t k_t k_t^T) + beta_t v_t k_t^T."""
    S = u.S0.copy()
    dk = S.shape[1]
    outs, cks = [], []
    for t in range(u.q.shape[0]):
        kt = u.k[t][:, None]
        M = np.exp(u.g[t]) * (np.eye(dk) - u.beta[t] * (kt @ kt.T))
        S = S @ M + u.beta[t] * (u.v[t][:, None] @ kt.T)
        outs.append(q_scale * (S @ u.q[t]))
        cks.append(S.copy())
    return S, np.array(outs), np.array(cks)


@pytest.mark.parametrize("n,dk,dv", [(4, 16, 16), (7, 32, 16), (3, 128, 128)])
def test_matches_dense_product_form(n, dk, dv):
    u = _rand_unit(n, dk, dv)
    S, o, ck = _run(u, q_scale=0.7)
    S2, o2, ck2 = dense_product_form(u, q_scale=0.7)
    np.testing.assert_allclose(S, S2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(o, o2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(ck, ck2, rtol=1e-12, atol=1e-13)


def test_tiny_workload_matches_dense_product_form():
    spec = sy.SPECS["tiny"]
    r = sy.ring_rows(spec, 0, 0, 4)
    S0 = sy.pool_state(spec)[0, 0]
    for u in oracle.head_units(r.q, r.k, r.v, r.g, r.beta, S0):
        S, o, ck = _run(u)
        S2, o2, ck2 = dense_product_form(u)
        np.testing.assert_allclose(S, S2, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(o, o2, rtol=1e-12, atol=1e-14)


def test_beta_zero_is_pure_decay():
    # beta = 0: S_t = e^{G_t} S_0 and o_t = e^{G_t} S_0 q_t (closed form).
    u = _rand_unit(6, 16, 8, s0_std=1.0, beta=np.zeros(6))
    S, o, ck = _run(u)
    G = np.cumsum(u.g)
    for t in range(6):
        np.testing.assert_allclose(ck[t], np.exp(G[t]) * u.S0, rtol=1e-13)
        np.testing.assert_allclose(o[t], np.exp(G[t]) * (u.S0 @ u.q[t]), rtol=1e-12, atol=1e-14)


def test_g_zero_beta_zero_leaves_state_unchanged():
    u = _rand_unit(5, 16, 16, s0_std=1.0, g=np.zeros(5), beta=np.zeros(5))
    S, o, ck = _run(u)
    assert np.array_equal(S, u.S0)
    for t in range(5):
        assert np.array_equal(ck[t], u.S0)


def test_single_row_from_zero_state():
    # S_0 = 0, one row: S_1 = beta v k^T and o = beta v (k . q).
    u = _rand_unit(1, 32, 16, s0_std=0.0)
    S, o, _ = _run(u, q_scale=1.5)
    np.testing.assert_allclose(S, u.beta[0] * np.outer(u.v[0], u.k[0]), rtol=1e-14, atol=1e-16)
    np.testing.assert_allclose(o[0], 1.5 * u.beta[0] * u.v[0] * (u.k[0] @ u.q[0]), rtol=1e-12, atol=1e-15)


def test_delta_rule_write_property():
    # beta = 1 and ||k|| = 1: the update writes v_t at key k_t exactly,
    # S_t k_t = v_t, whatever the decay and the previous state.
    u = _rand_unit(8, 16, 12, s0_std=1.0, unit_k=True, beta=np.ones(8))
    _, _, ck = _run(u)
    for t in range(8):
        np.testing.assert_allclose(ck[t] @ u.k[t], u.v[t], rtol=1e-12, atol=1e-12)


def test_associative_recall_with_orthonormal_keys():
    # alpha = 1, beta = 1, orthonormal keys: every stored pair is recalled,
    # S_n k_i = v_i, and directions orthogonal to all keys keep S_0's image.
    dk, dv, n = 16, 8, 6
    Qm, _ = np.linalg.qr(RNG.standard_normal((dk, dk)))
    keys = Qm[:, :n].T
    u = _rand_unit(n, dk, dv, s0_std=1.0, g=np.zeros(n), beta=np.ones(n))
    u.k = keys.copy()
    S, _, _ = _run(u)
    for i in range(n):
        np.testing.assert_allclose(S @ keys[i], u.v[i], atol=1e-12)
    for x in Qm[:, n:].T:
        np.testing.assert_allclose(S @ x, u.S0 @ x, atol=1e-12)


def test_gqa_head_mapping_consecutive_groups():
    # h_qk = 2, h_v = 4: v-heads 0,1 use qk-head 0; v-heads 2,3 use qk-head 1.
    n, dk, dv = 1, 8, 4
    q = RNG.standard_normal((n, 2, dk))
    k = RNG.standard_normal((n, 2, dk))
    v = RNG.standard_normal((n, 4, dv))
    g = np.zeros((n, 4))
    beta = np.full((n, 4), 0.5)
    S0 = np.zeros((4, dv, dk))
    S, o, _ = oracle.gdn_recurrent(q, k, v, g, beta, S0)
    for h in range(4):
        hq = h // 2
        np.testing.assert_allclose(o[0, h], 0.5 * v[0, h] * (k[0, hq] @ q[0, hq]), rtol=1e-12)
        np.testing.assert_allclose(S[h], 0.5 * np.outer(v[0, h], k[0, hq]), rtol=1e-14)


def test_state_norm_bound():
    # ||I - beta k k^T||_2 = 1 for unit k and beta in [0, 2], hence
    # ||S_t||_2 <= alpha_t ||S_{t-1}||_2 + beta_t ||v_t|| ||k_t||.
    u = _rand_unit(20, 16, 16, s0_std=1.0, unit_k=True)
    _, _, ck = _run(u)
    prev = u.S0
    for t in range(20):
        lhs = np.linalg.norm(ck[t], 2)
        rhs = np.exp(u.g[t]) * np.linalg.norm(prev, 2) + u.beta[t] * np.linalg.norm(u.v[t])
        assert lhs <= rhs * (1 + 1e-12)
        prev = ck[t]


def test_checkpoint_row_equals_prefix_run():
    # ckpt row j is the state after rows 0..j: rerunning the first j+1 rows
    # from S_0 gives the same state, and chaining single-row runs from the
    # previous checkpoint gives it too (verify == repeated decode, oracle side).
    u = _rand_unit(5, 16, 16)
    _, _, ck = _run(u)
    S = u.S0.copy()
    for j in range(5):
        one = oracle.Unit(u.q[j:j + 1], u.k[j:j + 1], u.v[j:j + 1], u.g[j:j + 1], u.beta[j:j + 1], S)
        S, _, _ = _run(one)
        np.testing.assert_allclose(S, ck[j], rtol=1e-14, atol=1e-16)


def test_many_units_in_one_call_are_independent():
    units = [_rand_unit(n, 16, 16) for n in (1, 3, 0, 5)]
    Sall, oall, _ = oracle.recurrent_units(units, want_ckpt=True)
    for i, u in enumerate(units):
        S, o, _ = oracle.recurrent_units([u], want_ckpt=True)
        assert np.array_equal(Sall[i], S[0])
        if u.q.shape[0]:
            assert np.array_equal(oall[i], o[0])


def test_inputs_widen_exactly():
    spec = sy.SPECS["tiny"]
    r = sy.ring_rows(spec, 0, 0, 4)
    q64 = oracle._f64(r.q)
    assert np.array_equal(q64.astype(np.float32), r.q.float().numpy())
    assert r.q.dtype == torch.bfloat16 and r.g.dtype == torch.float32


def _mutant_runs(u, variant):
    """Deliberately wrong variants of the rule, to check the pins bite."""
    S = u.S0.copy()
    outs, cks = [], []
    for t in range(u.q.shape[0]):
        a, b, k, v, q = np.exp(u.g[t]), u.beta[t], u.k[t], u.v[t], u.q[t]
        if variant == "no_decay_in_prediction":
            S = a * S + b * np.outer(v - S @ k, k)
        elif variant == "transposed_state":
            S = a * S + b * np.outer(v - a * (S.T @ k)[: len(v)], k)
        elif variant == "output_before_update":
            o = S @ q
            S = a * S + b * np.outer(v - a * S @ k, k)
            outs.append(o)
            cks.append(S.copy())
            continue
        elif variant == "no_beta":
            S = a * S + np.outer(v - a * S @ k, k)
        outs.append(S @ q)
        cks.append(S.copy())
    return S, np.array(outs), np.array(cks)


@pytest.mark.parametrize("variant", ["no_decay_in_prediction", "transposed_state",
                                     "output_before_update", "no_beta"])
def test_pins_catch_planted_mistakes(variant):
    """Each mutant disagrees with the dense product form or a closed form."""
    u = _rand_unit(4, 16, 16, s0_std=1.0)
    S2, o2, _ = dense_product_form(u)
    Sm, om, _ = _mutant_runs(u, variant)
    assert not (np.allclose(Sm, S2, rtol=1e-9) and np.allclose(om, o2, rtol=1e-9))

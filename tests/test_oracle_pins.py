"""Pins for the CPU oracle, against things other than the oracle itself.

The pages print no worked KDA example, so the oracle is pinned by:
brute-force matrix products of the recurrence's matrix form, the product
(closed) form of the state, the chunked (WY/UT) form reaching the same
result, the delta-rule invariant, closed-form special cases, a norm bound,
varlen/continuation structure, linearity, and a small example worked by hand.
Each check is chosen so that a dropped term, a wrong sign or index, or a
transposed operand in the oracle fails at least one of them.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def rand_problem(T, H, K, V, *, g_scale=0.3, s0=False, unit_k=True, seed=0):
    r = np.random.default_rng(seed)
    q = r.standard_normal((T, H, K))
    k = r.standard_normal((T, H, K))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.standard_normal((T, H, V))
    g = -g_scale * np.abs(r.standard_normal((T, H, K)))
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal((T, H))))
    S0 = r.standard_normal((1, H, K, V)) * 0.3 if s0 else None
    return q, k, v, g, beta, S0


def brute_force(q, k, v, g, beta, S0, scale=1.0):
    """The recurrence in its matrix form, one explicit K x K matrix per step."""
    T, H, K = q.shape
    V = v.shape[-1]
    o = np.zeros((T, H, V))
    S_all = np.zeros((H, K, V))
    for h in range(H):
        S = np.zeros((K, V)) if S0 is None else S0[0, h].copy()
        for t in range(T):
            M = (np.eye(K) - beta[t, h] * np.outer(k[t, h], k[t, h])) @ np.diag(np.exp(g[t, h]))
            S = M @ S + beta[t, h] * np.outer(k[t, h], v[t, h])
            o[t, h] = S.T @ (scale * q[t, h])
        S_all[h] = S
    return o, S_all


def rel(a, b):
    return np.linalg.norm(np.asarray(a) - np.asarray(b)) / max(np.linalg.norm(b), 1e-300)


# --- worked example -------------------------------------------------------------

def test_handworked_two_token_example():
    ex = json.load(open(os.path.join(GOLDEN, "handworked_d2.json")))
    q = np.array(ex["q"])[:, None, :]
    k = np.array(ex["k"])[:, None, :]
    v = np.array(ex["v"])[:, None, :]
    g = np.array(ex["g"])[:, None, :]
    beta = np.array(ex["beta"])[:, None]
    o, S = oracle.recurrent(q, k, v, g, beta)
    np.testing.assert_allclose(o[:, 0, :], np.array(ex["o"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(S[0, 0], np.array(ex["final_state"]), rtol=0, atol=1e-14)


# --- brute force and the product form ---------------------------------------------

@pytest.mark.parametrize("K,V,T,scale", [(4, 3, 9, 1.0), (8, 8, 17, 0.5), (16, 16, 64, 0.25)])
def test_recurrent_matches_matrix_form(K, V, T, scale):
    q, k, v, g, beta, S0 = rand_problem(T, 2, K, V, s0=True, seed=K + T)
    o_ref, S_ref = brute_force(q, k, v, g, beta, S0, scale)
    o, S = oracle.recurrent(q, k, v, g, beta, scale=scale, initial_state=S0)
    assert rel(o, o_ref) < 1e-12
    assert rel(S[0], S_ref) < 1e-12


def test_final_state_matches_product_form():
    """S_T = (M_T...M_1) S_0 + sum_s (M_T...M_{s+1}) beta_s k_s v_s^T."""
    T, K, V = 12, 6, 5
    q, k, v, g, beta, S0 = rand_problem(T, 1, K, V, s0=True, seed=7)
    Ms = [(np.eye(K) - beta[t, 0] * np.outer(k[t, 0], k[t, 0])) @ np.diag(np.exp(g[t, 0]))
          for t in range(T)]

    def prod(a, b):  # M_b ... M_a (b >= a), identity when empty
        P = np.eye(K)
        for t in range(a, b + 1):
            P = Ms[t] @ P
        return P

    closed = prod(0, T - 1) @ S0[0, 0]
    for s in range(T):
        closed = closed + prod(s + 1, T - 1) @ (beta[s, 0] * np.outer(k[s, 0], v[s, 0]))
    _, S = oracle.recurrent(q, k, v, g, beta, initial_state=S0)
    assert rel(S[0, 0], closed) < 1e-12


# --- chunked form -------------------------------------------------------------------

@pytest.mark.parametrize("chunk,frame,T", [(16, 16, 64), (16, 4, 50), (64, 16, 200), (64, 64, 131),
                                           (8, 8, 1), (64, 16, 64)])
def test_chunked_form_matches_recurrence(chunk, frame, T):
    q, k, v, g, beta, S0 = rand_problem(T, 2, 16, 12, s0=True, seed=T + chunk)
    o_ref, S_ref = oracle.recurrent(q, k, v, g, beta, scale=0.7, initial_state=S0)
    o, S = oracle.chunked(q, k, v, g, beta, scale=0.7, initial_state=S0, chunk=chunk, frame=frame)
    assert rel(o, o_ref) < 1e-10
    assert rel(S, S_ref) < 1e-10


def test_chunked_form_varlen_matches_recurrence():
    lens = [5, 64, 0, 70, 17]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(cu[-1])
    q, k, v, g, beta, _ = rand_problem(N, 3, 16, 16, seed=3)
    S0 = np.random.default_rng(5).standard_normal((len(lens), 3, 16, 16)) * 0.2
    o_ref, S_ref = oracle.recurrent(q, k, v, g, beta, cu_seqlens=cu, initial_state=S0)
    o, S = oracle.chunked(q, k, v, g, beta, cu_seqlens=cu, initial_state=S0, chunk=16, frame=8)
    assert rel(o, o_ref) < 1e-10
    assert rel(S, S_ref) < 1e-10


# --- delta-rule invariant and closed forms ---------------------------------------------

def test_delta_rule_invariant():
    """g = 0, beta = 1, |k| = 1: after each step S_t^T k_t = v_t (read via q_t = k_t)."""
    T, K, V = 40, 16, 16
    _, k, v, _, _, S0 = rand_problem(T, 2, K, V, s0=True, seed=11)
    g = np.zeros((T, 2, K))
    beta = np.ones((T, 2))
    o, _ = oracle.recurrent(k, k, v, g, beta, initial_state=S0)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-12)


def test_beta_zero_is_pure_decay():
    T, K, V = 20, 8, 6
    q, k, v, g, _, S0 = rand_problem(T, 2, K, V, s0=True, seed=13)
    beta = np.zeros((T, 2))
    o, S = oracle.recurrent(q, k, v, g, beta, initial_state=S0)
    Gam = np.cumsum(g, axis=0)  # [T,H,K]
    for h in range(2):
        np.testing.assert_allclose(S[0, h], np.exp(Gam[-1, h])[:, None] * S0[0, h], rtol=1e-13)
        for t in range(T):
            St = np.exp(Gam[t, h])[:, None] * S0[0, h]
            np.testing.assert_allclose(o[t, h], St.T @ q[t, h], rtol=1e-12, atol=1e-14)


def test_basis_keys_write_rows():
    """g = 0, beta = 1, k_t = e_t, S_0 = 0: row t of S_T is v_t."""
    K = V = 8
    T = K
    k = np.zeros((T, 1, K))
    for t in range(T):
        k[t, 0, t] = 1.0
    v = rng.standard_normal((T, 1, V))
    q = rng.standard_normal((T, 1, K))
    o, S = oracle.recurrent(q, k, v, np.zeros((T, 1, K)), np.ones((T, 1)))
    np.testing.assert_array_equal(S[0, 0], v[:, 0, :])


def test_frozen_state():
    """g = 0, beta = 0: S is constant and o_t = S_0^T q_t."""
    q, k, v, _, _, S0 = rand_problem(10, 2, 8, 8, s0=True, seed=17)
    o, S = oracle.recurrent(q, k, v, np.zeros_like(q), np.zeros((10, 2)), initial_state=S0)
    np.testing.assert_array_equal(S, S0)
    np.testing.assert_allclose(o, np.einsum("hkv,thk->thv", S0[0], q), rtol=1e-13)


def test_frobenius_norm_bound():
    """beta in [0,1], |k| <= 1, g <= 0 make the step non-expansive:
    |S_t|_F <= |S_{t-1}|_F + beta_t |k_t| |v_t|."""
    T, K, V = 60, 16, 16
    q, k, v, g, beta, S0 = rand_problem(T, 1, K, V, s0=True, seed=19, g_scale=0.05)
    k *= rng.uniform(0.2, 1.0, (T, 1, 1))
    S = S0
    for t in range(T):
        _, S1 = oracle.decode(q[t][None], k[t][None], v[t][None], g[t][None], beta[t][None], S)
        bound = np.linalg.norm(S) + beta[t, 0] * np.linalg.norm(k[t, 0]) * np.linalg.norm(v[t, 0])
        assert np.linalg.norm(S1) <= bound * (1 + 1e-12)
        S = S1


def test_raw_logit_beta_can_diverge_but_sigmoid_beta_cannot():
    """With raw logits as beta (> 2) the step is expansive; the norm bound is
    exactly what the beta-sigmoid requirement protects."""
    T, K, V = 200, 8, 8
    q, k, v, _, _, _ = rand_problem(T, 1, K, V, seed=23)
    g = np.zeros((T, 1, K))
    o_bad, S_bad = oracle.recurrent(q, k, v, g, np.full((T, 1), 3.5))
    o_ok, S_ok = oracle.recurrent(q, k, v, g, 1 / (1 + np.exp(-np.full((T, 1), 3.5))))
    assert np.linalg.norm(S_bad) > 1e6 * np.linalg.norm(S_ok)


# --- structure ------------------------------------------------------------------------

def test_varlen_is_concatenation():
    lens = [7, 0, 13, 1, 30]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(cu[-1])
    q, k, v, g, beta, _ = rand_problem(N, 2, 8, 8, seed=29)
    S0 = rng.standard_normal((len(lens), 2, 8, 8))
    o, S = oracle.recurrent(q, k, v, g, beta, cu_seqlens=cu, initial_state=S0)
    for i in range(len(lens)):
        a, b = cu[i], cu[i + 1]
        oi, Si = oracle.recurrent(q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b],
                                  initial_state=S0[i:i + 1])
        np.testing.assert_array_equal(o[a:b], oi)
        np.testing.assert_array_equal(S[i], Si[0])
    np.testing.assert_array_equal(S[1], S0[1])  # empty sequence: final = initial


def test_continuation_equals_one_long_run():
    T1, T2 = 23, 41
    q, k, v, g, beta, S0 = rand_problem(T1 + T2, 2, 8, 8, s0=True, seed=31)
    o, S = oracle.recurrent(q, k, v, g, beta, initial_state=S0)
    o1, S1 = oracle.recurrent(q[:T1], k[:T1], v[:T1], g[:T1], beta[:T1], initial_state=S0)
    o2, S2 = oracle.recurrent(q[T1:], k[T1:], v[T1:], g[T1:], beta[T1:], initial_state=S1)
    np.testing.assert_allclose(np.concatenate([o1, o2]), o, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(S2, S, rtol=1e-13, atol=1e-15)


def test_linearity_in_values_and_state():
    q, k, v1, g, beta, S01 = rand_problem(25, 2, 8, 8, s0=True, seed=37)
    _, _, v2, _, _, S02 = rand_problem(25, 2, 8, 8, s0=True, seed=41)
    o1, S1 = oracle.recurrent(q, k, v1, g, beta, initial_state=S01)
    o2, S2 = oracle.recurrent(q, k, v2, g, beta, initial_state=S02)
    o3, S3 = oracle.recurrent(q, k, v1 - 2 * v2, g, beta, initial_state=S01 - 2 * S02)
    np.testing.assert_allclose(o3, o1 - 2 * o2, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(S3, S1 - 2 * S2, rtol=1e-11, atol=1e-12)


def test_tiny_config_runs_and_agrees_with_chunked():
    from gated_delta_rule_33_gb300 import synth
    x = synth.tiny_config()
    g, beta = oracle.gate(x.f.numpy(), x.b.numpy(), x.A_log.numpy(), x.dt_bias.numpy(), x.alog_mode)
    args = (x.q.double().numpy(), x.k.double().numpy(), x.v.double().numpy(), g, beta)
    o, S = oracle.recurrent(*args)
    oc, Sc = oracle.chunked(*args, chunk=16, frame=16)
    assert np.isfinite(o).all() and np.isfinite(S).all()
    assert rel(oc, o) < 1e-12 and rel(Sc, S) < 1e-12

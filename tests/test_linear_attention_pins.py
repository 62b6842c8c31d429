"""Pins of the fp64 gated delta-rule oracle to facts outside itself (CPU only): closed forms,
the delta rule's exact-retrieval property, an unrolled matrix-product form of the state,
finite differences of the backward, and planted mistakes that one of these catches."""

import math

import numpy as np
import pytest

from oracle import linear_attention as LA


def _rand(seed, B=1, T=7, H=2, dk=4, dv=3):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, H, dk))
    k = rng.standard_normal((B, T, H, dk))
    v = rng.standard_normal((B, T, H, dv))
    beta = rng.uniform(0.05, 0.95, (B, T, H))
    g = -rng.uniform(0.0, 0.5, (B, T, H))
    return q, k, v, beta, g


def check_zero_write_strength():
    q, k, v, beta, g = _rand(1)
    o, S = LA.gated_delta_rule(q, k, v, 0 * beta, g)
    assert np.abs(o).max() == 0 and np.abs(S).max() == 0


def check_single_token_closed_form():
    # from a zero state: S_1 = beta v k^T / ||k||, o_1 = scale beta v (k . q) / (||k|| ||q||)
    q = np.array([[[[1.0, 2.0, 2.0, 0.0]]]])         # ||q|| = 3
    k = np.array([[[[0.0, 3.0, 0.0, 4.0]]]])         # ||k|| = 5
    v = np.array([[[[1.0, -2.0, 0.5]]]])
    beta = np.array([[[0.25]]])
    g = np.array([[[-0.3]]])
    o, S = LA.gated_delta_rule(q, k, v, beta, g)
    kq = (0 * 1 + 3 * 2 + 0 * 2 + 4 * 0) / (5 * 3)
    assert np.allclose(o[0, 0, 0], 0.5 * 0.25 * kq * np.array([1.0, -2.0, 0.5]), rtol=1e-14)
    assert np.allclose(S[0, 0], 0.25 * np.outer([1.0, -2.0, 0.5], [0, 0.6, 0, 0.8]), rtol=1e-14)


def check_full_strength_write_is_retrieved():
    # after any history, a step with beta = 1 makes S_t k^_t = v_t exactly, so querying
    # with the key just written returns scale * v_t (whatever the decay)
    q, k, v, beta, g = _rand(2, T=9)
    beta[:, 6] = 1.0
    q[:, 6] = 2.5 * k[:, 6]
    o, _ = LA.gated_delta_rule(q, k, v, beta, g)
    assert np.allclose(o[:, 6], 0.5 * v[:, 6], rtol=1e-12, atol=1e-12)


def check_orthonormal_keys_store_every_value():
    # keys e_0, e_1, e_2, e_3 (distinct basis vectors), no decay, beta = 1: each write leaves
    # the others untouched, so querying key s after all writes returns v_s
    T, dk, dv = 4, 4, 3
    rng = np.random.default_rng(3)
    k = np.eye(dk)[None, :, None, :]
    v = rng.standard_normal((1, T, 1, dv))
    q = k.copy()
    o, S = LA.gated_delta_rule(q, k, v, np.ones((1, T, 1)), np.zeros((1, T, 1)))
    assert np.allclose(S[0, 0], v[0, :, 0].T, rtol=1e-14)
    assert np.allclose(o[0, :, 0], 0.5 * v[0, :, 0], rtol=1e-14)


def check_decay_only():
    q, k, v, beta, g = _rand(4, T=6)
    rng = np.random.default_rng(5)
    S0 = rng.standard_normal((1, 2, 3, 4))
    o, S = LA.gated_delta_rule(q, k, v, 0 * beta, g, S0=S0)
    for h in range(2):
        assert np.allclose(S[0, h], math.exp(g[0, :, h].sum()) * S0[0, h], rtol=1e-13)
        qh = q[0, 3, h] / np.linalg.norm(q[0, 3, h])
        assert np.allclose(o[0, 3, h], 0.5 * math.exp(g[0, :4, h].sum()) * S0[0, h] @ qh,
                           rtol=1e-13)


def check_unrolled_product_form():
    # S_t = S_{t-1} M_t + beta_t v_t k^_t^T with M_t = alpha_t (I - beta_t k^_t k^_t^T), so
    # S_T = S_0 M_1 ... M_T + sum_t beta_t v_t k^_t^T M_{t+1} ... M_T
    q, k, v, beta, g = _rand(6, T=6, H=1, dv=4)
    rng = np.random.default_rng(7)
    S0 = rng.standard_normal((1, 1, 4, 4))
    _, S = LA.gated_delta_rule(q, k, v, beta, g, S0=S0)
    kh = k[0, :, 0] / np.linalg.norm(k[0, :, 0], axis=1, keepdims=True)
    M = [math.exp(g[0, t, 0]) * (np.eye(4) - beta[0, t, 0] * np.outer(kh[t], kh[t]))
         for t in range(6)]
    prod = lambda a, b: np.linalg.multi_dot([np.eye(4)] + M[a:b] + [np.eye(4)])
    ref = S0[0, 0] @ prod(0, 6)
    for t in range(6):
        ref = ref + beta[0, t, 0] * np.outer(v[0, t, 0], kh[t]) @ prod(t + 1, 6)
    assert np.allclose(S[0, 0], ref, rtol=1e-12)


def test_zero_write_strength():
    check_zero_write_strength()


def test_single_token_closed_form():
    check_single_token_closed_form()


def test_full_strength_write_is_retrieved():
    check_full_strength_write_is_retrieved()


def test_orthonormal_keys_store_every_value():
    check_orthonormal_keys_store_every_value()


def test_decay_only():
    check_decay_only()


def test_unrolled_product_form():
    check_unrolled_product_form()


# ---------------------------------------------------------------- backward

def _loss(q, k, v, beta, g, S0, do, dST):
    o, S = LA.gated_delta_rule(q, k, v, beta, g, S0=S0)
    return float(np.sum(o * do) + np.sum(S * dST))


def check_backward_finite_differences():
    q, k, v, beta, g = _rand(8, T=5)
    rng = np.random.default_rng(9)
    S0 = rng.standard_normal((1, 2, 3, 4))
    do = rng.standard_normal((1, 5, 2, 3))
    dST = rng.standard_normal((1, 2, 3, 4))
    G = LA.gated_delta_rule_backward(q, k, v, beta, g, do, dS_T=dST, S0=S0)
    args = dict(q=q, k=k, v=v, beta=beta, g=g, S0=S0)
    names = {"q": "dq", "k": "dk", "v": "dv", "beta": "dbeta", "g": "dg", "S0": "dS0"}
    eps = 1e-6
    for name, gname in names.items():
        x = args[name]
        num = np.zeros_like(x)
        for i in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[i] += eps
            xm[i] -= eps
            ap, am = dict(args), dict(args)
            ap[name], am[name] = xp, xm
            num[i] = (_loss(**ap, do=do, dST=dST) - _loss(**am, do=do, dST=dST)) / (2 * eps)
        err = np.linalg.norm(G[gname] - num) / np.linalg.norm(num)
        assert err < 1e-7, (name, err)


def test_backward_finite_differences():
    check_backward_finite_differences()


# ---------------------------------------------------------------- planted mistakes

def _expect_failure(check):
    with pytest.raises(AssertionError):
        check()


def _recurrence(update):
    """A forward that applies ``update(S, alpha, beta, k^, v)`` per token (planted mistakes)."""
    def fwd(q, k, v, beta, g, S0=None, scale=None):
        q, k, v, beta, g = (np.asarray(a, float) for a in (q, k, v, beta, g))
        B, T, H, dk = q.shape
        scale = dk ** -0.5 if scale is None else scale
        qh = q / np.linalg.norm(q, axis=-1, keepdims=True)
        kh = k / np.linalg.norm(k, axis=-1, keepdims=True)
        o = np.zeros(v.shape)
        Sout = np.zeros((B, H, v.shape[-1], dk))
        for b in range(B):
            for h in range(H):
                S = np.zeros((v.shape[-1], dk)) if S0 is None else np.array(S0[b, h], float)
                for t in range(T):
                    S = update(S, math.exp(g[b, t, h]), beta[b, t, h], kh[b, t, h], v[b, t, h])
                    o[b, t, h] = scale * (S @ qh[b, t, h])
                Sout[b, h] = S
        return o, Sout
    return fwd


def test_mutation_update_on_the_wrong_side_caught(monkeypatch):
    # the projection (I - beta k k^T) applied from the left instead of the right (square
    # state, dk = dv, so that the wrong form can be computed at all)
    def left(S, a, b, kt, vt):
        return a * (np.eye(len(kt)) - b * np.outer(kt, kt)) @ S + b * np.outer(vt, kt)
    monkeypatch.setattr(LA, "gated_delta_rule", _recurrence(left))
    _expect_failure(check_unrolled_product_form)


def test_mutation_decay_after_delta_caught(monkeypatch):
    # the delta computed against the undecayed state: S_t = alpha S + beta (v - S k) k^T
    def late(S, a, b, kt, vt):
        return a * S + b * np.outer(vt - S @ kt, kt)
    monkeypatch.setattr(LA, "gated_delta_rule", _recurrence(late))
    _expect_failure(check_full_strength_write_is_retrieved)


def test_mutation_unnormalised_keys_caught(monkeypatch):
    orig = LA._normalize
    monkeypatch.setattr(LA, "_normalize", lambda x: (x, np.ones(x.shape[:-1] + (1,))))
    _expect_failure(check_single_token_closed_form)


def test_mutation_backward_dropped_term_caught(monkeypatch):
    orig = LA.gated_delta_rule_backward

    def wrong(*a, **kw):
        G = orig(*a, **kw)
        G["dk"] = G["dk"] * 0.9
        return G
    monkeypatch.setattr(LA, "gated_delta_rule_backward", wrong)
    _expect_failure(check_backward_finite_differences)

"""fp64 reference of the gated delta-rule linear attention (test infrastructure only).

"Fine-Tuning Trillion-Parameter Sparse MoE Models: Challenges and Engineering Practices",
section 5 ("large forward fusion": normalization coefficients, gating and decay, intra-chunk
query-state interaction and output transformation in one kernel; chunked computation with
one small state recurrence between chunks; backward organised by chunk) and its chunked-
recurrence listing (per chunk: gating/decay coefficients and beta, query-state interaction,
then a delta update of the fixed-size state); "Adapting Ultra-Large MoE Models: Engineering
Practices and Optimization Pathways", section 3.2 (state recursion and chunked computation
fused into large forward and backward kernels).

The pages name the pieces but give no equations.  Reading taken (the plainest one the pieces
support): the gated delta rule, per sequence and head,

    q^_t = q_t / ||q_t||,  k^_t = k_t / ||k_t||          (L2 over the key width dk)
    alpha_t = exp(g_t)  (g_t <= 0: decay),  beta_t in (0, 1)  (write strength)
    S_t = alpha_t S_{t-1} (I - beta_t k^_t k^_t^T) + beta_t v_t k^_t^T       S_t: [dv, dk]
        = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k^_t) k^_t^T
    o_t = scale * S_t q^_t,  scale = dk^-1/2,  S_0 given (zero by default)

The oracle is that recurrence written out, one token at a time; the chunked evaluation is
the CUDA kernel's business.  Shapes: q, k [B, T, H, dk]; v [B, T, H, dv]; beta, g [B, T, H];
S0 [B, H, dv, dk].  Returns o [B, T, H, dv] and the final state S_T [B, H, dv, dk].
"""

from __future__ import annotations

import numpy as np

__all__ = ["gated_delta_rule", "gated_delta_rule_backward"]


def _f64(a):
    return None if a is None else np.asarray(a, dtype=np.float64)


def _normalize(x):
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return x / n, n


def gated_delta_rule(q, k, v, beta, g, S0=None, scale=None):
    q, k, v, beta, g = (_f64(a) for a in (q, k, v, beta, g))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    scale = dk ** -0.5 if scale is None else scale
    qh, _ = _normalize(q)
    kh, _ = _normalize(k)
    o = np.zeros((B, T, H, dv))
    S_out = np.zeros((B, H, dv, dk))
    for b in range(B):
        for h in range(H):
            S = np.zeros((dv, dk)) if S0 is None else _f64(S0)[b, h].copy()
            for t in range(T):
                a = np.exp(g[b, t, h])
                kt = kh[b, t, h]
                S = a * S
                S = S + beta[b, t, h] * np.outer(v[b, t, h] - S @ kt, kt)
                o[b, t, h] = scale * (S @ qh[b, t, h])
            S_out[b, h] = S
    return o, S_out


def gated_delta_rule_backward(q, k, v, beta, g, do, dS_T=None, S0=None, scale=None):
    """Gradients of <do, o> + <dS_T, S_T> with respect to q, k, v, beta, g and S0, by the
    reverse recurrence (reverse-mode differentiation of the forward above, derived by hand):
    with P_t = S_t after step t, the state gradient D_t = dL/dS_t flows backwards as
        D_t += scale do_t q^_t^T                       (from o_t = scale S_t q^_t)
        S_t = A_t + beta_t (v_t - A_t k^_t) k^_t^T,    A_t = alpha_t S_{t-1}
        dA_t = D_t (I - beta_t k^_t k^_t^T)            dv_t = beta_t D_t k^_t
        dbeta_t = <D_t, (v_t - A_t k^_t) k^_t^T>
        dk^_t = beta_t (D_t^T (v_t - A_t k^_t) - A_t^T D_t k^_t)
        D_{t-1} = alpha_t dA_t,  dg_t = alpha_t <dA_t, S_{t-1}>
    and the normalizations back-propagated: dx = (dx^ - x^ <dx^, x^>) / ||x||."""
    q, k, v, beta, g, do = (_f64(a) for a in (q, k, v, beta, g, do))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    scale = dk ** -0.5 if scale is None else scale
    qh, qn = _normalize(q)
    kh, kn = _normalize(k)
    dq = np.zeros_like(q)
    dk_ = np.zeros_like(k)
    dv_ = np.zeros_like(v)
    dbeta = np.zeros_like(beta)
    dg = np.zeros_like(g)
    dS0 = np.zeros((B, H, dv, dk))
    for b in range(B):
        for h in range(H):
            S = np.zeros((dv, dk)) if S0 is None else _f64(S0)[b, h].copy()
            states = [S]
            for t in range(T):
                a = np.exp(g[b, t, h])
                kt = kh[b, t, h]
                A = a * S
                S = A + beta[b, t, h] * np.outer(v[b, t, h] - A @ kt, kt)
                states.append(S)
            D = np.zeros((dv, dk)) if dS_T is None else _f64(dS_T)[b, h].copy()
            for t in range(T - 1, -1, -1):
                a = np.exp(g[b, t, h])
                kt, qt = kh[b, t, h], qh[b, t, h]
                St, Sprev = states[t + 1], states[t]
                A = a * Sprev
                bt = beta[b, t, h]
                D = D + scale * np.outer(do[b, t, h], qt)
                dqh = scale * St.T @ do[b, t, h]
                r = v[b, t, h] - A @ kt                 # the delta written this step
                dv_[b, t, h] = bt * D @ kt
                dbeta[b, t, h] = np.sum(D * np.outer(r, kt))
                dkh = bt * (D.T @ r - A.T @ (D @ kt))
                dA = D - bt * np.outer(D @ kt, kt)
                dg[b, t, h] = a * np.sum(dA * Sprev)
                D = a * dA
                dq[b, t, h] = (dqh - qt * (dqh @ qt)) / qn[b, t, h]
                dk_[b, t, h] = (dkh - kt * (dkh @ kt)) / kn[b, t, h]
            dS0[b, h] = D
    return dict(dq=dq, dk=dk_, dv=dv_, dbeta=dbeta, dg=dg, dS0=dS0)

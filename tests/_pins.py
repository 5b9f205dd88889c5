"""Pins for a KDA forward implementation, independent of the oracle's code.

Each pin builds a small fp64 case whose answer follows from the recurrence by
a different route (a closed form, a special case that reduces to textbook
linear algebra, an invariant) and checks an implementation ``fwd_unit``
against it.  ``fwd_unit(q, k, v, g, beta, s0) -> (o [T,dv], S_T [dk,dv])``
works on one (sequence, head).  Each pin returns (passed, error).

The gate used to build expected values is written here on its own, from
the textbook definition softplus(x) = log(1 + e^x) = logaddexp(0, x).
"""
from __future__ import annotations

import numpy as np

FLOOR = -5.0


def gate(x):
    return np.maximum(-np.logaddexp(0.0, np.asarray(x, dtype=np.float64)), FLOOR)


def _unit(rng, n, d):
    x = rng.standard_normal((n, d))
    return x / np.linalg.norm(x, axis=1, keepdims=True)


def _rel(a, b):
    den = max(np.max(np.abs(b)), 1e-300)
    return float(np.max(np.abs(np.asarray(a) - np.asarray(b))) / den)


def p1_retrieval(fwd_unit, seed=11, T=40, dk=8, dv=6):
    """beta_t = 1 and q_t = k_t with |k_t| = 1 give o_t = v_t exactly:
    k^T (I - k k^T) = 0, so S_t^T k_t = v_t whatever the history."""
    rng = np.random.default_rng(seed)
    q = _unit(rng, T, dk); k = _unit(rng, T, dk)
    v = rng.standard_normal((T, dv)); g = rng.standard_normal((T, dk)) * 2
    beta = rng.uniform(0.05, 0.95, T)
    s0 = rng.standard_normal((dk, dv))
    probe = np.arange(3, T, 5)
    beta[probe] = 1.0
    q[probe] = k[probe]
    o, _ = fwd_unit(q, k, v, g, beta, s0)
    err = _rel(o[probe], v[probe])
    return err < 1e-12, err


def p2_beta_zero(fwd_unit, seed=12, T=33, dk=7, dv=5):
    """beta = 0 freezes the write path: S_t = Diag(gamma_t) S0 with
    gamma_t = exp(sum_{s<=t} a_s), so o_t = S0^T (gamma_t * q_t); with
    alpha = 1 this is the plain product Q S0."""
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, dk)); k = _unit(rng, T, dk)
    v = rng.standard_normal((T, dv)); g = rng.standard_normal((T, dk)) * 3
    s0 = rng.standard_normal((dk, dv)); beta = np.zeros(T)
    o, S = fwd_unit(q, k, v, g, beta, s0)
    gam = np.exp(np.cumsum(gate(g), axis=0))
    e1 = max(_rel(o, (q * gam) @ s0), _rel(S, gam[-1][:, None] * s0))
    g1 = np.full((T, dk), -200.0)
    o1, S1 = fwd_unit(q, k, v, g1, beta, s0)
    e2 = max(_rel(o1, q @ s0), _rel(S1, s0))
    err = max(e1, e2)
    return err < 1e-12, err


def p3_deltanet(fwd_unit, seed=13, T=12, dk=6, dv=5):
    """alpha = 1 (x = -200) is DeltaNet; compare with explicit dk x dk
    transition matrices A_t = I - beta k k^T applied by matrix products."""
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, dk)); k = _unit(rng, T, dk)
    v = rng.standard_normal((T, dv)); beta = rng.uniform(0, 1, T)
    g = np.full((T, dk), -200.0); s0 = rng.standard_normal((dk, dv))
    S = s0.copy(); ref = np.zeros((T, dv))
    for t in range(T):
        A = np.eye(dk) - beta[t] * np.outer(k[t], k[t])
        S = A @ S + beta[t] * np.outer(k[t], v[t])
        ref[t] = S.T @ q[t]
    o, ST = fwd_unit(q, k, v, g, beta, s0)
    err = max(_rel(o, ref), _rel(ST, S))
    return err < 1e-12, err


def p4_orthonormal_keys(fwd_unit, seed=14, dk=10, dv=4):
    """Distinct basis keys k_t = e_{pi(t)}, S0 = 0: nothing is ever read back
    (p_t = 0), so the state is gated linear attention with beta-weighted
    values: o_t = sum_{i<=t} beta_i q_t[pi_i] e^{G_t[pi_i]-G_i[pi_i]} v_i."""
    rng = np.random.default_rng(seed)
    T = dk
    pi = rng.permutation(dk)
    k = np.eye(dk)[pi]
    q = rng.standard_normal((T, dk)); v = rng.standard_normal((T, dv))
    g = rng.standard_normal((T, dk)) * 2; beta = rng.uniform(0.1, 1, T)
    G = np.cumsum(gate(g), axis=0)
    ref = np.zeros((T, dv))
    for t in range(T):
        for i in range(t + 1):
            c = pi[i]
            ref[t] += beta[i] * q[t, c] * np.exp(G[t, c] - G[i, c]) * v[i]
    o, _ = fwd_unit(q, k, v, g, beta, np.zeros((dk, dv)))
    err = _rel(o, ref)
    return err < 1e-12, err


def p5_repeated_key(fwd_unit, seed=15, T=30, dk=6, dv=4, j=2):
    """One basis key e_j at every step: row j follows the scalar EMA
    S_j <- (1 - beta) alpha_j S_j + beta v, every other row only decays."""
    rng = np.random.default_rng(seed)
    k = np.zeros((T, dk)); k[:, j] = 1.0
    q = rng.standard_normal((T, dk)); v = rng.standard_normal((T, dv))
    g = rng.standard_normal((T, dk)); beta = rng.uniform(0, 1, T)
    s0 = rng.standard_normal((dk, dv))
    al = np.exp(gate(g))
    S = s0.copy(); ref = np.zeros((T, dv))
    for t in range(T):
        for i in range(dk):
            if i == j:
                S[i] = (1 - beta[t]) * al[t, i] * S[i] + beta[t] * v[t]
            else:
                S[i] = al[t, i] * S[i]
        ref[t] = q[t] @ S
    o, ST = fwd_unit(q, k, v, g, beta, s0)
    err = max(_rel(o, ref), _rel(ST, S))
    return err < 1e-12, err


def p6_small_beta(fwd_unit, seed=16, T=20, dk=8, dv=5, eps=1e-6):
    """S0 = 0, beta = eps: o/eps -> sum_{i<=t} (q_t . (e^{G_t-G_i} * k_i)) v_i
    (gated linear attention) with relative error O(eps); with alpha = 1
    the limit is causal linear attention tril(Q K^T) V."""
    rng = np.random.default_rng(seed)
    q = _unit(rng, T, dk); k = _unit(rng, T, dk); v = rng.standard_normal((T, dv))
    g = rng.standard_normal((T, dk)); beta = np.full(T, eps)
    G = np.cumsum(gate(g), axis=0)
    gla = np.zeros((T, dv))
    for t in range(T):
        for i in range(t + 1):
            gla[t] += (q[t] * np.exp(G[t] - G[i]) * k[i]).sum() * v[i]
    o, _ = fwd_unit(q, k, v, g, beta, np.zeros((dk, dv)))
    e1 = _rel(o / eps, gla)
    o2, _ = fwd_unit(q, k, v, np.full((T, dk), -200.0), beta, np.zeros((dk, dv)))
    e2 = _rel(o2 / eps, np.tril(q @ k.T) @ v)
    err = max(e1, e2)
    return err < 1e-4, err


def p8_affine(fwd_unit, seed=18, T=25, dk=6):
    """For fixed q, k, beta, alpha the map (V, S0) -> (O, S_T) is linear:
    o(V,S0) = o(V,0) + o(0,S0), and S_T(0,S0) = P S0 with P = S_T(0, I)
    the segment's cumulative transition (dv = dk so I is a valid state)."""
    rng = np.random.default_rng(seed)
    dv = dk
    q = rng.standard_normal((T, dk)); k = _unit(rng, T, dk)
    v = rng.standard_normal((T, dv)); g = rng.standard_normal((T, dk))
    beta = rng.uniform(0, 1, T); s0 = rng.standard_normal((dk, dv))
    o, S = fwd_unit(q, k, v, g, beta, s0)
    oa, Sa = fwd_unit(q, k, v, g, beta, np.zeros((dk, dv)))
    ob, Sb = fwd_unit(q, k, np.zeros_like(v), g, beta, s0)
    _, P = fwd_unit(q, k, np.zeros_like(v), g, beta, np.eye(dk))
    err = max(_rel(o, oa + ob), _rel(S, Sa + Sb), _rel(Sb, P @ s0))
    return err < 1e-12, err


def p10_split(fwd_unit, seed=20, T=150, dk=8, dv=6, cuts=(64, 77)):
    """Running [0, t0) then [t0, T) with the state handed over equals one run."""
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, dk)); k = _unit(rng, T, dk)
    v = rng.standard_normal((T, dv)); g = rng.standard_normal((T, dk)) * 2
    beta = rng.uniform(0, 1, T); s0 = rng.standard_normal((dk, dv))
    o, S = fwd_unit(q, k, v, g, beta, s0)
    err = 0.0
    for t0 in cuts:
        o1, S1 = fwd_unit(q[:t0], k[:t0], v[:t0], g[:t0], beta[:t0], s0)
        o2, S2 = fwd_unit(q[t0:], k[t0:], v[t0:], g[t0:], beta[t0:], S1)
        err = max(err, _rel(np.concatenate([o1, o2]), o), _rel(S2, S))
    return err < 1e-12, err


ALL = [p1_retrieval, p2_beta_zero, p3_deltanet, p4_orthonormal_keys, p5_repeated_key,
       p6_small_beta, p8_affine, p10_split]


def p11_scale(fwd_scaled, seed=21, T=18, dk=6, dv=5, s=0.37):
    """The q scale multiplies the read-out only: o_t = S_t^T (s q_t).  Checked
    against two routes that do not use the implementation's unscaled run:
    (a) DeltaNet (alpha = 1) by explicit dk x dk transition matrices, read out
    with s q_t; (b) the retrieval identity with beta = 1 and q = k, which gives
    o_t = s v_t.  The final state must not depend on s at all."""
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, dk)); k = _unit(rng, T, dk)
    v = rng.standard_normal((T, dv)); beta = rng.uniform(0, 1, T)
    g = np.full((T, dk), -200.0); s0 = rng.standard_normal((dk, dv))
    S = s0.copy(); ref = np.zeros((T, dv))
    for t in range(T):
        A = np.eye(dk) - beta[t] * np.outer(k[t], k[t])
        S = A @ S + beta[t] * np.outer(k[t], v[t])
        ref[t] = S.T @ (s * q[t])
    o, ST = fwd_scaled(q, k, v, g, beta, s0, s)
    e1 = max(_rel(o, ref), _rel(ST, S))
    # retrieval: beta = 1 and q = k at the probe steps, any gates
    g2 = rng.standard_normal((T, dk)) * 2
    beta2 = rng.uniform(0.05, 0.95, T)
    q2 = q.copy()
    probe = np.arange(2, T, 4)
    beta2[probe] = 1.0
    q2[probe] = k[probe]
    o2, S2 = fwd_scaled(q2, k, v, g2, beta2, s0, s)
    e2 = _rel(o2[probe], s * v[probe])
    _, S2u = fwd_scaled(q2, k, v, g2, beta2, s0, 1.0)
    e3 = _rel(S2, S2u)
    err = max(e1, e2, e3)
    return err < 1e-12, err

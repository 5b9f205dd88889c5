"""Chunkwise-parallel KDA forward in numpy fp64 -- TEST INFRASTRUCTURE.

A literal, step-by-step statement of the chunked form, used to pin the
chunked computation to the token loop (they must agree to rounding) and to
compare the GPU path's intermediate steps one by one.  Not blocked, fused or
reordered beyond the steps listed here.

Sources:
 * KDA can be rewritten in a chunk-parallel form and its decay logits pass
   through a negative-softplus map: Kimi K3 walkthrough (Towards AI,
   M. Zhao), section "Kimi Delta Attention (KDA)".
 * A chunked computation divides by the cumulative decay; the chunk is cut
   into 16-token tiles; with log-decay >= -5 per step the cumulative
   log-decay over one tile stays in (-80, 0], its inverse below
   e^80 ~ 5.5e34, so every tile of the intra-chunk matrices, diagonal ones
   included, is one dense product: Kimi K3 architecture (orkas.ai), section
   "A lower bound that erased a GPU code path".

Notation, for one chunk of C rows (0-based r, i), key channel j:
  a_r      = max(-softplus(x_r), -5)                       (per channel)
  Gam_r    = sum_{s <= r} a_s         (cumulative log-decay from chunk start)
  ref_tau  = Gam_{16 tau - 1}, 0 for tau = 0     (log-decay before tile tau)
  rows r of tile tau:      Qhat_r = q_r * e^{Gam_r - ref_tau}   in [e^-80, 1]
                           Khat_r = k_r * e^{Gam_r - ref_tau}
  columns i <= end of tau: Ktil_i = k_i * e^{ref_tau - Gam_i}   <= e^80
  A_qk[r,i] = Qhat_r . Ktil_i              (i <= r)
  A_kk[r,i] = beta_r Khat_r . Ktil_i       (i <  r)
  T  = (I + A_kk)^{-1}
  W  = T (beta * K * e^{Gam}),   U = T (beta * V)
  Delta = U - W S
  O  = (Q * e^{Gam}) S + A_qk Delta
  S <- e^{Gam_C} * S + (K * e^{Gam_C - Gam})^T Delta
A partial last chunk is padded with q = k = v = 0, beta = 0, a = 0.

Derivation from the recurrence S_t = (I - b k k^T) Diag(alpha) S + b k v^T:
with delta_t = b_t (v_t - (Diag(alpha_t) S_{t-1})^T k_t), unrolling the
chunk from its entry state S gives (I + A_kk) Delta = diag(b) V -
diag(b) (K*e^Gam) S, o_t = S^T(q_t*e^{Gam_t}) + sum_{i<=t} A_qk[t,i] delta_i
and the exit state above.
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular

TILE = 16
LOG_FLOOR = -5.0


def log_decay(x: np.ndarray) -> np.ndarray:
    """max(-softplus(x), -5), softplus in its overflow-free form."""
    x = np.asarray(x, dtype=np.float64)
    sp = np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))
    return np.maximum(-sp, LOG_FLOOR)


def chunk_step(Q, K, V, A, b, S, tile=TILE):
    """One chunk (already padded to C rows).  Returns (O, S_out, steps)."""
    C, dk = Q.shape
    Gam = np.cumsum(A, axis=0)
    ntile = (C + tile - 1) // tile
    Aqk = np.zeros((C, C))
    Akk = np.zeros((C, C))
    for tau in range(ntile):
        r0, r1 = tau * tile, min(C, (tau + 1) * tile)
        ref = Gam[r0 - 1] if r0 > 0 else np.zeros(dk)
        row_scale = np.exp(Gam[r0:r1] - ref)          # within [e^-80, 1]
        Qhat = Q[r0:r1] * row_scale
        Khat = K[r0:r1] * row_scale
        Ktil = K[:r1] * np.exp(ref - Gam[:r1])        # at most e^80
        Aqk[r0:r1, :r1] = Qhat @ Ktil.T
        Akk[r0:r1, :r1] = b[r0:r1, None] * (Khat @ Ktil.T)
    Aqk = np.tril(Aqk)
    Akk = np.tril(Akk, -1)
    I = np.eye(C)
    Tm = solve_triangular(I + Akk, I, lower=True, unit_diagonal=True)
    gam = np.exp(Gam)
    W = Tm @ (b[:, None] * K * gam)
    U = Tm @ (b[:, None] * V)
    Delta = U - W @ S
    O = (Q * gam) @ S + Aqk @ Delta
    gC = Gam[-1]
    S_out = np.exp(gC)[:, None] * S + (K * np.exp(gC - Gam)).T @ Delta
    steps = dict(Gam=Gam, Aqk=Aqk, Akk=Akk, T=Tm, W=W, U=U, Delta=Delta, S_in=S.copy())
    return O, S_out, steps


def forward_unit(q, k, v, g, beta, s0=None, chunk=64, tile=TILE, scale=1.0,
                 return_steps=False):
    """Chunked forward of one (sequence, head): q,k,g [T,dk], v [T,dv], beta [T]."""
    q = np.asarray(q, dtype=np.float64) * scale
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    A = log_decay(g)
    T, dk = q.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if s0 is None else np.array(s0, dtype=np.float64)
    out = np.zeros((T, dv))
    all_steps = []
    for c0 in range(0, T, chunk):
        L = min(chunk, T - c0)
        Qc = np.zeros((chunk, dk)); Qc[:L] = q[c0:c0 + L]
        Kc = np.zeros((chunk, dk)); Kc[:L] = k[c0:c0 + L]
        Vc = np.zeros((chunk, dv)); Vc[:L] = v[c0:c0 + L]
        Ac = np.zeros((chunk, dk)); Ac[:L] = A[c0:c0 + L]
        bc = np.zeros(chunk); bc[:L] = beta[c0:c0 + L]
        O, S, st = chunk_step(Qc, Kc, Vc, Ac, bc, S, tile)
        out[c0:c0 + L] = O[:L]
        if return_steps:
            all_steps.append(st)
    if return_steps:
        return out, S, all_steps
    return out, S


def forward(q, k, v, g, beta, init_state=None, cu_seqlens=None, chunk=64, tile=TILE,
            scale=1.0):
    """Batched chunked forward, same layouts as the C oracle's ``fwd``."""
    def f64(x):
        if x is None:
            return None
        if hasattr(x, "detach"):
            import torch
            return x.detach().cpu().to(torch.float64).numpy()
        return np.asarray(x, dtype=np.float64)
    q, k, v, g, beta, s0 = (f64(t) for t in (q, k, v, g, beta, init_state))
    rows, T, H, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is not None:
        cu = [int(c) for c in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist")
                               else cu_seqlens)]
        spans = [(0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]
    else:
        spans = [(n, 0, T) for n in range(rows)]
    out = np.zeros((rows, T, H, dv))
    fs = np.zeros((len(spans), H, dk, dv))
    for n, (row, t0, t1) in enumerate(spans):
        for h in range(H):
            o, S = forward_unit(q[row, t0:t1, h], k[row, t0:t1, h], v[row, t0:t1, h],
                                g[row, t0:t1, h], beta[row, t0:t1, h],
                                None if s0 is None else s0[n, h], chunk, tile, scale)
            out[row, t0:t1, h] = o
            fs[n, h] = S
    return out, fs

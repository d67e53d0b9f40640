"""Chunkwise form of the KDA recurrence, in plain float64 numpy.

TEST INFRASTRUCTURE.  It exists only to pin the chunk algebra that a parallel
implementation relies on ("Kimi K3, explained", section "Training in chunks"
and the question "How is KDA trained efficiently if it is a recurrence?":
inside a chunk the product of the per-token decay-and-erase matrices is
rewritten in the WY form, so most of the work becomes matrix products, and only
the state passes from one chunk to the next).  The oracle's tests check it
against the token-by-token recurrence of ``kda_oracle.c``; nothing in the CUDA
path imports it.

Derivation, per head, state S (d_k x d_v), chunk of L tokens r = 1..L that
starts from S_0:

* g_r = sum_{s<=r} log alpha_s (vector over d_k), Gamma_r = exp(g_r).
* By induction the state after token r is
      S_r = Diag(Gamma_r) S_0 + sum_{s<=r} Diag(Gamma_r / Gamma_s) k_s u_s^T
  with u_r = beta_r (v_r - (Diag(alpha_r) S_{r-1})^T k_r).
* Substituting S_{r-1} gives the unit lower triangular system
      (I + A) U = Diag(beta) V - Diag(beta) (Gamma . K) S_0,
      A_rs = beta_r sum_i k_ri k_si exp(g_ri - g_si)          (s < r),
  so U = Utilde - W S_0 with T = (I + A)^-1, W = T Diag(beta) (Gamma . K),
  Utilde = T Diag(beta) V  (the WY / UT form).
* Outputs:  O = (Gamma . Q) S_0 + P U,
      P_rs = sum_i q_ri k_si exp(g_ri - g_si)                  (s <= r).
* Carried state:  S_L = Diag(Gamma_L) S_0 + Khat^T U,  Khat_s = (Gamma_L / Gamma_s) . k_s.

Every exp(g_r - g_s) with s <= r is formed directly (never as a product of a
large and a small factor), so the form is exact up to f64 rounding for any
decay.
"""

from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular


def chunked_unit(q, k, v, beta, alpha, s0, C: int, scale: float = 1.0):
    """One (sequence, head): q, k [T, d_k]; v [T, d_v]; beta [T]; alpha [T, d_k]; s0 [d_k, d_v].

    Returns (o [T, d_v], S_T [d_k, d_v]), all float64.
    """
    q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
    beta, alpha = np.asarray(beta, np.float64), np.asarray(alpha, np.float64)
    T, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if s0 is None else np.array(s0, np.float64)
    o = np.empty((T, dv))
    for c0 in range(0, T, C):
        L = min(C, T - c0)
        Q, K, V = q[c0:c0 + L], k[c0:c0 + L], v[c0:c0 + L]
        b, a = beta[c0:c0 + L], alpha[c0:c0 + L]
        g = np.cumsum(np.log(a), axis=0)                      # [L, d_k]
        gam = np.exp(g)
        diff = g[:, None, :] - g[None, :, :]                 # g_r - g_s, [L, L, d_k]
        lower = np.tril(np.ones((L, L), dtype=bool))         # s <= r
        E = np.where(lower[:, :, None], np.exp(np.where(lower[:, :, None], diff, 0.0)), 0.0)
        A = np.tril(b[:, None] * np.einsum("ri,si,rsi->rs", K, K, E), -1)
        P = np.tril(np.einsum("ri,si,rsi->rs", Q, K, E))
        Tm = solve_triangular(np.eye(L) + A, np.eye(L), lower=True, unit_diagonal=True)
        W = Tm @ (b[:, None] * gam * K)
        Ut = Tm @ (b[:, None] * V)
        U = Ut - W @ S
        o[c0:c0 + L] = scale * ((gam * Q) @ S + P @ U)
        khat = np.exp(g[-1][None, :] - g) * K
        S = gam[-1][:, None] * S + khat.T @ U
    return o, S

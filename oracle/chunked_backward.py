"""Chunkwise (matrix) form of the KDA backward pass, in plain float64 numpy.

TEST INFRASTRUCTURE.  It exists only to pin the chunk algebra of the reverse mode, which a
tensor-core backward relies on: given a chunk's start state S_0 and the gradient dS_1 of its end
state, every gradient of the chunk follows from a fixed set of matrix products, with no per-token
state.  The oracle's tests check it against the token-by-token reverse mode of ``backward.py``;
nothing in the CUDA path imports it.

Forward of one chunk of L tokens ("Kimi K3, explained", section "Training in chunks"; the same
quantities as ``chunked.py``), with g_r = sum_{s<=r} ln alpha_s per key channel, Gamma_r = exp(g_r),
E_rsi = exp(g_ri - g_si) for s <= r:

    Qt = Gamma . Q,  Kt = Gamma . K,  Khat_s = (Gamma_L / Gamma_s) . k_s
    Bt_rs = sum_i k_ri k_si E_rsi (s < r),  A = Diag(beta) Bt,  T = (I + A)^-1
    P_rs  = sum_i q_ri k_si E_rsi (s <= r)
    W = T Diag(beta) Kt,  Ut = T Diag(beta) V,  U = Ut - W S_0
    O = Qt S_0 + P U,  S_1 = Diag(Gamma_L) S_0 + Khat^T U,  o = scale O

Reverse mode, dO = scale do:

    dU  = P^T dO + Khat dS_1                       dS_0 = Qt^T dO + Diag(Gamma_L) dS_1 - W^T dU
    dP  = (dO U^T) masked to s <= r                dW = -dU S_0^T,  dKhat = U dS_1^T
    dT  = dW (beta . Kt)^T + dU (beta . V)^T       dA = -(T^T dT T^T) masked to s < r
    dv  = beta . (T^T dU)                          dBt = Diag(beta) dA
    dq  = sum_s dP_rs k_s E_rs + (dO S_0^T) . Gamma
    dk  = sum_s dP_rs q_r E_rs (over r >= s) + sum_s dBt_rs k_s E_rs + sum_r dBt_rs k_r E_rs
          + beta . (T^T dW) . Gamma + dKhat . Gamma_L / Gamma
    dbeta_r = sum_s dA_rs Bt_rs + Kt_r . (T^T dW)_r + v_r . (T^T dU)_r
    dg  = q . (dP-term of dq) - k . (dP-term of dk) + k . (first dBt-term) - k . (second dBt-term)
          + (dO S_0^T) . Qt + beta . (T^T dW) . Kt - dKhat . Khat,
          and on the last row also sum_s dKhat_s . Khat_s + Gamma_L . rowsum(dS_1 . S_0)
    d ln alpha_s = sum_{r >= s} dg_r,  dalpha = d ln alpha / alpha

Each exp(g_r - g_s) with s <= r is formed directly, so the form is exact up to f64 rounding.
"""

from __future__ import annotations

import numpy as np

from . import oracle as O


def _f64(a, dtype):
    a = np.asarray(a)
    if dtype == "bf16" and a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def _chunk_forward(q, k, v, beta, alpha, s0):
    L = q.shape[0]
    g = np.cumsum(np.log(alpha), axis=0)
    gam = np.exp(g)
    E = np.exp(g[:, None, :] - g[None, :, :])                      # [r, s, i]
    strict, lower = np.tril(np.ones((L, L)), -1), np.tril(np.ones((L, L)))
    Bt = np.einsum("ri,si,rsi->rs", k, k, E) * strict
    P = np.einsum("ri,si,rsi->rs", q, k, E) * lower
    T = np.linalg.inv(np.eye(L) + beta[:, None] * Bt)
    Kt = k * gam
    W = T @ (beta[:, None] * Kt)
    U = T @ (beta[:, None] * v) - W @ s0
    Khat = k * np.exp(g[-1][None, :] - g)
    s1 = np.exp(g[-1])[:, None] * s0 + Khat.T @ U
    return dict(g=g, gam=gam, E=E, strict=strict, lower=lower, Bt=Bt, P=P, T=T, Kt=Kt, W=W, U=U, Khat=Khat,
                s1=s1)


def chunk_backward(q, k, v, beta, alpha, s0, dO, ds1):
    """Gradients of one chunk (all float64): q, k [L, d_k]; v, dO [L, d_v]; beta [L]; alpha [L, d_k];
    s0, ds1 [d_k, d_v].  Returns dq, dk, dv, dbeta, dalpha and ds0 (the gradient of the start state)."""
    f = _chunk_forward(q, k, v, beta, alpha, s0)
    E, T, W, U, P, Khat, Kt, gam, g = (f[n] for n in ("E", "T", "W", "U", "P", "Khat", "Kt", "gam", "g"))
    gL = g[-1]
    dU = P.T @ dO + Khat @ ds1
    ds0 = (q * gam).T @ dO + np.exp(gL)[:, None] * ds1 - W.T @ dU
    dP = (dO @ U.T) * f["lower"]
    dQs = dO @ s0.T
    dKhat = U @ ds1.T
    dW = -dU @ s0.T
    dT = dW @ (beta[:, None] * Kt).T + dU @ (beta[:, None] * v).T
    tdW, tdU = T.T @ dW, T.T @ dU
    dA = -(T.T @ dT @ T.T) * f["strict"]
    dBt = beta[:, None] * dA
    dq_p = np.einsum("rs,si,rsi->ri", dP, k, E)
    dk_p = np.einsum("rs,ri,rsi->si", dP, q, E)
    dk_r = np.einsum("rs,si,rsi->ri", dBt, k, E)
    dk_s = np.einsum("rs,ri,rsi->si", dBt, k, E)
    dq = dq_p + dQs * gam
    dk = dk_p + dk_r + dk_s + beta[:, None] * tdW * gam + dKhat * np.exp(gL[None, :] - g)
    dv = beta[:, None] * tdU
    dbeta = (dA * f["Bt"]).sum(1) + (Kt * tdW).sum(1) + (v * tdU).sum(1)
    dg = q * dq_p - k * dk_p + k * dk_r - k * dk_s + dQs * q * gam + beta[:, None] * tdW * Kt - dKhat * Khat
    dg[-1] += (dKhat * Khat).sum(0) + np.exp(gL) * (ds1 * s0).sum(1)
    dlna = np.cumsum(dg[::-1], axis=0)[::-1]
    return dict(dq=dq, dk=dk, dv=dv, dbeta=dbeta, dalpha=dlna / alpha, ds0=ds0)


def prefill_backward_chunked(inp: dict, do, d_state_out=None, scale: float = 1.0, C: int = 64) -> dict:
    """The backward pass of a packed varlen prefill (per-channel alpha), chunk by chunk: the chunk-start
    states come from the chunk forward, then the chunks are walked back with ``chunk_backward``.  Same
    arguments and result keys as ``backward.prefill_backward``."""
    inp = O.alpha_per_channel(inp)
    dt = inp["dtype"]
    q, k, v = _f64(inp["q"], dt), _f64(inp["k"], dt), _f64(inp["v"], dt)
    beta, alpha = np.asarray(inp["beta"], np.float64), np.asarray(inp["alpha"], np.float64)
    do = np.asarray(do, np.float64)
    cu = np.asarray(inp["cu_seqlens"], np.int64)
    N, H, dk_, dv_ = len(cu) - 1, inp["H"], inp["dk"], inp["dv"]
    s_in = inp.get("state_in")
    out = {"dq": np.zeros_like(q), "dk": np.zeros_like(k), "dv": np.zeros_like(v), "dbeta": np.zeros_like(beta),
           "dalpha": np.zeros_like(alpha), "d_state_in": np.zeros((N, H, dk_, dv_))}
    for n in range(N):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        starts = list(range(t0, t1, C))
        for h in range(H):
            s = np.zeros((dk_, dv_)) if s_in is None else np.asarray(s_in[n, h], np.float64).copy()
            s_starts = []
            for a in starts:                                        # chunk-start states
                b = min(a + C, t1)
                s_starts.append(s)
                s = _chunk_forward(q[a:b, h], k[a:b, h], v[a:b, h], beta[a:b, h], alpha[a:b, h], s)["s1"]
            G = np.zeros((dk_, dv_)) if d_state_out is None else np.asarray(d_state_out[n, h], np.float64).copy()
            for a, s0 in reversed(list(zip(starts, s_starts))):
                b = min(a + C, t1)
                r = chunk_backward(q[a:b, h], k[a:b, h], v[a:b, h], beta[a:b, h], alpha[a:b, h], s0,
                                   scale * do[a:b, h], G)
                for name in ("dq", "dk", "dv", "dbeta", "dalpha"):
                    out[name][a:b, h] = r[name]
                G = r["ds0"]
            out["d_state_in"][n, h] = G
    return out

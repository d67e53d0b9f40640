"""Float64 reverse-mode (backward) pass of the KDA recurrence, token by token.

TEST INFRASTRUCTURE.  Only ``tests/`` and ``bench.py``'s CPU legs may import this module; the product
path never does.

Forward, per head and token ("Kimi K3, explained", section "The math"; with the state S of size
d_k x d_v, key channel = row):

    S' = Diag(alpha_t) S_{t-1}                decay each key channel
    x  = S'^T k_t                             what the decayed state returns for k_t
    S_t = S' + beta_t k_t (v_t - x)^T         erase a beta share of x, write beta v_t
    o_t = scale S_t^T q_t                     read

Given the loss gradients do_t and dS_T (the gradient of the final state), the chain rule through one
token, from the last token back, with u = v_t - x and G = dS_t (already including later tokens):

    G  += scale q_t do_t^T                    (o_t depends on S_t)
    dq_t    = scale S_t do_t
    dbeta_t = k_t^T G u
    du      = beta_t G^T k_t  ->  dv_t = du,  dx = -du
    dk_t    = beta_t G u + S' dx              (through the write and through x)
    G'      = G + k_t dx^T                    (gradient of S')
    dalpha_t[i] = sum_j G'[i, j] S_{t-1}[i, j]
    dS_{t-1} = Diag(alpha_t) G'

Every product here is a library matrix-vector product; nothing is blocked or reordered.
"""

from __future__ import annotations

import numpy as np

from . import oracle as O


def _f64(a, dtype):
    a = np.asarray(a)
    if dtype == "bf16" and a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def prefill_backward(inp: dict, do, d_state_out=None, scale: float = 1.0) -> dict:
    """Gradients of the loss sum(o * do) + sum(state_out * d_state_out) with respect to q, k, v, beta,
    alpha (per key channel) and state_in.  Returns float64 arrays in a dict with keys dq, dk, dv, dbeta,
    dalpha, d_state_in; q, k, v, o take their storage dtypes' values (bf16 inputs are widened exactly)."""
    inp = O.alpha_per_channel(inp)
    dt = inp["dtype"]
    q, k, v = _f64(inp["q"], dt), _f64(inp["k"], dt), _f64(inp["v"], dt)
    beta, alpha = np.asarray(inp["beta"], np.float64), np.asarray(inp["alpha"], np.float64)
    do = np.asarray(do, np.float64)
    cu = np.asarray(inp["cu_seqlens"], np.int64)
    N, H, dk, dv = len(cu) - 1, inp["H"], inp["dk"], inp["dv"]
    s0 = inp.get("state_in")
    out = {"dq": np.zeros_like(q), "dk": np.zeros_like(k), "dv": np.zeros_like(v), "dbeta": np.zeros_like(beta),
           "dalpha": np.zeros_like(alpha), "d_state_in": np.zeros((N, H, dk, dv))}
    for n in range(N):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        for h in range(H):
            S = np.zeros((dk, dv)) if s0 is None else np.asarray(s0[n, h], np.float64).copy()
            states = [S]
            for t in range(t0, t1):                 # forward, keeping every state
                Sp = alpha[t, h][:, None] * S
                x = Sp.T @ k[t, h]
                S = Sp + beta[t, h] * np.outer(k[t, h], v[t, h] - x)
                states.append(S)
            G = np.zeros((dk, dv)) if d_state_out is None else np.asarray(d_state_out[n, h], np.float64).copy()
            for t in range(t1 - 1, t0 - 1, -1):     # backward
                S_prev, S_t = states[t - t0], states[t - t0 + 1]
                kt, qt, vt, bt, at = k[t, h], q[t, h], v[t, h], beta[t, h], alpha[t, h]
                G = G + scale * np.outer(qt, do[t, h])
                out["dq"][t, h] = scale * (S_t @ do[t, h])
                Sp = at[:, None] * S_prev
                u = vt - Sp.T @ kt
                out["dbeta"][t, h] = kt @ G @ u
                du = bt * (G.T @ kt)
                out["dv"][t, h] = du
                dx = -du
                out["dk"][t, h] = bt * (G @ u) + Sp @ dx
                Gp = G + np.outer(kt, dx)
                out["dalpha"][t, h] = (Gp * S_prev).sum(axis=1)
                G = at[:, None] * Gp
            out["d_state_in"][n, h] = G
    return out

"""Float64 models of the operand precision of two CUDA paths, against the float64 oracles.

Backward chunk pass at d = 128 (bf16 inputs): plain products on TF32 operands (10-bit significand,
rounded to nearest), decayed sums by 16-row blocks with a reference row inside each block.  On one head
of the prefill workload (its decay, a zero initial state): TF32 operands everywhere but in the decayed
sums that feed the decay gradient keep every gradient well inside the bf16 tolerance, while single TF32
operands in those sums do not (the terms of dg cancel almost exactly for the first rows of a sequence
that starts from zero), which is why they run in split (hi + lo) TF32.

Two-phase forward (one bf16 d = 128 sequence): fp16 records and operands with TF32 A/P factors stay
inside the tolerance for every decay, and fp16 (not bf16) M and Q' are what keep the state error low
when nothing decays.

Nothing here touches the CUDA path: these are models of its arithmetic, written from the same chunk
equations as the oracles."""

import numpy as np
import pytest

from kda_gated_delta_03_gb300 import inputs as I
from oracle import chunked_backward as CB

C = 64


def tf32(x):
    """Round float32 values to TF32 (10-bit significand), to nearest with ties away from zero."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return (((u + 0x1000) & 0xFFFFE000).astype(np.uint32)).view(np.float32).astype(np.float64)


def product(a, b, mode):
    """a @ b in float64 with the operands as the kernel stores them: exact ("f64"), TF32 ("tf32") or
    split into two TF32 parts, three products ("split")."""
    if mode == "f64":
        return a @ b
    if mode == "tf32":
        return tf32(a) @ tf32(b)
    ah, bh = tf32(a), tf32(b)
    return ah @ bh + ah @ tf32(b - bh) + tf32(a - ah) @ bh


def row_side(X, y, g, mode):
    """sum_{s} X_rs y_s exp(g_r - g_s) over 16-row blocks of r, reference row 16 b + 7."""
    out = np.zeros((C, y.shape[1]))
    for b in range(C // 16):
        ref, ns, rows = 16 * b + 7, 16 * (b + 1), slice(16 * b, 16 * b + 16)
        Y = y[:ns] * np.exp(g[ref] - g[:ns])
        out[rows] = np.exp(g[rows] - g[ref]) * product(X[rows, :ns], Y, mode)
    return out


def col_side(X, y, g, mode):
    """sum_{r >= s} X_rs y_r exp(g_r - g_s) over 16-row blocks of s."""
    out = np.zeros((C, y.shape[1]))
    for b in range(C // 16):
        ref, r0, cols = 16 * b + 7, 16 * b, slice(16 * b, 16 * b + 16)
        Y = y[r0:] * np.exp(g[r0:] - g[ref])
        out[cols] = np.exp(g[ref] - g[cols]) * product(X[r0:, cols].T, Y, mode)
    return out


def block_dots(a, c, g, mode, strict):
    """sum_i a_ri c_si exp(g_ri - g_si) for s <= r (s < r if strict), by 16-row blocks of r."""
    out = np.zeros((C, C))
    for b in range(C // 16):
        ref, ns, rows = 16 * b + 7, 16 * (b + 1), slice(16 * b, 16 * b + 16)
        A = a[rows] * np.exp(g[rows] - g[ref])
        out[rows, :ns] = product(A, (c[:ns] * np.exp(g[ref] - g[:ns])).T, mode)
    return out * np.tril(np.ones((C, C)), -1 if strict else 0)


def chunk_backward_model(q, k, v, beta, alpha, s0, dO, ds1, plain, decayed, ap):
    """The chunk pass's sequence of products ("Kimi K3, explained", section "Training in chunks", in
    reverse), each in the given operand precision."""
    g = np.cumsum(np.log(alpha), axis=0)
    gam = np.exp(g)
    strict, lower = np.tril(np.ones((C, C)), -1), np.tril(np.ones((C, C)))
    Bt, P = block_dots(k, k, g, ap, True), block_dots(q, k, g, ap, False)
    T = np.linalg.inv(np.eye(C) + beta[:, None] * Bt)
    Kt = k * gam
    W = product(T, beta[:, None] * Kt, plain)
    U = product(T, beta[:, None] * v, plain) - product(W, s0, plain)
    Khat = k * np.exp(g[-1] - g)
    dU = product(P.T, dO, plain) + product(Khat, ds1, plain)
    dP = product(dO, U.T, plain) * lower
    dQs, dKhat, dW = product(dO, s0.T, plain), product(U, ds1.T, plain), -product(dU, s0.T, plain)
    dT = (product(dW, (beta[:, None] * Kt).T, plain) + product(dU, (beta[:, None] * v).T, plain)) * strict
    tdW, tdU = product(T.T, dW, plain), product(T.T, dU, plain)
    dA = -product(T.T, product(dT, T.T, plain), plain) * strict
    dBt = beta[:, None] * dA
    dq_p, dk_r = row_side(dP, k, g, decayed), row_side(dBt, k, g, decayed)
    dk_p, dk_s = col_side(dP, q, g, decayed), col_side(dBt, k, g, decayed)
    dg = q * dq_p - k * dk_p + k * dk_r - k * dk_s + dQs * q * gam + beta[:, None] * tdW * Kt - dKhat * Khat
    dg[-1] += (dKhat * Khat).sum(0) + np.exp(g[-1]) * (ds1 * s0).sum(1)
    return dict(dq=dq_p + dQs * gam,
                dk=dk_p + dk_r + dk_s + beta[:, None] * tdW * gam + dKhat * np.exp(g[-1] - g),
                dv=beta[:, None] * tdU,
                dbeta=(dA * Bt).sum(1) + (Kt * tdW).sum(1) + (v * tdU).sum(1),
                dalpha=np.cumsum(dg[::-1], axis=0)[::-1] / alpha)


@pytest.fixture(scope="module")
def chunks():
    """Eight chunks of head 0 of the prefill workload, their start states and end-state gradients."""
    w = I.workload("prefill_8k")
    T = 8 * C
    inp = I.prefill_inputs([T], 1, 128, 128, "bf16", w["seed"], state="zero")
    f = lambda n: I.bf16_bits_to_f32(inp[n])[:, 0].astype(np.float64)
    q, k, v = f("q"), f("k"), f("v")
    beta, alpha = inp["beta"][:, 0].astype(np.float64), inp["alpha"][:, 0].astype(np.float64)
    dO = I.bf16_bits_to_f32(I.f32_to_bf16_bits(
        np.random.default_rng(8).standard_normal((T, 128)).astype(np.float32))).astype(np.float64)
    starts, s = [], np.zeros((128, 128))
    for c in range(8):
        sl = slice(C * c, C * c + C)
        starts.append(s)
        s = CB._chunk_forward(q[sl], k[sl], v[sl], beta[sl], alpha[sl], s)["s1"]
    ends, G = [None] * 8, np.zeros((128, 128))
    for c in reversed(range(8)):
        sl = slice(C * c, C * c + C)
        ends[c] = G
        G = CB.chunk_backward(q[sl], k[sl], v[sl], beta[sl], alpha[sl], starts[c], dO[sl], G)["ds0"]
    return [(q[C * c:C * c + C], k[C * c:C * c + C], v[C * c:C * c + C], beta[C * c:C * c + C],
             alpha[C * c:C * c + C], starts[c], dO[C * c:C * c + C], ends[c]) for c in range(8)]


def errors(chunks, plain, decayed, ap):
    got, ref = {}, {}
    for ch in chunks:
        r = CB.chunk_backward(*ch)
        m = chunk_backward_model(*ch, plain, decayed, ap)
        for n in m:
            got.setdefault(n, []).append(m[n])
            ref.setdefault(n, []).append(r[n])
    return {n: np.linalg.norm(np.concatenate(got[n]) - np.concatenate(ref[n])) / np.linalg.norm(np.concatenate(ref[n]))
            for n in got}


def test_model_in_float64_is_the_chunk_oracle(chunks):
    assert max(errors(chunks, "f64", "f64", "f64").values()) < 1e-9


def test_tf32_products_and_split_decayed_sums_stay_inside_the_bf16_tolerance(chunks):
    e = errors(chunks, "tf32", "split", "tf32")
    assert max(e.values()) < 1e-3, e


def test_single_tf32_decayed_sums_would_break_the_decay_gradient(chunks):
    e = errors(chunks, "tf32", "tf32", "tf32")
    assert e["dalpha"] > 3e-3, e
    assert max(v for n, v in e.items() if n != "dalpha") < 1e-3, e


# ---- the two-phase forward (one bf16 d = 128 sequence) ----

def f16(x):
    """Round to fp16, nearest-even."""
    return np.asarray(x, np.float64).astype(np.float32).astype(np.float16).astype(np.float64)


def f32(x):
    return np.asarray(x, np.float64).astype(np.float32).astype(np.float64)


def bf16(x):
    return I.bf16_bits_to_f32(I.f32_to_bf16_bits(np.asarray(x, np.float32))).astype(np.float64)


def two_phase_model(q, k, v, beta, alpha, s0, mq):
    """One head through the two-phase arithmetic: phase 1 per chunk (A and P on TF32 operands by 16-row
    blocks; T' = (I + A)^-1 Diag(beta), Gamma K, V, W, Utilde, Khat and P as fp16 operands; the record
    Q' = Gamma Q - P W, M = Khat^T W, B = Khat^T Utilde and P Utilde stored as fp16, M and Q' through `mq`),
    then the chain: o = Q' S + P Utilde and S <- Diag(Gamma_C) S + B - M S with S fp32 and its operand
    fp16 ("Kimi K3, explained", section "Training in chunks", with the chunk made affine in S)."""
    T = k.shape[0]
    S, o = s0.copy(), np.empty((T, v.shape[1]))
    for c0 in range(0, T, C):
        L = min(C, T - c0)
        Q, K, V, b = q[c0:c0 + L], k[c0:c0 + L], v[c0:c0 + L], beta[c0:c0 + L]
        g = np.cumsum(np.maximum(np.log2(alpha[c0:c0 + L]), -15.0), axis=0)
        gam = 2.0 ** g
        A, P = np.zeros((L, L)), np.zeros((L, L))
        for blk in range(0, L, 16):
            ref, rows, cols = g[min(blk + 7, L - 1)], slice(blk, min(blk + 16, L)), slice(0, min(blk + 16, L))
            R = tf32(K[cols] * 2.0 ** (ref - g[cols]))
            A[rows, cols] = b[rows, None] * (tf32(K[rows] * 2.0 ** (g[rows] - ref)) @ R.T)
            P[rows, cols] = tf32(Q[rows] * 2.0 ** (g[rows] - ref)) @ R.T
        A, P = np.tril(A, -1), f16(np.tril(P))
        Tp = f16(np.linalg.inv(np.eye(L) + A) * b[None, :])
        W, Ut = f16(Tp @ f16(gam * K)), f16(Tp @ f16(V))
        Kh = f16(2.0 ** (g[-1][None, :] - g) * K)
        M, B = mq(f32(Kh.T @ W)), f16(Kh.T @ Ut)
        Qp, Oi = mq(f32(gam * Q - P @ W)), f16(P @ Ut)
        o[c0:c0 + L] = Qp @ f16(S) + Oi
        S = f32(2.0 ** g[-1][:, None] * S + B - M @ f16(S))
    return o, S


def two_phase_errors(decay, mq):
    """Relative Frobenius errors of o (rounded to bf16) and of the final state against the float64 token
    oracle, over two heads of a 1,024-token sequence with a random initial state."""
    from oracle import oracle as O
    inp = I.prefill_inputs([1024], 2, 128, 128, "bf16", 3, decay=decay, state="randn")
    o_ref, s_ref = O.prefill(inp)
    f = lambda x: I.bf16_bits_to_f32(x).astype(np.float64)
    os_, ss_ = [], []
    for h in range(2):
        o, s = two_phase_model(f(inp["q"][:, h]), f(inp["k"][:, h]), f(inp["v"][:, h]),
                               inp["beta"][:, h].astype(np.float64), inp["alpha"][:, h].astype(np.float64),
                               inp["state_in"][0, h].astype(np.float64), mq)
        os_.append(o)
        ss_.append(s)
    eo = np.linalg.norm(bf16(np.stack(os_, 1)) - o_ref) / np.linalg.norm(o_ref)
    es = np.linalg.norm(np.stack(ss_) - s_ref[0]) / np.linalg.norm(s_ref[0])
    return eo, es


@pytest.mark.parametrize("decay", ["one", "slow", "config"])
def test_two_phase_forward_precision_model_within_tolerance(decay):
    """fp16 records and operands, TF32 A/P factors: o and the final state against the float64 token oracle,
    inside the bf16 tolerance (3e-3) with margin, for no decay, slow decay and the workload's decay (about
    1.7e-3 on o, most of it the bf16 rounding of o itself)."""
    eo, es = two_phase_errors(decay, f16)
    assert eo < 2.5e-3 and es < 1.0e-3, (eo, es)


def test_fp16_records_beat_bf16_records_without_decay():
    """M and Q' in bf16 (8-bit significand) instead of fp16 more than double the state error when nothing
    decays (the chain then compounds every chunk's rounding); the reason the records are fp16."""
    eo16, es16 = two_phase_errors("one", f16)
    eob, esb = two_phase_errors("one", bf16)
    assert esb > 2 * es16 and eob > eo16, (es16, esb, eo16, eob)

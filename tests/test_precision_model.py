"""A float64 model of the backward chunk pass's operand precision, against the float64 chunk oracle.

The d = 128 backward chunk pass (bf16 inputs) runs its plain products with TF32 operands (10-bit
significand, rounded to nearest) and its decayed sums by 16-row blocks with a reference row inside each
block.  This model repeats that arithmetic in numpy on one head of the prefill workload (its decay,
a zero initial state) and checks the two facts the kernel's design rests on: TF32 operands everywhere
but in the decayed sums that feed the decay gradient keep every gradient well inside the bf16
tolerance, while single TF32 operands in those sums do not (the terms of dg cancel almost exactly for
the first rows of a sequence that starts from zero), which is why they run in split (hi + lo) TF32.
Nothing here touches the CUDA path."""

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

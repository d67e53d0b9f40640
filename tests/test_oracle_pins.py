"""Pins of the float64 oracle against what the pages and the mathematics fix.

CPU only.  None of these compares the oracle with itself: each checks it
against a worked example the pages print, a closed form, a special case that
reduces to a textbook rule, an invariant, or an independent derivation
(the chunkwise form).  ``test_mutants_are_caught`` plants each plausible
mistake in the oracle (compiled variants of the C file) and checks that at least
one pin fails.
"""

import json
import os

import numpy as np
import pytest

from oracle import oracle as O
from oracle.chunked import chunked_unit
from kda_gated_delta_03_gb300 import inputs as I


def mk(q, k, v, beta, alpha, seqlens, state_in=None):
    """Token arrays for the oracle, stored float32 (values chosen so storage is exact where it matters)."""
    q, k, v = (np.ascontiguousarray(x, dtype=np.float32) for x in (q, k, v))
    T, H, dk = k.shape
    return dict(q=q, k=k, v=v, beta=np.ascontiguousarray(beta, np.float32),
                alpha=np.ascontiguousarray(alpha, np.float32), cu_seqlens=I.cu_seqlens_of(seqlens),
                state_in=None if state_in is None else np.ascontiguousarray(state_in, np.float64),
                dtype="f32", H=H, dk=dk, dv=v.shape[2])


def f64(x):
    return np.asarray(x, dtype=np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# pins, each usable against a planted-mistake build (mutant)
# ---------------------------------------------------------------------------
def pin_worked_overwrite(golden_dir, mutant=None):
    """The page's worked example: write (k, a) then (k, b) with beta = 1; reading k gives b, plain
    linear accumulation gives a + b."""
    g = json.load(open(os.path.join(golden_dir, "overwrite_example.json")))
    D = g["D"]
    key = np.zeros(D)
    key[g["key_index"]] = 1.0
    a, b = np.array(g["a"]), np.array(g["b"])
    q = np.stack([key, key])[:, None, :]
    v = np.stack([a, b])[:, None, :]
    inp = mk(q, q, v, np.full((2, 1), g["beta"]), np.full((2, 1, D), g["alpha"]), [2])
    o, _ = O.prefill(inp, mutant=mutant)
    assert np.array_equal(o[0, 0], a), o[0, 0]                       # write-then-read returns the value
    assert np.array_equal(o[1, 0], np.array(g["delta_read_after_both_writes"])), o[1, 0]
    o_lin, _ = O.prefill(inp, erase=False, mutant=mutant)
    assert np.array_equal(o_lin[1, 0], np.array(g["linear_read_after_both_writes"])), o_lin[1, 0]


def pin_overwrite_any_state(mutant=None):
    """beta = 1 and a unit key: right after the write, reading the key returns exactly v_t, whatever
    the state and the decay were (section 'The math')."""
    rng = np.random.default_rng(11)
    dk, dv = 5, 3
    s0 = rng.standard_normal((1, 1, dk, dv))
    keys = np.array([[0.5, -0.5, 0.5, 0.5, 0.0], [0.0, 0.5, 0.5, -0.5, 0.5], [0.5, 0.5, 0.5, 0.0, -0.5]])
    T = len(keys)
    v = f64(rng.standard_normal((T, 1, dv)))
    alpha = f64(rng.uniform(0.2, 0.95, (T, 1, dk)))
    inp = mk(keys[:, None, :], keys[:, None, :], v, np.ones((T, 1)), alpha, [T], s0)
    o, _ = O.prefill(inp, mutant=mutant)
    np.testing.assert_allclose(o[:, 0], v[:, 0], rtol=0, atol=1e-14)


def pin_non_interference(mutant=None):
    """Orthonormal keys, no decay, beta = 1: each later read returns its own value (the runnable's
    third assertion).  The reads are tokens with beta = 0, which write nothing."""
    h = 0.5 * np.array([[1, 1, 1, 1], [1, -1, 1, -1], [1, 1, -1, -1], [1, -1, -1, 1]], dtype=np.float64)
    rng = np.random.default_rng(12)
    vals = f64(rng.standard_normal((4, 3)))
    keys = np.concatenate([h, h])[:, None, :]
    v = np.concatenate([vals, np.zeros((4, 3))])[:, None, :]
    beta = np.concatenate([np.ones(4), np.zeros(4)])[:, None]
    inp = mk(keys, keys, v, beta, np.ones((8, 1, 4)), [8])
    o, _ = O.prefill(inp, mutant=mutant)
    np.testing.assert_allclose(o[4:, 0], vals, rtol=0, atol=1e-13)


def pin_deltanet_special_case(mutant=None):
    """alpha == 1 is plain DeltaNet: S <- S - beta (S k - v) k^T, o = S q, with S of size d_v x d_k
    (the page's orientation), run here as a textbook loop with non-unit keys and d_k != d_v."""
    rng = np.random.default_rng(13)
    T, dk, dv = 20, 6, 5
    q, k, v = (f64(rng.standard_normal((T, 1, d))) for d in (dk, dk, dv))
    beta = f64(rng.uniform(0.05, 0.95, (T, 1)))
    inp = mk(q, k, v, beta, np.ones((T, 1, dk)), [T])
    o, st = O.prefill(inp, mutant=mutant)
    S = np.zeros((dv, dk))
    ref = np.empty((T, dv))
    for t in range(T):
        kt, vt, qt = k[t, 0], v[t, 0], q[t, 0]
        S = S - beta[t, 0] * np.outer(S @ kt - vt, kt)
        ref[t] = S @ qt
    np.testing.assert_allclose(o[:, 0], ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(st[0, 0], S.T, rtol=1e-12, atol=1e-12)


def pin_decay_only(golden_dir, mutant=None):
    """beta = 0: nothing is written and the state only fades, S_t = Diag(prod alpha) S_0, o_t = S_t^T q_t;
    and the page's channel with alpha = 0.5 keeps 0.5^10 of its content after 10 tokens."""
    rng = np.random.default_rng(14)
    T, dk, dv = 9, 6, 4
    s0 = rng.standard_normal((1, 1, dk, dv))
    q = f64(rng.standard_normal((T, 1, dk)))
    k = f64(rng.standard_normal((T, 1, dk)))
    v = f64(rng.standard_normal((T, 1, dv)))
    alpha = f64(rng.uniform(0.3, 1.0, (T, 1, dk)))
    inp = mk(q, k, v, np.zeros((T, 1)), alpha, [T], s0)
    o, st = O.prefill(inp, mutant=mutant)
    cum = np.cumprod(alpha[:, 0, :], axis=0)
    for t in range(T):
        St = cum[t][:, None] * s0[0, 0]
        np.testing.assert_allclose(o[t, 0], St.T @ q[t, 0], rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(st[0, 0], cum[-1][:, None] * s0[0, 0], rtol=1e-14, atol=0)

    g = json.load(open(os.path.join(golden_dir, "decay_example.json")))
    n = g["tokens"]
    a = np.array([[g["alpha_fast"], g["alpha_slow"], 1.0, 1.0]] * n)[:, None, :]
    inp = mk(np.zeros((n, 1, 4)), np.zeros((n, 1, 4)), np.zeros((n, 1, 2)), np.zeros((n, 1)), a, [n],
             np.ones((1, 1, 4, 2)))
    _, st = O.prefill(inp, mutant=mutant)
    assert st[0, 0, 0, 0] == g["remaining_fast_exact"]
    assert abs(st[0, 0, 0, 1] - g["remaining_fast_approx"]) < 5e-5
    assert st[0, 0, 1, 0] == g["remaining_slow"]


def pin_linear_sum(mutant=None):
    """Dropping the erase factor with no decay gives plain (gated) linear attention: the state is the
    sum of the writes, S_T = S_0 + sum_t beta_t k_t v_t^T."""
    rng = np.random.default_rng(15)
    T, dk, dv = 7, 5, 3
    s0 = rng.standard_normal((1, 1, dk, dv))
    q, k, v = (f64(rng.standard_normal((T, 1, d))) for d in (dk, dk, dv))
    beta = f64(rng.uniform(0.1, 1.0, (T, 1)))
    inp = mk(q, k, v, beta, np.ones((T, 1, dk)), [T], s0)
    o, st = O.prefill(inp, erase=False, mutant=mutant)
    S = s0[0, 0].copy()
    for t in range(T):
        S = S + beta[t, 0] * np.outer(k[t, 0], v[t, 0])
        np.testing.assert_allclose(o[t, 0], S.T @ q[t, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(st[0, 0], S, rtol=0, atol=1e-12)


def pin_page_orientation(mutant=None):
    """The page's form S_t = S_{t-1} Diag(alpha_t) (I - beta_t k_t k_t^T) + beta_t v_t k_t^T, o_t = S_t q_t
    (S of size d_v x d_k), with per-channel alpha, equals the oracle's transposed state and outputs."""
    rng = np.random.default_rng(16)
    T, dk, dv = 12, 6, 4
    q, k, v = (f64(rng.standard_normal((T, 1, d))) for d in (dk, dk, dv))
    beta = f64(rng.uniform(0.05, 1.0, (T, 1)))
    alpha = f64(rng.uniform(0.2, 1.0, (T, 1, dk)))
    s0 = rng.standard_normal((1, 1, dk, dv))
    inp = mk(q, k, v, beta, alpha, [T], s0)
    o, st = O.prefill(inp, mutant=mutant)
    S = s0[0, 0].T.copy()
    for t in range(T):
        kt = k[t, 0]
        S = S @ np.diag(alpha[t, 0]) @ (np.eye(dk) - beta[t, 0] * np.outer(kt, kt)) + beta[t, 0] * np.outer(v[t, 0], kt)
        np.testing.assert_allclose(o[t, 0], S @ q[t, 0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(st[0, 0], S.T, rtol=1e-12, atol=1e-12)


def pin_chunked_form(mutant=None):
    """The chunkwise WY form computes the same result as the recurrence (to f64 rounding) for several
    chunk sizes, ragged lengths, a carried initial state and both slow and strong decay."""
    for decay, seed in (("slow", 21), ("config", 22), ("scalar", 23)):
        seqlens = [1, 63, 64, 65, 130]
        inp = I.prefill_inputs(seqlens, 2, 16, 8, "f32", seed, decay=decay, state="randn")
        o, st = O.prefill(inp, mutant=mutant)
        cu = inp["cu_seqlens"]
        for C in (4, 16, 64):
            for n in range(len(seqlens)):
                for h in range(2):
                    sl = slice(cu[n], cu[n + 1])
                    oc, sc = chunked_unit(f64(inp["q"][sl, h]), f64(inp["k"][sl, h]), f64(inp["v"][sl, h]),
                                          f64(inp["beta"][sl, h]), f64(inp["alpha"][sl, h]),
                                          inp["state_in"][n, h].astype(np.float64), C)
                    np.testing.assert_allclose(oc, o[sl, h], rtol=1e-10, atol=1e-12)
                    np.testing.assert_allclose(sc, st[n, h], rtol=1e-10, atol=1e-12)


ALL_PINS = [pin_worked_overwrite, pin_overwrite_any_state, pin_non_interference, pin_deltanet_special_case,
            pin_decay_only, pin_linear_sum, pin_page_orientation, pin_chunked_form]


def _call(pin, golden_dir, mutant=None):
    if "golden_dir" in pin.__code__.co_varnames[:pin.__code__.co_argcount]:
        return pin(golden_dir, mutant=mutant)
    return pin(mutant=mutant)


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin, golden_dir):
    _call(pin, golden_dir)


@pytest.mark.parametrize("mutant", [1, 2, 3, 4, 5, 6])
def test_mutants_are_caught(mutant, golden_dir):
    failed = []
    for pin in ALL_PINS:
        try:
            _call(pin, golden_dir, mutant=mutant)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"planted mistake {mutant} passed every pin"


# ---------------------------------------------------------------------------
# invariants of the oracle's entry points
# ---------------------------------------------------------------------------
def test_append_equals_one_shot():
    """prefill(T1) then prefill(T2) from the carried state equals prefill(T1 + T2), bit for bit."""
    inp = I.prefill_inputs([150], 2, 16, 16, "bf16", 31, decay="slow", state="randn")
    o_full, s_full = O.prefill(inp)
    cut = 97

    def part(t0, t1, s_in):
        d = dict(inp)
        for kk in ("q", "k", "v", "beta", "alpha"):
            d[kk] = np.ascontiguousarray(inp[kk][t0:t1])
        d["cu_seqlens"] = I.cu_seqlens_of([t1 - t0])
        return O.prefill(d, state_in=s_in)

    o1, s1 = part(0, cut, inp["state_in"])
    o2, s2 = part(cut, 150, s1)
    assert np.array_equal(np.concatenate([o1, o2]), o_full)
    assert np.array_equal(s2, s_full)


def test_scale_is_linear_in_output_only():
    inp = I.prefill_inputs([40], 2, 8, 8, "f32", 32, decay="slow")
    o1, s1 = O.prefill(inp, scale=1.0)
    o2, s2 = O.prefill(inp, scale=0.5)
    assert np.array_equal(o2, 0.5 * o1)
    assert np.array_equal(s1, s2)


def test_state_size_independent_of_length(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "state_size_example.json")))
    assert g["d_k"] * g["d_v"] == g["state_numbers"]
    assert 2 * g["d_k"] * 1_000_000 == g["softmax_cache_numbers_at_1M_tokens"]
    assert abs(g["softmax_cache_numbers_at_1M_tokens"] / g["state_numbers"] - g["ratio_approx"]) < 100
    for T in (1, 5, 77):
        inp = I.prefill_inputs([T], 1, 128, 128, "bf16", 33)
        _, st = O.prefill(inp)
        assert st.shape == (1, 1, 128, 128) and st[0, 0].size == g["state_numbers"]


def test_decode_entry_matches_one_token_prefill():
    """The decode entry point is one token of the same recurrence on each resident state, with slots
    chosen through state_idx."""
    rng = np.random.default_rng(34)
    B, H, dk, dv, P = 6, 2, 16, 8, 9
    pool = 0.3 * rng.standard_normal((P, H, dk, dv))
    idx = np.array([4, 0, 8, 2, 7, 5], np.int32)
    step = I.decode_step_inputs(B, H, dk, dv, "bf16", 35, 0, decay="slow")
    pool2 = pool.copy()
    o = O.decode_step(step, pool2, idx)
    for b in range(B):
        d = dict(step)
        for kk in ("q", "k", "v", "beta", "alpha"):
            d[kk] = np.ascontiguousarray(step[kk][b:b + 1])
        d["cu_seqlens"] = I.cu_seqlens_of([1])
        ob, sb = O.prefill(d, state_in=pool[idx[b]][None])
        assert np.array_equal(ob[0], o[b])
        assert np.array_equal(sb[0], pool2[idx[b]])
    untouched = sorted(set(range(P)) - set(idx.tolist()))
    assert np.array_equal(pool2[untouched], pool[untouched])


# ---- bf16-stored decode state ----

def test_round_bf16_is_nearest_even_at_eight_significant_bits():
    """bf16 keeps 8 significant bits: spacing 2^-7 at 1.0.  Halfway cases go to the even neighbour."""
    x = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -20, -(1 + 2 ** -8), 3.0, 2 ** -130,
                  65504.0, 1 + 2 ** -7])
    want = np.array([1.0, 1.0, 1 + 2 ** -6, 1 + 2 ** -7, -1.0, 3.0, 0.0, 65536.0, 1 + 2 ** -7])
    got = O.round_bf16(x)
    assert np.array_equal(got[np.arange(9) != 6], want[np.arange(9) != 6])
    assert abs(got[6]) < 2 ** -125                     # below bf16's (and float32's) normal range


def test_bf16_state_overwrite_example(golden_dir):
    """The page's overwrite example with the state stored in bf16: writing (k, a) then (k, b) at beta = 1
    leaves the key's row equal to b exactly (b is a bf16 number) and the read returns b."""
    g = json.load(open(os.path.join(golden_dir, "overwrite_example.json")))
    d = 16
    pool = np.zeros((1, 1, d, d))
    for vec in (g["a"], g["b"]):
        key = np.zeros(d, np.float32)
        key[g["key_index"]] = 1.0
        v = np.zeros(d, np.float32)
        v[:4] = vec
        step = dict(q=key[None, None].copy(), k=key[None, None].copy(), v=v[None, None].copy(),
                    beta=np.ones((1, 1), np.float32), alpha=np.ones((1, 1, d), np.float32), dtype="f32", H=1, dk=d,
                    dv=d)
        o = O.decode_step(step, pool, state_dtype="bf16")
    assert np.array_equal(pool[0, 0, g["key_index"], :4], g["b"])
    assert np.array_equal(o[0, 0, :4], g["delta_read_after_both_writes"])


def test_bf16_state_is_stored_in_bf16_and_unchanged_without_a_write():
    rng = np.random.default_rng(36)
    B, H, d = 3, 2, 16
    pool = O.round_bf16(0.3 * rng.standard_normal((B, H, d, d)))
    step = I.decode_step_inputs(B, H, d, d, "bf16", 37, 0, decay="slow")
    frozen = dict(step, beta=np.zeros_like(step["beta"]), alpha=np.ones_like(step["alpha"]))
    p0 = pool.copy()
    O.decode_step(frozen, p0, state_dtype="bf16")
    assert np.array_equal(p0, pool)                   # no decay, no write: bit-identical
    p1 = pool.copy()
    O.decode_step(step, p1, state_dtype="bf16")
    low = p1.astype(np.float32).view(np.uint32) & 0xFFFF
    assert not low.any()                              # every stored value is a bf16 number
    p2 = pool.copy()
    O.decode_step(step, p2)                           # the same step with an f64 state
    assert np.max(np.abs(p1 - p2)) <= 2 ** -8 * np.max(np.abs(p2))


# ---- state snapshots ----

def test_snapshots_are_prefix_states_and_the_last_is_state_out():
    """A snapshot after m tokens is the final state of the prefill of the first m tokens (computed here by
    a separate one-shot prefill of that prefix), and one at the sequence end equals state_out."""
    inp = I.prefill_inputs([256, 100, 128, 0], 2, 16, 16, "f32", 38, decay="slow", state="randn")
    snaps, offs = O.prefill_snapshots(inp, 64)
    assert offs.tolist() == [0, 4, 5, 7, 7]
    _, st = O.prefill(inp)
    cu = inp["cu_seqlens"]
    for n, m in ((0, 3), (2, 1)):                     # snapshots at the sequence ends
        assert np.allclose(snaps[offs[n] + m], st[n], rtol=1e-12, atol=1e-12)
    pre = dict(inp)                                   # sequence 0's first 128 tokens in one shot
    for key in ("q", "k", "v", "beta", "alpha"):
        pre[key] = np.ascontiguousarray(inp[key][cu[0]:cu[0] + 128])
    pre["cu_seqlens"] = I.cu_seqlens_of([128])
    pre["state_in"] = np.ascontiguousarray(inp["state_in"][0:1])
    _, s128 = O.prefill(pre)
    assert np.allclose(snaps[1], s128[0], rtol=1e-12, atol=1e-12)


# ---- alpha layouts (Gated DeltaNet, DeltaNet) ----

def test_gated_deltanet_one_token_closed_form():
    """One token with one forget value per head: S_1 = alpha (I - beta k k^T) S_0 + beta k v^T.  With
    k = e_0, beta = 1, alpha = 1/2: row 0 of S_1 is v, every other row is half of S_0's."""
    d = 4
    S0 = np.arange(1.0, 17.0).reshape(1, 1, d, d)
    k = np.zeros((1, 1, d), np.float32); k[0, 0, 0] = 1.0
    v = np.array([[[1.0, 2.0, 3.0, 4.0]]], np.float32)
    step = dict(q=k.copy(), k=k, v=v, beta=np.ones((1, 1), np.float32), alpha=np.full((1, 1), 0.5, np.float32),
                alpha_mode=1, dtype="f32", H=1, dk=d, dv=d)
    pool = S0.copy()
    o = O.decode_step(step, pool)
    assert np.array_equal(pool[0, 0, 0], v[0, 0])
    assert np.array_equal(pool[0, 0, 1:], 0.5 * S0[0, 0, 1:])
    assert np.array_equal(o[0, 0], v[0, 0])           # q = k reads row 0 back


def test_deltanet_layout_equals_unit_decay():
    """alpha_mode 2 (no decay, alpha not read) equals per-channel alpha = 1 exactly."""
    inp = I.prefill_inputs([70, 5], 2, 16, 16, "f32", 39, decay="one", state="randn")
    o1, s1 = O.prefill(inp)
    o2, s2 = O.prefill(dict(inp, alpha=None, alpha_mode=2))
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)


# ---- backward pass ----

def test_backward_matches_finite_differences_of_the_forward_oracle():
    """The reverse-mode gradients of loss = sum(o * do) + sum(state_out * dS) equal central differences
    of the (independently pinned) forward oracle, element by element, for q, k, v, beta, alpha and the
    initial state."""
    from oracle.backward import prefill_backward
    rng = np.random.default_rng(41)
    inp = I.prefill_inputs([7, 5], 1, 8, 8, "f32", 42, decay="config", state="randn")
    T, H, dv = inp["v"].shape
    do = rng.standard_normal((T, H, dv))
    dS = rng.standard_normal((2, H, 8, 8))
    g = prefill_backward(inp, do, dS)

    def loss(x):
        o, st = O.prefill(x)
        return float((o * do).sum() + (st * dS).sum())

    eps = 2.0 ** -12
    names = {"q": "dq", "k": "dk", "v": "dv", "beta": "dbeta", "alpha": "dalpha", "state_in": "d_state_in"}
    for name, gname in names.items():
        arr = inp[name]
        for flat in rng.choice(arr.size, size=6, replace=False):
            idx = np.unravel_index(flat, arr.shape)
            hi, lo = dict(inp), dict(inp)
            hi[name], lo[name] = arr.copy(), arr.copy()
            hi[name][idx] += eps
            lo[name][idx] -= eps
            fd = (loss(hi) - loss(lo)) / (2 * eps)
            assert abs(fd - g[gname][idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, g[gname][idx])


@pytest.mark.parametrize("C", [1, 4, 16, 64])
def test_chunked_backward_equals_token_backward(C):
    """The chunkwise (matrix) backward equals the token-by-token reverse mode to f64 rounding, for any
    chunk size, on ragged sequences with initial states, a final-state gradient and a query scale."""
    from oracle.backward import prefill_backward
    from oracle.chunked_backward import prefill_backward_chunked
    rng = np.random.default_rng(43)
    inp = I.prefill_inputs([37, 0, 70], 2, 8, 8, "bf16", 44, decay="slow", state="randn")
    T, H, dv = inp["v"].shape
    do = rng.standard_normal((T, H, dv))
    dS = rng.standard_normal((3, H, 8, 8))
    ref = prefill_backward(inp, do, dS, scale=0.75)
    got = prefill_backward_chunked(inp, do, dS, scale=0.75, C=C)
    for name in ref:
        err = np.abs(got[name] - ref[name]).max() / max(np.abs(ref[name]).max(), 1e-30)
        assert err <= 1e-12, (name, err)

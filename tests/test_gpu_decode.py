"""Parity of kda_decode_step (CUDA, through the C ABI) with the float64 oracle."""

import numpy as np
import pytest
import torch

from kda_gated_delta_03_gb300 import inputs as I
from oracle import oracle as O
from kda_testutil import TOL, rel_frob, to_dev

pytestmark = pytest.mark.gpu


def run_steps(B, H, d, dtype, steps, seed, P=None, idx=None, decay="config", state_dtype="f32"):
    import kda_gated_delta_03_gb300 as kda
    P = P or B
    pool = I.random_state(P, H, d, d, seed)
    if state_dtype == "bf16":                         # a bf16 pool: the same seeded values, stored in 2 bytes
        pool = I.bf16_bits_to_f32(I.f32_to_bf16_bits(pool))
        pool_d = to_dev(I.f32_to_bf16_bits(pool), True)
    else:
        pool_d = to_dev(pool)
    pool64 = pool.astype(np.float64)
    idx_d = None if idx is None else to_dev(np.asarray(idx, np.int32))
    bf = dtype == "bf16"
    os_gpu, os_ref = [], []
    for s in range(steps):
        st = I.decode_step_inputs(B, H, d, d, dtype, seed, s, decay=decay)
        o = kda.kda_decode_step(*(to_dev(st[n], bf) for n in ("q", "k", "v")), to_dev(st["beta"]),
                                to_dev(st["alpha"]), pool_d, idx_d)
        os_gpu.append(o.double().cpu().numpy())
        os_ref.append(O.decode_step(st, pool64, idx, state_dtype=state_dtype))
    torch.cuda.synchronize()
    return np.stack(os_gpu), np.stack(os_ref), pool_d.double().cpu().numpy(), pool64


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [16, 64, 128])
@pytest.mark.parametrize("decay", ["config", "slow"])
def test_decode_steps(dtype, d, decay):
    o, o_ref, pool, pool_ref = run_steps(5, 3, d, dtype, 6, 40 + d, decay=decay)
    assert rel_frob(o, o_ref) <= TOL[dtype]
    assert rel_frob(pool, pool_ref) <= TOL[dtype]


def test_decode_state_idx_and_untouched_slots():
    idx = [6, 1, 3, 0]
    o, o_ref, pool, pool_ref = run_steps(4, 2, 128, "bf16", 3, 50, P=8, idx=idx)
    assert rel_frob(o, o_ref) <= 3e-3
    assert rel_frob(pool, pool_ref) <= 3e-3
    untouched = [2, 4, 5, 7]
    assert np.array_equal(pool[untouched], pool_ref[untouched])


def test_decode_bad_slot_is_reported_not_faulted():
    import kda_gated_delta_03_gb300 as kda
    pool = to_dev(I.random_state(4, 2, 16, 16, 1))
    before = pool.clone()
    st = I.decode_step_inputs(2, 2, 16, 16, "f32", 1, 0)
    idx = to_dev(np.array([1, 9], np.int32))
    kda.kda_decode_step(*(to_dev(st[n]) for n in ("q", "k", "v", "beta", "alpha")), pool, idx)
    assert kda.kda_get_device_error() & 0x2
    assert torch.equal(pool[[0, 2, 3]], before[[0, 2, 3]])
    assert not torch.equal(pool[1], before[1])


def test_decode_equals_prefill_of_one_token():
    """A decode step is one token of the recurrence: it matches kda_prefill with T = 1 per sequence."""
    import kda_gated_delta_03_gb300 as kda
    B, H, d = 3, 2, 128
    st = I.decode_step_inputs(B, H, d, d, "f32", 60, 0, decay="slow")
    pool = I.random_state(B, H, d, d, 61)
    pool_d = to_dev(pool)
    o_dec = kda.kda_decode_step(*(to_dev(st[n]) for n in ("q", "k", "v", "beta", "alpha")), pool_d)
    cu = to_dev(np.arange(B + 1, dtype=np.int32))
    o_pre, s_pre = kda.kda_prefill(*(to_dev(st[n]) for n in ("q", "k", "v", "beta", "alpha")), cu, to_dev(pool))
    torch.cuda.synchronize()
    assert rel_frob(o_dec.cpu().numpy(), o_pre.cpu().numpy()) <= 1e-5
    assert rel_frob(pool_d.cpu().numpy(), s_pre.cpu().numpy()) <= 1e-5


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [16, 64, 128])
def test_decode_steps_bf16_state(dtype, d):
    """kda_decode_step_bf16_state against the oracle's bf16-stored state (rounded to nearest-even bf16
    after every step), over 8 steps."""
    o, o_ref, pool, pool_ref = run_steps(5, 3, d, dtype, 8, 80 + d, decay="slow", state_dtype="bf16")
    assert rel_frob(o, o_ref) <= 3e-3
    assert rel_frob(pool, pool_ref) <= 3e-3
    low = pool.astype(np.float32).view(np.uint32) & 0xFFFF
    assert not low.any()


def test_decode_bf16_state_idx_and_untouched_slots():
    idx = [6, 1, 3, 0]
    o, o_ref, pool, pool_ref = run_steps(4, 2, 128, "bf16", 3, 51, P=8, idx=idx, state_dtype="bf16")
    assert rel_frob(o, o_ref) <= 3e-3
    assert rel_frob(pool, pool_ref) <= 3e-3
    untouched = [2, 4, 5, 7]
    assert np.array_equal(pool[untouched], pool_ref[untouched])


def test_decode_bf16_state_many_states_per_cta():
    """Thousands of states, so that every CTA of the d = 128 bf16-state kernel streams several of them
    through its ring of shared-memory stages (and wraps around it), with a state_idx permutation."""
    B, H, d, P = 300, 8, 128, 310
    rng = np.random.default_rng(52)
    idx = rng.permutation(P)[:B].astype(np.int32)
    o, o_ref, pool, pool_ref = run_steps(B, H, d, "bf16", 3, 52, P=P, idx=idx, decay="slow", state_dtype="bf16")
    assert rel_frob(o, o_ref) <= 3e-3
    assert rel_frob(pool, pool_ref) <= 3e-3
    untouched = np.setdiff1d(np.arange(P), idx)
    assert np.array_equal(pool[untouched], pool_ref[untouched])


def test_decode_bf16_state_bad_slots_are_skipped():
    """Out-of-range slots among many valid ones: the error word says so, those rows touch nothing, and
    every other row is still stepped correctly."""
    import kda_gated_delta_03_gb300 as kda
    B, H, d, P = 700, 1, 128, 800
    rng = np.random.default_rng(53)
    idx = rng.permutation(P)[:B].astype(np.int32)
    bad = [5, 300, 699]
    idx[bad] = [-1, P, P + 7]
    good = np.setdiff1d(np.arange(B), bad)
    pool = I.bf16_bits_to_f32(I.f32_to_bf16_bits(I.random_state(P, H, d, d, 54)))
    pool_d = to_dev(I.f32_to_bf16_bits(pool), True)
    st = I.decode_step_inputs(B, H, d, d, "bf16", 55, 0, decay="slow")
    o = kda.kda_decode_step(*(to_dev(st[n], n in ("q", "k", "v")) for n in ("q", "k", "v", "beta", "alpha")),
                            pool_d, to_dev(idx))
    torch.cuda.synchronize()
    assert kda.kda_get_device_error() & 0x2
    sub = dict(st)
    for n in ("q", "k", "v", "beta", "alpha"):
        sub[n] = np.ascontiguousarray(st[n][good])
    ref = pool.astype(np.float64)
    o_ref = O.decode_step(sub, ref, idx[good], state_dtype="bf16")
    got = pool_d.double().cpu().numpy()
    assert rel_frob(o.double().cpu().numpy()[good], o_ref) <= 3e-3
    assert rel_frob(got[idx[good]], ref[idx[good]]) <= 3e-3
    untouched = np.setdiff1d(np.arange(P), idx[good])
    assert np.array_equal(got[untouched], ref[untouched])

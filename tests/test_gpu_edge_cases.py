"""Edge cases of the method on every prefill path at d = 128, against the float64 oracle.

Each case runs through the paths a kda_prefill call can take at d_k = d_v = 128:
  - "two_phase":     one bf16 sequence (per-chunk records, then the state chain);
  - "single_kernel": one bf16 sequence with the single_kernel option (tcgen05 chunk kernel);
  - "varlen":        several bf16 sequences (records of every sequence's chunks, one chain per sequence);
  - "varlen_single": several bf16 sequences with the single_kernel option (the tcgen05 chunk kernel,
                     longest-first order);
  - "fp32":          float32 inputs (the FFMA chunk kernel, 1e-4 tolerance).

The cases ("Kimi K3, explained", section "The math" and "Check yourself"):
  - the page's worked overwrite example, zero-padded to d = 128;
  - a unit key written with beta = 1 overwrites whatever the state held for that key (any state, any
    decay), placed inside long random sequences at chunk starts, chunk middles and chunk ends;
  - beta exactly 0 (nothing written) and exactly 1 on a share of the tokens;
  - decays far below the kernels' clamp (alpha = 1e-8 on some channels: every kernel treats
    alpha < 2^-15 as 2^-15), whose effect must stay inside the tolerances.
"""

import json
import os

import numpy as np
import pytest
import torch

from kda_gated_delta_03_gb300 import inputs as I
from oracle import oracle as O
from kda_testutil import TOL, rel_frob, to_dev

pytestmark = pytest.mark.gpu

PATHS = ["two_phase", "single_kernel", "varlen", "varlen_single", "fp32"]
SINGLE = ("single_kernel", "varlen_single")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import kda_gated_delta_03_gb300 as kda
    from kda_gated_delta_03_gb300 import build
    build.build()
    kda.load()
    yield
    assert kda.kda_get_device_error() == 0


def run_gpu(inp, single_kernel=False):
    import kda_gated_delta_03_gb300 as kda
    bf = inp["dtype"] == "bf16"
    o, st = kda.kda_prefill(to_dev(inp["q"], bf), to_dev(inp["k"], bf), to_dev(inp["v"], bf),
                            to_dev(inp["beta"]), to_dev(inp["alpha"]), to_dev(inp["cu_seqlens"]),
                            None if inp["state_in"] is None else to_dev(inp["state_in"]),
                            single_kernel=single_kernel)
    torch.cuda.synchronize()
    assert kda.kda_get_device_error() == 0
    return o.double().cpu().numpy(), st.double().cpu().numpy()


def path_inputs(path, seqlens, H, seed, state="randn"):
    """Seeded inputs for one path: a single sequence for the one-sequence paths, the same tokens split
    into several sequences for "varlen"."""
    dtype = "f32" if path == "fp32" else "bf16"
    if path.startswith("varlen"):
        T = sum(seqlens)
        cuts = [T // 3, T // 3 + 1, T - T // 3 - (T // 3 + 1)]
        seqlens = [c for c in cuts if c > 0] + [0]
    return I.prefill_inputs(seqlens, H, 128, 128, dtype, seed, decay="config", state=state)


def unit_bits(i, d, dtype):
    """A unit vector e_i in the storage dtype (bf16 bits or float32)."""
    e = np.zeros(d, np.float32)
    e[i] = 1.0
    return I.to_storage(e.astype(np.float64), dtype)


def check_oracle(inp, o, st):
    o_ref, st_ref = O.prefill(inp)
    tol = TOL[inp["dtype"]]
    e_o, e_s = rel_frob(o, o_ref), rel_frob(st, st_ref)
    assert e_o <= tol and e_s <= tol, (e_o, e_s)
    return o_ref


@pytest.mark.parametrize("path", PATHS)
def test_worked_overwrite_example_at_d128(path, golden_dir):
    """Write (k, a), then (k, b), with beta = 1, no decay and a zero state: reading k returns b, not the
    a + b that plain accumulation gives (values are exact in bf16)."""
    g = json.load(open(os.path.join(golden_dir, "overwrite_example.json")))
    dtype = "f32" if path == "fp32" else "bf16"
    d = 128
    key = unit_bits(g["key_index"], d, dtype)
    a = np.zeros(d)
    b = np.zeros(d)
    a[:4], b[:4] = g["a"], g["b"]
    reps = 2 if path.startswith("varlen") else 1          # two identical sequences for the batch paths
    q = np.stack([key, key] * reps)[:, None, :].copy()
    v = np.stack([I.to_storage(a, dtype), I.to_storage(b, dtype)] * reps)[:, None, :].copy()
    inp = dict(q=q, k=q.copy(), v=v, beta=np.ones((2 * reps, 1), np.float32),
               alpha=np.ones((2 * reps, 1, d), np.float32), cu_seqlens=I.cu_seqlens_of([2] * reps),
               state_in=None, dtype=dtype, H=1, dk=d, dv=d)
    o, st = run_gpu(inp, single_kernel=path in SINGLE)
    for r in range(reps):
        np.testing.assert_allclose(o[2 * r, 0, :4], g["a"], rtol=0, atol=1e-6)
        np.testing.assert_allclose(o[2 * r + 1, 0, :4], g["delta_read_after_both_writes"], rtol=0, atol=1e-6)
        assert np.all(o[2 * r + 1, 0, 4:] == 0)
        assert not np.allclose(o[2 * r + 1, 0, :4], g["linear_read_after_both_writes"])
    check_oracle(inp, o, st)


@pytest.mark.parametrize("path", PATHS)
def test_unit_key_overwrites_any_state(path):
    """Inside long random sequences with random initial states and the workload's per-channel decay,
    tokens whose key is a unit vector e_i, with beta = 1 and the query equal to the key, read back exactly
    their own value: S_t^T k_t = v_t for any S_{t-1} and alpha ("The math": beta = 1 with a unit key is a
    full overwrite).  Such tokens sit at chunk starts, middles and ends."""
    T = 700
    inp = path_inputs(path, [T], 2, 911)
    dtype = inp["dtype"]
    rows = [0, 37, 63, 64, 100, 127, 128, 250, 383, 511, 640, 699]
    for n, t in enumerate(rows):
        for h in range(2):
            e = unit_bits((17 * n + 5 * h) % 128, 128, dtype)
            inp["k"][t, h] = e
            inp["q"][t, h] = e
            inp["beta"][t, h] = 1.0
    o, st = run_gpu(inp, single_kernel=path in SINGLE)
    v = I.storage_to_f64(inp["v"], dtype)
    tol = 1e-4 if dtype == "f32" else 1e-2            # bf16: o is rounded to bf16 once
    for t in rows:
        np.testing.assert_allclose(o[t], v[t], rtol=tol, atol=tol)
    check_oracle(inp, o, st)


@pytest.mark.parametrize("path", PATHS)
def test_beta_exactly_zero_and_one(path):
    """A third of the tokens with beta = 0 (nothing is written: the state is only decayed) and a third
    with beta = 1 (the key's old content is fully erased before the write)."""
    inp = path_inputs(path, [600], 3, 912)
    rng = np.random.default_rng(912)
    u = rng.random(inp["beta"].shape)
    inp["beta"][u < 1 / 3] = 0.0
    inp["beta"][u > 2 / 3] = 1.0
    o, st = run_gpu(inp, single_kernel=path in SINGLE)
    check_oracle(inp, o, st)


@pytest.mark.parametrize("path", PATHS)
def test_decay_below_the_clamp(path):
    """alpha = 1e-8 on 5% of the (token, head, channel) entries, and on every channel of a few whole
    tokens: the kernels clamp log2 alpha at -15 (alpha >= 2^-15 ~= 3.1e-5), the oracle does not.  The
    departure is at most 2^-15 of the affected state rows and must stay inside the tolerances."""
    inp = path_inputs(path, [640], 2, 913)
    rng = np.random.default_rng(913)
    mask = rng.random(inp["alpha"].shape) < 0.05
    inp["alpha"][mask] = 1e-8
    inp["alpha"][[5, 64, 130, 400]] = 1e-8
    o, st = run_gpu(inp, single_kernel=path in SINGLE)
    check_oracle(inp, o, st)

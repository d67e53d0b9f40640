"""kda_prefill_backward against the float64 backward oracle (itself pinned to finite differences of the
forward oracle), on every forward path the recompute takes: CUDA-core fp32, single-kernel tensor-core
(several bf16 d=128 sequences) and two-phase (one bf16 d=128 sequence)."""

import numpy as np
import pytest
import torch

from kda_gated_delta_03_gb300 import inputs as I
from oracle.backward import prefill_backward
from kda_testutil import TOL, rel_frob, to_dev

pytestmark = pytest.mark.gpu


def run(seqlens, H, d, dtype, seed, decay="slow", with_states=True):
    import kda_gated_delta_03_gb300 as kda
    inp = I.prefill_inputs(seqlens, H, d, d, dtype, seed, decay=decay, state="randn" if with_states else "zero")
    rng = np.random.default_rng(seed + 1)
    T = inp["v"].shape[0]
    N = len(seqlens)
    do = rng.standard_normal((T, H, d)).astype(np.float32)
    if dtype == "bf16":                               # grad_o in the storage dtype, as the oracle sees it
        do_store = I.f32_to_bf16_bits(do)
        do = I.bf16_bits_to_f32(do_store)
    else:
        do_store = do
    dS = (0.1 * rng.standard_normal((N, H, d, d))).astype(np.float32) if with_states else None
    bf = dtype == "bf16"
    args = [to_dev(inp[n], bf and n in ("q", "k", "v")) for n in ("q", "k", "v", "beta", "alpha", "cu_seqlens")]
    gq, gk, gv, gb, ga, gs = kda.kda_prefill_backward(
        *args, to_dev(do_store, bf), to_dev(inp["state_in"]) if with_states else None,
        to_dev(dS) if with_states else None, want_state_grad=with_states)
    torch.cuda.synchronize()
    assert kda.kda_get_device_error() == 0
    got = dict(dq=gq, dk=gk, dv=gv, dbeta=gb, dalpha=ga)
    if with_states:
        got["d_state_in"] = gs
    else:
        assert gs is None
    ref = prefill_backward(inp, do, dS)
    return {n: (got[n].double().cpu().numpy(), ref[n]) for n in got}


@pytest.mark.parametrize("case", [([70, 1, 0, 130], 2, 16, "f32"), ([200], 2, 64, "f32"),
                                  ([100, 64, 129], 2, 128, "bf16"), ([300], 2, 128, "bf16"),
                                  ([700, 1100], 3, 128, "bf16"), ([2000], 1, 128, "bf16"),
                                  ([64, 128, 191], 2, 64, "bf16"), ([130, 64], 2, 128, "f32")],
                         ids=["cuda_core_d16", "cuda_core_d64", "tensor_core_varlen", "two_phase",
                              "tensor_core_many_chunks", "two_phase_many_chunks", "cuda_core_bf16_boundaries",
                              "matrix_form_fp32"])
def test_backward_matches_oracle(case):
    seqlens, H, d, dtype = case
    res = run(seqlens, H, d, dtype, 61 + d)
    tol = TOL[dtype]
    for name, (got, ref) in res.items():
        assert rel_frob(got, ref) <= tol, (name, rel_frob(got, ref))


def test_backward_zero_states():
    """No initial state, no final-state gradient, no state gradient requested."""
    res = run([150, 80], 2, 64, "f32", 77, with_states=False)
    for name, (got, ref) in res.items():
        assert rel_frob(got, ref) <= TOL["f32"], (name, rel_frob(got, ref))


def test_backward_bad_cu_seqlens_is_reported_not_faulted():
    """A cu_seqlens that is not non-decreasing within [0, T] (here two sequences both span all 200
    tokens, so their 64-token boundaries would need twice the slots the workspace holds) is caught on
    the device: the error word says so and every write stays inside the workspace's slots."""
    import kda_gated_delta_03_gb300 as kda
    inp = I.prefill_inputs([100, 100], 1, 16, 16, "f32", 78)
    cu = to_dev(np.array([0, 200, 0, 200], np.int32))
    args = [to_dev(inp[n]) for n in ("q", "k", "v", "beta", "alpha")]
    do = torch.zeros_like(args[2])
    kda.kda_prefill_backward(*args, cu, do)
    torch.cuda.synchronize()
    assert kda.kda_get_device_error() & 0x1
    assert kda.kda_get_device_error() == 0


def test_backward_workload_decay_from_a_zero_state():
    """The workload's decay (strong: about a factor 10 per token) from a zero initial state, over several
    chunks at d = 128: the decay gradient of the first rows is a sum whose terms cancel almost exactly
    (alpha of the first token multiplies a zero state), which is where a low-precision chunk form shows."""
    res = run([1024], 2, 128, "bf16", 84, decay="config", with_states=False)
    for name, (got, ref) in res.items():
        assert rel_frob(got, ref) <= TOL["bf16"], (name, rel_frob(got, ref))


@pytest.mark.parametrize("case", [([300], 2, 128, "bf16"), ([100, 64, 129], 2, 128, "bf16"), ([70, 1, 130], 2, 16, "f32")],
                         ids=["two_phase", "tensor_core_varlen", "cuda_core_d16"])
def test_backward_is_bit_reproducible(case):
    """Two calls on the same inputs give the same bits: every sum of the backward has a fixed order (no
    floating-point atomics), so a training step can be replayed exactly."""
    import kda_gated_delta_03_gb300 as kda
    seqlens, H, d, dtype = case
    inp = I.prefill_inputs(seqlens, H, d, d, dtype, 91, state="randn")
    T, N, bf = inp["v"].shape[0], len(seqlens), dtype == "bf16"
    rng = np.random.default_rng(92)
    do = rng.standard_normal((T, H, d)).astype(np.float32)
    do = I.f32_to_bf16_bits(do) if bf else do
    dS = (0.1 * rng.standard_normal((N, H, d, d))).astype(np.float32)
    args = [to_dev(inp[n], bf and n in ("q", "k", "v")) for n in ("q", "k", "v", "beta", "alpha", "cu_seqlens")]
    outs = []
    for _ in range(2):
        r = kda.kda_prefill_backward(*args, to_dev(do, bf), to_dev(inp["state_in"]), to_dev(dS), want_state_grad=True)
        torch.cuda.synchronize()
        outs.append([t.contiguous().view(torch.uint8).cpu().numpy() for t in r])
    assert kda.kda_get_device_error() == 0
    for a, b in zip(*outs):
        assert np.array_equal(a, b)

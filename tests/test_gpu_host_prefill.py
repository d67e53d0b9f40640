"""kda_prefill_host (inputs and outputs in host memory, transfers overlapped with the compute) against
the device-buffer kda_prefill and the oracle."""

import numpy as np
import pytest
import torch

from kda_gated_delta_03_gb300 import inputs as I
from oracle import oracle as O
from kda_testutil import TOL, prefill_gpu, rel_frob

pytestmark = pytest.mark.gpu


def to_host(a, bf16=False, pin=True):
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if bf16 else torch.from_numpy(a)
    return t.pin_memory() if pin else t.clone()


def host_run(inp, pin=True, state=True):
    import kda_gated_delta_03_gb300 as kda
    bf = inp["dtype"] == "bf16"
    args = [to_host(inp[n], bf and n in ("q", "k", "v"), pin) for n in ("q", "k", "v", "beta", "alpha")]
    cu = torch.from_numpy(np.ascontiguousarray(inp["cu_seqlens"]))
    s0 = None if inp["state_in"] is None or not state else to_host(np.asarray(inp["state_in"], np.float32), pin=pin)
    o, st = kda.kda_prefill_host(*args, cu, s0)
    torch.cuda.synchronize()
    return o.double().numpy(), st.double().numpy()


def test_one_sequence_equals_the_device_call_bit_for_bit():
    """One sequence is cut at multiples of 64 tokens with its state carried: the chunks are those of one
    kda_prefill call, so o and the final state are identical."""
    inp = I.prefill_inputs([3000], 2, 128, 128, "bf16", 91, decay="slow", state="randn")
    o_h, s_h = host_run(inp)
    o_d, s_d = prefill_gpu(inp)
    assert np.array_equal(o_h, o_d)
    assert np.array_equal(s_h, s_d)
    o_ref, s_ref = O.prefill(inp)
    assert rel_frob(o_h, o_ref) <= TOL["bf16"] and rel_frob(s_h, s_ref) <= TOL["bf16"]


@pytest.mark.parametrize("case", [([700, 1500, 30, 0, 900, 2100], 2, 128, "bf16"), ([70, 1, 0, 130], 2, 16, "f32"),
                                  ([1200, 64, 900], 2, 64, "bf16")],
                         ids=["tensor_core_groups", "cuda_core_fp32", "cuda_core_bf16"])
def test_several_sequences_match_the_oracle(case):
    seqlens, H, d, dt = case
    inp = I.prefill_inputs(seqlens, H, d, d, dt, 92, decay="slow", state="randn")
    o_h, s_h = host_run(inp)
    o_ref, s_ref = O.prefill(inp)
    assert rel_frob(o_h, o_ref) <= TOL[dt] and rel_frob(s_h, s_ref) <= TOL[dt]


def test_pageable_buffers_and_no_initial_state():
    inp = I.prefill_inputs([500, 260], 2, 128, 128, "bf16", 93, decay="slow")
    o_h, s_h = host_run(inp, pin=False)
    o_ref, s_ref = O.prefill(inp)
    assert rel_frob(o_h, o_ref) <= TOL["bf16"] and rel_frob(s_h, s_ref) <= TOL["bf16"]


def test_zero_tokens_copies_the_state():
    inp = I.prefill_inputs([0, 0], 2, 16, 16, "f32", 94, state="randn")
    o_h, s_h = host_run(inp)
    assert o_h.shape == (0, 2, 16)
    assert np.array_equal(s_h, np.asarray(inp["state_in"], np.float32).astype(np.float64))

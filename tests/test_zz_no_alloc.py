"""The allocation-free prefill entry point, kda_prefill_noalloc.

Some callers cannot allocate device memory: a serving process whose memory manager reserves the GPU's
memory up front and hands out no scratch, or a host program that reaches libkda only through its C ABI
and has no device allocator.  kda_prefill_noalloc serves them: it takes no workspace and keeps its
scratch (the longest-first order of the sequences) in a fixed static device array instead.

These tests call it through the C ABI and check its results against kda_prefill on the same inputs, on
two calls in a row (the static array keeps the previous call's contents).  The file is named so that
pytest collects it last.
"""

import ctypes
import os
import shutil

import numpy as np
import pytest
import torch

from kda_gated_delta_03_gb300 import binding, build
from kda_gated_delta_03_gb300 import inputs as I
from kda_testutil import TOL, rel_frob, to_dev
from oracle import oracle as O

HAVE_NVCC = shutil.which("nvcc") is not None or os.path.exists("/usr/local/cuda/bin/nvcc")


def _device_inputs(inp):
    bf = inp["dtype"] == "bf16"
    t = {n: to_dev(inp[n], bf and n in ("q", "k", "v")) for n in ("q", "k", "v", "beta", "alpha", "cu_seqlens")}
    t["state_in"] = None if inp["state_in"] is None else to_dev(inp["state_in"])
    return t


@pytest.mark.gpu
def test_noalloc_matches_prefill_on_two_calls_in_a_row():
    """Several sequences: the no-alloc call runs the same kernels as kda_prefill with the single-kernel
    option (no records); only the home of the longest-first sequence order differs.  So its results must be
    bit-identical, on two calls in a row with different sequence counts (an order left stale by the first
    call would skip or repeat sequences), and within tolerance of the float64 oracle."""
    build.build()
    binding.load()
    cases = [
        I.prefill_inputs([70, 150, 33, 0, 200], 2, 128, 128, "bf16", 71, decay="slow", state="randn"),
        I.prefill_inputs([9, 300, 64, 65], 3, 64, 64, "f32", 72, decay="config", state="randn"),
    ]
    devs = [_device_inputs(inp) for inp in cases]
    # outputs allocated up front, so the no-alloc calls themselves allocate nothing
    outs = []
    for inp, d in zip(cases, devs):
        T, H, dv = inp["v"].shape
        N = len(inp["cu_seqlens"]) - 1
        outs.append((torch.empty((T, H, dv), dtype=d["q"].dtype, device="cuda:0"),
                     torch.empty((N, H, inp["dk"], dv), dtype=torch.float32, device="cuda:0")))
    for d, (o, st) in zip(devs, outs):          # two no-alloc calls back to back
        binding.kda_prefill_noalloc(d["q"], d["k"], d["v"], d["beta"], d["alpha"], d["cu_seqlens"], d["state_in"],
                                    o=o, state_out=st)
    torch.cuda.synchronize()
    for inp, d, (o, st) in zip(cases, devs, outs):
        # bf16 d=128 batches take kda_prefill's record-based path by default; the single-kernel option selects
        # the path the no-alloc call runs
        o_ref, st_ref = binding.kda_prefill(d["q"], d["k"], d["v"], d["beta"], d["alpha"], d["cu_seqlens"],
                                            d["state_in"], single_kernel=inp["dtype"] == "bf16")
        torch.cuda.synchronize()
        assert torch.equal(o.view(torch.int16) if o.dtype == torch.bfloat16 else o,
                           o_ref.view(torch.int16) if o_ref.dtype == torch.bfloat16 else o_ref)
        assert torch.equal(st, st_ref)
        o64, st64 = O.prefill(inp)
        tol = TOL[inp["dtype"]]
        assert rel_frob(o.double().cpu().numpy(), o64) <= tol
        assert rel_frob(st.double().cpu().numpy(), st64) <= tol
    assert binding.kda_get_device_error() == 0


@pytest.mark.gpu
def test_noalloc_one_sequence_runs_the_single_kernel_path():
    """One bf16 d=128 sequence: without a workspace for per-chunk records, the no-alloc call takes the
    single-kernel chunkwise path.  It must equal kda_prefill_ex with single_kernel set, bit for bit, on two
    calls in a row, and the float64 oracle within the bf16 tolerance."""
    build.build()
    binding.load()
    inp = I.prefill_inputs([709], 3, 128, 128, "bf16", 73, decay="config", state="randn")
    d = _device_inputs(inp)
    T, H, dv = inp["v"].shape
    o = torch.empty((T, H, dv), dtype=torch.bfloat16, device="cuda:0")
    st = torch.empty((1, H, 128, dv), dtype=torch.float32, device="cuda:0")
    o_ref, st_ref = binding.kda_prefill(d["q"], d["k"], d["v"], d["beta"], d["alpha"], d["cu_seqlens"],
                                        d["state_in"], single_kernel=True)
    for _ in range(2):
        o.zero_()
        st.zero_()
        binding.kda_prefill_noalloc(d["q"], d["k"], d["v"], d["beta"], d["alpha"], d["cu_seqlens"], d["state_in"],
                                    o=o, state_out=st)
        torch.cuda.synchronize()
        assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
        assert torch.equal(st, st_ref)
    o64, st64 = O.prefill(inp)
    assert rel_frob(o.double().cpu().numpy(), o64) <= TOL["bf16"]
    assert rel_frob(st.double().cpu().numpy(), st64) <= TOL["bf16"]
    assert binding.kda_get_device_error() == 0


@pytest.mark.skipif(not HAVE_NVCC, reason="nvcc not available")
def test_noalloc_rejects_more_sequences_than_its_scratch_holds():
    """More than KDA_NOALLOC_MAX_SEQS sequences is refused on the host, before anything is launched."""
    build.build()
    L = binding.load()
    P = ctypes.c_void_p(0x10000)
    n = binding.KDA_NOALLOC_MAX_SEQS + 1
    rc = L.kda_prefill_noalloc(P, P, P, P, P, P, n, n, 2, 16, 16, 0, 1.0, None, P, P, None)
    assert rc == binding.KDA_ERR_TOO_LARGE
    assert binding.kda_status_string(rc) == "KDA_ERR_TOO_LARGE"

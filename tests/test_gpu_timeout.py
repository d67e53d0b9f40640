"""A bounded device wait that runs out: the give-up path of the tcgen05 prefill kernels.

Every mbarrier wait in the tensor-core prefill kernels is bounded; when one gives up, the kernel records
KDA_DEVERR_TIMEOUT in the device error word, stops its work, waits (bounded) for the copies it already
issued, frees its tensor memory and returns, so the CUDA context stays usable.  Nothing in a correct run
ever makes a wait run out, so this test uses a second build of the library with test hooks compiled in
(-DKDA_TEST_HOOKS): kda_test_stall_prefill(1) makes each prefill kernel wait, right after issuing its
first copies, on a barrier that nothing completes, with a limit of about 1 ms.

It runs in a child process that loads only that build, and checks, for the two-phase path (one
sequence), the single-kernel path and the several-sequence path:
  - the call returns and the stream completes promptly (no hang);
  - KDA_DEVERR_TIMEOUT is reported through kda_get_device_error;
  - with the hook disarmed, the next call on the same context is clean and matches the float64 oracle.
"""

import os
import subprocess
import sys

import pytest

from kda_gated_delta_03_gb300 import build

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import ctypes, sys, time
sys.path.insert(0, ROOT); sys.path.insert(0, ROOT + "/tests")
import numpy as np, torch
from kda_gated_delta_03_gb300 import binding, inputs as I
from oracle import oracle as O
from kda_testutil import TOL, rel_frob, to_dev

L = binding.load()
assert L._name.endswith("libkda_test.so"), L._name
L.kda_test_stall_prefill.argtypes = [ctypes.c_int32]
L.kda_test_stall_prefill.restype = None
TIMEOUT = 0x4

def run(inp, single_kernel):
    o, st = binding.kda_prefill(to_dev(inp["q"], True), to_dev(inp["k"], True), to_dev(inp["v"], True),
                                to_dev(inp["beta"]), to_dev(inp["alpha"]), to_dev(inp["cu_seqlens"]),
                                to_dev(inp["state_in"]), single_kernel=single_kernel)
    return o, st

cases = [("two_phase", [300], False), ("single_kernel", [300], True), ("varlen", [100, 70, 130], False)]
for name, seqlens, sk in cases:
    inp = I.prefill_inputs(seqlens, 2, 128, 128, "bf16", 931, decay="config", state="randn")
    L.kda_test_stall_prefill(1)
    t0 = time.perf_counter()
    run(inp, sk)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    bits = binding.kda_get_device_error()
    assert bits & TIMEOUT, (name, bits)
    assert dt < 30.0, (name, dt)
    L.kda_test_stall_prefill(0)
    o, st = run(inp, sk)
    torch.cuda.synchronize()
    assert binding.kda_get_device_error() == 0, name
    o_ref, st_ref = O.prefill(inp)
    e_o = rel_frob(o.double().cpu().numpy(), o_ref)
    e_s = rel_frob(st.double().cpu().numpy(), st_ref)
    assert e_o <= TOL["bf16"] and e_s <= TOL["bf16"], (name, e_o, e_s)
    print(name, "gave up in %.3f s, then clean: o %.2e, state %.2e" % (dt, e_o, e_s))
print("OK")
"""


def test_a_wait_that_runs_out_is_reported_and_the_next_call_is_clean():
    lib = build.build_test_variant()
    env = dict(os.environ, KDA_LIBRARY=lib)
    r = subprocess.run([sys.executable, "-c", f"ROOT = {ROOT!r}\n" + CHILD], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("OK"), r.stdout + r.stderr

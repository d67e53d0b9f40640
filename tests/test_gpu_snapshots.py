"""State snapshots of kda_prefill_ex (the state after every `snapshot_every` tokens of each sequence)
against the float64 oracle, on the three prefill paths: two-phase (one bf16 d=128 sequence, with and
without multiple windows), single-kernel tensor-core (several bf16 sequences) and CUDA-core (fp32)."""

import numpy as np
import pytest
import torch

from kda_gated_delta_03_gb300 import inputs as I
from oracle import oracle as O
from kda_testutil import TOL, rel_frob, to_dev

pytestmark = pytest.mark.gpu


def run(inp, every, workspace_chunks=None):
    import kda_gated_delta_03_gb300 as kda
    bf = inp["dtype"] == "bf16"
    args = [to_dev(inp[n], bf and n in ("q", "k", "v")) for n in ("q", "k", "v", "beta", "alpha", "cu_seqlens")]
    s0 = None if inp["state_in"] is None else to_dev(inp["state_in"])
    ref, offs = O.prefill_snapshots(inp, every)
    snaps = torch.full((max(len(ref), 1), inp["H"], inp["dk"], inp["dv"]), float("nan"), device="cuda:0")
    ws = None
    if workspace_chunks:
        ws = torch.empty(workspace_chunks * inp["H"] * 99072, dtype=torch.uint8, device="cuda:0")
    o, st = kda.kda_prefill(*args, s0, workspace=ws, snapshot_every=every, snapshots=snaps,
                            snapshot_offsets=to_dev(offs))
    torch.cuda.synchronize()
    assert kda.kda_get_device_error() == 0
    return o.double().cpu().numpy(), st.double().cpu().numpy(), snaps.double().cpu().numpy()[:len(ref)], ref


@pytest.mark.parametrize("workspace_chunks,H", [(None, 2), (3, 2), (3, 12)])
def test_snapshots_two_phase(workspace_chunks, H):
    """H = 2 runs the chain on 16-column slices, H = 12 on 32-column slices."""
    inp = I.prefill_inputs([700], H, 128, 128, "bf16", 90, decay="slow", state="randn")
    o, st, snaps, ref = run(inp, 128, workspace_chunks)
    assert ref.shape[0] == 5
    assert rel_frob(snaps, ref) <= TOL["bf16"]
    o_ref, st_ref = O.prefill(inp)
    assert rel_frob(o, o_ref) <= TOL["bf16"] and rel_frob(st, st_ref) <= TOL["bf16"]


def test_snapshots_tensor_core_varlen():
    inp = I.prefill_inputs([300, 64, 129, 0, 256], 2, 128, 128, "bf16", 91, decay="config", state="randn")
    o, st, snaps, ref = run(inp, 64)
    assert ref.shape[0] == 4 + 1 + 2 + 0 + 4
    assert rel_frob(snaps, ref) <= TOL["bf16"]


def test_snapshots_cuda_core_fp32():
    inp = I.prefill_inputs([200, 384, 17], 2, 64, 64, "f32", 92, decay="slow", state="randn")
    o, st, snaps, ref = run(inp, 128)
    assert ref.shape[0] == 1 + 3 + 0
    assert rel_frob(snaps, ref) <= TOL["f32"]
    assert np.array_equal(snaps[3], st[1])            # a snapshot at a sequence's end is its state_out


def test_snapshot_offsets_that_disagree_are_reported():
    import kda_gated_delta_03_gb300 as kda
    inp = I.prefill_inputs([128, 128], 1, 16, 16, "f32", 93)
    args = [to_dev(inp[n]) for n in ("q", "k", "v", "beta", "alpha", "cu_seqlens")]
    snaps = torch.zeros((4, 1, 16, 16), device="cuda:0")
    bad = to_dev(np.array([0, 1, 4], np.int32))       # sequence 0 has 2 snapshot points, not 1
    kda.kda_prefill(*args, None, snapshot_every=64, snapshots=snaps, snapshot_offsets=bad)
    assert kda.kda_get_device_error() & 0x8
    assert kda.kda_get_device_error() == 0

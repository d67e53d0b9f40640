"""Gated DeltaNet (one alpha per token and head) and DeltaNet (no decay) layouts of alpha, on every
prefill path and on decode, against the float64 oracle."""

import numpy as np
import pytest
import torch

from kda_gated_delta_03_gb300 import inputs as I
from oracle import oracle as O
from kda_testutil import TOL, rel_frob, to_dev

pytestmark = pytest.mark.gpu
PER_HEAD, NONE = 1, 2


def with_layout(inp, mode):
    """The same inputs with alpha in layout `mode` ("scalar" decay draws one value per (token, head),
    repeated over the key channels, so its first channel is the per-head alpha)."""
    if mode == PER_HEAD:
        return dict(inp, alpha=np.ascontiguousarray(inp["alpha"][..., 0]), alpha_mode=PER_HEAD)
    return dict(inp, alpha=None, alpha_mode=NONE)


def run_prefill(inp):
    import kda_gated_delta_03_gb300 as kda
    bf = inp["dtype"] == "bf16"
    args = [to_dev(inp[n], bf and n in ("q", "k", "v")) if inp[n] is not None else None
            for n in ("q", "k", "v", "beta", "alpha", "cu_seqlens")]
    s0 = None if inp["state_in"] is None else to_dev(inp["state_in"])
    o, st = kda.kda_prefill(*args, s0, alpha_mode=inp["alpha_mode"])
    torch.cuda.synchronize()
    return o.double().cpu().numpy(), st.double().cpu().numpy()


CASES = [([700], 2, 128, "bf16"),                   # two-phase path
         ([300, 64, 129, 0], 2, 128, "bf16"),        # single-kernel tensor-core path
         ([200, 77], 2, 64, "f32")]                  # CUDA-core path


@pytest.mark.parametrize("case", CASES, ids=["two_phase", "tensor_core", "cuda_core"])
@pytest.mark.parametrize("mode", [PER_HEAD, NONE], ids=["gated_deltanet", "deltanet"])
def test_prefill_alpha_layouts(case, mode):
    import kda_gated_delta_03_gb300 as kda
    seqlens, H, d, dtype = case
    base = I.prefill_inputs(seqlens, H, d, d, dtype, 95, decay="scalar" if mode == PER_HEAD else "one",
                            state="randn")
    inp = with_layout(base, mode)
    o, st = run_prefill(inp)
    o_ref, st_ref = O.prefill(inp)
    assert rel_frob(o, o_ref) <= TOL[dtype] and rel_frob(st, st_ref) <= TOL[dtype]
    assert kda.kda_get_device_error() == 0


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("mode", [PER_HEAD, NONE], ids=["gated_deltanet", "deltanet"])
def test_decode_alpha_layouts(mode, state_dtype):
    import kda_gated_delta_03_gb300 as kda
    B, H, d = 5, 3, 128
    pool = I.random_state(B, H, d, d, 96)
    if state_dtype == "bf16":
        pool = I.bf16_bits_to_f32(I.f32_to_bf16_bits(pool))
        pool_d = to_dev(I.f32_to_bf16_bits(pool), True)
    else:
        pool_d = to_dev(pool)
    ref = pool.astype(np.float64)
    og, orf = [], []
    for s in range(4):
        st = with_layout(I.decode_step_inputs(B, H, d, d, "bf16", 97, s,
                                              decay="scalar" if mode == PER_HEAD else "one"), mode)
        o = kda.kda_decode_step(*(to_dev(st[n], n in ("q", "k", "v")) for n in ("q", "k", "v", "beta")),
                                None if st["alpha"] is None else to_dev(st["alpha"]), pool_d, alpha_mode=mode)
        og.append(o.double().cpu().numpy())
        orf.append(O.decode_step(st, ref, state_dtype=state_dtype))
    torch.cuda.synchronize()
    assert rel_frob(np.stack(og), np.stack(orf)) <= 3e-3
    assert rel_frob(pool_d.double().cpu().numpy(), ref) <= 3e-3

"""Host checks of the seeded input generator shared by the CUDA path and the oracle."""

import numpy as np
import torch

from kda_gated_delta_03_gb300 import inputs as I


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100_000).astype(np.float32),
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.005859375, 3.4e38, -1e-40], np.float32)])
    ours = I.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = I.bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_reproducible_and_block_independent():
    a = I.token_inputs(I.BLOCK + 100, 2, 16, 8, "bf16", 7)
    b = I.token_inputs(I.BLOCK + 100, 2, 16, 8, "bf16", 7, threads=1)
    for key in a:
        assert np.array_equal(a[key], b[key])
    c = I.token_inputs(I.BLOCK + 100, 2, 16, 8, "bf16", 8)
    assert not np.array_equal(a["q"], c["q"])


def test_distributions():
    d = I.token_inputs(5000, 4, 128, 64, "bf16", 1)
    q = I.bf16_bits_to_f32(d["q"]).astype(np.float64)
    norms = np.linalg.norm(q, axis=-1)
    assert np.all(np.abs(norms - 1) < 1e-2)
    assert np.all((d["beta"] > 0) & (d["beta"] < 1))
    assert np.all((d["alpha"] > 0) & (d["alpha"] < 1))
    la = np.log(d["alpha"].astype(np.float64))
    assert abs(la.mean() + 2.18) < 0.03          # E[softplus(N(0,1) + 2)] ~= 2.18
    v = I.bf16_bits_to_f32(d["v"])
    assert abs(v.std() - 1) < 0.02
    s = I.random_state(2, 4, 16, 16, 3)
    assert abs(s.std() - 0.02) < 0.002


def test_decay_modes():
    one = I.token_inputs(10, 2, 8, 8, "f32", 1, decay="one")
    assert np.all(one["alpha"] == 1)
    sc = I.token_inputs(10, 2, 8, 8, "f32", 1, decay="scalar")
    assert np.all(sc["alpha"] == sc["alpha"][:, :, :1])
    slow = I.token_inputs(2000, 2, 8, 8, "f32", 1, decay="slow")
    assert abs(np.log(slow["alpha"].astype(np.float64)).mean() + 2.18 / 64) < 0.002


def test_varlen_workload_lengths():
    s, lens = I.varlen_lengths()
    assert s == 4 and len(lens) == 64 and sum(lens) == 291_042
    assert min(lens) >= 128 and max(lens) <= 16384
    w = I.workload("varlen_64")
    assert w["seqlens"] == lens

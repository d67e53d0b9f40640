"""Parity at the full workload sizes, in the launch configuration the benchmark times.

The oracle computes every output where it finishes in seconds (prefill_8k); for the larger workloads it
computes a sample of whole (sequence, head) units or decode rows, which the CUDA results must match to the
same relative Frobenius bound."""

import numpy as np
import pytest
import torch

from kda_gated_delta_03_gb300 import inputs as I
from oracle import oracle as O
from kda_testutil import prefill_gpu, rel_frob, to_dev

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
TOL = 3e-3


def test_prefill_8k_full():
    w = I.workload("prefill_8k")
    inp = I.prefill_inputs(w["seqlens"], w["H"], w["dk"], w["dv"], w["dtype"], w["seed"], state=w["state"])
    o, st = prefill_gpu(inp)
    o_ref, st_ref = O.prefill(inp)
    assert rel_frob(o, o_ref) <= TOL
    assert rel_frob(st, st_ref) <= TOL


def test_varlen_64_sampled_units():
    w = I.workload("varlen_64")
    inp = I.prefill_inputs(w["seqlens"], w["H"], w["dk"], w["dv"], w["dtype"], w["seed"], state=w["state"])
    o, st = prefill_gpu(inp)
    lens = np.array(w["seqlens"])
    order = np.argsort(-lens)
    seqs = [int(order[0]), int(order[1]), int(order[len(order) // 2]), int(order[-1])]   # longest .. shortest
    units = [(n, h) for n in seqs for h in (0, 13, 31)]
    res = O.prefill_units(inp, units)
    cu = inp["cu_seqlens"]
    o_s = np.concatenate([o[cu[n]:cu[n + 1], h] for n, h in units])
    o_r = np.concatenate([res[u][0] for u in units])
    assert rel_frob(o_s, o_r) <= TOL
    assert rel_frob(np.stack([st[n, h] for n, h in units]), np.stack([res[u][1] for u in units])) <= TOL


def test_decode_512x32_sampled_rows():
    """All 256 steps over the full 512 x 32 pool; the oracle follows 16 of the 512 sequences."""
    import kda_gated_delta_03_gb300 as kda
    w = I.workload("decode_512x32")
    B, H, d = w["B"], w["H"], w["dk"]
    rows = np.arange(0, B, B // 16)
    pool = np.concatenate([I.random_state(64, H, d, d, (w["seed"], b0)) for b0 in range(0, B, 64)])
    pool_d = to_dev(pool)
    ref = pool[rows].astype(np.float64)
    og, orf = [], []
    for s in range(w["steps"]):
        st = I.decode_step_inputs(B, H, d, d, w["dtype"], w["seed"], s)
        o = kda.kda_decode_step(*(to_dev(st[n], n in ("q", "k", "v")) for n in ("q", "k", "v")),
                                to_dev(st["beta"]), to_dev(st["alpha"]), pool_d)
        og.append(o[torch.from_numpy(rows).to(o.device)].double().cpu().numpy())
        sub = dict(st)
        for n in ("q", "k", "v", "beta", "alpha"):
            sub[n] = np.ascontiguousarray(st[n][rows])
        orf.append(O.decode_step(sub, ref))
    torch.cuda.synchronize()
    assert rel_frob(np.stack(og), np.stack(orf)) <= TOL
    assert rel_frob(pool_d[torch.from_numpy(rows).to(pool_d.device)].double().cpu().numpy(), ref) <= TOL


def test_append_1m_sampled_heads():
    """1,032,192-token prefill then a 16,384-token append from the carried state; the oracle runs two of
    the eight heads over the whole million tokens.  The append must also equal the one-shot prefill."""
    w = I.workload("append_1m")
    T1, T2 = w["seqlens"][0], w["append"]
    full = I.prefill_inputs([T1 + T2], w["H"], w["dk"], w["dv"], w["dtype"], w["seed"])

    def part(t0, t1):
        d = dict(full)
        for n in ("q", "k", "v", "beta", "alpha"):
            d[n] = np.ascontiguousarray(full[n][t0:t1])
        d["cu_seqlens"] = I.cu_seqlens_of([t1 - t0])
        return d

    o1, s1 = prefill_gpu(part(0, T1))
    o2, s2 = prefill_gpu(part(T1, T1 + T2), state_in=s1.astype(np.float32))
    heads = [0, 5]
    res = O.prefill_units(full, [(0, h) for h in heads])
    for h in heads:
        o_ref, s_ref = res[(0, h)]
        assert rel_frob(o1[:, h], o_ref[:T1]) <= TOL
        assert rel_frob(o2[:, h], o_ref[T1:]) <= TOL
        assert rel_frob(s2[0, h], s_ref) <= TOL
    o_one, s_one = prefill_gpu(full)
    assert np.array_equal(np.concatenate([o1, o2]), o_one)          # chunk-aligned split: identical chunking
    assert np.array_equal(s2, s_one)


def test_prefill_8k_backward_sampled_heads():
    """The backward pass at the full prefill_8k size, in the configuration the benchmark times (no initial
    state, no final-state gradient, 4,096 chunk units on every SM); the float64 backward oracle follows two
    of the 32 heads, each of which depends on its own head's inputs only."""
    import kda_gated_delta_03_gb300 as kda
    from oracle.backward import prefill_backward
    w = I.workload("prefill_8k")
    inp = I.prefill_inputs(w["seqlens"], w["H"], w["dk"], w["dv"], w["dtype"], w["seed"], state=w["state"])
    T, H, d = inp["v"].shape
    do = I.f32_to_bf16_bits(np.random.default_rng(8).standard_normal((T, H, d)).astype(np.float32))
    args = [to_dev(inp[n], n in ("q", "k", "v")) for n in ("q", "k", "v", "beta", "alpha", "cu_seqlens")]
    gq, gk, gv, gb, ga, gs = kda.kda_prefill_backward(*args, to_dev(do, True))
    torch.cuda.synchronize()
    assert kda.kda_get_device_error() == 0
    heads = [0, 21]
    sub = dict(inp, H=len(heads))
    for n in ("q", "k", "v", "beta", "alpha"):
        sub[n] = np.ascontiguousarray(inp[n][:, heads])
    ref = prefill_backward(sub, I.bf16_bits_to_f32(np.ascontiguousarray(do[:, heads])))
    got = dict(dq=gq, dk=gk, dv=gv, dbeta=gb, dalpha=ga, d_state_in=gs)
    for name, t in got.items():
        g = t.double().cpu().numpy()[:, heads]
        assert rel_frob(g, ref[name]) <= TOL, (name, rel_frob(g, ref[name]))

"""Parity of kda_prefill (CUDA, through the C ABI) with the float64 oracle, element by element,
on seeded inputs that span several chunks, ragged tails and the degenerate cases."""

import json
import os

import numpy as np
import pytest
import torch

from kda_gated_delta_03_gb300 import inputs as I
from oracle import oracle as O
from kda_testutil import TOL, prefill_gpu, rel_frob, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import kda_gated_delta_03_gb300 as kda
    from kda_gated_delta_03_gb300 import build
    build.build()
    kda.load()
    yield
    assert kda.kda_get_device_error() == 0


def check(inp, tol=None, scale=1.0):
    tol = tol or TOL[inp["dtype"]]
    o, st = prefill_gpu(inp, scale=scale)
    o_ref, st_ref = O.prefill(inp, scale=scale)
    e_o, e_s = rel_frob(o, o_ref), rel_frob(st, st_ref)
    assert e_o <= tol and e_s <= tol, (e_o, e_s)
    return e_o, e_s


def test_tiny_fp32_workload():
    """B=1, H=2, T=64, d=16, fp32 throughout, zero initial state (the tiny correctness workload)."""
    w = I.workload("tiny_fp32")
    inp = I.prefill_inputs(w["seqlens"], w["H"], w["dk"], w["dv"], w["dtype"], w["seed"], state=w["state"])
    check(inp, 1e-4)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [16, 64, 128])
@pytest.mark.parametrize("decay", ["config", "slow", "one", "scalar"])
def test_ragged_varlen(dtype, d, decay):
    """Lengths 1, 63, 64, 65, 0 and 200 packed together, random initial states."""
    inp = I.prefill_inputs([1, 63, 64, 65, 0, 200], 3, d, d, dtype, 100 + d, decay=decay, state="randn")
    check(inp)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_long_carry_slow_decay(dtype):
    """Slow decay over 1000 tokens, so the carried state matters across many chunks."""
    inp = I.prefill_inputs([1000], 2, 128, 128, dtype, 7, decay="slow", state="randn")
    check(inp)


def test_many_units_wide_slices():
    """At least 148 (sequence, head) units: the bf16 d=128 path carries 64 value columns per CTA."""
    rng = np.random.default_rng(77)
    seqlens = [int(x) for x in rng.integers(1, 200, size=40)]
    inp = I.prefill_inputs(seqlens, 4, 128, 128, "bf16", 78, decay="slow", state="randn")
    check(inp)


@pytest.mark.parametrize("seqlens,H", [([int(x) for x in np.random.default_rng(77).integers(1, 200, size=40)], 4),
                                         ([1, 63, 64, 65, 0, 200], 3)])
def test_single_kernel_path_for_several_sequences(seqlens, H):
    """The single-kernel option runs several bf16 d=128 sequences on the tcgen05 chunk kernel (64-column
    slices once sequences x heads >= 148, 32-column slices below), matching the oracle."""
    import kda_gated_delta_03_gb300 as kda
    inp = I.prefill_inputs(seqlens, H, 128, 128, "bf16", 78, decay="slow", state="randn")
    args = [to_dev(inp[n], n in ("q", "k", "v")) for n in ("q", "k", "v", "beta", "alpha", "cu_seqlens")]
    o, st = kda.kda_prefill(*args, to_dev(inp["state_in"]), single_kernel=True)
    torch.cuda.synchronize()
    o_ref, st_ref = O.prefill(inp)
    assert rel_frob(o.double().cpu().numpy(), o_ref) <= 3e-3
    assert rel_frob(st.double().cpu().numpy(), st_ref) <= 3e-3


def test_records_path_for_several_sequences():
    """Several bf16 d=128 sequences take the record-based path: every sequence's chunks get their records,
    then one chain CTA per (sequence, head, value slice) walks its own chunks.  Each sequence's o and state
    equal, bit for bit, a one-sequence call on it; a workspace of only a few chunks (many windows, sequences
    split across windows, their state carried through state_out, also in place) gives identical results;
    and the oracle agrees."""
    import kda_gated_delta_03_gb300 as kda
    seqlens = [300, 0, 65, 1, 700, 64, 129]
    H = 2
    inp = I.prefill_inputs(seqlens, H, 128, 128, "bf16", 41, decay="slow", state="randn")
    cu = inp["cu_seqlens"]
    args = [to_dev(inp[n], n in ("q", "k", "v")) for n in ("q", "k", "v", "beta", "alpha", "cu_seqlens")]
    s0 = to_dev(inp["state_in"])
    o, st = kda.kda_prefill(*args, s0)
    torch.cuda.synchronize()
    o_ref, st_ref = O.prefill(inp)
    assert rel_frob(o.double().cpu().numpy(), o_ref) <= 3e-3
    assert rel_frob(st.double().cpu().numpy(), st_ref) <= 3e-3
    for n in range(len(seqlens)):
        one = _sub_batch(inp, [n])
        o1, st1 = kda.kda_prefill(*[to_dev(one[m], m in ("q", "k", "v")) for m in ("q", "k", "v", "beta", "alpha",
                                                                                    "cu_seqlens")],
                                  to_dev(one["state_in"]))
        torch.cuda.synchronize()
        assert torch.equal(o1.view(torch.int16), o[cu[n]:cu[n + 1]].view(torch.int16)), n
        assert torch.equal(st1, st[n:n + 1]), n
    up = lambda x: (x + 255) // 256 * 256
    hdr = up(4 * (len(seqlens) + 1)) + up(4 * len(seqlens))
    for chunks in (1, 3):
        ws = torch.empty(hdr + chunks * H * 99072, dtype=torch.uint8, device="cuda:0")
        o2, st2 = kda.kda_prefill(*args, s0, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(o2.view(torch.int16), o.view(torch.int16)) and torch.equal(st2, st), chunks
    st3 = s0.clone()
    ws = torch.empty(hdr + 2 * H * 99072, dtype=torch.uint8, device="cuda:0")
    o3, _ = kda.kda_prefill(*args, st3, state_out=st3, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o3.view(torch.int16), o.view(torch.int16)) and torch.equal(st3, st)


@pytest.mark.parametrize("N", [127, 128, 200])
def test_records_path_for_many_sequences(N):
    """Up to 127 sequences, phase 1 looks chunks up in copies of the chunk offsets and cu_seqlens in shared
    memory; beyond that, in global memory.  Both sides of that limit match the oracle, with short and
    empty sequences mixed in, and a workspace of a few chunks (many windows) gives the same bits."""
    import kda_gated_delta_03_gb300 as kda
    rng = np.random.default_rng(700 + N)
    seqlens = [int(x) for x in rng.integers(0, 90, N)]
    seqlens[3] = 0
    seqlens[N - 1] = 129
    H = 2
    inp = I.prefill_inputs(seqlens, H, 128, 128, "bf16", 42, decay="config", state="randn")
    args = [to_dev(inp[n], n in ("q", "k", "v")) for n in ("q", "k", "v", "beta", "alpha", "cu_seqlens")]
    s0 = to_dev(inp["state_in"])
    o, st = kda.kda_prefill(*args, s0)
    torch.cuda.synchronize()
    assert kda.kda_get_device_error() == 0
    o_ref, st_ref = O.prefill(inp)
    assert rel_frob(o.double().cpu().numpy(), o_ref) <= 3e-3
    assert rel_frob(st.double().cpu().numpy(), st_ref) <= 3e-3
    up = lambda x: (x + 255) // 256 * 256
    ws = torch.empty(up(4 * (N + 1)) + up(4 * N) + 5 * H * 99072, dtype=torch.uint8, device="cuda:0")
    o2, st2 = kda.kda_prefill(*args, s0, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o2.view(torch.int16), o.view(torch.int16)) and torch.equal(st2, st)


def test_scale_and_zero_state():
    inp = I.prefill_inputs([130, 7], 2, 64, 64, "f32", 8, decay="slow")
    check(inp, scale=0.125)


def test_worked_overwrite_on_gpu(golden_dir):
    """The page's overwrite example (write (k, a) then (k, b), beta = 1, no decay) at d = 16 with zero
    padding: reading k returns b."""
    g = json.load(open(os.path.join(golden_dir, "overwrite_example.json")))
    d = 16
    key = np.zeros(d, np.float32)
    key[g["key_index"]] = 1.0
    a = np.zeros(d, np.float32)
    b = np.zeros(d, np.float32)
    a[:4], b[:4] = g["a"], g["b"]
    inp = dict(q=np.stack([key, key])[:, None, :].copy(), k=np.stack([key, key])[:, None, :].copy(),
               v=np.stack([a, b])[:, None, :].copy(), beta=np.ones((2, 1), np.float32),
               alpha=np.ones((2, 1, d), np.float32), cu_seqlens=I.cu_seqlens_of([2]), state_in=None,
               dtype="f32", H=1, dk=d, dv=d)
    o, _ = prefill_gpu(inp)
    np.testing.assert_allclose(o[0, 0, :4], g["a"], rtol=0, atol=1e-5)
    np.testing.assert_allclose(o[1, 0, :4], g["delta_read_after_both_writes"], rtol=0, atol=1e-5)


def _sub_batch(inp, seqs):
    cu = inp["cu_seqlens"]
    sub = dict(inp)
    for key in ("q", "k", "v", "beta", "alpha"):
        sub[key] = np.ascontiguousarray(np.concatenate([inp[key][cu[n]:cu[n + 1]] for n in seqs]))
    sub["cu_seqlens"] = I.cu_seqlens_of([int(cu[n + 1] - cu[n]) for n in seqs])
    sub["state_in"] = np.ascontiguousarray(inp["state_in"][list(seqs)])
    return sub


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_packing_independence(dtype, d):
    """Each sequence's results do not depend on which other sequences share the batch (or where in it)."""
    inp = I.prefill_inputs([70, 150, 33], 2, d, d, dtype, 9, decay="slow", state="randn")
    o, st = prefill_gpu(inp)
    cu = inp["cu_seqlens"]
    for pair in ((1, 0), (2, 1), (0, 2)):
        o1, st1 = prefill_gpu(_sub_batch(inp, pair))
        c1 = cu[pair[0] + 1] - cu[pair[0]]
        for part, n in ((slice(0, c1), pair[0]), (slice(c1, None), pair[1])):
            assert np.array_equal(o1[part], o[cu[n]:cu[n + 1]])
        assert np.array_equal(st1, st[list(pair)])


# One sequence with few heads runs the chain on 16-column slices, with more heads on 32-column slices (the
# chain of 16-column slices must leave half of the GB300's 152 SMs to phase 1: H <= 9); H = 12 takes the latter.
CHAIN_WIDTHS = [2, 12]


@pytest.mark.parametrize("T", [1, 63, 64, 65, 200, 700])
@pytest.mark.parametrize("decay", ["config", "slow", "one", "scalar"])
def test_single_sequence_two_phase(T, decay):
    """One bf16 d=128 sequence takes the two-phase path (per-chunk records, then the state chain)."""
    inp = I.prefill_inputs([T], 3, 128, 128, "bf16", 300 + T, decay=decay, state="randn")
    check(inp)


@pytest.mark.parametrize("T", [65, 700])
def test_single_sequence_two_phase_wide_chain(T):
    """The same with twelve heads, whose chain runs on 32-column slices."""
    inp = I.prefill_inputs([T], 12, 128, 128, "bf16", 400 + T, decay="config", state="randn")
    check(inp)


@pytest.mark.parametrize("H", CHAIN_WIDTHS)
def test_two_phase_windows_give_identical_results(H):
    """A workspace smaller than the recommended size walks the sequence in more windows of chunks, the
    state passing between windows through state_out; the results are bit-identical, in place too."""
    import kda_gated_delta_03_gb300 as kda
    inp = I.prefill_inputs([1000], H, 128, 128, "bf16", 15, decay="slow", state="randn")
    args = [to_dev(inp[n], n in ("q", "k", "v")) for n in ("q", "k", "v", "beta", "alpha", "cu_seqlens")]
    s0 = to_dev(inp["state_in"])
    rec = H * 99072                                           # one chunk of records
    assert kda.kda_prefill_workspace_size(1, 1000, H, 128, 128, torch.bfloat16) == 16 * rec
    runs = []
    for chunks in (16, 5, 1):
        ws = torch.empty(chunks * rec, dtype=torch.uint8, device="cuda:0")
        runs.append(kda.kda_prefill(*args, s0, workspace=ws))
    st = s0.clone()
    ws = torch.empty(3 * rec, dtype=torch.uint8, device="cuda:0")
    o_ip, _ = kda.kda_prefill(*args, st, state_out=st, workspace=ws)
    torch.cuda.synchronize()
    for o, s in runs[1:] + [(o_ip, st)]:
        assert torch.equal(o, runs[0][0]) and torch.equal(s, runs[0][1])
    o_ref, s_ref = O.prefill(inp)
    assert rel_frob(runs[0][0].double().cpu().numpy(), o_ref) <= 3e-3
    assert rel_frob(runs[0][1].double().cpu().numpy(), s_ref) <= 3e-3


@pytest.mark.parametrize("H,T", [(1, 200), (48, 300)])
def test_single_sequence_two_phase_head_counts(H, T):
    """One head (eight 16-column chain CTAs) and 48 heads (192 chain CTAs of 32 columns: more than the
    GB300's 152 SMs, so the chain runs in two waves)."""
    inp = I.prefill_inputs([T], H, 128, 128, "bf16", 500 + H, decay="config", state="randn")
    check(inp)


def test_two_phase_bad_cu_seqlens_is_reported():
    import kda_gated_delta_03_gb300 as kda
    inp = I.prefill_inputs([100], 2, 128, 128, "bf16", 16)
    inp["cu_seqlens"] = np.array([0, 90], np.int32)
    prefill_gpu(inp)
    assert kda.kda_get_device_error() & 0x1
    assert kda.kda_get_device_error() == 0


def test_append_equals_one_shot():
    """prefill(T1) then prefill(T2) from the carried state equals prefill(T1 + T2) when T1 is a whole
    number of chunks (identical chunking), and matches the oracle otherwise."""
    inp = I.prefill_inputs([320], 2, 128, 128, "bf16", 10, decay="slow", state="randn")
    o_full, s_full = prefill_gpu(inp)
    for cut in (192, 100):
        a, b = dict(inp), dict(inp)
        for key in ("q", "k", "v", "beta", "alpha"):
            a[key] = np.ascontiguousarray(inp[key][:cut])
            b[key] = np.ascontiguousarray(inp[key][cut:])
        a["cu_seqlens"], b["cu_seqlens"] = I.cu_seqlens_of([cut]), I.cu_seqlens_of([320 - cut])
        o1, s1 = prefill_gpu(a)
        o2, s2 = prefill_gpu(b, state_in=s1.astype(np.float32))
        if cut % 64 == 0:
            assert np.array_equal(np.concatenate([o1, o2]), o_full)
            assert np.array_equal(s2, s_full.astype(np.float32).astype(np.float64))
        else:
            o_ref, s_ref = O.prefill(inp)
            assert rel_frob(np.concatenate([o1, o2]), o_ref) <= 3e-3
            assert rel_frob(s2, s_ref) <= 3e-3


def test_in_place_state():
    import kda_gated_delta_03_gb300 as kda
    inp = I.prefill_inputs([90, 40], 2, 64, 64, "f32", 11, decay="slow", state="randn")
    st = to_dev(inp["state_in"])
    kda.kda_prefill(*(to_dev(inp[n]) for n in ("q", "k", "v", "beta", "alpha", "cu_seqlens")), st, state_out=st)
    torch.cuda.synchronize()
    _, s_ref = O.prefill(inp)
    assert rel_frob(st.cpu().numpy(), s_ref) <= 1e-4


def test_empty_and_all_zero_length():
    import kda_gated_delta_03_gb300 as kda
    inp = I.prefill_inputs([0, 0], 2, 16, 16, "f32", 12, state="randn")
    o, st = prefill_gpu(inp)
    assert o.shape == (0, 2, 16)
    assert np.array_equal(st, inp["state_in"].astype(np.float64))
    o, st = prefill_gpu(I.prefill_inputs([0], 2, 16, 16, "f32", 12))
    assert np.all(st == 0)
    assert kda.kda_get_device_error() == 0


def test_bad_cu_seqlens_is_reported_not_faulted():
    """Inconsistent cu_seqlens contents are caught on the device: the affected sequences are skipped and
    the error word says so; nothing reads or writes out of bounds."""
    import kda_gated_delta_03_gb300 as kda
    inp = I.prefill_inputs([10, 20, 30], 1, 16, 16, "f32", 13)
    inp["cu_seqlens"] = np.array([0, 25, 20, 60], np.int32)
    prefill_gpu(inp)
    assert kda.kda_get_device_error() & 0x1
    assert kda.kda_get_device_error() == 0


def _run_one(inp, single):
    import kda_gated_delta_03_gb300 as kda
    args = [to_dev(inp[n], n in ("q", "k", "v")) for n in ("q", "k", "v", "beta", "alpha", "cu_seqlens")]
    o, st = kda.kda_prefill(*args, to_dev(inp["state_in"]), single_kernel=single)
    torch.cuda.synchronize()
    return o.double().cpu().numpy(), st.double().cpu().numpy()


def _scaled_v(inp, factor, rows=slice(None)):
    v = I.bf16_bits_to_f32(inp["v"]).copy()
    v[rows] *= factor
    return I.f32_to_bf16_bits(v)


@pytest.mark.parametrize("H", CHAIN_WIDTHS)
def test_large_values_and_states_on_the_two_phase_path(H):
    """The two-phase path keeps its per-chunk records and its state operand in fp16 (range 65,504) and
    holds large magnitudes inside that range with exact power-of-two scales: per chunk for v, and for the
    carried state a scale chosen before every chunk from the largest state entry.  With v and the initial
    state 1e6 times larger, with every |v| just above the point where scaling starts, and with only a
    large initial state that then decays to O(1) (the state's scale must come back down), the default call
    matches the float64 oracle (over the first and the later tokens separately, so that the large part
    does not hide the small one) and reports nothing; the single-kernel path agrees too."""
    import kda_gated_delta_03_gb300 as kda
    base = I.prefill_inputs([700], H, 128, 128, "bf16", 95, decay="slow", state="randn")
    fast = I.prefill_inputs([700], H, 128, 128, "bf16", 96, decay="config", state="randn")
    cases = {
        "all_x1e6": dict(base, v=_scaled_v(base, 1e6), state_in=base["state_in"] * 1e6),
        "just_above": dict(base, v=_scaled_v(base, 70.0)),
        "state_x1e4": dict(fast, state_in=fast["state_in"] * 1e4),
    }
    for name, inp in cases.items():
        o_ref, s_ref = O.prefill(inp)
        for single in (False, True):
            o, st = _run_one(inp, single)
            assert kda.kda_get_device_error() == 0, (name, single)
            for part in (slice(0, 128), slice(128, 700)):
                e = rel_frob(o[part], o_ref[part])
                assert e <= 3e-3, (name, single, part, e)
            assert rel_frob(st, s_ref) <= 3e-3, (name, single)


def test_single_kernel_option_matches_the_oracle():
    """kda_prefill_options.single_kernel computes one sequence on the single-kernel path (TF32 / bf16
    operands) instead of the two-phase path."""
    import kda_gated_delta_03_gb300 as kda
    inp = I.prefill_inputs([300], 2, 128, 128, "bf16", 95, decay="slow", state="randn")
    o_ref, s_ref = O.prefill(inp)
    o1, s1 = _run_one(inp, True)
    assert kda.kda_get_device_error() == 0
    assert rel_frob(o1, o_ref) <= 3e-3 and rel_frob(s1, s_ref) <= 3e-3


def test_chain_widths_agree_bit_for_bit():
    """Heads are independent, so two heads taken out of a twelve-head sequence (chain on 32-column slices)
    and run on their own (chain on 16-column slices) give the same bits: the slice width changes only how
    the value columns are split over CTAs, not the arithmetic of any element."""
    import kda_gated_delta_03_gb300 as kda
    inp = I.prefill_inputs([700], 12, 128, 128, "bf16", 97, decay="config", state="randn")
    names = ("q", "k", "v", "beta", "alpha")
    full = [to_dev(inp[n], n in ("q", "k", "v")) for n in names] + [to_dev(inp["cu_seqlens"])]
    o12, st12 = kda.kda_prefill(*full, to_dev(inp["state_in"]))
    heads = slice(5, 7)
    part = [to_dev(np.ascontiguousarray(inp[n][:, heads]), n in ("q", "k", "v")) for n in names]
    o2, st2 = kda.kda_prefill(*part, to_dev(inp["cu_seqlens"]), to_dev(np.ascontiguousarray(inp["state_in"][:, heads])))
    torch.cuda.synchronize()
    assert kda.kda_get_device_error() == 0
    assert torch.equal(o2, o12[:, heads]) and torch.equal(st2, st12[:, heads])


@pytest.mark.parametrize("case", [([700], 3, "two_phase"), ([300, 0, 129, 64], 2, "records_several"),
                                  ([70, 130], 2, "cuda_core")], ids=["two_phase", "records_several", "cuda_core"])
def test_prefill_is_bit_reproducible(case):
    """Two calls on the same inputs give the same bits on every path (no sum depends on the order of
    atomic updates or on which CTA took which unit)."""
    seqlens, H, path = case
    d, dtype = (128, "bf16") if path != "cuda_core" else (16, "f32")
    inp = I.prefill_inputs(seqlens, H, d, d, dtype, 77, state="randn")
    a = prefill_gpu(inp)
    b = prefill_gpu(inp)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])

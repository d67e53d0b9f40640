"""Host-side checks of the C ABI: the library builds for sm_103a, exports every symbol the header
declares, and rejects bad arguments on the host before touching the CUDA runtime (no GPU needed)."""

import ctypes
import os
import re
import shutil
import subprocess

import pytest

from kda_gated_delta_03_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc not available")


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"KDA_API\s+[\w\s\*]+?\b(kda_\w+)\s*\(", text)


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def test_header_declares_the_abi():
    names = declared_functions()
    assert set(names) == set(binding.SIGNATURES), names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_library_targets_sm103a():
    assert "arch=compute_103a,code=sm_103a" in " ".join(build.ARCH)


def test_status_strings(lib):
    assert binding.kda_status_string(0) == "KDA_OK"
    assert binding.kda_status_string(3) == "KDA_ERR_WORKSPACE"
    assert binding.kda_status_string(99) == "KDA_ERR_UNKNOWN"


def test_workspace_size(lib):
    # one bf16 d=128 sequence: 99,072 bytes of records per (chunk, head), at most 1 GiB of them
    assert lib.kda_prefill_workspace_size(1, 8192, 32, 128, 128, 1) == 128 * 32 * 99072
    assert lib.kda_prefill_workspace_size(1, 1_032_192, 8, 128, 128, 1) == 1354 * 8 * 99072
    assert lib.kda_prefill_workspace_size(1, 1 << 20, 32, 128, 128, 1) == 338 * 32 * 99072
    assert lib.kda_prefill_workspace_size(1, 65, 4, 128, 128, 1) == (2 * 4 * 99072 + 255) // 256 * 256
    assert lib.kda_prefill_workspace_size(1, 8192, 32, 128, 128, 0) == 0      # fp32: single-kernel path
    assert lib.kda_prefill_workspace_size(1, 8192, 32, 64, 64, 1) == 0
    # several bf16 d=128 sequences: their chunk offsets and longest-first order, then the records of at most
    # T // 64 + N chunks (each sequence's last chunk may be partial), at most 16 GiB of them
    up = lambda x: (x + 255) // 256 * 256
    hdr = lambda n: up(4 * (n + 1)) + up(4 * n)
    assert lib.kda_prefill_workspace_size(64, 300000, 32, 128, 128, 1) == up(hdr(64) + (300000 // 64 + 64) * 32 * 99072)
    assert lib.kda_prefill_workspace_size(65, 300000, 32, 128, 128, 1) == up(hdr(65) + (300000 // 64 + 65) * 32 * 99072)
    cap = (16 << 30) // (32 * 99072)
    assert lib.kda_prefill_workspace_size(64, 1 << 20, 32, 128, 128, 1) == up(hdr(64) + cap * 32 * 99072)
    assert lib.kda_prefill_workspace_size(3, 700, 2, 128, 128, 1) == up(hdr(3) + (700 // 64 + 3) * 2 * 99072)
    # other sequence batches: the longest-first order only
    assert lib.kda_prefill_workspace_size(64, 300000, 32, 64, 64, 1) == 256
    assert lib.kda_prefill_workspace_size(65, 300000, 32, 128, 128, 0) == 512


def test_backward_workspace_size(lib):
    """The backward workspace: offsets, the recompute's snapshots and the state gradients at every 64-token
    boundary, the recompute's o and state_out, its own prefill workspace, and the chunk pass's per-CTA
    scratch (one CTA per SM, at most 160): ten 64 x 128 fp32 matrices for the matrix form at d = 128,
    63 states for the token walk at d = 16 and 64."""
    def up(x):
        return (x + 255) // 256 * 256

    def expected(N, T, H, d, dt):
        dd, es = d * d * 4, 2 if dt == 1 else 4
        ctas = min((T // 64 + N) * H, 160)
        # the recompute: one sequence as kda_prefill, several on the single-kernel path (their order only)
        fwd = lib.kda_prefill_workspace_size(N, T, H, d, d, dt) if N == 1 else 4 * N
        parts = [(N + 1) * 8, (T // 64) * H * dd, (T // 64) * H * dd, T * H * d * es, N * H * dd, fwd,
                 ctas * (10 * 64 * 128 * 4 if d == 128 else 63 * dd)]
        return sum(up(x) for x in parts)

    for args in ((1, 8192, 32, 128, 1), (3, 700, 2, 128, 1), (2, 1000, 4, 64, 0), (4, 300, 2, 16, 0)):
        N, T, H, d, dt = args
        assert lib.kda_prefill_backward_workspace_size(N, T, H, d, d, dt) == expected(*args), args
    assert lib.kda_prefill_backward_workspace_size(1, 8192, 32, 32, 32, 1) == 0        # unsupported head size


def test_launch_count_host_paths(lib):
    """Launch counts that need no device: rejected arguments, the single-kernel paths."""
    assert lib.kda_prefill_launch_count(0, 0, 2, 16, 16, 0, 0) == 0
    assert lib.kda_prefill_launch_count(0, 5, 2, 16, 16, 0, 0) == -1
    assert lib.kda_prefill_launch_count(1, 64, 2, 32, 32, 0, 0) == -1
    assert lib.kda_prefill_launch_count(1, 64, 2, 16, 16, 0, 0) == 1
    assert lib.kda_prefill_launch_count(3, 640, 2, 64, 64, 1, 256) == 2
    assert lib.kda_prefill_launch_count(1, 640, 2, 128, 128, 1, 100) == -1      # below one chunk's records


# Fake, suitably aligned device addresses: every call below must be rejected before any CUDA call.
P = ctypes.c_void_p(0x10000)


def prefill(lib, **over):
    a = dict(q=P, k=P, v=P, beta=P, alpha=P, cu=P, N=1, T=64, H=2, dk=16, dv=16, dt=0, scale=1.0, s_in=None,
             s_out=P, o=P, ws=None, wsb=0, stream=None)
    a.update(over)
    return lib.kda_prefill(a["q"], a["k"], a["v"], a["beta"], a["alpha"], a["cu"], a["N"], a["T"], a["H"], a["dk"],
                           a["dv"], a["dt"], a["scale"], a["s_in"], a["s_out"], a["o"], a["ws"], a["wsb"],
                           a["stream"])


def decode(lib, fn="kda_decode_step", **over):
    a = dict(q=P, k=P, v=P, beta=P, alpha=P, state=P, idx=None, slots=4, o=P, B=4, H=2, dk=16, dv=16, dt=1,
             scale=1.0, stream=None)
    a.update(over)
    return getattr(lib, fn)(a["q"], a["k"], a["v"], a["beta"], a["alpha"], a["state"], a["idx"], a["slots"],
                            a["o"], a["B"], a["H"], a["dk"], a["dv"], a["dt"], a["scale"], a["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(H=0), binding.KDA_ERR_INVALID_ARG),
    (dict(N=-1), binding.KDA_ERR_INVALID_ARG),
    (dict(T=-5), binding.KDA_ERR_INVALID_ARG),
    (dict(T=2**31), binding.KDA_ERR_INVALID_ARG),
    (dict(dk=32, dv=32), binding.KDA_ERR_UNSUPPORTED),
    (dict(dk=128, dv=64), binding.KDA_ERR_UNSUPPORTED),
    (dict(dt=7), binding.KDA_ERR_INVALID_ARG),
    (dict(q=None), binding.KDA_ERR_INVALID_ARG),
    (dict(alpha=None), binding.KDA_ERR_INVALID_ARG),
    (dict(cu=None), binding.KDA_ERR_INVALID_ARG),
    (dict(s_out=None), binding.KDA_ERR_INVALID_ARG),
    (dict(q=ctypes.c_void_p(0x10008)), binding.KDA_ERR_INVALID_ARG),
    (dict(cu=ctypes.c_void_p(0x10002)), binding.KDA_ERR_INVALID_ARG),
    (dict(s_in=ctypes.c_void_p(0x10004)), binding.KDA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), binding.KDA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), binding.KDA_ERR_INVALID_ARG),
    (dict(N=4), binding.KDA_ERR_WORKSPACE),
    (dict(N=4, ws=P, wsb=255), binding.KDA_ERR_WORKSPACE),
    (dict(N=4, ws=ctypes.c_void_p(0x10010), wsb=4096), binding.KDA_ERR_WORKSPACE),
    # one bf16 d=128 sequence needs at least one chunk's records (H x 99,072 bytes)
    (dict(dk=128, dv=128, dt=1), binding.KDA_ERR_WORKSPACE),
    (dict(dk=128, dv=128, dt=1, ws=P, wsb=2 * 99072 - 1), binding.KDA_ERR_WORKSPACE),
    (dict(dk=128, dv=128, dt=1, ws=ctypes.c_void_p(0x10010), wsb=2 * 99072), binding.KDA_ERR_WORKSPACE),
    (dict(N=0, T=5), binding.KDA_ERR_INVALID_ARG),
    (dict(N=0, T=0), binding.KDA_OK),
])
def test_prefill_host_validation(lib, over, code):
    assert prefill(lib, **over) == code


@pytest.mark.parametrize("over,code", [
    (dict(H=0), binding.KDA_ERR_INVALID_ARG),
    (dict(B=-1), binding.KDA_ERR_INVALID_ARG),
    (dict(dk=48, dv=48), binding.KDA_ERR_UNSUPPORTED),
    (dict(state=None), binding.KDA_ERR_INVALID_ARG),
    (dict(o=ctypes.c_void_p(0x10001)), binding.KDA_ERR_INVALID_ARG),
    (dict(slots=3), binding.KDA_ERR_INVALID_ARG),
    (dict(idx=ctypes.c_void_p(0x10002)), binding.KDA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), binding.KDA_ERR_INVALID_ARG),
    (dict(B=0), binding.KDA_OK),
])
def test_decode_host_validation(lib, over, code):
    assert decode(lib, **over) == code


@pytest.mark.parametrize("over,code", [
    (dict(H=0), binding.KDA_ERR_INVALID_ARG),
    (dict(dk=48, dv=48), binding.KDA_ERR_UNSUPPORTED),
    (dict(state=None), binding.KDA_ERR_INVALID_ARG),
    (dict(state=ctypes.c_void_p(0x10008)), binding.KDA_ERR_INVALID_ARG),
    (dict(slots=3), binding.KDA_ERR_INVALID_ARG),
    (dict(B=0), binding.KDA_OK),
])
def test_decode_bf16_state_host_validation(lib, over, code):
    assert decode(lib, "kda_decode_step_bf16_state", **over) == code


def test_prefill_ex_validates_snapshot_options(lib):
    """kda_prefill_ex rejects bad snapshot options on the host; NULL options is kda_prefill."""
    def call(opts):
        return lib.kda_prefill_ex(P, P, P, P, P, P, 1, 64, 2, 16, 16, 0, 1.0, None, P, P, None, 0, None,
                                  None if opts is None else ctypes.byref(opts))
    assert call(binding.PrefillOptions(100, P, P)) == binding.KDA_ERR_INVALID_ARG     # not a multiple of 64
    assert call(binding.PrefillOptions(-64, P, P)) == binding.KDA_ERR_INVALID_ARG
    assert call(binding.PrefillOptions(64, None, P)) == binding.KDA_ERR_INVALID_ARG
    assert call(binding.PrefillOptions(64, ctypes.c_void_p(0x10004), P)) == binding.KDA_ERR_INVALID_ARG
    assert call(binding.PrefillOptions(64, P, None)) == binding.KDA_ERR_INVALID_ARG


def test_alpha_layout_validation(lib):
    """An unknown alpha layout, or an alpha pointer that the layout's alignment rules out, is rejected on
    the host (KDA_ALPHA_PER_HEAD needs 4 bytes, KDA_ALPHA_PER_CHANNEL 16)."""
    def pre(mode, alpha):
        opts = binding.PrefillOptions(0, None, None, mode)
        return lib.kda_prefill_ex(P, P, P, P, alpha, P, 1, 64, 2, 16, 16, 0, 1.0, None, P, P, None, 0, None,
                                  ctypes.byref(opts))
    assert pre(3, P) == binding.KDA_ERR_INVALID_ARG
    assert pre(binding.KDA_ALPHA_PER_HEAD, ctypes.c_void_p(0x10002)) == binding.KDA_ERR_INVALID_ARG
    assert pre(binding.KDA_ALPHA_PER_CHANNEL, ctypes.c_void_p(0x10004)) == binding.KDA_ERR_INVALID_ARG
    assert pre(binding.KDA_ALPHA_PER_HEAD, None) == binding.KDA_ERR_INVALID_ARG

    def dec(mode, alpha, sdt=0):
        opts = binding.DecodeOptions(mode, sdt)
        return lib.kda_decode_step_ex(P, P, P, P, alpha, P, None, 4, P, 4, 2, 16, 16, 1, 1.0, None,
                                      ctypes.byref(opts))
    assert dec(7, P) == binding.KDA_ERR_INVALID_ARG
    assert dec(binding.KDA_ALPHA_PER_HEAD, ctypes.c_void_p(0x10001)) == binding.KDA_ERR_INVALID_ARG
    assert dec(binding.KDA_ALPHA_PER_CHANNEL, None) == binding.KDA_ERR_INVALID_ARG
    assert dec(binding.KDA_ALPHA_PER_CHANNEL, P, 5) == binding.KDA_ERR_INVALID_ARG   # unknown state dtype


# ---- kda_prefill_host: cu_seqlens is host memory, so all of it is checked on the host ----
def host_prefill(lib, cu, N, T, d=128, dt=1, state_out=P, buf=P, buf_bytes=1 << 40, scale=1.0):
    arr = (ctypes.c_int32 * len(cu))(*cu)
    return lib.kda_prefill_host(P, P, P, P, P, arr, N, T, 2, d, d, dt, scale, None, state_out, P, buf, buf_bytes,
                                None)


def test_host_prefill_buffer_size(lib):
    # bf16 d=128, one sequence of 8192 tokens, H=32: device copies of q, k, v, beta, alpha, o, two states,
    # the cu_seqlens area and the workspace of one 1024-token segment
    rows = 8192 * 32
    a = lambda x: (x + 255) // 256 * 256
    want = a(rows * 256) * 3 + a(rows * 4) + a(rows * 512) + a(rows * 256) + 2 * a(32 * 128 * 128 * 4) + a(36 * 4)
    want += a(lib.kda_prefill_workspace_size(1, 1024, 32, 128, 128, 1))
    assert lib.kda_prefill_host_buffer_size(1, 8192, 32, 128, 128, 1) == want
    assert lib.kda_prefill_host_buffer_size(0, 10, 2, 16, 16, 0) == 0
    assert lib.kda_prefill_host_buffer_size(1, 10, 2, 32, 32, 0) == 0
    assert lib.kda_prefill_host_buffer_size(2, 0, 2, 16, 16, 0) > 0


def test_host_prefill_rejects_bad_arguments(lib):
    OK_, INV, UNS, WS = 0, 1, 2, 3
    assert host_prefill(lib, [1, 10], 1, 10) == INV                  # cu[0] != 0
    assert host_prefill(lib, [0, 10, 5, 20], 3, 20) == INV           # decreasing
    assert host_prefill(lib, [0, 10, 20], 2, 21) == INV              # cu[N] != T
    assert host_prefill(lib, [0, 10], 1, 10, d=32) == UNS
    assert host_prefill(lib, [0, 10], 1, 10, state_out=None) == INV
    assert host_prefill(lib, [0, 10], 1, 10, buf=None) == WS
    assert host_prefill(lib, [0, 10], 1, 10, buf=ctypes.c_void_p(0x10010)) == WS     # not 256-byte aligned
    assert host_prefill(lib, [0, 10], 1, 10, buf_bytes=1024) == WS
    # a non-finite scale is refused before any copy is queued (without a GPU, any CUDA call would give
    # KDA_ERR_CUDA instead)
    assert host_prefill(lib, [0, 10], 1, 10, scale=float("nan")) == INV
    assert host_prefill(lib, [0, 10], 1, 10, scale=float("inf")) == INV
    assert lib.kda_prefill_host(P, P, P, P, P, None, 1, 10, 2, 16, 16, 0, 1.0, None, P, P, P, 1 << 40, None) == INV
    assert lib.kda_prefill_host(None, P, P, P, P, (ctypes.c_int32 * 2)(0, 10), 1, 10, 2, 16, 16, 0, 1.0, None, P,
                                P, P, 1 << 40, None) == INV

"""Thin Python binding of libkda (``include/kda.h``), through ctypes.

Argument marshalling only: shape/dtype checks, pointer extraction, default
output allocation through PyTorch, and the caller's current CUDA stream.  Every
step of the operator runs in the CUDA kernels behind the C ABI; when the library
is missing or fails to load, every call raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_WORKSPACE, KDA_ERR_CUDA, KDA_ERR_DEVICE = range(6)
KDA_ERR_TOO_LARGE = 6
KDA_NOALLOC_MAX_SEQS = 16384
KDA_DTYPE_F32, KDA_DTYPE_BF16 = 0, 1
KDA_DEVERR_CU_SEQLENS, KDA_DEVERR_STATE_IDX = 0x1, 0x2

class PrefillOptions(ctypes.Structure):
    """kda_prefill_options (include/kda.h)."""
    _fields_ = [("snapshot_every", ctypes.c_int32), ("snapshots", ctypes.c_void_p),
                ("snapshot_offsets", ctypes.c_void_p), ("alpha_mode", ctypes.c_int32),
                ("single_kernel", ctypes.c_int32)]


class DecodeOptions(ctypes.Structure):
    """kda_decode_options (include/kda.h)."""
    _fields_ = [("alpha_mode", ctypes.c_int32), ("state_dtype", ctypes.c_int32)]


KDA_ALPHA_PER_CHANNEL, KDA_ALPHA_PER_HEAD, KDA_ALPHA_NONE = 0, 1, 2


# Every function include/kda.h declares, with its ctypes signature.
_vp, _i32, _i64, _sz, _f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
SIGNATURES = {
    "kda_prefill_workspace_size": (_sz, [_i32, _i64, _i32, _i32, _i32, ctypes.c_int]),
    "kda_prefill_launch_count": (_i64, [_i32, _i64, _i32, _i32, _i32, ctypes.c_int, _sz]),
    "kda_prefill": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32, _i32, ctypes.c_int,
                                   _f32, _vp, _vp, _vp, _vp, _sz, _vp]),
    "kda_prefill_ex": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32, _i32, ctypes.c_int,
                                      _f32, _vp, _vp, _vp, _vp, _sz, _vp, _vp]),
    "kda_decode_step": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32,
                                       ctypes.c_int, _f32, _vp]),
    "kda_prefill_backward_workspace_size": (_sz, [_i32, _i64, _i32, _i32, _i32, ctypes.c_int]),
    "kda_prefill_backward": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32, _i32,
                                            ctypes.c_int, _f32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                            _vp, _sz, _vp]),
    "kda_decode_step_ex": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32,
                                          ctypes.c_int, _f32, _vp, _vp]),
    "kda_decode_step_bf16_state": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32,
                                                  _i32, ctypes.c_int, _f32, _vp]),
    "kda_prefill_noalloc": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32, _i32,
                                           ctypes.c_int, _f32, _vp, _vp, _vp, _vp]),
    "kda_prefill_host_buffer_size": (_sz, [_i32, _i64, _i32, _i32, _i32, ctypes.c_int]),
    "kda_prefill_host": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32, _i32, ctypes.c_int,
                                        _f32, _vp, _vp, _vp, _vp, _sz, _vp]),
    "kda_get_device_error": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_uint32)]),
    "kda_status_string": (ctypes.c_char_p, [ctypes.c_int]),
}


class KdaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {kda_status_string(code)} ({code})")
        self.code = code


_LIB = None


def lib_path() -> str:
    """The in-tree libkda, or the library named by the KDA_LIBRARY environment variable."""
    return os.environ.get("KDA_LIBRARY") or _build.LIB


def load():
    """Load libkda (built in-tree by ``build.build()``); raises if it is missing."""
    global _LIB
    if _LIB is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libkda is not built ({path} missing); run kda_gated_delta_03_gb300.build.build()")
        L = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _LIB = L
    return _LIB


def kda_status_string(code: int) -> str:
    return load().kda_status_string(int(code)).decode()


def _dt(t: torch.dtype) -> int:
    if t == torch.bfloat16:
        return KDA_DTYPE_BF16
    if t == torch.float32:
        return KDA_DTYPE_F32
    raise TypeError(f"unsupported q/k/v dtype {t}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(name, t, dtype, shape, device):
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def kda_prefill_workspace_size(num_seqs: int, total_tokens: int, H: int, d_k: int, d_v: int,
                               dtype: torch.dtype = torch.bfloat16) -> int:
    return int(load().kda_prefill_workspace_size(num_seqs, total_tokens, H, d_k, d_v, _dt(dtype)))


def kda_prefill_launch_count(num_seqs: int, total_tokens: int, H: int, d_k: int, d_v: int,
                             dtype: torch.dtype = torch.bfloat16, workspace_bytes: int = None) -> int:
    """Kernel launches of one kda_prefill call (with the recommended workspace when none is given)."""
    if workspace_bytes is None:
        workspace_bytes = kda_prefill_workspace_size(num_seqs, total_tokens, H, d_k, d_v, dtype)
    return int(load().kda_prefill_launch_count(num_seqs, total_tokens, H, d_k, d_v, _dt(dtype), workspace_bytes))


def _alpha_shape(mode, lead, dk):
    return {KDA_ALPHA_PER_CHANNEL: (*lead, dk), KDA_ALPHA_PER_HEAD: tuple(lead)}.get(mode)


def kda_prefill(q, k, v, beta, alpha, cu_seqlens, state_in=None, *, scale: float = 1.0, state_out=None,
                o=None, workspace=None, stream=None, snapshot_every: int = 0, snapshots=None, snapshot_offsets=None,
                alpha_mode: int = KDA_ALPHA_PER_CHANNEL, single_kernel: bool = False):
    """Chunkwise prefill over packed sequences; returns (o, state_out).

    q, k [T, H, d_k], v [T, H, d_v] (bf16 or f32); beta [T, H] f32; alpha [T, H, d_k] f32;
    cu_seqlens [N + 1] int32 (device); state_in [N, H, d_k, d_v] f32 or None.
    With snapshot_every > 0 (a multiple of 64): snapshots [S, H, d_k, d_v] f32 and snapshot_offsets
    [N + 1] int32 (device) receive the state of sequence n after each multiple of snapshot_every tokens
    (kda_prefill_ex).  alpha_mode: KDA_ALPHA_PER_CHANNEL (alpha [T, H, d_k]), KDA_ALPHA_PER_HEAD (Gated
    DeltaNet, alpha [T, H]) or KDA_ALPHA_NONE (DeltaNet, alpha may be None).  single_kernel: run one bf16
    d=128 sequence on the single-kernel path instead of the two-phase path (whose fp16 operands end at
    65,504; KDA_DEVERR_RANGE reports values beyond).
    """
    L = load()
    T, H, dk = q.shape
    dv = v.shape[2]
    dev = q.device
    N = cu_seqlens.shape[0] - 1
    _check("q", q, q.dtype, (T, H, dk), dev)
    _check("k", k, q.dtype, (T, H, dk), dev)
    _check("v", v, q.dtype, (T, H, dv), dev)
    _check("beta", beta, torch.float32, (T, H), dev)
    if alpha_mode != KDA_ALPHA_NONE or alpha is not None:
        _check("alpha", alpha, torch.float32, _alpha_shape(alpha_mode, (T, H), dk), dev)
    _check("cu_seqlens", cu_seqlens, torch.int32, (N + 1,), dev)
    if state_in is not None:
        _check("state_in", state_in, torch.float32, (N, H, dk, dv), dev)
    if state_out is None:
        state_out = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    _check("state_out", state_out, torch.float32, (N, H, dk, dv), dev)
    if o is None:
        o = torch.empty((T, H, dv), dtype=q.dtype, device=dev)
    _check("o", o, q.dtype, (T, H, dv), dev)
    need = int(L.kda_prefill_workspace_size(N, T, H, dk, dv, _dt(q.dtype)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(alpha), _ptr(cu_seqlens), N, T, H, dk, dv, _dt(q.dtype),
            float(scale), _ptr(state_in), _ptr(state_out), _ptr(o), _ptr(workspace), wbytes, _stream(stream))
    if snapshot_every or alpha_mode != KDA_ALPHA_PER_CHANNEL or single_kernel:
        if snapshot_every:
            S = snapshots.shape[0]
            _check("snapshots", snapshots, torch.float32, (S, H, dk, dv), dev)
            _check("snapshot_offsets", snapshot_offsets, torch.int32, (N + 1,), dev)
        opts = PrefillOptions(int(snapshot_every), _ptr(snapshots), _ptr(snapshot_offsets), int(alpha_mode),
                              int(bool(single_kernel)))
        rc = L.kda_prefill_ex(*args, ctypes.byref(opts))
        name = "kda_prefill_ex"
    else:
        rc = L.kda_prefill(*args)
        name = "kda_prefill"
    if rc != KDA_OK:
        raise KdaError(name, rc)
    return o, state_out


def kda_prefill_noalloc(q, k, v, beta, alpha, cu_seqlens, state_in=None, *, scale: float = 1.0, state_out=None,
                        o=None, stream=None):
    """kda_prefill for callers that cannot allocate device memory: no workspace argument; the library
    uses a fixed static device array (at most KDA_NOALLOC_MAX_SEQS sequences) and allocates nothing.

    Pass preallocated `state_out` and `o` to keep the whole call allocation-free; when they are None,
    this wrapper allocates them through PyTorch.  Returns (o, state_out).
    """
    L = load()
    T, H, dk = q.shape
    dv = v.shape[2]
    dev = q.device
    N = cu_seqlens.shape[0] - 1
    _check("q", q, q.dtype, (T, H, dk), dev)
    _check("k", k, q.dtype, (T, H, dk), dev)
    _check("v", v, q.dtype, (T, H, dv), dev)
    _check("beta", beta, torch.float32, (T, H), dev)
    _check("alpha", alpha, torch.float32, (T, H, dk), dev)
    _check("cu_seqlens", cu_seqlens, torch.int32, (N + 1,), dev)
    if state_in is not None:
        _check("state_in", state_in, torch.float32, (N, H, dk, dv), dev)
    if state_out is None:
        state_out = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    _check("state_out", state_out, torch.float32, (N, H, dk, dv), dev)
    if o is None:
        o = torch.empty((T, H, dv), dtype=q.dtype, device=dev)
    _check("o", o, q.dtype, (T, H, dv), dev)
    rc = L.kda_prefill_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(alpha), _ptr(cu_seqlens), N, T, H, dk,
                               dv, _dt(q.dtype), float(scale), _ptr(state_in), _ptr(state_out), _ptr(o),
                               _stream(stream))
    if rc != KDA_OK:
        raise KdaError("kda_prefill_noalloc", rc)
    return o, state_out


def kda_prefill_host(q, k, v, beta, alpha, cu_seqlens, state_in=None, *, scale: float = 1.0, state_out=None,
                     o=None, device_buffer=None, stream=None):
    """kda_prefill with every tensor in host memory (CPU tensors; pin them for the copies to overlap with
    the compute).  The library streams the inputs to the device and the outputs back, segment by segment,
    through `device_buffer` (a uint8 CUDA tensor of kda_prefill_host_buffer_size bytes, allocated here when
    None).  Asynchronous on `stream`: synchronise it before reading the returned (o, state_out)."""
    L = load()
    T, H, dk = q.shape
    dv = v.shape[2]
    cpu = torch.device("cpu")
    N = cu_seqlens.shape[0] - 1
    _check("q", q, q.dtype, (T, H, dk), cpu)
    _check("k", k, q.dtype, (T, H, dk), cpu)
    _check("v", v, q.dtype, (T, H, dv), cpu)
    _check("beta", beta, torch.float32, (T, H), cpu)
    _check("alpha", alpha, torch.float32, (T, H, dk), cpu)
    _check("cu_seqlens", cu_seqlens, torch.int32, (N + 1,), cpu)
    if state_in is not None:
        _check("state_in", state_in, torch.float32, (N, H, dk, dv), cpu)
    pin = q.is_pinned()
    if state_out is None:
        state_out = torch.empty((N, H, dk, dv), dtype=torch.float32, pin_memory=pin)
    _check("state_out", state_out, torch.float32, (N, H, dk, dv), cpu)
    if o is None:
        o = torch.empty((T, H, dv), dtype=q.dtype, pin_memory=pin)
    _check("o", o, q.dtype, (T, H, dv), cpu)
    need = int(L.kda_prefill_host_buffer_size(N, T, H, dk, dv, _dt(q.dtype)))
    if device_buffer is None:
        device_buffer = torch.empty(max(need, 1), dtype=torch.uint8, device=torch.device("cuda",
                                                                                           torch.cuda.current_device()))
    rc = L.kda_prefill_host(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(alpha), _ptr(cu_seqlens), N, T, H, dk, dv,
                            _dt(q.dtype), float(scale), _ptr(state_in), _ptr(state_out), _ptr(o), _ptr(device_buffer),
                            device_buffer.numel() * device_buffer.element_size(), _stream(stream))
    if rc != KDA_OK:
        raise KdaError("kda_prefill_host", rc)
    return o, state_out


def kda_decode_step(q, k, v, beta, alpha, state, state_idx=None, *, scale: float = 1.0, o=None, stream=None,
                    alpha_mode: int = KDA_ALPHA_PER_CHANNEL):
    """One fused decode step; updates `state` ([P, H, d_k, d_v] f32, or bf16 for the bf16-stored state) in
    place and returns o [B, H, d_v]."""
    L = load()
    B, H, dk = q.shape
    dv = v.shape[2]
    dev = q.device
    P = state.shape[0]
    _check("q", q, q.dtype, (B, H, dk), dev)
    _check("k", k, q.dtype, (B, H, dk), dev)
    _check("v", v, q.dtype, (B, H, dv), dev)
    _check("beta", beta, torch.float32, (B, H), dev)
    if alpha_mode != KDA_ALPHA_NONE or alpha is not None:
        _check("alpha", alpha, torch.float32, _alpha_shape(alpha_mode, (B, H), dk), dev)
    bf16_state = state.dtype == torch.bfloat16
    _check("state", state, torch.bfloat16 if bf16_state else torch.float32, (P, H, dk, dv), dev)
    if state_idx is not None:
        _check("state_idx", state_idx, torch.int32, (B,), dev)
    if o is None:
        o = torch.empty((B, H, dv), dtype=q.dtype, device=dev)
    _check("o", o, q.dtype, (B, H, dv), dev)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(alpha), _ptr(state), _ptr(state_idx), P, _ptr(o), B, H,
            dk, dv, _dt(q.dtype), float(scale), _stream(stream))
    if alpha_mode != KDA_ALPHA_PER_CHANNEL:
        name = "kda_decode_step_ex"
        rc = L.kda_decode_step_ex(*args, ctypes.byref(DecodeOptions(int(alpha_mode), int(bf16_state))))
    else:
        name = "kda_decode_step_bf16_state" if bf16_state else "kda_decode_step"
        rc = getattr(L, name)(*args)
    if rc != KDA_OK:
        raise KdaError(name, rc)
    return o


def kda_prefill_backward(q, k, v, beta, alpha, cu_seqlens, grad_o, state_in=None, grad_state_out=None, *,
                         scale: float = 1.0, want_state_grad: bool = True, workspace=None, stream=None):
    """Backward pass of kda_prefill (per-channel alpha).  Returns (grad_q, grad_k, grad_v, grad_beta,
    grad_alpha, grad_state_in or None) for the loss sum(o * grad_o) + sum(state_out * grad_state_out)."""
    L = load()
    T, H, dk = q.shape
    dv = v.shape[2]
    dev = q.device
    N = cu_seqlens.shape[0] - 1
    for name, t, dt_, shape in (("q", q, q.dtype, (T, H, dk)), ("k", k, q.dtype, (T, H, dk)),
                                ("v", v, q.dtype, (T, H, dv)), ("beta", beta, torch.float32, (T, H)),
                                ("alpha", alpha, torch.float32, (T, H, dk)),
                                ("cu_seqlens", cu_seqlens, torch.int32, (N + 1,)),
                                ("grad_o", grad_o, q.dtype, (T, H, dv))):
        _check(name, t, dt_, shape, dev)
    for name, t in (("state_in", state_in), ("grad_state_out", grad_state_out)):
        if t is not None:
            _check(name, t, torch.float32, (N, H, dk, dv), dev)
    gq, gk, gv = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    gb = torch.empty((T, H), dtype=torch.float32, device=dev)
    ga = torch.empty((T, H, dk), dtype=torch.float32, device=dev)
    gs = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev) if want_state_grad else None
    need = int(L.kda_prefill_backward_workspace_size(N, T, H, dk, dv, _dt(q.dtype)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    wbytes = workspace.numel() * workspace.element_size()
    rc = L.kda_prefill_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(alpha), _ptr(cu_seqlens), N, T, H, dk,
                                dv, _dt(q.dtype), float(scale), _ptr(state_in), _ptr(grad_o), _ptr(grad_state_out),
                                _ptr(gq), _ptr(gk), _ptr(gv), _ptr(gb), _ptr(ga), _ptr(gs), _ptr(workspace), wbytes,
                                _stream(stream))
    if rc != KDA_OK:
        raise KdaError("kda_prefill_backward", rc)
    return gq, gk, gv, gb, ga, gs


def kda_get_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error bits."""
    bits = ctypes.c_uint32(0)
    rc = load().kda_get_device_error(_stream(stream), ctypes.byref(bits))
    if rc not in (KDA_OK, KDA_ERR_DEVICE):
        raise KdaError("kda_get_device_error", rc)
    return int(bits.value)

"""Python front end of the float64 KDA oracle (``kda_oracle.c``).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this module.  The product path (the
CUDA library and its binding) never imports or calls it.

The recurrence lives in ``kda_oracle.c`` ("Kimi K3, explained", section "The
math"); this module compiles it with gcc, marshals the seeded storage arrays
into it and spreads independent (sequence, head) units, or decode rows, over
host threads (ctypes releases the GIL during the call).  What happens here
besides marshalling is plain composition and storage: the alpha layouts of
Gated DeltaNet and DeltaNet are expanded to per-channel alpha, a bf16-stored
decode state is rounded to bf16 after each step, and snapshots are prefills of
successive segments.  The backward pass is ``backward.py`` (token by token) and
``chunked_backward.py`` (its chunkwise matrix form, pinned against it).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIBS: dict = {}

_DT = {"f32": 0, "bf16": 1}


def build(mutant: int | None = None, force: bool = False) -> str:
    """Compile the oracle into a shared library (plain C, double precision, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    name = "libkda_oracle.so" if mutant is None else f"libkda_oracle_m{mutant}.so"
    out = os.path.join(_BUILD, name)
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
               _SRC, "-o", out + ".tmp"]
        if mutant is not None:
            cmd.insert(1, f"-DKDA_ORACLE_MUTANT={int(mutant)}")
        subprocess.run(cmd, check=True)
        os.replace(out + ".tmp", out)
    return out


def _lib(mutant: int | None = None):
    with _LOCK:
        if mutant in _LIBS:
            return _LIBS[mutant]
        lib = ctypes.CDLL(build(mutant))
        vp, i32, i64, f64p = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
        lib.kda_oracle_unit.argtypes = [vp, vp, vp, ctypes.c_int, vp, vp, i64, i64, i32, i32, i32, i32,
                                        ctypes.c_double, i32, f64p, f64p, f64p, i64]
        lib.kda_oracle_unit.restype = ctypes.c_int
        lib.kda_oracle_decode.argtypes = [vp, vp, vp, ctypes.c_int, vp, vp, f64p, vp, i32, i32, i32, i32,
                                          i32, ctypes.c_double, f64p, i32, i32]
        lib.kda_oracle_decode.restype = ctypes.c_int
        _LIBS[mutant] = lib
        return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


def _threads(threads):
    return threads or max(1, os.cpu_count() or 1)


def _check_token_arrays(inp: dict):
    for name in ("q", "k", "v", "beta", "alpha"):
        a = inp[name]
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError(f"{name} must be C-contiguous")
    dt = inp["dtype"]
    want = np.uint16 if dt == "bf16" else np.float32
    for name in ("q", "k", "v"):
        if inp[name].dtype != want:
            raise ValueError(f"{name} dtype {inp[name].dtype} does not match storage dtype {dt}")


def alpha_per_channel(inp: dict) -> dict:
    """The inputs with alpha in the per-channel layout.  "Kimi K3, explained", section "The math": Gated
    DeltaNet's one forget value per head (alpha_mode 1, alpha [T, H]) decays every key channel by it, and
    DeltaNet (alpha_mode 2) has no decay, alpha = 1."""
    mode = inp.get("alpha_mode", 0)
    if mode == 0:
        return inp
    out = dict(inp)
    lead = inp["beta"].shape
    if mode == 1:
        out["alpha"] = np.ascontiguousarray(np.repeat(np.asarray(inp["alpha"], np.float32)[..., None], inp["dk"], -1))
    elif mode == 2:
        out["alpha"] = np.ones((*lead, inp["dk"]), np.float32)
    else:
        raise ValueError("alpha_mode must be 0, 1 or 2")
    out["alpha_mode"] = 0
    return out


def prefill_units(inp: dict, units, scale: float = 1.0, erase: bool = True, want_o: bool = True,
                  threads: int | None = None, mutant: int | None = None, state_in=None):
    """Run selected (sequence, head) units of a packed varlen prefill.

    Returns {(n, h): (o [T_n, d_v] float64 or None, state_out [d_k, d_v] float64)}.
    ``state_in`` overrides ``inp['state_in']`` (float32 or float64, [N, H, d_k, d_v]).
    """
    inp = alpha_per_channel(inp)
    _check_token_arrays(inp)
    lib = _lib(mutant)
    H, dk, dv = inp["H"], inp["dk"], inp["dv"]
    cu = np.asarray(inp["cu_seqlens"], dtype=np.int64)
    s0 = inp.get("state_in") if state_in is None else state_in
    s0 = None if s0 is None else np.ascontiguousarray(s0, dtype=np.float64)
    res = {}

    def run(u):
        n, h = u
        T = int(cu[n + 1] - cu[n])
        so = np.empty((dk, dv), np.float64)
        o = np.empty((T, dv), np.float64) if want_o else None
        si = None if s0 is None else np.ascontiguousarray(s0[n, h])
        rc = lib.kda_oracle_unit(_ptr(inp["q"]), _ptr(inp["k"]), _ptr(inp["v"]), _DT[inp["dtype"]],
                                 _ptr(inp["beta"]), _ptr(inp["alpha"]), int(cu[n]), T, H, h, dk, dv,
                                 float(scale), int(bool(erase)), _ptr(si), _ptr(so), _ptr(o), dv)
        if rc != 0:
            raise RuntimeError("kda_oracle_unit failed")
        res[(n, h)] = (o, so)

    units = list(units)
    if len(units) == 1:
        run(units[0])
    else:
        with ThreadPoolExecutor(_threads(threads)) as ex:
            list(ex.map(run, units))
    return res


def prefill(inp: dict, scale: float = 1.0, erase: bool = True, threads: int | None = None,
            mutant: int | None = None, state_in=None):
    """Full packed varlen prefill: returns (o [T, H, d_v], state_out [N, H, d_k, d_v]), float64."""
    H, dv, dk = inp["H"], inp["dv"], inp["dk"]
    cu = np.asarray(inp["cu_seqlens"], dtype=np.int64)
    N = len(cu) - 1
    res = prefill_units(inp, [(n, h) for n in range(N) for h in range(H)], scale, erase, True,
                        threads, mutant, state_in)
    o = np.empty((int(cu[-1]), H, dv), np.float64)
    st = np.empty((N, H, dk, dv), np.float64)
    for (n, h), (ou, su) in res.items():
        o[cu[n]:cu[n + 1], h, :] = ou
        st[n, h] = su
    return o, st


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Nearest bf16 number (ties to even) of each float64 value, as float64.  The value is first rounded to
    float32 (nearest); bf16 keeps the top 16 bits of a float32, so the low 16 bits are rounded away with
    the usual add-half-minus-one-plus-lsb carry."""
    f = np.ascontiguousarray(x, dtype=np.float64).astype(np.float32)
    bits = f.view(np.uint32).astype(np.uint64)
    bits = (bits + 0x7FFF + ((bits >> 16) & 1)) & 0xFFFF0000
    return bits.astype(np.uint32).view(np.float32).astype(np.float64)


def decode_step(step: dict, pool: np.ndarray, state_idx=None, scale: float = 1.0,
                threads: int | None = None, mutant: int | None = None, state_dtype: str = "f32") -> np.ndarray:
    """One decode step on a float64 state pool [P, H, d_k, d_v], updated in place; returns o [B, H, d_v].

    state_dtype "bf16" models a pool stored in bf16: after the step each updated state is rounded to the
    nearest bf16 (ties to even), as storing it in 2 bytes per element does ("Kimi K3 changed the memory
    math for agentic AI forever", section "Linear Attention's Promise", sizes the state at 2 bytes)."""
    step = alpha_per_channel(step)
    _check_token_arrays(step)
    if pool.dtype != np.float64 or not pool.flags["C_CONTIGUOUS"]:
        raise ValueError("pool must be a C-contiguous float64 array")
    lib = _lib(mutant)
    B, H = step["q"].shape[0], step["H"]
    dk, dv = step["dk"], step["dv"]
    P = pool.shape[0]
    idx = None if state_idx is None else np.ascontiguousarray(state_idx, dtype=np.int32)
    o = np.empty((B, H, dv), np.float64)
    nt = min(_threads(threads), max(1, B))
    edges = np.linspace(0, B, nt + 1).astype(int)

    def run(i):
        rc = lib.kda_oracle_decode(_ptr(step["q"]), _ptr(step["k"]), _ptr(step["v"]), _DT[step["dtype"]],
                                   _ptr(step["beta"]), _ptr(step["alpha"]), _ptr(pool), _ptr(idx), P, B, H,
                                   dk, dv, float(scale), _ptr(o), int(edges[i]), int(edges[i + 1]))
        if rc != 0:
            raise RuntimeError("kda_oracle_decode failed")

    if nt == 1:
        run(0)
    else:
        with ThreadPoolExecutor(nt) as ex:
            list(ex.map(run, range(nt)))
    if state_dtype == "bf16":
        slots = np.arange(B) if idx is None else idx
        pool[slots] = round_bf16(pool[slots])
    elif state_dtype != "f32":
        raise ValueError("state_dtype must be f32 or bf16")
    return o


def prefill_snapshots(inp: dict, every: int, scale: float = 1.0, threads: int | None = None):
    """State snapshots of a prefill: for each sequence n, the state after its first (m + 1) * every tokens,
    m = 0 .. floor(len_n / every) - 1, in order; returns (snapshots [S, H, d_k, d_v] float64, offsets
    [N + 1]).  Each snapshot is the prefill of that prefix, taken segment by segment: the recurrence is
    sequential, so continuing from a segment's final state is the prefix's state ("Kimi K3 changed the
    memory math for agentic AI forever", section "But KDA State Is Not Additive", restartable checkpoints
    at fixed token intervals)."""
    cu = inp["cu_seqlens"]
    N = len(cu) - 1
    H, dk, dv = inp["H"], inp["dk"], inp["dv"]
    snaps, offsets = [], [0]
    for n in range(N):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        state = None if inp["state_in"] is None else np.ascontiguousarray(inp["state_in"][n:n + 1])
        for a in range(t0, t1 - (t1 - t0) % every, every):
            seg = dict(inp)
            for key in ("q", "k", "v", "beta", "alpha"):
                seg[key] = np.ascontiguousarray(inp[key][a:a + every])
            seg["cu_seqlens"] = np.array([0, every], np.int32)
            seg["state_in"] = state                  # the previous segment's final state (or the initial one)
            _, st = prefill(seg, scale=scale, threads=threads)
            state = st
            snaps.append(st[0])
        offsets.append(len(snaps))
    out = np.stack(snaps) if snaps else np.zeros((0, H, dk, dv))
    return out, np.array(offsets, np.int32)

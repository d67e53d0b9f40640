"""Seeded synthetic inputs for the Kimi Delta Attention (KDA) operator.

This module is shared by both sides of every parity check: the CUDA path (tests,
bench) and the float64 oracle (tests, CPU baseline).  It holds none of the
operator's arithmetic -- only random draws, the input-side L2 normalisation of q
and k that the projection step performs ("Kimi K3, explained", section "How Kimi
Delta Attention works, step by step": queries and keys are L2-normalised), the
gate parametrisations of the workloads, and rounding to the storage dtypes.

Recipe (all draws float64, then rounded once to the storage dtype):

* q, k ~ N(0, 1), L2-normalised per (token, head) over d_k, stored bf16 (or f32).
* v ~ N(0, 1), stored bf16 (or f32).
* beta = sigmoid(N(0, 1)), stored f32, shape [T, H].
* alpha = exp(-softplus(N(0, 1) + 2)), one value per key channel, stored f32,
  shape [T, H, d_k].  Other decay modes exist for tests: "slow" divides the
  softplus by 64 so that the state survives across many chunks, "one" is
  alpha == 1 (plain DeltaNet), "scalar" draws one value per (token, head) and
  broadcasts it over the channels (Gated DeltaNet).
* initial state ~ N(0, 0.02) (standard deviation 0.02) in f32, or zero.

Every array is drawn in blocks of ``BLOCK`` tokens; block ``b`` of stream ``s``
uses ``Generator(PCG64(SeedSequence([*seed, s, b])))``, so large workloads can
be generated in parallel and any token range regenerates identically.
"""

from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
import os

import numpy as np

BLOCK = 4096

# stream ids, in the draw order of the recipe
_Q, _K, _V, _BETA, _ALPHA, _STATE = range(6)

DECAY_MODES = ("config", "slow", "one", "scalar")


# ----------------------------------------------------------------------------
# storage rounding
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest even); returns uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bits (uint16) to float32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_storage(x64: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 draws to the storage dtype: 'f32' -> float32, 'bf16' -> uint16 bits."""
    x32 = x64.astype(np.float32)
    if dtype == "f32":
        return x32
    if dtype == "bf16":
        return f32_to_bf16_bits(x32)
    raise ValueError(f"unknown dtype {dtype!r}")


def storage_to_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of stored values to float64."""
    if dtype == "bf16":
        return bf16_bits_to_f32(x).astype(np.float64)
    return np.asarray(x, dtype=np.float64)


# ----------------------------------------------------------------------------
# draws
# ----------------------------------------------------------------------------
def _seed_list(seed) -> list:
    return list(seed) if isinstance(seed, (tuple, list)) else [int(seed)]


def _rng(seed, stream: int, block: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(_seed_list(seed) + [stream, block])))


def _softplus(x: np.ndarray) -> np.ndarray:
    return np.logaddexp(0.0, x)


def _unit_rows(x: np.ndarray) -> np.ndarray:
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return x / np.maximum(n, 1e-300)


def _fill_block(seed, b: int, t0: int, t1: int, H: int, dk: int, dv: int, dtype: str,
                decay: str, out: dict) -> None:
    n = t1 - t0
    q = _unit_rows(_rng(seed, _Q, b).standard_normal((n, H, dk)))
    k = _unit_rows(_rng(seed, _K, b).standard_normal((n, H, dk)))
    v = _rng(seed, _V, b).standard_normal((n, H, dv))
    out["q"][t0:t1] = to_storage(q, dtype)
    out["k"][t0:t1] = to_storage(k, dtype)
    out["v"][t0:t1] = to_storage(v, dtype)
    zb = _rng(seed, _BETA, b).standard_normal((n, H))
    out["beta"][t0:t1] = (1.0 / (1.0 + np.exp(-zb))).astype(np.float32)
    if decay == "one":
        out["alpha"][t0:t1] = 1.0
    elif decay == "scalar":
        za = _rng(seed, _ALPHA, b).standard_normal((n, H, 1))
        out["alpha"][t0:t1] = np.broadcast_to(np.exp(-_softplus(za + 2.0)), (n, H, dk)).astype(np.float32)
    else:
        za = _rng(seed, _ALPHA, b).standard_normal((n, H, dk))
        sp = _softplus(za + 2.0)
        if decay == "slow":
            sp = sp / 64.0
        out["alpha"][t0:t1] = np.exp(-sp).astype(np.float32)


def _threads(threads):
    return threads or max(1, min(32, os.cpu_count() or 1))


def token_inputs(T: int, H: int, dk: int, dv: int, dtype: str, seed, decay: str = "config",
                 threads: int | None = None) -> dict:
    """q, k, v, beta, alpha for T packed tokens and H heads (storage dtypes)."""
    if decay not in DECAY_MODES:
        raise ValueError(f"unknown decay mode {decay!r}")
    sdt = np.uint16 if dtype == "bf16" else np.float32
    out = {
        "q": np.empty((T, H, dk), sdt),
        "k": np.empty((T, H, dk), sdt),
        "v": np.empty((T, H, dv), sdt),
        "beta": np.empty((T, H), np.float32),
        "alpha": np.empty((T, H, dk), np.float32),
    }
    nblk = (T + BLOCK - 1) // BLOCK
    jobs = [(b, b * BLOCK, min(T, (b + 1) * BLOCK)) for b in range(nblk)]
    if nblk <= 1:
        for b, t0, t1 in jobs:
            _fill_block(seed, b, t0, t1, H, dk, dv, dtype, decay, out)
    else:
        with ThreadPoolExecutor(_threads(threads)) as ex:
            list(ex.map(lambda j: _fill_block(seed, j[0], j[1], j[2], H, dk, dv, dtype, decay, out), jobs))
    return out


def random_state(N: int, H: int, dk: int, dv: int, seed, std: float = 0.02) -> np.ndarray:
    """Initial states ~ N(0, std^2), float32, layout [N, H, d_k, d_v]."""
    out = np.empty((N, H, dk, dv), np.float32)
    for n in range(N):
        out[n] = (std * _rng(seed, _STATE, n).standard_normal((H, dk, dv))).astype(np.float32)
    return out


def cu_seqlens_of(seqlens) -> np.ndarray:
    cu = np.zeros(len(seqlens) + 1, np.int32)
    cu[1:] = np.cumsum(np.asarray(seqlens, dtype=np.int64))
    return cu


def prefill_inputs(seqlens, H: int, dk: int, dv: int, dtype: str, seed, decay: str = "config",
                   state: str = "zero", threads: int | None = None) -> dict:
    """Packed varlen prefill inputs: token arrays, cu_seqlens and (optionally) state_in."""
    seqlens = [int(x) for x in seqlens]
    T = int(sum(seqlens))
    d = token_inputs(T, H, dk, dv, dtype, seed, decay, threads)
    d["cu_seqlens"] = cu_seqlens_of(seqlens)
    d["state_in"] = random_state(len(seqlens), H, dk, dv, seed) if state == "randn" else None
    d.update(dtype=dtype, H=H, dk=dk, dv=dv)
    return d


def decode_step_inputs(B: int, H: int, dk: int, dv: int, dtype: str, seed: int, step: int,
                       decay: str = "config") -> dict:
    """Per-step decode inputs (one token for each of B sequences); step s uses seed (seed, 1 + s)."""
    d = token_inputs(B, H, dk, dv, dtype, (seed, 1 + step), decay, threads=1)
    d.update(dtype=dtype, H=H, dk=dk, dv=dv)
    return d


# ----------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------
def varlen_lengths(n: int = 64, lo: int = 128, hi: int = 16384, total_lo: int = 285_000,
                   total_hi: int = 315_000) -> tuple[int, list[int]]:
    """Log-uniform lengths in [lo, hi]; the first seed s >= 2 whose total lies in [total_lo, total_hi].

    The workload is described as 64 sequences, log-uniform in [128, 16384], "about 300K
    tokens"; the log-uniform mean for 64 draws is nearer 214K, so the seed is searched.
    """
    for s in range(2, 10_000):
        u = np.random.Generator(np.random.PCG64(s)).uniform(math.log(lo), math.log(hi), n)
        lens = [int(x) for x in np.floor(np.exp(u))]
        if total_lo <= sum(lens) <= total_hi:
            return s, lens
    raise RuntimeError("no seed found")


WORKLOADS = {
    # tiny correctness case, fp32 throughout
    "tiny_fp32": dict(kind="prefill", seqlens=[64], H=2, dk=16, dv=16, dtype="f32", seed=0, state="zero"),
    # single-sequence prefill, H=32, T=8192
    "prefill_8k": dict(kind="prefill", seqlens=[8192], H=32, dk=128, dv=128, dtype="bf16", seed=1, state="zero"),
    # 64 packed sequences, log-uniform lengths, random initial states
    "varlen_64": dict(kind="prefill", seqlens=None, H=32, dk=128, dv=128, dtype="bf16", seed=2, state="randn"),
    # batched decode: 512 sequences x 32 heads, 256 steps, resident fp32 states
    "decode_512x32": dict(kind="decode", B=512, H=32, dk=128, dv=128, dtype="bf16", seed=3, steps=256),
    # long-context append-prefill: 1,032,192-token prefill then a 16,384-token append
    "append_1m": dict(kind="append", seqlens=[1_032_192], append=16_384, H=8, dk=128, dv=128, dtype="bf16",
                      seed=4, state="zero"),
}


def workload(name: str) -> dict:
    w = dict(WORKLOADS[name])
    if name == "varlen_64":
        w["lengths_seed"], w["seqlens"] = varlen_lengths()
    return w

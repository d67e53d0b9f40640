"""Benchmark of the KDA operator on one GB300 (or N independent replicas under torchrun).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Default workload: the single-sequence prefill (B=1, H=32, T=8192, d_k=d_v=128, bf16 q/k/v, fp32
gates and state).  One step is one kda_prefill call over that batch; `value` is prefill tokens/s
with the inputs resident in HBM.  The same JSON line carries the other workloads as objects, each with
its roofline and the float64 oracle timed on a bounded sample beside it: `decode` (512 sequences x 32
heads of 128x128 fp32 state, 256 steps: steps/s and achieved state-HBM GB/s against the measured copy
bandwidth), `decode_bf16_state`, `varlen_64` (64 packed sequences), `append_1m` (both phases),
`prefill_backward` and `prefill_gated_deltanet`.

Other workloads (`--workload`): varlen_64 (64 packed sequences, ~291K tokens), append_1m (a
1,032,192-token prefill followed by a 16,384-token append, H=8), decode_512x32.

`--impl reference` times the float64 CPU oracle (a deliberately slow baseline) on the host cores on
the same workload, metric and unit.
"""

from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from kda_gated_delta_03_gb300 import inputs as I  # noqa: E402

CSRC = "kda_gated_delta_03_gb300/csrc/"
# sources of each path: the DRAM traffic in profiles/traffic.json is used only while they are unchanged
PREFILL_2P_SRC = [CSRC + "kda_prefill_2p.cu", CSRC + "kda_tc_util.cuh"]
PREFILL_TC_SRC = [CSRC + "kda_prefill_tc.cu", CSRC + "kda_tc_util.cuh"]
DECODE_KERNEL_SRC = [CSRC + "kda_decode.cu"]
DECODE_BF16S_SRC = [CSRC + "kda_decode.cu", CSRC + "kda_decode_bf16s.cu"]
PREFILL_2P_LABEL = "kda_prefill_prep_kernel + kda_prefill_chain_kernel (one call, all windows)"
PREFILL_TC_LABEL = "kda_order_kernel + kda_prefill_tc_kernel (one call)"
DECODE_LABEL = "kda_decode_cols_kernel (fp32 state, two CTAs per state)"
DECODE_BF16S_LABEL = "kda_decode_bf16s_stream_kernel (bf16-stored state, streamed through shared memory)"


PREFILL_2P_MULTI_LABEL = ("kda_chunk_offsets_kernel + kda_order_kernel + kda_prefill_prep_kernel + "
                          "kda_prefill_chain_kernel (one call, all windows)")


def prefill_path(N, dtype, dk):
    """(traffic key, sources, label) of the kernels one kda_prefill call of this shape launches."""
    if dtype == "bf16" and dk == 128:
        if N == 1:
            return "prefill_2p", PREFILL_2P_SRC, PREFILL_2P_LABEL
        return "prefill_2p_multi", PREFILL_2P_SRC, PREFILL_2P_MULTI_LABEL
    return "prefill_tc", PREFILL_TC_SRC, PREFILL_TC_LABEL
METRIC = "KDA prefill tokens/s (H=32,d=128); decode steps/s and state HBM GB/s vs peak"
# what the bf16 prefill computes in: bf16 q/k/v in HBM, tensor-core products on fp16 and TF32 operands with
# fp32 accumulation, the state and every carried sum in fp32
PREFILL_DTYPE = "bf16 in; fp16/tf32 tensor-core operands; fp32 accumulate and state"
DECODE_DTYPE = "bf16 q/k/v; fp32 arithmetic and state"


# ----------------------------------------------------------------------------
# distributed plumbing (replicas only: no data-path collective)
# ----------------------------------------------------------------------------
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def dist_init(world: int):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group("gloo")


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest value of x over all ranks (timing of the slowest replica)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# measurement helpers
# ----------------------------------------------------------------------------
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def code_only(text: str) -> str:
    """A C/CUDA source without its comments and blank lines (string literals here hold no comment
    markers), so that a comment edit does not invalidate a capture taken on the same code."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def source_sha(paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kind: str, paths, workload: str):
    """DRAM bytes per timed launch from the committed ncu summary, if it was taken on the current kernel
    source and on this workload."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    entry = json.load(open(path)).get(kind)
    if not entry or entry.get("source_sha") != source_sha(paths) or entry.get("workload_key") != workload:
        return None
    return entry.get("bytes_per_launch")


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        loaded = [s for s in sm if mx and s >= 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(power) if power else None}


# ----------------------------------------------------------------------------
# workloads on the GPU
# ----------------------------------------------------------------------------
def to_dev(a, bf16=False, dev=None, pin=False):
    import torch
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if bf16 else torch.from_numpy(a)
    if pin:
        return t.pin_memory()
    return t.to(dev)


def prefill_bytes(tokens: int, H: int, dk: int, dv: int, esize: int, n_states_in: int, n_states_out: int) -> int:
    """Algorithmic HBM bytes of one prefill: q, k, v, o in the storage dtype, fp32 alpha and beta, fp32 states."""
    per_token_head = (2 * dk + dv) * esize + 4 * dk + 4 + dv * esize
    return tokens * H * per_token_head + (n_states_in + n_states_out) * H * dk * dv * 4


def decode_bytes_per_step(B: int, H: int, d: int, esize: int, state_esize: int = 4) -> int:
    """Algorithmic HBM bytes of one decode step: state read + write, q, k, v, o, alpha, beta."""
    return B * H * (2 * d * d * state_esize + 4 * d * esize + 4 * d + 4)


def gpu_prefill(inp, steps, warmup, dev, e2e_steps, snapshot_every=0, alpha_mode=0):
    import torch
    import kda_gated_delta_03_gb300 as kda
    bf = inp["dtype"] == "bf16"
    names = ("q", "k", "v", "beta", "alpha", "cu_seqlens") if alpha_mode != 2 else ("q", "k", "v", "beta",
                                                                                     "cu_seqlens")
    host = {n: to_dev(inp[n], bf and n in ("q", "k", "v"), pin=True) for n in names}
    d = {n: host[n].to(dev) for n in names}
    s_in = None if inp["state_in"] is None else to_dev(inp["state_in"], dev=dev)
    T, H, dv = inp["v"].shape
    N = len(inp["cu_seqlens"]) - 1
    dk = inp["dk"]
    o = torch.empty((T, H, dv), dtype=d["q"].dtype, device=dev)
    st = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    ws_bytes = kda.kda_prefill_workspace_size(N, T, H, dk, dv, d["q"].dtype)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    launches_per_call = kda.kda_prefill_launch_count(N, T, H, dk, dv, d["q"].dtype, ws_bytes)
    stream = torch.cuda.current_stream()
    snap = {}
    if snapshot_every:                                # one sequence: floor(T / every) snapshots
        cnt = T // snapshot_every
        snap = dict(snapshot_every=snapshot_every,
                    snapshots=torch.empty((max(cnt, 1), H, dk, dv), dtype=torch.float32, device=dev),
                    snapshot_offsets=torch.tensor([0, cnt], dtype=torch.int32, device=dev))

    def call():
        kda.kda_prefill(d["q"], d["k"], d["v"], d["beta"], d.get("alpha"), d["cu_seqlens"], s_in, state_out=st, o=o,
                        workspace=ws, alpha_mode=alpha_mode, **snap)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(steps):
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    total_ms = start.elapsed_time(end)
    kernel_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)

    # end to end: pinned host inputs -> device, the C-ABI call, outputs -> pinned host
    o_h = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    st_h = torch.empty(st.shape, dtype=st.dtype).pin_memory()
    s_in_h = None if s_in is None else s_in.cpu().pin_memory()
    h2d = sum(host[n].numel() * host[n].element_size() for n in names) + (
        0 if s_in_h is None else s_in_h.numel() * 4)
    d2h = o.numel() * o.element_size() + st.numel() * 4

    if alpha_mode == 0 and not snapshot_every:
        # the C-ABI entry with host buffers: the library streams the inputs in and the outputs out,
        # overlapped with the compute
        dbuf = torch.empty(kda.load().kda_prefill_host_buffer_size(N, T, H, dk, dv, 1 if bf else 0),
                           dtype=torch.uint8, device=dev)

        def e2e_call():
            kda.kda_prefill_host(host["q"], host["k"], host["v"], host["beta"], host["alpha"], host["cu_seqlens"],
                                 s_in_h, o=o_h, state_out=st_h, device_buffer=dbuf)
    else:
        def e2e_call():
            for n in names:
                d[n].copy_(host[n], non_blocking=True)
            if s_in is not None:
                s_in.copy_(s_in_h, non_blocking=True)
            call()
            o_h.copy_(o, non_blocking=True)
            st_h.copy_(st, non_blocking=True)

    for _ in range(2):
        e2e_call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_call()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    return dict(total_ms=total_ms, ms_per_step=total_ms / steps, kernel_ms=kernel_ms, e2e_ms=e2e_ms, h2d=h2d,
                d2h=d2h, launches=steps * launches_per_call, T=T, H=H, N=N)


def gpu_backward(inp, steps, warmup, dev):
    """kda_prefill_backward on the workload (gradients of q, k, v, beta, alpha and state_in), inputs and
    the output gradient resident on the device."""
    import torch
    import kda_gated_delta_03_gb300 as kda
    bf = inp["dtype"] == "bf16"
    d = {n: to_dev(inp[n], bf and n in ("q", "k", "v"), dev=dev) for n in ("q", "k", "v", "beta", "alpha",
                                                                          "cu_seqlens")}
    T, H, dv = inp["v"].shape
    N = len(inp["cu_seqlens"]) - 1
    go = torch.randn((T, H, dv), device=dev).to(d["q"].dtype)
    need = kda.load().kda_prefill_backward_workspace_size(N, T, H, inp["dk"], dv, 1 if bf else 0)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def call():
        kda.kda_prefill_backward(d["q"], d["k"], d["v"], d["beta"], d["alpha"], d["cu_seqlens"], go, workspace=ws)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    return dict(ms_per_step=e0.elapsed_time(e1) / steps, T=T, H=H, N=N)


def gpu_decode(w, steps, warmup, dev, distinct=16, state_dtype="f32"):
    """Batched decode: `steps` fused steps over the resident pool; step s uses input set s mod `distinct`.
    state_dtype "bf16" runs the bf16-stored state (kda_decode_step_bf16_state)."""
    import torch
    import kda_gated_delta_03_gb300 as kda
    B, H, d, dt = w["B"], w["H"], w["dk"], w["dtype"]
    bf = dt == "bf16"
    pool = torch.empty((B, H, d, d), dtype=torch.bfloat16 if state_dtype == "bf16" else torch.float32, device=dev)
    for b0 in range(0, B, 64):   # seeded N(0, 0.02) states, generated in slices to bound host memory
        pool[b0:b0 + 64] = to_dev(I.random_state(min(64, B - b0), H, d, d, (w["seed"], b0)), dev=dev)
    sets = []
    for s in range(distinct):
        st = I.decode_step_inputs(B, H, d, d, dt, w["seed"], s)
        sets.append({n: to_dev(st[n], bf and n in ("q", "k", "v"), dev=dev) for n in ("q", "k", "v", "beta", "alpha")})
    o = torch.empty((B, H, d), dtype=sets[0]["q"].dtype, device=dev)
    stream = torch.cuda.current_stream()

    def call(i):
        x = sets[i % distinct]
        kda.kda_decode_step(x["q"], x["k"], x["v"], x["beta"], x["alpha"], pool, o=o)

    for i in range(warmup):
        call(i)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(steps):
        ev[i][0].record(stream)
        call(i)
        ev[i][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    total_ms = start.elapsed_time(end)
    kernel_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    return dict(total_ms=total_ms, ms_per_step=total_ms / steps, kernel_ms=kernel_ms, launches=steps,
                bytes_per_step=decode_bytes_per_step(B, H, d, 2 if bf else 4, 2 if state_dtype == "bf16" else 4))


# ----------------------------------------------------------------------------
# CPU oracle leg
# ----------------------------------------------------------------------------
def oracle_prefill_time(inp, threads):
    from oracle import oracle as O
    t0 = time.perf_counter()
    O.prefill(inp, threads=threads)
    return time.perf_counter() - t0


def cpu_threads():
    return max(1, os.cpu_count() or 1)


def sub_sequences(inp, seqs):
    """The inputs of a subset of the packed sequences (same values), for a bounded oracle sample."""
    cu = inp["cu_seqlens"]
    sub = dict(inp)
    for key in ("q", "k", "v", "beta", "alpha"):
        sub[key] = np.ascontiguousarray(np.concatenate([inp[key][cu[n]:cu[n + 1]] for n in seqs]))
    sub["cu_seqlens"] = I.cu_seqlens_of([int(cu[n + 1] - cu[n]) for n in seqs])
    if inp["state_in"] is not None:
        sub["state_in"] = np.ascontiguousarray(inp["state_in"][list(seqs)])
    return sub


def oracle_varlen_baseline(inp, threads, min_tokens=16_000):
    """The oracle on the first sequences of the packed batch whose lengths add up to at least min_tokens
    (all heads), in tokens/s."""
    cu = inp["cu_seqlens"]
    seqs, tok = [], 0
    for n in range(len(cu) - 1):
        seqs.append(n)
        tok += int(cu[n + 1] - cu[n])
        if tok >= min_tokens:
            break
    secs = oracle_prefill_time(sub_sequences(inp, seqs), threads)
    H = inp["v"].shape[1]
    return {"value": round(tok / secs, 1), "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"the first {len(seqs)} of the {len(cu) - 1} sequences ({tok} tokens x {H} heads, "
                      f"{tok / int(cu[-1]):.3f} of the workload), float64, {threads} threads"}


def oracle_decode_baseline(w, threads, rows=64, steps=2):
    """The oracle's decode step on `rows` of the batch's sequences (all heads), scaled to the full batch."""
    from oracle import oracle as O
    pool = I.random_state(rows, w["H"], w["dk"], w["dv"], (w["seed"], 0)).astype(np.float64)
    sts = [I.decode_step_inputs(rows, w["H"], w["dk"], w["dv"], w["dtype"], w["seed"], s_) for s_ in range(steps)]
    t0 = time.perf_counter()
    for st in sts:
        O.decode_step(st, pool, threads=threads)
    per_step = (time.perf_counter() - t0) / steps * w["B"] / rows
    return {"value": round(1.0 / per_step, 3), "unit": "steps/s", "cores": threads, "kind": "oracle",
            "sample": f"{steps} steps of {rows} of the {w['B']} sequences x {w['H']} heads, scaled to the "
                      f"full batch, float64, {threads} threads"}


# ----------------------------------------------------------------------------
# main
# ----------------------------------------------------------------------------
def prefill_workload_inputs(name):
    w = I.workload(name)
    return w, I.prefill_inputs(w["seqlens"], w["H"], w["dk"], w["dv"], w["dtype"], w["seed"], state=w["state"])


def roofline_obj(alg_bytes, kernel_ms, peaks, kind, src, label, workload):
    """HBM roofline of the timed launch sequence: algorithmic bytes / CUDA-event time per call."""
    achieved = alg_bytes / (kernel_ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": ncu_traffic(kind, src, workload),
            "kernel": label, "alg_bytes_per_launch": int(alg_bytes), "kernel_ms": round(kernel_ms, 4),
            "peak_source": peaks["source"]}


def decode_object(wd, dev, peaks, world, state_dtype="f32"):
    """The decode_512x32 workload (all 256 steps) as a sub-object of the default line."""
    rd = gpu_decode(wd, wd["steps"], 3, dev, state_dtype=state_dtype)
    dms = max_over_ranks(rd["ms_per_step"], world)
    bf = state_dtype == "bf16"
    roof = roofline_obj(rd["bytes_per_step"], rd["kernel_ms"], peaks, "decode_bf16" if bf else "decode",
                        DECODE_BF16S_SRC if bf else DECODE_KERNEL_SRC, DECODE_BF16S_LABEL if bf else DECODE_LABEL,
                        "decode_512x32_bf16_state" if bf else "decode_512x32")
    return {"workload": "decode_512x32" + (", state stored in bf16" if bf else ""), "steps": wd["steps"],
            "steps_per_s": round(world * 1e3 / dms, 2), "tokens_per_s": round(world * wd["B"] * 1e3 / dms, 1),
            "ms_per_step": round(dms, 4), "state_hbm_gbs": roof["achieved"], "roofline": roof,
            "dtype": DECODE_DTYPE if not bf else "bf16 q/k/v and state; fp32 arithmetic",
            "gpu_launches": rd["launches"]}


def varlen_object(dev, peaks, world, steps, warmup, with_oracle):
    """The varlen_64 workload (64 packed sequences, about 291K tokens, random initial states)."""
    w, inp = prefill_workload_inputs("varlen_64")
    r = gpu_prefill(inp, steps, warmup, dev, 2)
    ms = max_over_ranks(r["ms_per_step"], world)
    e2e_ms = max_over_ranks(r["e2e_ms"], world)
    alg = prefill_bytes(r["T"], r["H"], inp["dk"], inp["dv"], 2, r["N"], r["N"])
    obj = {"workload": "varlen_64", "seqs": r["N"], "tokens": r["T"], "H": r["H"], "steps": steps,
           "tokens_per_s": round(world * r["T"] * 1e3 / ms, 1), "ms_per_step": round(ms, 4),
           "roofline": roofline_obj(alg, r["kernel_ms"], peaks, *prefill_path(r["N"], "bf16", inp["dk"]), "varlen_64"),
           "e2e": {"value": round(world * r["T"] * 1e3 / e2e_ms, 1), "unit": "tokens/s",
                   "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
           "gpu_launches": r["launches"]}
    if with_oracle:
        obj["cpu_baseline"] = oracle_varlen_baseline(inp, cpu_threads())
    return obj


def append_object(dev, peaks, world, steps, warmup, with_oracle):
    """The append_1m workload: both phases (prefill and append), without the snapshot variant."""
    w = I.workload("append_1m")
    a = append_measure(w, steps, warmup, dev, peaks, world, snapshots=False)
    obj = {"workload": "append_1m", "H": w["H"], "steps": steps,
           "prefill": {"tokens": a["T1"], "tokens_per_s": round(world * a["T1"] * 1e3 / a["ms1"], 1),
                       "ms_per_step": round(a["ms1"], 4), "roofline": a["roof1"],
                       "e2e": {"value": round(world * a["T1"] * 1e3 / a["r1"]["e2e_ms"], 1), "unit": "tokens/s",
                               "h2d_bytes_per_step": a["r1"]["h2d"], "d2h_bytes_per_step": a["r1"]["d2h"]}},
           "append": {"tokens": a["T2"], "tokens_per_s": round(world * a["T2"] * 1e3 / a["ms2"], 1),
                      "ms_per_step": round(a["ms2"], 4), "roofline": a["roof2"]},
           "gpu_launches": a["r1"]["launches"] + a["r2"]["launches"]}
    if with_oracle:
        obj["cpu_baseline"] = oracle_append_baseline(a["prefix"], cpu_threads())
    return obj


def run_ours(args, rank, world, local_rank):
    import torch
    import kda_gated_delta_03_gb300 as kda
    from kda_gated_delta_03_gb300 import build
    build.build()
    kda.load()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    name = args.workload
    oracle_here = rank == 0 and not args.no_cpu_baseline
    line = {"metric": METRIC, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "data": "synthetic"}
    if name in ("decode_512x32", "decode_512x32_bf16_state"):
        sdt = "bf16" if name.endswith("bf16_state") else "f32"
        w = I.workload("decode_512x32")
        barrier(world)
        with ClockSampler(local_rank) as clk:
            r = gpu_decode(w, args.steps, args.warmup, dev, state_dtype=sdt)
        ms = max_over_ranks(r["ms_per_step"], world)
        steps_s = world * 1e3 / ms
        line.update(metric="KDA decode steps/s (512 seqs x 32 heads, d=128)", value=round(steps_s, 2),
                    unit="steps/s", ms_per_step=round(ms, 4),
                    dtype=DECODE_DTYPE if sdt == "f32" else "bf16 q/k/v and state; fp32 arithmetic",
                    config=workload_config(name, world),
                    roofline=roofline_obj(r["bytes_per_step"], r["kernel_ms"], peaks,
                                          "decode_bf16" if sdt == "bf16" else "decode",
                                          DECODE_BF16S_SRC if sdt == "bf16" else DECODE_KERNEL_SRC,
                                          DECODE_BF16S_LABEL if sdt == "bf16" else DECODE_LABEL, name),
                    gpu_launches=r["launches"], clocks=clk.summary())
        if oracle_here:
            line["cpu_baseline"] = oracle_decode_baseline(w, cpu_threads())
        return line

    if name == "append_1m":
        return run_append(args, I.workload(name), dev, peaks, line, world, local_rank)
    w, inp = prefill_workload_inputs(name)
    barrier(world)
    with ClockSampler(local_rank) as clk:
        r = gpu_prefill(inp, args.steps, args.warmup, dev, args.e2e_steps)
    ms = max_over_ranks(r["ms_per_step"], world)
    e2e_ms = max_over_ranks(r["e2e_ms"], world)
    tokens = r["T"]
    esize = 2 if inp["dtype"] == "bf16" else 4
    alg = prefill_bytes(tokens, r["H"], inp["dk"], inp["dv"], esize, 0 if inp["state_in"] is None else r["N"], r["N"])
    line.update(value=round(world * tokens * 1e3 / ms, 1), unit="tokens/s", ms_per_step=round(ms, 4),
                dtype=PREFILL_DTYPE if inp["dtype"] == "bf16" else "f32",
                config=workload_config(name, world),
                roofline=roofline_obj(alg, r["kernel_ms"], peaks, *prefill_path(r["N"], inp["dtype"], inp["dk"]), name),
                e2e={"value": round(world * tokens * 1e3 / e2e_ms, 1), "unit": "tokens/s",
                     "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
                gpu_launches=r["launches"], clocks=clk.summary())
    if name == "prefill_8k" and args.steady_steps > 0:
        # the same call back to back over a longer region (inputs larger than L2), to show the number is steady
        rs = gpu_prefill(inp, args.steady_steps, 3, dev, 1)
        line["steady"] = {"steps": args.steady_steps, "ms_per_step": round(rs["ms_per_step"], 4),
                          "timed_region_s": round(rs["total_ms"] / 1e3, 3),
                          "tokens_per_s": round(tokens * 1e3 / rs["ms_per_step"], 1)}
    if name == "prefill_8k" and not args.no_decode:
        wd = I.workload("decode_512x32")
        line["decode"] = decode_object(wd, dev, peaks, world)
        if oracle_here:
            line["decode"]["cpu_baseline"] = oracle_decode_baseline(wd, cpu_threads())
        line["gpu_launches"] += line["decode"]["gpu_launches"]
        line["decode_bf16_state"] = decode_object(wd, dev, peaks, world, state_dtype="bf16")
        line["gpu_launches"] += line["decode_bf16_state"]["gpu_launches"]
    if name == "prefill_8k" and not args.no_backward:
        # the backward pass of the same prefill (per-channel alpha)
        rw = gpu_backward(inp, 5, 3, dev)
        wms = max_over_ranks(rw["ms_per_step"], world)
        dk_, dv_ = inp["dk"], inp["dv"]
        # reads q, k, v, alpha, beta, grad_o; writes grad_q, grad_k, grad_v, grad_alpha, grad_beta
        bwd_bytes = tokens * r["H"] * (2 * (2 * dk_ + dv_) * esize + 2 * (4 * dk_ + 4) + dv_ * esize)
        line["prefill_backward"] = {"workload": name + ", gradients of q, k, v, beta, alpha (forward recompute "
                                                       "with a snapshot every 64 tokens, state-gradient chain, "
                                                       "then one unit per (chunk, head))",
                                    "tokens_per_s": round(world * tokens * 1e3 / wms, 1), "ms_per_step": round(wms, 4),
                                    "alg_bytes_per_step": int(bwd_bytes),
                                    "hbm_gbs": round(bwd_bytes / (wms * 1e-3) / 1e9, 1)}
    if name == "prefill_8k" and not args.no_gdn:
        # the same prefill with one forget value per (token, head): Gated DeltaNet's layout of alpha
        gd = dict(inp, alpha=np.ascontiguousarray(inp["alpha"][..., 0]))
        rg = gpu_prefill(gd, args.steps, args.warmup, dev, 1, alpha_mode=1)
        gms = max_over_ranks(rg["ms_per_step"], world)
        algg = alg - tokens * r["H"] * (inp["dk"] - 1) * 4
        line["prefill_gated_deltanet"] = {"workload": name + ", alpha one value per (token, head)",
                                          "tokens_per_s": round(world * tokens * 1e3 / gms, 1),
                                          "ms_per_step": round(gms, 4),
                                          "roofline": roofline_obj(algg, rg["kernel_ms"], peaks, "prefill_2p_gdn",
                                                                   PREFILL_2P_SRC, PREFILL_2P_LABEL, name + "_gdn"),
                                          "gpu_launches": rg["launches"]}
    if oracle_here:
        threads = cpu_threads()
        if name == "varlen_64":
            line["cpu_baseline"] = oracle_varlen_baseline(inp, threads)
        else:
            secs = oracle_prefill_time(inp, threads)
            line["cpu_baseline"] = {"value": round(tokens / secs, 1), "unit": "tokens/s", "cores": threads,
                                    "kind": "oracle", "sample": f"the whole {name} workload once ({tokens} tokens x "
                                                                f"{r['H']} heads), float64, {threads} threads"}
    if name == "prefill_8k" and not args.no_varlen:
        del inp
        line["varlen_64"] = varlen_object(dev, peaks, world, args.sub_steps, 3, oracle_here)
        line["gpu_launches"] += line["varlen_64"]["gpu_launches"]
        torch.cuda.empty_cache()
    if name == "prefill_8k" and not args.no_append:
        line["append_1m"] = append_object(dev, peaks, world, args.sub_steps, 3, oracle_here)
        line["gpu_launches"] += line["append_1m"]["gpu_launches"]
        torch.cuda.empty_cache()
    return line


def append_measure(w, steps, warmup, dev, peaks, world, snapshots=True, e2e_steps=1):
    """append_1m: the 1,032,192-token prefill from a zero state, then the 16,384-token append from the
    carried state (timed from a state of the same shape), and optionally the prefill writing snapshots."""
    T1, T2 = w["seqlens"][0], w["append"]
    full = I.prefill_inputs([T1 + T2], w["H"], w["dk"], w["dv"], w["dtype"], w["seed"])

    def part(t0, t1):
        d = dict(full)
        for k in ("q", "k", "v", "beta", "alpha"):
            d[k] = full[k][t0:t1]
        d["cu_seqlens"] = I.cu_seqlens_of([t1 - t0])
        return d

    p1 = part(0, T1)
    r1 = gpu_prefill(p1, steps, warmup, dev, e2e_steps)
    p2 = part(T1, T1 + T2)
    p2["state_in"] = np.zeros((1, w["H"], w["dk"], w["dv"]), np.float32)
    r2 = gpu_prefill(p2, steps, warmup, dev, 1)
    ms1 = max_over_ranks(r1["ms_per_step"], world)
    ms2 = max_over_ranks(r2["ms_per_step"], world)
    alg1 = prefill_bytes(T1, w["H"], w["dk"], w["dv"], 2, 0, 1)
    alg2 = prefill_bytes(T2, w["H"], w["dk"], w["dv"], 2, 1, 1)
    out = {"T1": T1, "T2": T2, "r1": r1, "r2": r2, "ms1": ms1, "ms2": ms2,
           "roof1": roofline_obj(alg1, r1["kernel_ms"], peaks, *prefill_path(1, "bf16", w["dk"]), "append_1m"),
           "roof2": roofline_obj(alg2, r2["kernel_ms"], peaks, *prefill_path(1, "bf16", w["dk"]), "append_1m/append"),
           "prefix": p1}
    if snapshots:
        every = 312 * 64                              # restartable checkpoints about every 20,000 tokens
        r3 = gpu_prefill(p1, steps, warmup, dev, 1, snapshot_every=every)
        ms3 = max_over_ranks(r3["ms_per_step"], world)
        out["snapshots"] = {"every_tokens": every, "count": T1 // every,
                            "bytes": (T1 // every) * w["H"] * w["dk"] * w["dv"] * 4,
                            "tokens_per_s": round(world * T1 * 1e3 / ms3, 1), "ms_per_step": round(ms3, 4),
                            "overhead": round(ms3 / ms1 - 1.0, 4), "gpu_launches": r3["launches"]}
    return out


def oracle_append_baseline(prefix, threads, tokens=16_384):
    """The oracle on the first `tokens` tokens of the long sequence (all heads): the append phase's size.
    The oracle's cost per token does not depend on the state it starts from."""
    d = dict(prefix)
    for k in ("q", "k", "v", "beta", "alpha"):
        d[k] = prefix[k][:tokens]
    d["cu_seqlens"] = I.cu_seqlens_of([tokens])
    secs = oracle_prefill_time(d, threads)
    H = prefix["v"].shape[1]
    used = min(threads, H)
    return {"value": round(tokens / secs, 1), "unit": "tokens/s", "cores": used, "kind": "oracle",
            "sample": f"the first {tokens} tokens x {H} heads of the sequence (the append phase's size), "
                      f"float64, {used} threads (one per head)"}


def run_append(args, w, dev, peaks, line, world, local_rank):
    barrier(world)
    with ClockSampler(local_rank) as clk:
        a = append_measure(w, args.steps, args.warmup, dev, peaks, world)
    r1, r2 = a["r1"], a["r2"]
    T1, T2 = a["T1"], a["T2"]
    line.update(metric="KDA append-prefill tokens/s (H=8, d=128): 1,032,192-token prefill",
                value=round(world * T1 * 1e3 / a["ms1"], 1), unit="tokens/s", ms_per_step=round(a["ms1"], 4),
                dtype=PREFILL_DTYPE,
                config=workload_config("append_1m", world),
                roofline=a["roof1"],
                e2e={"value": round(world * T1 * 1e3 / r1["e2e_ms"], 1), "unit": "tokens/s",
                     "h2d_bytes_per_step": r1["h2d"], "d2h_bytes_per_step": r1["d2h"]},
                append={"tokens_per_s": round(world * T2 * 1e3 / a["ms2"], 1), "ms_per_step": round(a["ms2"], 4),
                        "roofline": a["roof2"]},
                snapshots=a["snapshots"], gpu_launches=r1["launches"] + r2["launches"], clocks=clk.summary())
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_append_baseline(a["prefix"], cpu_threads())
    return line


def workload_config(name, world):
    """The `config` object of a workload's bench line: the workload itself (the GPU arm's keys), whatever
    sample of it an arm times."""
    if name.startswith("decode_512x32"):
        w = I.workload("decode_512x32")
        bf = name.endswith("bf16_state")
        return {"workload": name, "B": w["B"], "H": w["H"], "d": w["dk"], "qkv": w["dtype"],
                "state": "bf16" if bf else "f32", "l2": f"state pool ({'0.5' if bf else '1'} GiB) larger than L2"}
    w = I.workload(name)
    if name == "append_1m":
        return {"workload": name, "prefill_tokens": int(sum(w["seqlens"])), "append_tokens": int(w["append"]),
                "H": w["H"], "d": w["dk"], "l2": "inputs larger than L2 (no flush)"}
    return {"workload": name, "seqs": len(w["seqlens"]), "tokens": int(sum(w["seqlens"])), "H": w["H"], "d": w["dk"],
            "qkv": w["dtype"], "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas{world}"}


def run_reference(args, rank, world):
    """The float64 CPU oracle on the host cores, one bounded sample of the workload per step."""
    if rank != 0:
        return None
    name = args.workload
    threads = cpu_threads()
    if name.startswith("decode_512x32"):
        w = I.workload("decode_512x32")
        times = []
        for i in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            b = oracle_decode_baseline(w, threads, rows=16, steps=1)
            if i >= args.warmup:
                times.append(time.perf_counter() - t0)
        value, unit = b["value"], "steps/s"
        metric, sample = "KDA decode steps/s (512 seqs x 32 heads, d=128)", b["sample"]
        ms = 1e3 / value
    else:
        if name == "append_1m":
            w = I.workload(name)
            sample_inp = I.prefill_inputs([16_384], w["H"], w["dk"], w["dv"], w["dtype"], w["seed"])
            sample = f"the first 16384 tokens x {w['H']} heads of the sequence (the append phase's size)"
            metric = "KDA append-prefill tokens/s (H=8, d=128): 1,032,192-token prefill"
        elif name == "varlen_64":
            w, inp = prefill_workload_inputs(name)
            cu = inp["cu_seqlens"]
            seqs, tok = [], 0
            for n in range(len(cu) - 1):
                seqs.append(n)
                tok += int(cu[n + 1] - cu[n])
                if tok >= 16_000:
                    break
            sample_inp = sub_sequences(inp, seqs)
            del inp
            sample = f"the first {len(seqs)} of the 64 sequences ({tok} tokens x {w['H']} heads)"
            metric = METRIC
        else:
            w, sample_inp = prefill_workload_inputs(name)
            sample = f"the whole {name} workload ({int(sample_inp['cu_seqlens'][-1])} tokens x {w['H']} heads)"
            metric = METRIC
        tokens = int(sample_inp["cu_seqlens"][-1])
        times = []
        for i in range(args.warmup + args.steps):
            s_ = oracle_prefill_time(sample_inp, threads)
            if i >= args.warmup:
                times.append(s_)
        secs = statistics.mean(times)
        value, unit = tokens / secs, "tokens/s"
        sample += " per step, float64"
        ms = secs * 1e3
    return {"impl": "reference", "metric": metric, "value": round(value, 3), "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(name, world),
            "cpu_baseline": {"value": round(value, 3), "unit": unit, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 3), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="prefill_8k",
                    choices=["prefill_8k", "varlen_64", "decode_512x32", "decode_512x32_bf16_state", "append_1m"])
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-decode", action="store_true", help="skip the decode lines of the prefill_8k run")
    ap.add_argument("--no-backward", action="store_true", help="skip the backward line of the prefill_8k run")
    ap.add_argument("--no-gdn", action="store_true", help="skip the Gated DeltaNet line of the prefill_8k run")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-varlen", action="store_true", help="skip the varlen_64 object of the prefill_8k run")
    ap.add_argument("--no-append", action="store_true", help="skip the append_1m object of the prefill_8k run")
    ap.add_argument("--sub-steps", type=int, default=5,
                    help="timed calls of the varlen_64 and append_1m objects of the prefill_8k run")
    ap.add_argument("--steady-steps", type=int, default=1000,
                    help="calls of the steadiness run of prefill_8k (0 = none)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    rank, world, local_rank = dist_env()
    dist_init(world)
    line = run_reference(args, rank, world) if args.impl == "reference" else run_ours(args, rank, world, local_rank)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

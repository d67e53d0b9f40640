"""Shared helpers of the tests: device transfer of the seeded storage arrays and the error metric."""

import numpy as np
import torch

# Relative Frobenius error bounds, per storage dtype of q, k, v, o: 1e-4 with float32 inputs, 3e-3 with bf16
# inputs and float32 state.
TOL = {"f32": 1e-4, "bf16": 3e-3}


def to_dev(a, bf16: bool = False, dev="cuda:0"):
    a = np.ascontiguousarray(a)
    if bf16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(a).to(dev)


def rel_frob(x, ref) -> float:
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300))


def prefill_gpu(inp, state_in="from_inputs", scale=1.0, dev="cuda:0"):
    """Run kda_prefill on the seeded inputs; returns (o float64 [T,H,dv], state float64 [N,H,dk,dv])."""
    import kda_gated_delta_03_gb300 as kda
    bf = inp["dtype"] == "bf16"
    s0 = inp["state_in"] if isinstance(state_in, str) else state_in
    o, st = kda.kda_prefill(to_dev(inp["q"], bf, dev), to_dev(inp["k"], bf, dev), to_dev(inp["v"], bf, dev),
                            to_dev(inp["beta"], dev=dev), to_dev(inp["alpha"], dev=dev),
                            to_dev(inp["cu_seqlens"], dev=dev),
                            None if s0 is None else to_dev(np.asarray(s0, np.float32), dev=dev), scale=scale)
    torch.cuda.synchronize()
    return o.double().cpu().numpy(), st.double().cpu().numpy()

"""Kimi Delta Attention (KDA) operator for one GB300 GPU (sm_103a).

The operator runs in hand-written CUDA kernels behind the C ABI of libkda
(``include/kda.h``); this package is its thin Python binding plus the seeded
input generator (``inputs``) and the build step (``build``).
"""

from .binding import (KdaError, kda_decode_step, kda_get_device_error, kda_prefill, kda_prefill_backward,
                      kda_prefill_host, kda_prefill_launch_count, kda_prefill_noalloc, kda_prefill_workspace_size,
                      kda_status_string, load)

__all__ = ["KdaError", "kda_decode_step", "kda_get_device_error", "kda_prefill", "kda_prefill_backward",
           "kda_prefill_host", "kda_prefill_launch_count", "kda_prefill_noalloc", "kda_prefill_workspace_size", "kda_status_string",
           "load"]

"""Host-side logic of bench.py that needs no GPU: both arms describe a workload with the same config object,
and it names the workload's own sizes."""

import pytest

import bench
from kda_gated_delta_03_gb300 import inputs as I


@pytest.mark.parametrize("name", ["prefill_8k", "varlen_64", "append_1m", "decode_512x32", "decode_512x32_bf16_state"])
def test_workload_config_names_the_workload(name):
    c = bench.workload_config(name, 1)
    assert c["workload"] == name
    w = I.workload("decode_512x32" if name.startswith("decode") else name)
    assert c["H"] == w["H"] and c["d"] == w["dk"]
    if name.startswith("decode"):
        assert c["B"] == w["B"] and c["state"] == ("bf16" if name.endswith("bf16_state") else "f32")
    elif name == "append_1m":
        assert c["prefill_tokens"] == sum(w["seqlens"]) and c["append_tokens"] == w["append"]
    else:
        assert c["seqs"] == len(w["seqlens"]) and c["tokens"] == sum(w["seqlens"])
        assert c["parallelism"] == "replicas1" and bench.workload_config(name, 4)["parallelism"] == "replicas4"

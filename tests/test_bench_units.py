"""bench.py's launch units (no GPU): which GEMVs of a workload share one grouped launch,
and the algorithmic bytes each launch is charged."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402
from quantized_weight_dequant_gb300 import synth  # noqa: E402


def test_plain_workloads_launch_every_gemv_alone():
    g = bench.WORKLOADS["q4k_llama8b_decode"]
    units = bench.launch_units("q4k_llama8b_decode", g)
    assert units == [("qkv", [0], False), ("gate_up", [1], False), ("down", [2], False)]
    assert sum(bench.unit_bytes(g, i, s) for _, i, s in units) == sum(bench.gemv_bytes(*x[1:4]) for x in g)


def test_grouped_layer_shares_x_and_pairs_gate_with_up():
    g = bench.WORKLOADS["layer_mixed_grouped"]
    units = bench.launch_units("layer_mixed_grouped", g)
    assert [(u[0], [g[i][0] for i in u[1]], u[2]) for u in units] == [
        ("qkv", ["q", "k", "v"], False), ("o", ["o"], False), ("mlp", ["gate", "up"], True), ("down", ["down"], False)]
    # one x per launch; the SwiGLU pair writes one output per row
    qkv = bench.unit_bytes(g, units[0][1], False)
    assert qkv == sum(synth.packed_bytes(g[i][1], g[i][2], g[i][3]) for i in (0, 1, 2)) + 2 * 4096 + 4 * (4096 + 2048)
    mlp = bench.unit_bytes(g, units[2][1], True)
    assert mlp == 2 * synth.packed_bytes(synth.Q4_K, 12288, 4096) + 2 * 4096 + 4 * 12288


def test_swiglu_group_must_hold_two_matrices(monkeypatch):
    monkeypatch.setitem(bench.GROUPS, "q4k_llama8b_decode", {"qkv": "mlp"})
    with pytest.raises(ValueError):
        bench.launch_units("q4k_llama8b_decode", bench.WORKLOADS["q4k_llama8b_decode"])


def test_prefill_option_is_validated():
    """--prefill takes a row count >= 0; the oracle arm has no prefill measurement."""
    import bench
    with pytest.raises(SystemExit):
        bench.main(["--prefill", "-1"])

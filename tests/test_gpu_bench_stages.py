"""The benchmark's single-stage and A/B modes run end to end on the tiny and a
small skewed workload and print one well-formed JSON line each (the modes the
profile summaries' numbers come from)."""
import json

import pytest
import torch

import bench

pytestmark = pytest.mark.gpu


def _run(capsys, argv):
    assert bench.main(argv) == 0
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    return json.loads(lines[0])


def test_router_stage(capsys):
    j = _run(capsys, ["--stage", "router", "--workload", "tiny", "--steps", "3", "--warmup", "1",
                      "--no-clocks"])
    assert j["stage"] == "router" and j["kernel_ms"]["router"] > 0.0
    assert 0.0 < j["router_frac_of_hbm"] < 2.0


def test_ffn_stage(capsys):
    j = _run(capsys, ["--stage", "ffn", "--workload", "tiny", "--steps", "3", "--warmup", "1",
                      "--no-clocks", "--tune", "tail_max_n=-1"])
    assert j["stage"] == "ffn" and j["tune"] == {"tail_max_n": -1}
    assert j["kernel_ms"]["gemm_swiglu"] > 0.0 and j["kernel_ms"]["gemm_down"] > 0.0
    assert sum(j["rows"]) == 64 * 2


def test_ab_stage_same_bits_for_a_pure_scheduling_change(capsys):
    """Two layers that differ only in the order of their tiles give the same
    bits, and each call of both is timed."""
    j = _run(capsys, ["--stage", "ab", "--workload", "tiny", "--steps", "4", "--warmup", "1",
                      "--tune", "n_block=1", "--tune-b", "n_block=2", "--tune-b",
                      "block_min_rows=1"])
    assert j["A"] == {"n_block": 1} and j["B"] == {"n_block": 2, "block_min_rows": 1}
    assert j["calls_each"] == 4 and all(t > 0.0 for t in j["layer_ms"])
    assert set(j["kernel_us"][0]) >= {"router", "scatter", "gemm_swiglu", "gemm_down", "combine"}
    assert j["same_y"] is True
    torch.cuda.synchronize()


def test_dense_stage(capsys):
    """The dense gate/up comparison runs both tile shapes and the library GEMM
    of torch and reports a time for each."""
    j = _run(capsys, ["--stage", "dense", "--workload", "tiny", "--rows", "256", "--steps", "3",
                      "--warmup", "1", "--no-clocks"])
    assert j["stage"] == "dense" and j["shape"] == {"rows": 256, "d": 64, "two_M": 256}
    assert set(j["gate_up_ms"]) == {"single_cta", "cta_pair", "cublas"}
    assert all(t > 0.0 for t in j["gate_up_ms"].values())
    torch.cuda.synchronize()

"""Host-side pieces of the benchmark: the algorithmic work that the roofline
and the stage bandwidths divide by, checked against the totals of the layer's
FLOP formula (6 R d M routed + 6 T d Ms shared) written out per workload, and
the argument defaults the timing rules require.  CPU only."""
import pytest

import bench
import synth


@pytest.mark.parametrize("name,tflop", [
    ("mixtral", 2.886),          # 6 * 8192 * 4096 * 14336
    ("deepseekmoe16b", 1.134),   # 6 * 49152 * 2048 * 1408 + 6 * 8192 * 2048 * 2816
    ("deepseekv2", 3.092),       # 6 * 49152 * 5120 * 1536 + 6 * 8192 * 5120 * 3072
])
def test_ffn_flops_match_the_layer_totals(name, tflop):
    w = synth.WORKLOADS[name]
    R = w.T * w.k  # dropless: every pair is a row
    flops, _ = bench.algorithmic_work(w, R)
    total = flops["gemm_swiglu"] + flops["gemm_down"]
    assert total / 1e12 == pytest.approx(tflop, abs=5e-4)
    # the gate/up projection carries two thirds of it
    assert flops["gemm_swiglu"] == pytest.approx(2 * flops["gemm_down"], rel=1e-12)


def test_memory_stage_bytes():
    w = synth.WORKLOADS["mixtral"]
    R = w.T * w.k
    _, b = bench.algorithmic_work(w, R)
    x = w.T * w.d * 2
    assert b["router"] == x + w.E * w.d * 2 + w.T * w.k * 8
    assert b["scatter"] == x + R * w.d * 2 + w.T * w.k * 5 + R * 4
    assert b["combine"] == R * w.d * 2 + x + w.T * w.k * 8   # no shared experts


def test_attainable_bound_is_at_least_the_flop_and_byte_floors():
    w = synth.WORKLOADS["deepseekv2"]
    peaks = dict(bench.FALLBACK_PEAKS)
    kept = [300] * w.E
    t = bench.attainable_ffn_ms(w, kept, peaks)
    flops = 6.0 * (sum(kept) * w.d * w.M + w.T * w.d * w.Ms)
    weights = 3 * w.d * 2 * (w.E * w.M + w.Ms)
    assert t >= 1000 * flops / (peaks["bf16_tflops"] * 1e12) * (1 - 1e-12)
    assert t >= 1000 * weights / (peaks["hbm_gbs"] * 1e9) * (1 - 1e-12)


def test_defaults_follow_the_timing_rules():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.warmup >= 3 and a.steps >= 1
    assert bench.FLUSH_BYTES > 126 * 2**20    # larger than the L2


def test_ab_stage_arguments():
    """`--stage ab` takes the tuning of each layer as field=value pairs; the
    fields are moe_tuning_t's and unknown ones fail when the shape is built."""
    import top_routing_expert_lb_b300 as moe
    args = bench.parse_args(["--stage", "ab", "--tune", "n_block=8", "--tune", "block_min_rows=2048",
                             "--tune-b", "gemm1_tile=256"])
    assert args.stage == "ab"
    a, b = bench.parse_tune(args.tune), bench.parse_tune(args.tune_b)
    assert a == {"n_block": 8, "block_min_rows": 2048} and b == {"gemm1_tile": 256}
    s = moe.Shape.of(64, 64, 128, 8, 2, **a)
    assert s.tuning.n_block == 8 and s.tuning.block_min_rows == 2048
    with pytest.raises(TypeError):
        moe.Shape.of(64, 64, 128, 8, 2, no_such_field=1)
    with pytest.raises(TypeError):
        s.tuned(gemm_tile=128)


def test_dense_stage_arguments():
    """`--stage dense` takes the expert's row count; it defaults to 8192."""
    assert bench.parse_args(["--stage", "dense"]).rows == 8192
    args = bench.parse_args(["--stage", "dense", "--rows", "1024", "--workload", "mixtral"])
    assert args.stage == "dense" and args.rows == 1024

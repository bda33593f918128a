"""GPU parity of the whole layer (moe_layer_forward through the C ABI) against
the oracle, on seeded inputs: small cases that span several 128-token tiles
with ragged tails, the degenerate cases of the method, and the tiny workload."""
import numpy as np
import pytest
import torch

import synth
import top_routing_expert_lb_b300 as moe
from parity import check_layer, guard_layer, run_layer, shape_of, np_of
from top_routing_expert_lb_b300 import build as mbuild

pytestmark = pytest.mark.gpu

W = synth.Workload
CASES = {
    "tiny": synth.WORKLOADS["tiny"],
    "ragged_shared": W("ragged_shared", T=300, d=256, E=8, k=2, M=256, n_shared=1,
                       offsets="normal"),
    "capacity_k4": W("capacity_k4", T=517, d=192, E=16, k=4, M=128, capacity_factor=0.9,
                     offsets="normal"),
    "fine_bias_shared": W("fine_bias_shared", T=389, d=128, E=64, k=6, M=128, n_shared=2,
                          offsets="normal", sel_bias="uniform", bias_range=0.02),
    "top1_capacity": W("top1_capacity", T=1000, d=64, E=32, k=1, M=128,
                       capacity_factor=1.25, offsets="normal"),
    "wide_E160": W("wide_E160", T=260, d=320, E=160, k=6, M=256, sel_bias="uniform",
                   bias_range=0.005),
    "E1_k1_dense": W("E1_k1_dense", T=150, d=128, E=1, k=1, M=128),
    "k_equals_E": W("k_equals_E", T=140, d=64, E=4, k=4, M=128),
    "k0_shared_only": W("k0_shared_only", T=130, d=128, E=8, k=0, M=128, n_shared=1),
    "k0_no_experts": W("k0_no_experts", T=70, d=64, E=8, k=0, M=128),
    "single_token": W("single_token", T=1, d=64, E=8, k=2, M=128, n_shared=1),
    "E256_k8": W("E256_k8", T=200, d=64, E=256, k=8, M=128, offsets="normal"),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mbuild.ensure_built()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("name", list(CASES))
def test_layer_parity(name):
    inp = synth.make_inputs(CASES[name], "cuda")
    g, ref = check_layer(inp)
    if name == "k0_no_experts":
        assert torch.count_nonzero(g.y) == 0
    if CASES[name].capacity_factor > 0:
        assert ref.disp.dropped.any(), "capacity case should drop pairs"


@pytest.mark.parametrize("dynamic", ["0", "1"])
@pytest.mark.parametrize("name", ["ragged_shared", "capacity_k4", "fine_bias_shared",
                                  "k0_shared_only", "E1_k1_dense", "wide_E160"])
def test_layer_parity_paired_tiles(name, dynamic):
    """The same cases with the expert GEMMs forced onto 256-row CTA-pair tiles,
    in the static and in the dynamic (tile counter) order."""
    inp = synth.make_inputs(CASES[name], "cuda")
    tune = dict(gemm1_tile=256, tile_order=2 if dynamic == "1" else 1)
    if CASES[name].d % 256 == 0:
        tune["gemm2_tile"] = 256
    g, ref = check_layer(inp, tuning=tune)
    if name == "k0_no_experts":
        assert torch.count_nonzero(g.y) == 0
    if CASES[name].capacity_factor > 0:
        assert ref.disp.dropped.any(), "capacity case should drop pairs"


@pytest.mark.parametrize("name", ["ragged_shared", "capacity_k4", "fine_bias_shared",
                                  "top1_capacity", "wide_E160", "single_token"])
def test_layer_parity_fused_gather(name):
    """The same cases with GEMM-1 gathering the token rows itself (TMA 4-row
    gathers by row_token) instead of reading the scatter's x_perm."""
    check_layer(synth.make_inputs(CASES[name], "cuda"),
                tuning=dict(options=moe.MOE_TUNE_FUSED_GATHER))


@pytest.mark.parametrize("name", ["ragged_shared", "capacity_k4", "fine_bias_shared",
                                  "top1_capacity", "E1_k1_dense", "k_equals_E"])
def test_layer_parity_split_gate_up(name):
    """The same cases with the gate/up projection split into CTA-pair tiles for
    whole 256-row blocks and single-CTA tiles for the rest."""
    check_layer(synth.make_inputs(CASES[name], "cuda"),
                tuning=dict(options=moe.MOE_TUNE_GEMM1_SPLIT))


@pytest.mark.parametrize("name,tile2", [("ragged_shared", "128"), ("ragged_shared", "256"),
                                        ("capacity_k4", "128"), ("fine_bias_shared", "128"),
                                        ("wide_E160", "128"), ("k_equals_E", "128"),
                                        ("single_token", "128"), ("top1_capacity", "128")])
def test_layer_parity_gate_in_epilogue(name, tile2):
    """The same cases with each routed row scaled by its gate in the down
    projection's epilogue and a combine that only adds rows."""
    check_layer(synth.make_inputs(CASES[name], "cuda"),
                tuning=dict(options=moe.MOE_TUNE_GATE_IN_EPILOGUE, gemm2_tile=int(tile2)))


@pytest.mark.parametrize("name", ["ragged_shared", "capacity_k4", "fine_bias_shared", "wide_E160"])
def test_two_ctas_per_sm_gives_the_same_bits(name):
    """The single-CTA GEMMs run two CTAs per SM (MOE_TUNE_TWO_CTAS_PER_SM): the
    oracle's results, and the bits of the default launch (the same tiles, run
    by other CTAs)."""
    inp = synth.make_inputs(CASES[name], "cuda")
    g, _ = check_layer(inp, tuning=dict(options=moe.MOE_TUNE_TWO_CTAS_PER_SM))
    plain = run_layer(inp)
    assert torch.equal(g.y.view(torch.int16), plain.y.view(torch.int16))


def test_fused_and_materialised_rows_agree_bitwise():
    """Gathering the rows inside GEMM-1 stages the same bytes as the scatter's
    copy, so the two paths give bit-identical outputs."""
    w = CASES["fine_bias_shared"]
    inp = synth.make_inputs(w, "cuda")
    outs = []
    for opts in (moe.MOE_TUNE_FUSED_GATHER, 0):
        outs.append(run_layer(inp, tuning=dict(options=opts)).y)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_one_expert_takes_every_row():
    w = W("hot", T=333, d=128, E=8, k=1, M=128, n_shared=0)
    inp = synth.make_inputs(w, "cuda")
    off = torch.zeros(8, dtype=torch.float32)
    off[5] = 30.0
    inp.offset = off.cuda()
    g, ref = check_layer(inp)
    assert g.counts.tolist() == [0, 0, 0, 0, 0, 333, 0, 0]


def test_capacity_drops_all_but_first_tokens():
    # a single hot expert with capacity C = ceil(0.25 * 1 * 260 / 4) = 17:
    # only its first 17 tokens (token order) are kept, all others output 0
    w = W("cap_hot", T=260, d=64, E=4, k=1, M=128, capacity_factor=0.25)
    inp = synth.make_inputs(w, "cuda")
    off = torch.tensor([0.0, 40.0, 0.0, 0.0], dtype=torch.float32)
    inp.offset = off.cuda()
    g, ref = check_layer(inp)
    assert ref.C == 17
    assert g.drop[:17].sum() == 0 and g.drop[17:].all()
    assert torch.count_nonzero(g.y[17:]) == 0


def test_empty_batch():
    w = W("empty", T=0, d=64, E=8, k=2, M=128)
    s = shape_of(w)
    dev = "cuda"
    ws = moe._binding.alloc_workspace(s, dev)
    wr = torch.zeros((8, 64), dtype=torch.bfloat16, device=dev)
    counts = torch.full((8,), 7, dtype=torch.int32, device=dev)
    f = torch.full((8,), 7.0, device=dev)
    P = torch.full((8,), 7.0, device=dev)
    lb = torch.full((1,), 7.0, device=dev)
    lz = torch.full((1,), 7.0, device=dev)
    moe.moe_layer_forward(s, None, wr, None, None, None, None, None, None, None, None, None,
                          counts, None, f, P, lb, lz, ws)
    torch.cuda.synchronize()
    assert counts.sum().item() == 0 and f.abs().sum().item() == 0 and P.abs().sum().item() == 0
    assert lb.item() == 0.0 and lz.item() == 0.0


def test_deterministic_bitwise():
    w = CASES["capacity_k4"]
    inp = synth.make_inputs(w, "cuda")
    layer = moe.MoELayer(shape_of(w), inp.wr, inp.w1, inp.w3, inp.w2, inp.ws1, inp.ws3,
                         inp.ws2, inp.offset, inp.sel_bias)
    a = run_layer(inp, layer)
    b = run_layer(inp, layer)
    assert torch.equal(a.y.view(torch.int16), b.y.view(torch.int16))
    for fld in ("ids", "gates", "counts", "drop", "f", "P"):
        np.testing.assert_array_equal(getattr(a, fld), getattr(b, fld))
    assert a.bal == b.bal and a.z == b.z


def test_host_io_entry_matches_device_entry():
    w = CASES["ragged_shared"]
    inp = synth.make_inputs(w, "cuda")
    layer = moe.MoELayer(shape_of(w), inp.wr, inp.w1, inp.w3, inp.w2, inp.ws1, inp.ws3,
                         inp.ws2, inp.offset, inp.sel_bias)
    dev_out = run_layer(inp, layer)
    x_host = inp.x.cpu().pin_memory()
    y_host = torch.empty_like(x_host).pin_memory()
    losses = torch.empty(2, dtype=torch.float32).pin_memory()
    x_dev = torch.empty_like(inp.x)
    y_dev = torch.empty_like(inp.x)
    moe.moe_layer_forward_host(layer.shape, x_host, x_dev, layer.w_router, layer.logit_offset,
                               layer.sel_bias, layer.w13, layer.w2, layer.w13_shared,
                               layer.w2_shared, y_dev, y_host, losses, layer.ids, layer.gates,
                               layer.counts, layer.drop_mask, layer.f, layer.P,
                               layer.losses[0:1], layer.losses[1:2], layer.ws)
    assert torch.equal(y_host.view(torch.int16), dev_out.y.cpu().view(torch.int16))
    assert losses[0].item() == dev_out.bal and losses[1].item() == dev_out.z


@pytest.mark.parametrize("n_batches,same_stream", [(5, False), (1, False), (3, True)])
def test_host_batches_stream_matches_per_batch_calls(n_batches, same_stream):
    """The double-buffered host stream (copy-in, layer and copy-out on three
    streams) gives, batch for batch, the bits of separate layer calls."""
    w = CASES["ragged_shared"]
    inp = synth.make_inputs(w, "cuda")
    layer = moe.MoELayer(shape_of(w), inp.wr, inp.w1, inp.w3, inp.w2, inp.ws1, inp.ws3,
                         inp.ws2, inp.offset, inp.sel_bias)
    xs = [synth.make_inputs(w.replace(seed=w.seed + 100 + i), "cuda").x for i in range(n_batches)]
    expect = []
    for x in xs:
        layer.forward(x)
        torch.cuda.synchronize()
        expect.append((layer.y.cpu().clone(), layer.losses.cpu().clone()))
    x_host = torch.stack([x.cpu() for x in xs]).pin_memory()
    y_host = torch.zeros_like(x_host).pin_memory()
    losses = torch.zeros(n_batches, 2, dtype=torch.float32).pin_memory()
    x_dev = torch.empty((2,) + tuple(inp.x.shape), dtype=inp.x.dtype, device="cuda")
    y_dev = torch.empty_like(x_dev)
    loss_dev = torch.empty(2, 2, dtype=torch.float32, device="cuda")
    main = torch.cuda.current_stream()
    h2d = main if same_stream else torch.cuda.Stream()
    d2h = main if same_stream else torch.cuda.Stream()
    moe.moe_layer_forward_host_batches(
        layer.shape, x_host, y_host, losses, x_dev, y_dev, loss_dev, layer.w_router,
        layer.logit_offset, layer.sel_bias, layer.w13, layer.w2, layer.w13_shared,
        layer.w2_shared, layer.ids, layer.gates, layer.counts, layer.drop_mask, layer.f,
        layer.P, layer.ws, main, h2d, d2h)
    for i, (y, l) in enumerate(expect):
        assert torch.equal(y_host[i].view(torch.int16), y.view(torch.int16)), i
        assert torch.equal(losses[i], l), i
    # the device outputs hold the last batch's routing
    ref_last = run_layer(synth.make_inputs(w.replace(seed=w.seed + 100 + n_batches - 1), "cuda"),
                         layer)
    assert torch.equal(y_host[-1].view(torch.int16), ref_last.y.cpu().view(torch.int16))


def test_bounded_wait_reports_timeout():
    s = shape_of(CASES["tiny"])
    ws = moe._binding.alloc_workspace(s)
    try:
        moe.moe_set_wait_timeout_ns(1_000_000)          # 1 ms
        moe.moe_debug_timeout_probe(ws)
        assert moe.moe_check_status(ws) == moe._binding.MOE_ERR_TIMEOUT
        assert moe.moe_check_status(ws) == 0             # read clears it
    finally:
        moe.moe_set_wait_timeout_ns(2_000_000_000)
    # the context is still usable afterwards
    inp = synth.make_inputs(CASES["tiny"], "cuda")
    check_layer(inp)


def test_cuda_graph_capture_and_replay():
    """The whole layer forward is stream-ordered work with no host
    synchronisation, so it can be captured once into a CUDA graph and replayed;
    replays give the same bits as direct calls and pass parity."""
    w = CASES["fine_bias_shared"]
    inp = synth.make_inputs(w, "cuda")
    layer = moe.MoELayer(shape_of(w), inp.wr, inp.w1, inp.w3, inp.w2, inp.ws1, inp.ws3,
                         inp.ws2, inp.offset, inp.sel_bias, device="cuda")
    layer.forward(inp.x)                      # first call sets kernel attributes
    torch.cuda.synchronize()
    direct = layer.y.clone()
    x_static = inp.x.clone()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            layer.forward(x_static)
    torch.cuda.current_stream().wait_stream(side)
    layer.y.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert moe.moe_check_status(layer.ws) == 0
    assert torch.equal(layer.y.view(torch.int16), direct.view(torch.int16))
    check_layer(inp, layer=None)


@pytest.mark.parametrize("name", ["ragged_shared", "capacity_k4", "wide_E160"])
def test_programmatic_dependent_launch_gives_the_same_bits(name):
    """Each kernel of the layer may start while the one before it finishes
    (the default) or only after it (MOE_TUNE_NO_PDL): the same bits either way,
    also when calls follow each other on the stream with no host sync between."""
    inp = synth.make_inputs(CASES[name], "cuda")
    layer = guard_layer(moe.MoELayer(shape_of(inp.w), inp.wr, inp.w1, inp.w3, inp.w2, inp.ws1,
                                     inp.ws3, inp.ws2, inp.offset, inp.sel_bias,
                                     device=inp.x.device))
    g, _ = check_layer(inp, layer=layer)
    serial = run_layer(inp, tuning=dict(options=moe.MOE_TUNE_NO_PDL))
    assert torch.equal(g.y.view(torch.int16), serial.y.view(torch.int16))
    for _ in range(5):
        layer.forward(inp.x)
    torch.cuda.synchronize()
    assert torch.equal(layer.y.view(torch.int16), serial.y.view(torch.int16))
    assert np.array_equal(np_of(layer.ids), serial.ids)
    assert moe.moe_check_status(layer.ws) == 0

"""moe_route_noalloc is the router for callers that cannot allocate device
memory: code running under a host framework that owns all device memory
through its own pool, plug-ins loaded into such a process, or paths where an
allocation (and the synchronisation it may bring) is not allowed.  It takes no
workspace; its scratch is a static device array inside the library.

Checked here, through the C ABI: on consecutive calls of different shapes it
gives the same results as moe_route (the workspace entry point) and the
oracle's routing; it handles the largest shape its array allows and T = 0; it
changes neither the device memory in use nor torch's allocations; shapes
beyond its array are refused.  This file is collected last, so that a run
stopping at the first failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import synth
import top_routing_expert_lb_b300 as moe
from parity import GATE_ABS, LOSS_REL, assert_routing_parity, np_of, oracle_routing, shape_of, \
    GpuOut
from top_routing_expert_lb_b300 import _binding as B
from top_routing_expert_lb_b300 import build as mbuild

pytestmark = pytest.mark.gpu
W = synth.Workload


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mbuild.ensure_built()
    assert torch.cuda.is_available()


def _outs(w, dev="cuda"):
    return dict(ids=torch.full((max(w.T, 1), max(w.k, 1)), -5, dtype=torch.int32, device=dev),
                gates=torch.full((max(w.T, 1), max(w.k, 1)), -5.0, device=dev),
                counts=torch.full((w.E,), -5, dtype=torch.int32, device=dev),
                f=torch.full((w.E,), -5.0, device=dev), P=torch.full((w.E,), -5.0, device=dev),
                lb=torch.full((1,), -5.0, device=dev), lz=torch.full((1,), -5.0, device=dev))


def _noalloc(s, inp, o):
    moe.moe_route_noalloc(s, inp.x, inp.wr, inp.offset, inp.sel_bias, o["ids"], o["gates"],
                          o["counts"], o["f"], o["P"], o["lb"], o["lz"])


def _route_both(w):
    inp = synth.make_inputs(w, "cuda", experts=False)
    s = shape_of(w)
    ref, got = _outs(w), _outs(w)
    ws = B.alloc_workspace(s)
    moe.moe_route(s, inp.x, inp.wr, inp.offset, inp.sel_bias, ref["ids"], ref["gates"],
                  ref["counts"], ref["f"], ref["P"], ref["lb"], ref["lz"], ws)
    _noalloc(s, inp, got)
    torch.cuda.synchronize()
    return inp, ref, got


def _assert_same(ref, got):
    assert torch.equal(ref["ids"], got["ids"])
    assert torch.equal(ref["counts"], got["counts"])
    assert (ref["gates"] - got["gates"]).abs().max().item() <= GATE_ABS
    torch.testing.assert_close(got["f"], ref["f"], rtol=1e-6, atol=0)
    torch.testing.assert_close(got["P"], ref["P"], rtol=LOSS_REL, atol=1e-7)
    for key in ("lb", "lz"):
        a, b = got[key].item(), ref[key].item()
        assert abs(a - b) <= LOSS_REL * max(abs(b), 1e-30), (key, a, b)


def _assert_oracle(inp, got):
    """The no-allocation router's outputs against the oracle (dropless: the
    drop mask is all zeros), with the near-tie protocol of the other tests."""
    w = inp.w
    g = GpuOut(None, np_of(got["ids"]), np_of(got["gates"]), np_of(got["counts"]),
               np.zeros((w.T, w.k), np.uint8), np_of(got["f"]), np_of(got["P"]),
               got["lb"].item(), got["lz"].item())
    assert_routing_parity(g, oracle_routing(inp, g.ids), w)


def test_noalloc_router_matches_workspace_router_and_oracle_on_consecutive_calls():
    shapes = [
        W("na_bias", T=700, d=1024, E=160, k=6, M=128, offsets="normal", sel_bias="uniform"),
        W("na_small", T=129, d=256, E=8, k=2, M=128),
        W("na_top1", T=3000, d=512, E=64, k=1, M=128, offsets="normal"),
    ]
    for w in shapes:           # consecutive calls reuse the same static scratch
        inp, ref, got = _route_both(w)
        _assert_same(ref, got)
        _assert_oracle(inp, got)
    inp, ref, got = _route_both(shapes[0])  # and back to the first shape
    _assert_same(ref, got)
    _assert_oracle(inp, got)


def test_noalloc_router_at_its_size_limit():
    """T = 65536 tokens and E = 256 experts fill every per-tile and per-expert
    region of the static array."""
    w = W("na_limit", T=65536, d=64, E=256, k=8, M=128, offsets="normal")
    inp, ref, got = _route_both(w)
    _assert_same(ref, got)
    _assert_oracle(inp, got)


def test_noalloc_router_with_no_tokens():
    """T = 0: no router launch, only the reduction, which writes zero counts,
    f, P and losses."""
    w = W("na_empty", T=0, d=128, E=16, k=2, M=128)
    inp = synth.make_inputs(w, "cuda", experts=False)
    got = _outs(w)
    _noalloc(shape_of(w), inp, got)
    torch.cuda.synchronize()
    assert got["counts"].tolist() == [0] * w.E
    assert got["f"].abs().max().item() == 0.0 and got["P"].abs().max().item() == 0.0
    assert got["lb"].item() == 0.0 and got["lz"].item() == 0.0


def test_noalloc_router_allocates_nothing():
    """After a first call on the device (which may load the library's kernels
    and its static array), further calls leave the device's free memory and
    torch's allocations unchanged."""
    w = W("na_mem", T=1000, d=256, E=32, k=4, M=128, offsets="normal")
    inp = synth.make_inputs(w, "cuda", experts=False)
    s = shape_of(w)
    got = _outs(w)
    _noalloc(s, inp, got)
    torch.cuda.synchronize()
    torch_before = torch.cuda.memory_allocated()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        _noalloc(s, inp, got)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == torch_before
    assert free_after == free_before
    _assert_oracle(inp, got)


def test_noalloc_router_rejects_shapes_beyond_its_scratch():
    s = moe.Shape.of(65537, 64, 128, 8, 2)          # one token past the maximum
    dummy = torch.empty(16, dtype=torch.float32, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    rc = B.lib().moe_route_noalloc(ctypes.byref(s), p, p, None, None, p, p, p, p, p, p, p, None)
    assert rc == B.MOE_ERR_UNSUPPORTED

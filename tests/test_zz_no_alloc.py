"""moe_route_noalloc — the router entry point for callers that cannot allocate
device memory (no workspace; the library's static device scratch is used) —
must give the same results as moe_route, the workspace entry point, on
consecutive calls of different shapes.  This file is collected last so that a
run stopping at the first failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import synth
import top_routing_expert_lb_b300 as moe
from parity import GATE_ABS, LOSS_REL, shape_of
from top_routing_expert_lb_b300 import _binding as B
from top_routing_expert_lb_b300 import build as mbuild

pytestmark = pytest.mark.gpu
W = synth.Workload


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mbuild.ensure_built()
    assert torch.cuda.is_available()


def _outs(w, dev="cuda"):
    return dict(ids=torch.full((w.T, w.k), -5, dtype=torch.int32, device=dev),
                gates=torch.full((w.T, w.k), -5.0, device=dev),
                counts=torch.full((w.E,), -5, dtype=torch.int32, device=dev),
                f=torch.full((w.E,), -5.0, device=dev), P=torch.full((w.E,), -5.0, device=dev),
                lb=torch.full((1,), -5.0, device=dev), lz=torch.full((1,), -5.0, device=dev))


def _route_both(w):
    inp = synth.make_inputs(w, "cuda", experts=False)
    s = shape_of(w)
    ref, got = _outs(w), _outs(w)
    ws = B.alloc_workspace(s)
    moe.moe_route(s, inp.x, inp.wr, inp.offset, inp.sel_bias, ref["ids"], ref["gates"],
                  ref["counts"], ref["f"], ref["P"], ref["lb"], ref["lz"], ws)
    moe.moe_route_noalloc(s, inp.x, inp.wr, inp.offset, inp.sel_bias, got["ids"], got["gates"],
                          got["counts"], got["f"], got["P"], got["lb"], got["lz"])
    torch.cuda.synchronize()
    return ref, got


def _assert_same(ref, got):
    assert torch.equal(ref["ids"], got["ids"])
    assert torch.equal(ref["counts"], got["counts"])
    assert (ref["gates"] - got["gates"]).abs().max().item() <= GATE_ABS
    torch.testing.assert_close(got["f"], ref["f"], rtol=1e-6, atol=0)
    torch.testing.assert_close(got["P"], ref["P"], rtol=LOSS_REL, atol=1e-7)
    for key in ("lb", "lz"):
        a, b = got[key].item(), ref[key].item()
        assert abs(a - b) <= LOSS_REL * max(abs(b), 1e-30), (key, a, b)


def test_noalloc_router_matches_workspace_router_on_consecutive_calls():
    shapes = [
        W("na_bias", T=700, d=1024, E=160, k=6, M=128, offsets="normal", sel_bias="uniform"),
        W("na_small", T=129, d=256, E=8, k=2, M=128),
        W("na_top1", T=3000, d=512, E=64, k=1, M=128, offsets="normal"),
    ]
    for w in shapes:           # consecutive calls reuse the same static scratch
        ref, got = _route_both(w)
        _assert_same(ref, got)
    ref, got = _route_both(shapes[0])  # and back to the first shape
    _assert_same(ref, got)


def test_noalloc_router_rejects_shapes_beyond_its_scratch():
    s = moe.Shape.of(65537, 64, 128, 8, 2)          # one token past the maximum
    dummy = torch.empty(16, dtype=torch.float32, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    rc = B.lib().moe_route_noalloc(ctypes.byref(s), p, p, None, None, p, p, p, p, p, p, p, None)
    assert rc == B.MOE_ERR_UNSUPPORTED

"""GPU parity of the routing variants (sigmoid scores, un-renormalised gates)
and of the optional router side outputs (importance and its CV^2, mean router
entropy) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
import top_routing_expert_lb_b300 as moe
from guard import guarded
from parity import GATE_ABS, LOSS_REL, check_layer, guarded_workspace, np_of, oracle_routing, rel_close, \
    shape_of
from top_routing_expert_lb_b300 import build as mbuild

pytestmark = pytest.mark.gpu
W = synth.Workload
SIG, NOR = moe.MOE_FLAG_SIGMOID, moe.MOE_FLAG_NO_RENORM


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mbuild.ensure_built()
    assert torch.cuda.is_available()


ROUTE_CASES = [
    W("v_soft", T=300, d=256, E=16, k=4, M=128, offsets="normal"),
    W("v_sig", T=300, d=256, E=16, k=4, M=128, offsets="normal", flags=SIG),
    W("v_noren", T=517, d=192, E=64, k=6, M=128, offsets="normal", sel_bias="uniform",
      bias_range=0.01, flags=NOR),
    W("v_sig_noren", T=1000, d=512, E=160, k=6, M=128, flags=SIG | NOR),
    W("v_sig_split", T=256, d=2048, E=8, k=2, M=128, flags=SIG),      # cluster split-K path
    W("v_top1_many", T=4097, d=128, E=128, k=1, M=128, offsets="normal"),
]


@pytest.mark.parametrize("w", ROUTE_CASES, ids=lambda w: w.name)
def test_route_ex_variants_and_side_outputs(w):
    inp = synth.make_inputs(w, "cuda", experts=False)
    s = shape_of(w)
    dev = "cuda"
    out = dict(ids=guarded((w.T, w.k), torch.int32, dev, label="ids"),
               gates=guarded((w.T, w.k), torch.float32, dev, label="gates"),
               counts=guarded(w.E, torch.int32, dev, label="counts"),
               f=guarded(w.E, torch.float32, dev, label="f"),
               P=guarded(w.E, torch.float32, dev, label="P"),
               bal_loss=guarded(1, torch.float32, dev, label="bal_loss"),
               z_loss=guarded(1, torch.float32, dev, label="z_loss"),
               importance=guarded(w.E, torch.float32, dev, label="importance"),
               importance_cv2=guarded(1, torch.float32, dev, label="importance_cv2"),
               entropy_mean=guarded(1, torch.float32, dev, label="entropy_mean"))
    ws = guarded_workspace(s)
    moe.moe_route_ex(s, inp.x, inp.wr, inp.offset, inp.sel_bias, ws, **out)
    torch.cuda.synchronize()
    assert moe.moe_check_status(ws) == 0
    ref = oracle_routing(inp, np_of(out["ids"]))
    np.testing.assert_array_equal(np_of(out["ids"]), ref.routing.ids)
    assert np.abs(np_of(out["gates"]) - ref.routing.gates).max() <= GATE_ABS
    np.testing.assert_array_equal(np_of(out["counts"]), ref.disp.counts)
    np.testing.assert_allclose(np_of(out["P"]), ref.loss.P, rtol=LOSS_REL, atol=1e-7)
    rel_close(out["bal_loss"].item(), ref.loss.L_bal, LOSS_REL, "balance loss")
    rel_close(out["z_loss"].item(), ref.loss.L_z, LOSS_REL, "z-loss")
    imp, cv2 = oracle.importance(ref.routing.ids, ref.routing.gates, w.E)
    np.testing.assert_allclose(np_of(out["importance"]), imp, rtol=LOSS_REL, atol=1e-4)
    rel_close(out["importance_cv2"].item(), cv2, 1e-3, "importance CV^2")
    rel_close(out["entropy_mean"].item(), float(ref.routing.entropy.mean()), LOSS_REL,
              "mean router entropy")


@pytest.mark.parametrize("flags", [SIG, NOR, SIG | NOR])
def test_layer_variants(flags):
    w = W("lv", T=389, d=128, E=16, k=4, M=256, n_shared=1, offsets="normal",
          capacity_factor=1.0, flags=flags)
    g, ref = check_layer(synth.make_inputs(w, "cuda"))
    if flags & NOR:
        # un-renormalised gates sum to the selected scores' mass, not to 1
        assert not np.allclose(ref.routing.gates.sum(1), 1.0)

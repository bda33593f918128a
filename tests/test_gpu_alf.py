"""ALF-LB bias update on the GPU: each step's update equals the oracle's from
the same counts bit for bit, and a multi-step run over seeded token batches
reduces the load imbalance of the GPU router."""
import numpy as np
import pytest
import torch

import oracle
import synth
import top_routing_expert_lb_b300 as moe
from parity import np_of, oracle_routing, shape_of
from top_routing_expert_lb_b300 import build as mbuild

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mbuild.ensure_built()
    assert torch.cuda.is_available()


def test_alf_bias_update_balances_load_over_steps():
    w = synth.Workload("alf", T=2048, d=256, E=32, k=4, M=128, offsets="normal", w_std=0.05)
    s = shape_of(w)
    dev = "cuda"
    wr = synth.normal_bf16(w.seed, synth.TID_WR, (w.E, w.d), w.w_std, dev)
    off = synth.make_offsets(w, dev)                  # skewed loads (CV of counts ~1.8)
    bias = torch.zeros(w.E, dtype=torch.float32, device=dev)
    ws = moe.alloc_workspace(s)
    ids = torch.empty((w.T, w.k), dtype=torch.int32, device=dev)
    gates = torch.empty((w.T, w.k), device=dev)
    counts = torch.empty(w.E, dtype=torch.int32, device=dev)
    f, P = torch.empty(w.E, device=dev), torch.empty(w.E, device=dev)
    lb, lz = torch.empty(1, device=dev), torch.empty(1, device=dev)
    cvs = []
    for step in range(100):
        x = synth.normal_bf16(1000 + step, synth.TID_X, (w.T, w.d), 1.0, dev)
        moe.moe_route(s, x, wr, off, bias, ids, gates, counts, f, P, lb, lz, ws)
        before = np_of(bias).copy()
        moe.moe_alf_bias_update(s, counts, 0.002, bias)
        torch.cuda.synchronize()
        n = np_of(counts)
        want = oracle.alf_bias_update(n, w.T, w.k, 0.002, before)
        np.testing.assert_array_equal(np_of(bias), want)
        cvs.append(n.std() / n.mean())
        if step in (0, 99):     # the routing with the current bias matches the oracle
            inp = synth.Inputs(w.replace(sel_bias="given"), x, wr, None, None, None,
                               offset=off, sel_bias=torch.from_numpy(before).to(dev))
            oracle_routing(inp, np_of(ids))
    assert moe.moe_check_status(ws) == 0
    # coefficient of variation of the loads: ~1.8 at the start, a few tenths after
    assert cvs[0] > 1.0 and np.mean(cvs[-10:]) < 0.25 * cvs[0], cvs[::10]

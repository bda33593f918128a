"""Full-size parity: every workload at its full size, run exactly as the
benchmark runs it (moe_layer_forward through the C ABI), checked against the
oracle on everything: routing, counts, drop masks, f, P and both losses, and
the layer output of every token (about three minutes of oracle work on the
host cores for all five workloads)."""
import numpy as np
import pytest
import torch

import synth
from parity import assert_routing_parity, assert_y_close, bf16_to_f64, np_of, oracle_routing, \
    oracle_y, run_layer
from top_routing_expert_lb_b300 import build as mbuild

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mbuild.ensure_built()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("name", ["tiny", "mixtral", "deepseekmoe16b", "deepseekv2", "switch"])
def test_full_size(name):
    w = synth.WORKLOADS[name]
    inp = synth.make_inputs(w, "cuda")
    g = run_layer(inp)
    ref = oracle_routing(inp, g.ids)
    assert_routing_parity(g, ref, w)
    if w.k and ref.disp.dropped.any() and w.n_shared == 0:
        # a token with every pair dropped and no shared expert outputs exact zeros
        all_dropped = np.nonzero(ref.disp.dropped.all(axis=1))[0]
        assert torch.count_nonzero(g.y[torch.from_numpy(all_dropped).cuda()]) == 0
    # every token, in chunks (each chunk's tolerance is checked on its own, which
    # is stricter than one check over the whole output for the max-abs bound)
    y_gpu = bf16_to_f64(g.y)
    host_w = (np_of(inp.w1), np_of(inp.w3), np_of(inp.w2))
    chunk = 1024
    for t0 in range(0, w.T, chunk):
        sel = np.arange(t0, min(w.T, t0 + chunk), dtype=np.int32)
        y_ref = oracle_y(inp, ref, sel, host_w)
        assert_y_close(y_gpu[sel], y_ref, f"{name} y[{t0}:{t0 + len(sel)}]")
    n = ref.disp.counts
    print(f"{name}: max/mean load {n.max() / max(n.mean(), 1e-9):.2f}, empty experts "
          f"{int((n == 0).sum())}, dropped pairs {int(ref.disp.dropped.sum())}, "
          f"near-tie or reordered tokens {int(ref.exempt.sum())}")

"""Full-size parity: every workload at its full size, run exactly as the
benchmark runs it (moe_layer_forward through the C ABI), checked against the
oracle on everything the oracle can afford: routing, counts, drop masks, f, P
and both losses for every token, and the layer output for a seeded sample of
tokens (plus the first and last token, and every token whose pairs were all
dropped)."""
import numpy as np
import pytest
import torch

import synth
from parity import assert_routing_parity, assert_y_close, bf16_to_f64, oracle_routing, \
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
    rng = np.random.default_rng(1234)
    sel = set(rng.choice(w.T, size=min(w.T, 16), replace=False).tolist()) | {0, w.T - 1}
    if w.k and ref.disp.dropped.any():
        all_dropped = np.nonzero(ref.disp.dropped.all(axis=1))[0]
        sel |= set(all_dropped[:4].tolist())
        if w.n_shared == 0:
            # a token with every pair dropped and no shared expert outputs exact zeros
            assert torch.count_nonzero(g.y[torch.from_numpy(all_dropped).cuda()]) == 0
    sel = np.array(sorted(sel), dtype=np.int32)
    y_ref = oracle_y(inp, ref, sel)
    assert_y_close(bf16_to_f64(g.y)[sel], y_ref, f"{name} y (sampled)")
    # loads reported for the record
    n = ref.disp.counts
    print(f"{name}: max/mean load {n.max() / max(n.mean(), 1e-9):.2f}, empty experts "
          f"{int((n == 0).sum())}, dropped pairs {int(ref.disp.dropped.sum())}, "
          f"near-tie tokens {int(ref.exempt.sum())}")

"""Randomised GPU parity: seeded draws of small layer shapes and routing
variants (token choice with or without capacity, probability-priority
capacity, sigmoid scores, un-renormalised gates, shared experts, selection
bias, expert choice), each checked against the oracle on every token."""
import numpy as np
import pytest
import torch

import synth
import top_routing_expert_lb_b300 as moe
from parity import check_ec_layer, check_layer
from top_routing_expert_lb_b300 import build as mbuild

pytestmark = pytest.mark.gpu

SIG, NOR = moe.MOE_FLAG_SIGMOID, moe.MOE_FLAG_NO_RENORM
PRIO, EC = moe.MOE_FLAG_PRIORITY_CAPACITY, moe.MOE_FLAG_EXPERT_CHOICE


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mbuild.ensure_built()
    assert torch.cuda.is_available()


def draw(seed: int) -> synth.Workload:
    rng = np.random.default_rng(1000 + seed)
    E = int(rng.choice([1, 2, 5, 8, 16, 33, 64, 130]))
    k = int(rng.integers(0, min(E, 8) + 1))
    T = int(rng.choice([1, 7, 128, 129, 300, 511, 700]))
    d = int(rng.choice([64, 128, 192, 256, 320, 512]))
    M = int(rng.choice([128, 256, 384]))
    n_shared = int(rng.choice([0, 0, 1, 2]))
    mode = rng.choice(["dropless", "capacity", "priority", "expert_choice"])
    cap = 0.0
    flags = 0
    if mode == "capacity":
        cap = float(np.float32(rng.uniform(0.3, 2.0)))
    elif mode == "priority":
        cap = float(np.float32(rng.uniform(0.3, 1.5)))
        flags |= PRIO
    elif mode == "expert_choice":
        cap = float(np.float32(rng.choice([0.0, rng.uniform(0.3, 3.0)])))
        flags |= EC
    if rng.random() < 0.3:
        flags |= SIG
    if rng.random() < 0.3 and not flags & EC:
        flags |= NOR
    offsets = str(rng.choice(["none", "normal"]))
    sel_bias = "uniform" if (rng.random() < 0.3 and not flags & EC) else "none"
    return synth.Workload(f"rand{seed}", T=T, d=d, E=E, k=k, M=M, n_shared=n_shared,
                          capacity_factor=cap, offsets=offsets, sel_bias=sel_bias,
                          bias_range=0.02, flags=flags, seed=seed)


@pytest.mark.parametrize("seed", range(24))
def test_random_layer(seed):
    w = draw(seed)
    inp = synth.make_inputs(w, "cuda")
    if w.flags & EC:
        check_ec_layer(inp)
    else:
        check_layer(inp)

"""GPU parity of the score-ordered selections against the oracle:
probability-priority capacity (an over-full expert keeps its highest-score
pairs) and expert-choice routing (each expert takes its top-r tokens), both
through the C ABI, at small sizes that span several tiles with ragged tails,
with exact score ties (duplicated token rows), the degenerate cases (r = 0,
r = T, empty batch) and at full workload sizes with sampled outputs."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import (assert_routing_parity, assert_y_close, bf16_to_f64, check_ec_layer,
                    check_layer, oracle_routing, oracle_y, run_layer)
import top_routing_expert_lb_b300 as moe
from top_routing_expert_lb_b300 import build as mbuild

pytestmark = pytest.mark.gpu
W = synth.Workload
PRIO, EC, SIG = moe.MOE_FLAG_PRIORITY_CAPACITY, moe.MOE_FLAG_EXPERT_CHOICE, moe.MOE_FLAG_SIGMOID


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mbuild.ensure_built()
    assert torch.cuda.is_available()


def with_duplicate_rows(inp: synth.Inputs, distinct: int) -> synth.Inputs:
    """Token t takes the row of token t % distinct: equal scores everywhere, so
    every cut falls inside a group of exact ties."""
    idx = torch.arange(inp.w.T, device=inp.x.device) % distinct
    inp.x = inp.x[idx].contiguous()
    return inp


PRIO_CASES = [
    W("p_k2", T=1000, d=256, E=16, k=2, M=128, offsets="normal", capacity_factor=1.0,
      flags=PRIO),
    W("p_k1", T=2049, d=128, E=32, k=1, M=128, offsets="normal", capacity_factor=1.25,
      flags=PRIO),
    W("p_k6_shared", T=517, d=192, E=64, k=6, M=128, n_shared=1, offsets="normal",
      capacity_factor=0.6, sel_bias="uniform", bias_range=0.01, flags=PRIO),
    W("p_sigmoid", T=389, d=128, E=16, k=4, M=256, offsets="normal", capacity_factor=0.8,
      flags=PRIO | SIG),
    W("p_split", T=256, d=2048, E=8, k=2, M=128, offsets="normal", capacity_factor=0.5,
      flags=PRIO),                                   # cluster split-K router
    W("p_no_cut", T=300, d=128, E=8, k=2, M=128, capacity_factor=8.0, flags=PRIO),
]


@pytest.mark.parametrize("w", PRIO_CASES, ids=lambda w: w.name)
def test_priority_capacity(w):
    g, ref = check_layer(synth.make_inputs(w, "cuda"))
    C = ref.C
    if C < ref.disp.counts.max():
        assert ref.disp.dropped.any()
        # the cut really is by score: some kept pair comes after a dropped one
        # of the same expert in token order
        tok = oracle_routing(synth.make_inputs(w.replace(flags=w.flags & ~PRIO), "cuda"),
                             g.ids)
        assert (tok.disp.dropped != ref.disp.dropped).any()


@pytest.mark.parametrize("k,distinct", [(1, 7), (2, 13)])
def test_priority_capacity_exact_ties(k, distinct):
    w = W("p_ties", T=640, d=128, E=8, k=k, M=128, offsets="normal", capacity_factor=0.5,
          flags=PRIO)
    inp = with_duplicate_rows(synth.make_inputs(w, "cuda"), distinct)
    g, ref = check_layer(inp)
    # exact ties at the cut are broken identically on both sides (token order)
    free = oracle.dispatch_priority(ref.routing.ids, ref.routing.p, w.E, ref.C)
    np.testing.assert_array_equal(g.drop.astype(np.uint8), free.dropped)
    assert free.dropped.any()


def test_priority_capacity_full_switch():
    w = synth.WORKLOADS["switch"].replace(flags=PRIO)
    inp = synth.make_inputs(w, "cuda")
    g = run_layer(inp)
    ref = oracle_routing(inp, g.ids, g.drop)
    assert_routing_parity(g, ref, w)
    rng = np.random.default_rng(99)
    sel = set(rng.choice(w.T, size=16, replace=False).tolist()) | {0, w.T - 1}
    sel |= set(np.nonzero(ref.disp.dropped.all(axis=1))[0][:4].tolist())
    sel = np.array(sorted(sel), dtype=np.int32)
    assert_y_close(bf16_to_f64(g.y)[sel], oracle_y(inp, ref, sel), "switch priority y")


EC_CASES = [
    W("ec_soft", T=300, d=256, E=16, k=2, M=128, offsets="normal", capacity_factor=1.0,
      flags=EC),
    W("ec_sigmoid", T=517, d=192, E=64, k=6, M=128, offsets="normal", flags=EC | SIG),
    W("ec_shared", T=389, d=128, E=16, k=4, M=256, n_shared=1, capacity_factor=1.0, flags=EC),
    W("ec_r_is_T", T=200, d=128, E=8, k=2, M=128, capacity_factor=8.0, flags=EC),
    W("ec_k0_shared", T=130, d=128, E=8, k=0, M=128, n_shared=2, flags=EC),
    W("ec_split", T=256, d=2048, E=8, k=2, M=128, capacity_factor=0.5, flags=EC),
    W("ec_many", T=4097, d=128, E=128, k=1, M=128, offsets="normal", flags=EC),
]


@pytest.mark.parametrize("w", EC_CASES, ids=lambda w: w.name)
def test_expert_choice(w):
    g, ref = check_ec_layer(synth.make_inputs(w, "cuda"))
    if w.k > 0 and g.r < w.T:
        # a token may be taken by several experts or by none
        hits = np.bincount(g.row_token, minlength=w.T)
        assert hits.max() >= 2 or hits.min() == 0


@pytest.mark.parametrize("distinct", [5, 17])
def test_expert_choice_exact_ties(distinct):
    w = W("ec_ties", T=640, d=128, E=8, k=2, M=128, offsets="normal", flags=EC)
    inp = with_duplicate_rows(synth.make_inputs(w, "cuda"), distinct)
    g, ref = check_ec_layer(inp)
    assert ref.forced > 0      # the cuts do fall inside groups of equal scores
    assert ref.flipped == 0    # and both sides break those ties identically


def test_expert_choice_empty_batch():
    w = W("ec_empty", T=0, d=128, E=8, k=2, M=128, n_shared=1, flags=EC)
    s = moe.Shape.of(w.T, w.d, w.M, w.E, w.k, w.n_shared, w.capacity_factor, w.balance_coef,
                     w.flags)
    assert moe.moe_ec_capacity(s) == 0
    inp = synth.make_inputs(w, "cuda")
    layer = moe.MoELayer(s, inp.wr, inp.w1, inp.w3, inp.w2, inp.ws1, inp.ws3, inp.ws2,
                         device="cuda")
    layer.forward(inp.x)
    torch.cuda.synchronize()
    assert moe.moe_check_status(layer.ws) == 0
    assert layer.counts.cpu().tolist() == [0] * w.E


@pytest.mark.parametrize("name", ["mixtral", "deepseekv2"])
def test_expert_choice_full_size(name):
    base = synth.WORKLOADS[name]
    w = base.replace(flags=EC, sel_bias="none")
    inp = synth.make_inputs(w, "cuda")
    rng = np.random.default_rng(7)
    sel = np.array(sorted(set(rng.choice(w.T, size=12, replace=False).tolist())
                          | {0, w.T - 1}), dtype=np.int32)
    g, ref = check_ec_layer(inp, sel)
    print(f"{name} expert choice: r = {g.r}, near-cut picks {ref.forced} (flipped "
          f"{ref.flipped}), tokens picked by none {int((np.bincount(g.row_token, minlength=w.T) == 0).sum())}")


@pytest.mark.parametrize("w", [PRIO_CASES[0], PRIO_CASES[2], EC_CASES[1], EC_CASES[2]],
                         ids=lambda w: w.name)
def test_select_paths_with_fused_gather(w):
    """Priority capacity and expert choice with GEMM-1 gathering token rows by
    row_token instead of the gather kernel's x_perm."""
    tune = dict(options=moe.MOE_TUNE_FUSED_GATHER)
    if w.flags & EC:
        check_ec_layer(synth.make_inputs(w, "cuda"), tuning=tune)
    else:
        check_layer(synth.make_inputs(w, "cuda"), tuning=tune)


@pytest.mark.parametrize("w", [PRIO_CASES[0], PRIO_CASES[2], EC_CASES[0], EC_CASES[2]],
                         ids=lambda w: w.name)
def test_select_paths_gate_in_epilogue(w):
    """Priority capacity and expert choice with the gates applied in the down
    projection's epilogue."""
    tune = dict(options=moe.MOE_TUNE_GATE_IN_EPILOGUE)
    if w.flags & EC:
        check_ec_layer(synth.make_inputs(w, "cuda"), tuning=tune)
    else:
        check_layer(synth.make_inputs(w, "cuda"), tuning=tune)


def test_deterministic_bitwise_select():
    for w in (PRIO_CASES[0], EC_CASES[0]):
        inp = synth.make_inputs(w, "cuda")
        s = moe.Shape.of(w.T, w.d, w.M, w.E, w.k, w.n_shared, w.capacity_factor,
                         w.balance_coef, w.flags)
        layer = moe.MoELayer(s, inp.wr, inp.w1, inp.w3, inp.w2, inp.ws1, inp.ws3, inp.ws2,
                             inp.offset, inp.sel_bias if not (w.flags & EC) else None,
                             device="cuda")
        outs = []
        for _ in range(2):
            layer.forward(inp.x)
            torch.cuda.synchronize()
            outs.append(layer.y.clone())
        assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))

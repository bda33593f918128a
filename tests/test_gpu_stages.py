"""GPU parity of each entry point on its own, with synthetic stage inputs
(never inputs produced by another GPU stage): moe_route, moe_permute,
moe_grouped_ffn, moe_combine, moe_pack_w13."""
import numpy as np
import pytest
import torch

import oracle
import synth
import top_routing_expert_lb_b300 as moe
from guard import guarded
from parity import (guarded_workspace, GATE_ABS, LOSS_REL, assert_y_close, bf16_to_f64, np_of, oracle_routing,
                    rel_close, shape_of)
from top_routing_expert_lb_b300 import build as mbuild

pytestmark = pytest.mark.gpu
W = synth.Workload


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mbuild.ensure_built()
    assert torch.cuda.is_available()


def _ws(s):
    return guarded_workspace(s)


# --------------------------------------------------------------------------- route
@pytest.mark.parametrize("w", [
    W("r_small", T=257, d=128, E=8, k=2, M=128),
    W("r_offset", T=1000, d=512, E=64, k=6, M=128, offsets="normal"),
    W("r_bias", T=700, d=1024, E=160, k=6, M=128, offsets="normal", sel_bias="uniform"),
    W("r_top1", T=129, d=64, E=128, k=1, M=128, offsets="normal"),
    W("r_k0", T=200, d=64, E=8, k=0, M=128),
    W("r_E256", T=300, d=192, E=256, k=8, M=128),
], ids=lambda w: w.name)
def test_route(w):
    inp = synth.make_inputs(w, "cuda", experts=False)
    s = shape_of(w)
    dev = "cuda"
    ids = guarded((w.T, w.k), torch.int32, dev, label="ids")
    gates = guarded((w.T, w.k), torch.float32, dev, label="gates")
    counts = guarded(w.E, torch.int32, dev, label="counts")
    f = guarded(w.E, torch.float32, dev, label="f")
    P = guarded(w.E, torch.float32, dev, label="P")
    lb = guarded(1, torch.float32, dev, label="bal_loss")
    lz = guarded(1, torch.float32, dev, label="z_loss")
    ws = _ws(s)
    moe.moe_route(s, inp.x, inp.wr, inp.offset, inp.sel_bias, ids, gates, counts, f, P, lb, lz,
                  ws)
    torch.cuda.synchronize()
    assert moe.moe_check_status(ws) == 0
    ref = oracle_routing(inp, np_of(ids))
    if w.k:
        np.testing.assert_array_equal(np_of(ids), ref.routing.ids)
        assert np.abs(np_of(gates) - ref.routing.gates).max() <= GATE_ABS
    np.testing.assert_array_equal(np_of(counts), ref.disp.counts)
    np.testing.assert_allclose(np_of(f), ref.loss.f, rtol=1e-6)
    np.testing.assert_allclose(np_of(P), ref.loss.P, rtol=LOSS_REL, atol=1e-7)
    rel_close(lb.item(), ref.loss.L_bal, LOSS_REL, "balance loss")
    rel_close(lz.item(), ref.loss.L_z, LOSS_REL, "z-loss")


@pytest.mark.parametrize("d", [256, 4096])
def test_route_exact_expert_ties_break_to_lower_index(d):
    """Pairs of experts with identical router rows and offsets tie exactly in
    every token; the lower index must be chosen first (listed before the
    higher one with the same gate, and never left out while the higher one is
    in).  The pairs sit in the same and in different 16-column groups, so the
    tie is decided inside one thread's list and in the merge of the four
    per-row lists; d = 4096 splits each tile's K across CTAs."""
    w = W("r_ties", T=1000, d=d, E=80, k=6, M=128, offsets="normal")
    inp = synth.make_inputs(w, "cuda", experts=False)
    pairs = [(3, 20), (17, 50), (5, 37), (2, 10), (64, 79)]
    wr = inp.wr.clone()
    off = inp.offset.clone()
    for lo, hi in pairs:
        wr[hi] = wr[lo]
        off[lo] = off[hi] = 2.5   # popular, so both members are often selected
    inp.wr, inp.offset = wr, off
    s = shape_of(w)
    dev = "cuda"
    ids = guarded((w.T, w.k), torch.int32, dev, label="ids")
    gates = guarded((w.T, w.k), torch.float32, dev, label="gates")
    counts = guarded(w.E, torch.int32, dev, label="counts")
    f, P = torch.empty(w.E, device=dev), torch.empty(w.E, device=dev)
    lb, lz = torch.empty(1, device=dev), torch.empty(1, device=dev)
    ws = _ws(s)
    moe.moe_route(s, inp.x, inp.wr, inp.offset, inp.sel_bias, ids, gates, counts, f, P, lb, lz,
                  ws)
    torch.cuda.synchronize()
    assert moe.moe_check_status(ws) == 0
    g_ids, g_gates = np_of(ids), np_of(gates)
    for lo, hi in pairs:
        has_lo, has_hi = (g_ids == lo).any(1), (g_ids == hi).any(1)
        assert has_hi.sum() > 0 and (has_lo & ~has_hi).sum() > 0, "the tie is not exercised"
        assert not (has_hi & ~has_lo).any(), f"expert {hi} chosen without its tie partner {lo}"
        for t in np.nonzero(has_hi)[0]:
            jl, jh = int(np.nonzero(g_ids[t] == lo)[0][0]), int(np.nonzero(g_ids[t] == hi)[0][0])
            assert jl < jh, f"token {t}: {hi} listed before its tie partner {lo}"
            assert g_gates[t, jl] == g_gates[t, jh]
    ref = oracle_routing(inp, g_ids)
    np.testing.assert_array_equal(g_ids, ref.routing.ids)
    np.testing.assert_array_equal(np_of(counts), ref.disp.counts)


# --------------------------------------------------------------------------- permute
def _synthetic_ids(T, E, k, seed, hot_frac=0.4):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    hot = rng.random(T) < hot_frac                  # skew: many tokens pick expert 1 first
    for t in np.nonzero(hot)[0]:
        if 1 not in ids[t]:
            ids[t, 0] = 1
    return ids


@pytest.mark.parametrize("T,E,k,c,d", [
    (1, 4, 2, 0.0, 64), (129, 8, 2, 0.0, 128), (300, 16, 3, 0.0, 192),
    (517, 16, 4, 0.8, 64), (1000, 32, 1, 1.25, 128), (2048, 160, 6, 0.0, 256),
    (640, 8, 8, 0.5, 64), (130, 256, 8, 1.0, 64),
])
def test_permute(T, E, k, c, d):
    ids_np = _synthetic_ids(T, E, k, seed=T * 7 + E)
    w = W("p", T=T, d=d, E=E, k=k, M=128, capacity_factor=c)
    s = shape_of(w)
    x = synth.normal_bf16(3, synth.TID_X, (T, d), 1.0, "cuda")
    ids = torch.from_numpy(ids_np).cuda()
    R_max = moe.moe_max_rows(s)
    offsets = guarded(E + 1, torch.int32, fill=-7, label="offsets")
    slot_row = guarded((T, k), torch.int32, label="slot_row")
    row_token = guarded(max(R_max, 1), torch.int32, fill=-7, label="row_token")
    drop = guarded((T, k), torch.uint8, label="drop_mask")
    x_perm = guarded((max(R_max, 1), d), torch.bfloat16, fill=0, label="x_perm")
    ws = _ws(s)
    moe.moe_permute(s, x, ids, offsets, slot_row, row_token, drop, x_perm, ws)
    torch.cuda.synchronize()
    assert moe.moe_check_status(ws) == 0
    C = oracle.capacity(float(np.float32(c)), k, T, E)
    ref = oracle.dispatch(ids_np, E, C)
    R = int(ref.offsets[-1])
    np.testing.assert_array_equal(np_of(offsets), ref.offsets)
    np.testing.assert_array_equal(np_of(slot_row), ref.slot_row)
    np.testing.assert_array_equal(np_of(row_token)[:R], ref.row_token)
    np.testing.assert_array_equal(np_of(drop), ref.dropped)
    xp = np_of(x_perm)[:R]
    np.testing.assert_array_equal(xp, np_of(x)[ref.row_token])


# --------------------------------------------------------------------------- grouped FFN
def _tuning_for(tile: str) -> dict:
    """moe_tuning_t fields of a grouped-FFN variant name.
    128: single-CTA 128-row tiles; 256: CTA-pair 256-row tiles; 128-split: the
    gate/up projection's whole 256-row blocks on CTA pairs, the remaining rows
    on single CTAs; *-block: every group of more than 100 rows in blocks of two
    n-tiles, m-tile major inside a block (otherwise n-tile major throughout);
    CTA pairs take their tiles from the workspace counter except with
    256-static; a group's last pair tile of at most 128 rows runs as an M = 128
    pair MMA except with 256-nohalf.  With 256* and d % 256 == 0 the down
    projection runs on CTA pairs too.  Single-CTA tiles transpose the tail of
    a group of one m-tile; with 128-swapall the tail of every group.  128-twosm
    runs two CTAs per SM (one accumulator, 2-stage ring each) where BN = 256."""
    opts = 0
    if tile.endswith("swapall"):
        opts |= moe.MOE_TUNE_SWAP_ALL_TAILS
    if tile.endswith("twosm"):
        opts |= moe.MOE_TUNE_TWO_CTAS_PER_SM
    if tile.endswith("nohalf"):
        opts |= moe.MOE_TUNE_NO_HALF_TILES
    if tile.endswith("split"):
        opts |= moe.MOE_TUNE_GEMM1_SPLIT
    return dict(gemm1_tile=int(tile.split("-")[0]), tile_order=1 if tile.endswith("static") else 2,
                n_block=2 if tile.endswith("block") else 1, block_min_rows=100, options=opts)


@pytest.mark.parametrize("tile", ["128", "128-swapall", "128-twosm", "256", "256-static",
                                  "256-nohalf",
                                  "128-split", "128-block", "256-block"])
@pytest.mark.parametrize("rows,d,M,n_shared,T", [
    ([0, 1, 127, 128, 129, 300], 128, 256, 1, 200),    # empty, single, tile edges
    ([5, 0, 0, 260], 64, 128, 0, 0),                   # d = 64 (second projection N = 64)
    ([130, 70, 2], 256, 128, 2, 131),                  # d = 256, 2 shared experts
    ([0, 0, 0], 192, 128, 1, 77),                      # routed rows all empty, shared only
    ([400], 320, 384, 0, 0),                           # one group, d = 320 (N tile 64)
    ([255, 256, 257, 511, 1], 512, 256, 1, 300),       # 256-row tile edges, d = 512
    # tails of 1..112 rows run transposed (weights as the MMA's M) in groups of
    # one m-tile (every group with 128-swapall); 113..127 never
    ([16, 17, 111, 112, 113, 240, 33, 128], 256, 256, 1, 200),  # second projection N = 256
    ([48, 200, 97, 1], 384, 128, 0, 0),                # second projection N = 128
])
def test_grouped_ffn(rows, d, M, n_shared, T, tile):
    E = len(rows)
    R = int(sum(rows))
    Ms = n_shared * M
    # the shape's T is the shared group's row count; T*k bounds the routed rows
    Tshape = T if n_shared else max(R, 1)
    k = max(1, -(-R // Tshape))
    assert k <= min(E, 8)
    tune = _tuning_for(tile)
    if tile.startswith("256") and d % 256 == 0:
        tune["gemm2_tile"] = 256   # the down projection on CTA pairs as well
    s_ffn = moe.Shape.of(Tshape, d, M, E, k, n_shared, **tune)
    dev = "cuda"
    R_max = moe.moe_max_rows(s_ffn)
    assert R <= R_max
    x_perm = torch.zeros((max(R_max, 1), d), dtype=torch.bfloat16, device=dev)
    if R:
        x_perm[:R] = synth.normal_bf16(5, synth.TID_X, (R, d), 1.0, dev)
    offsets = torch.tensor(np.concatenate([[0], np.cumsum(rows)]).astype(np.int32), device=dev)
    w1 = synth.normal_bf16(5, synth.TID_W1, (E, M, d), 0.05, dev)
    w3 = synth.normal_bf16(5, synth.TID_W3, (E, M, d), 0.05, dev)
    w2 = synth.normal_bf16(5, synth.TID_W2, (E, d, M), 0.05, dev)
    w13 = moe.moe_pack_w13(w1, w3)
    y_perm = guarded((max(R_max, 1), d), torch.bfloat16, dev, fill=0, label="y_perm")
    x = ws1 = ws3 = ws2 = w13s = y_s = None
    if n_shared:
        x = synth.normal_bf16(6, synth.TID_X, (T, d), 1.0, dev)
        ws1 = synth.normal_bf16(5, synth.TID_WS1, (Ms, d), 0.05, dev)
        ws3 = synth.normal_bf16(5, synth.TID_WS3, (Ms, d), 0.05, dev)
        ws2 = synth.normal_bf16(5, synth.TID_WS2, (d, Ms), 0.05, dev)
        w13s = moe.moe_pack_w13(ws1, ws3)
        y_s = guarded((T, d), torch.bfloat16, dev, fill=0, label="y_shared")
    ws = _ws(s_ffn)
    moe.moe_grouped_ffn(s_ffn, x_perm, offsets, w13, w2, y_perm, x, w13s, ws2, y_s, ws)
    torch.cuda.synchronize()
    assert moe.moe_check_status(ws) == 0
    expert = np.repeat(np.arange(E, dtype=np.int32), rows)
    if R:
        ref = oracle.expert_rows(np_of(x_perm)[:R], expert, np_of(w1), np_of(w3), np_of(w2))
        assert_y_close(bf16_to_f64(y_perm)[:R], ref, "y_perm")
    if n_shared:
        ref_s = oracle.expert_rows(np_of(x), np.zeros(T, np.int32), np_of(ws1)[None],
                                   np_of(ws3)[None], np_of(ws2)[None])
        assert_y_close(bf16_to_f64(y_s), ref_s, "y_shared")


def test_grouped_ffn_dynamic_order_repeats():
    """CTA-pair launches that take tiles from the workspace counter leave it at
    zero: back-to-back calls on one workspace (and a run of a different shape
    on it in between) give the same bits, and the oracle's values."""
    dev = "cuda"
    rows = [300, 0, 513, 77, 256, 129]
    E, d, M = len(rows), 256, 256
    R = sum(rows)
    s_ffn = moe.Shape.of(R, d, M, E, 1, 0, gemm1_tile=256, tile_order=2)
    x_perm = synth.normal_bf16(7, synth.TID_X, (R, d), 1.0, dev)
    offsets = torch.tensor(np.concatenate([[0], np.cumsum(rows)]).astype(np.int32), device=dev)
    w1 = synth.normal_bf16(7, synth.TID_W1, (E, M, d), 0.05, dev)
    w3 = synth.normal_bf16(7, synth.TID_W3, (E, M, d), 0.05, dev)
    w2 = synth.normal_bf16(7, synth.TID_W2, (E, d, M), 0.05, dev)
    w13 = moe.moe_pack_w13(w1, w3)
    ws = _ws(s_ffn)
    outs = []
    for i in range(3):
        y = guarded((R, d), torch.bfloat16, dev, fill=0, label="y_perm")
        moe.moe_grouped_ffn(s_ffn, x_perm, offsets, w13, w2, y, None, None, None, None, ws)
        if i == 1:   # another grouping on the same workspace in between
            off2 = torch.tensor([0, R // 2, R, R, R, R, R], dtype=torch.int32, device=dev)
            y2 = torch.zeros_like(y)
            moe.moe_grouped_ffn(s_ffn, x_perm, off2, w13, w2, y2, None, None, None, None, ws)
        torch.cuda.synchronize()
        assert moe.moe_check_status(ws) == 0
        outs.append(y)
    for y in outs[1:]:
        assert torch.equal(y.view(torch.int16), outs[0].view(torch.int16))
    expert = np.repeat(np.arange(E, dtype=np.int32), rows)
    ref = oracle.expert_rows(np_of(x_perm), expert, np_of(w1), np_of(w3), np_of(w2))
    assert_y_close(bf16_to_f64(outs[-1]), ref, "y_perm after repeated dynamic launches")


# --------------------------------------------------------------------------- combine
@pytest.mark.parametrize("T,d,E,k,c,shared", [
    (1, 64, 4, 2, 0.0, False), (300, 256, 8, 2, 0.0, True), (517, 128, 16, 4, 0.7, True),
    (999, 64, 32, 1, 1.25, False), (64, 512, 8, 8, 0.0, True),
])
def test_combine(T, d, E, k, c, shared):
    ids_np = _synthetic_ids(T, E, k, seed=T + d)
    C = oracle.capacity(float(np.float32(c)), k, T, E)
    disp = oracle.dispatch(ids_np, E, C)
    R = max(int(disp.offsets[-1]), 1)
    rng = np.random.default_rng(T)
    g = rng.random((T, k)).astype(np.float32) + 0.05
    g /= g.sum(1, keepdims=True)
    y_perm = synth.normal_bf16(9, synth.TID_X, (R, d), 1.0, "cuda")
    y_s = synth.normal_bf16(10, synth.TID_X, (T, d), 1.0, "cuda") if shared else None
    y = guarded((T, d), torch.bfloat16, label="y")
    s = moe.Shape.of(T, d, 128, E, k, 1 if shared else 0, c)
    moe.moe_combine(s, y_perm, torch.from_numpy(disp.slot_row).cuda(), torch.from_numpy(g).cuda(),
                    y_s, y)
    torch.cuda.synchronize()
    ref = oracle.combine(np_of(y_perm), disp.slot_row, g.astype(np.float64), np_of(y_s))
    yg = bf16_to_f64(y)
    # one bf16 rounding of an fp32 sum: |err| <= 2^-8 |ref| + small
    assert np.all(np.abs(yg - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5)


def test_pack_w13():
    G, Mw, d = 3, 384, 128
    w1 = synth.normal_bf16(1, synth.TID_W1, (G, Mw, d), 1.0, "cuda")
    w3 = synth.normal_bf16(1, synth.TID_W3, (G, Mw, d), 1.0, "cuda")
    out = np_of(moe.moe_pack_w13(w1, w3))
    a, b = np_of(w1), np_of(w3)
    for g in range(G):
        for j in range(Mw // 128):
            np.testing.assert_array_equal(out[g, 256 * j:256 * j + 128], a[g, 128 * j:128 * j + 128])
            np.testing.assert_array_equal(out[g, 256 * j + 128:256 * j + 256],
                                          b[g, 128 * j:128 * j + 128])

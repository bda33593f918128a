"""Shared helpers of the GPU parity tests: run the CUDA layer through the C ABI,
run the oracle on the same seeded inputs, compare with the stated tolerances.

Tolerances (fixed by the benchmark spec of the layer and restated here):
  * expert ids, counts, drop masks, offsets, permutation: bit-exact, except
    tokens whose k-th and (k+1)-th selection keys differ by less than 1e-5
    ("near ties"), whose choice may differ between fp32 and fp64; for those the
    oracle is re-run with the GPU's choice forced, after checking that the
    oracle's own gap really is below the threshold (so both choices are valid);
  * layer output y: relative Frobenius error <= 1e-2 and
    max |y - ref| <= 3e-2 * max |ref|;
  * balance loss, z-loss and P: 1e-4 relative; f exact up to fp32 rounding;
  * gates (fp32 softmax / renormalisation): 1e-5 absolute;
  * score-ordered cuts (probability-priority capacity, expert choice):
    kept sets bit-exact except entries whose score lies within a relative
    1e-5 of the cut score, where the GPU's decision is taken after checking
    that its kept set has the right size and keeps everything clearly above
    the cut and nothing clearly below.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

import oracle
import synth
import top_routing_expert_lb_b300 as moe
from guard import guarded, guarded_like

TIE = 1e-5
CUT_REL = 1e-5   # near-cut band of score-ordered selections, relative to the cut score
Y_REL_FRO = 1e-2
Y_MAX_ABS = 3e-2
LOSS_REL = 1e-4
GATE_ABS = 1e-5


def shape_of(w: synth.Workload, **tuning) -> moe.Shape:
    """The workload's moe_shape_t; keyword arguments set moe_tuning_t fields."""
    return moe.Shape.of(w.T, w.d, w.M, w.E, w.k, w.n_shared, w.capacity_factor,
                        w.balance_coef, w.flags, **tuning)


def guarded_workspace(shape: moe.Shape, device="cuda") -> torch.Tensor:
    """A zeroed workspace with canary guards on both sides."""
    n = max(moe.moe_workspace_size(shape), 256)
    return guarded((n,), torch.uint8, device, fill=0, label="workspace")


def guard_layer(layer: moe.MoELayer) -> moe.MoELayer:
    """Replaces the layer's outputs and workspace by canary-guarded buffers."""
    names = ["y", "ids", "gates", "drop_mask", "counts", "f", "P", "losses"]
    if layer.expert_choice:
        names += ["row_token", "row_gate"]
    for name in names:
        setattr(layer, name, guarded_like(getattr(layer, name), label=f"layer.{name}"))
    layer.ws = guarded_workspace(layer.shape, layer.ws.device)
    return layer


def np_of(t: Optional[torch.Tensor]):
    if t is None:
        return None
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


@dataclass
class GpuOut:
    y: torch.Tensor
    ids: np.ndarray
    gates: np.ndarray
    counts: np.ndarray
    drop: np.ndarray
    f: np.ndarray
    P: np.ndarray
    bal: float
    z: float


def run_layer(inp: synth.Inputs, layer: Optional[moe.MoELayer] = None,
              tuning: Optional[dict] = None) -> GpuOut:
    w = inp.w
    if layer is None:
        layer = guard_layer(moe.MoELayer(shape_of(w, **(tuning or {})), inp.wr, inp.w1, inp.w3,
                                         inp.w2, inp.ws1, inp.ws3, inp.ws2, inp.offset,
                                         inp.sel_bias, device=inp.x.device))
    layer.forward(inp.x)
    torch.cuda.synchronize()
    assert moe.moe_check_status(layer.ws) == 0
    return GpuOut(layer.y.clone(), np_of(layer.ids), np_of(layer.gates), np_of(layer.counts),
                  np_of(layer.drop_mask), np_of(layer.f), np_of(layer.P),
                  float(layer.losses[0]), float(layer.losses[1]))


def topk_choice_problems(key: np.ndarray, ids: np.ndarray, k: int, tol: float = TIE):
    """Why ``ids`` is not a valid Top-k of one token's selection keys ``key``
    (fp64, the oracle's) within ``tol``; an empty list when it is.

    A valid choice names k distinct experts in [0, E); each selected key is at
    least the k-th largest key minus tol, each unselected key at most the
    (k+1)-th largest plus tol, and the selected keys descend up to tol.  With
    a gap of at least tol between the k-th and (k+1)-th keys this leaves only
    the oracle's set (in any order of keys closer than tol)."""
    E = key.shape[0]
    ids = np.asarray(ids)
    out = []
    if len(ids) != k or len(set(ids.tolist())) != k:
        out.append(f"ids {ids.tolist()} are not {k} distinct experts")
        return out
    if ids.min() < 0 or ids.max() >= E:
        out.append(f"ids {ids.tolist()} outside [0, {E})")
        return out
    srt = np.sort(key)[::-1]
    kth = srt[k - 1]
    nxt = srt[k] if k < E else -np.inf
    sel = key[ids]
    if np.any(sel < kth - tol):
        out.append(f"selected key {sel.min():.9g} below the k-th key {kth:.9g} - {tol}")
    rest = np.delete(key, ids)
    if rest.size and np.any(rest > nxt + tol):
        out.append(f"unselected key {rest.max():.9g} above the (k+1)-th key {nxt:.9g} + {tol}")
    if np.any(np.diff(sel) > tol):
        out.append(f"selected keys {sel.tolist()} not descending up to {tol}")
    return out


def routing_force_mask(free: oracle.Routing, gpu_ids: np.ndarray, bias) -> np.ndarray:
    """Tokens whose GPU selection the oracle takes over, after checking it.

    The selected set is unique unless the k-th and (k+1)-th keys are within
    1e-5 (a near tie at the cut: such tokens are exempt).  Inside the set, the
    order of two keys closer than 1e-5 is not unique either.  Every token whose
    GPU choice differs from the oracle's must be a valid Top-k of the oracle's
    fp64 keys within 1e-5 (``topk_choice_problems``); a token outside the
    near-tie band must in addition have the oracle's set.  Any other
    difference fails.  (Slot order inside one token cannot change drops or
    rows: a token sends at most one pair to an expert.)"""
    key = free.p + (0.0 if bias is None else np.asarray(bias, np.float64)[None, :])
    k = free.ids.shape[1]
    exempt = free.gap < TIE
    diff = np.any(free.ids != gpu_ids, axis=1)
    bad = []
    for t in np.nonzero(diff)[0]:
        why = topk_choice_problems(key[t], gpu_ids[t], k)
        if not exempt[t] and sorted(free.ids[t].tolist()) != sorted(gpu_ids[t].tolist()):
            why.append("a different set outside the near-tie band")
        if why:
            bad.append((t, why))
    assert not bad, (f"{len(bad)} tokens routed to an invalid choice, e.g. token {bad[0][0]}: "
                     f"gpu {gpu_ids[bad[0][0]]} oracle {free.ids[bad[0][0]]} gap "
                     f"{free.gap[bad[0][0]]}: {'; '.join(bad[0][1])}")
    return diff


@dataclass
class OracleRef:
    routing: oracle.Routing
    disp: oracle.Dispatch
    loss: oracle.Losses
    exempt: np.ndarray
    C: int


def cut_force(score: np.ndarray, want: int, gpu_keep: np.ndarray, what: str) -> np.ndarray:
    """Near-cut protocol of a score-ordered selection (keep the ``want``
    largest of ``score``).  The kept set is unique except for scores within a
    relative 1e-5 of the cut value (the want-th largest, fp64): the GPU's fp32
    scores carry a relative error of a few 1e-6 (fp32 logit accumulation and
    softmax), so there fp32 and fp64 may decide differently.  Scores span many
    orders of magnitude across experts, hence relative rather than absolute.
    Checks that the GPU kept exactly ``want`` entries, every entry clearly
    above the cut and none clearly below; returns the int8 force vector (+1
    kept / -1 dropped on the near-cut entries, else 0) that makes the oracle
    take the GPU's decisions there."""
    n = len(score)
    force = np.zeros(n, np.int8)
    if want >= n:
        assert gpu_keep.all(), f"{what}: dropped an entry with no cut"
        return force
    thr = np.sort(score)[::-1][want - 1] if want > 0 else np.inf
    tol = CUT_REL * thr if want > 0 else 0.0
    assert int(gpu_keep.sum()) == want, f"{what}: kept {int(gpu_keep.sum())}, want {want}"
    assert gpu_keep[score > thr + tol].all(), f"{what}: dropped a score above the cut"
    assert not gpu_keep[score < thr - tol].any(), f"{what}: kept a score below the cut"
    band = np.abs(score - thr) <= tol
    force[band] = np.where(gpu_keep[band], 1, -1)
    return force


def priority_force(r: oracle.Routing, E: int, C: int, gpu_drop: np.ndarray) -> np.ndarray:
    """cut_force over each over-full expert's pairs (probability priority)."""
    T, k = r.ids.shape
    flat = r.ids.reshape(-1)
    score = r.p[np.repeat(np.arange(T), k), flat]
    keep = np.asarray(gpu_drop).reshape(-1) == 0
    force = np.zeros(T * k, np.int8)
    for e in range(E):
        pos = np.nonzero(flat == e)[0]
        if len(pos) > C:
            force[pos] = cut_force(score[pos], C, keep[pos], f"expert {e}")
    return force.reshape(T, k)


def oracle_routing(inp: synth.Inputs, gpu_ids: np.ndarray,
                   gpu_drop: Optional[np.ndarray] = None) -> OracleRef:
    """Oracle routing / dispatch / losses for all tokens; near-tie tokens take
    the GPU's ids after the non-tie tokens were checked bit-exactly (and, with
    probability-priority capacity, near-cut pairs the GPU's keep decision)."""
    w = inp.w
    x, wr = np_of(inp.x), np_of(inp.wr)
    off = np_of(inp.offset)
    bias = np_of(inp.sel_bias)
    logits = oracle.router_logits(x, wr, off)
    rflags = w.flags & (oracle.SIGMOID | oracle.NO_RENORM)
    free = oracle.route(logits, w.k, bias, flags=rflags)
    exempt = free.gap < TIE
    if w.k > 0:
        force = routing_force_mask(free, gpu_ids, bias)
        r = oracle.route(logits, w.k, bias, force_ids=gpu_ids, force_mask=force, flags=rflags)
        exempt = force | exempt
    else:
        r = free
    C = oracle.capacity(float(np.float32(w.capacity_factor)), w.k, w.T, w.E)
    if (w.flags & oracle.PRIORITY) and C >= 0 and w.k > 0:
        assert gpu_drop is not None
        pf = priority_force(r, w.E, C, gpu_drop)
        disp = oracle.dispatch_priority(r.ids, r.p, w.E, C, force=pf)
    else:
        disp = oracle.dispatch(r.ids, w.E, C)
    ls = oracle.losses(disp.counts, r.p, r.lse, w.k, float(np.float32(w.balance_coef)))
    return OracleRef(r, disp, ls, exempt, C)


def oracle_y(inp: synth.Inputs, ref: OracleRef, sel: np.ndarray,
             host_weights: Optional[tuple] = None) -> np.ndarray:
    """Oracle layer output for the tokens in ``sel``, copying to the host only
    the expert weights those tokens use (or using ``host_weights``, the full
    (w1, w3, w2) as uint16 arrays, when given)."""
    w = inp.w
    sel = np.asarray(sel, np.int32)
    x = np_of(inp.x)
    ids = ref.routing.ids[sel]
    if host_weights is not None:
        w1, w3, w2 = host_weights
        ids_c = np.ascontiguousarray(ids, np.int32)
    else:
        used = sorted(set(ids.reshape(-1).tolist())) if w.k > 0 else []
        remap = {e: i for i, e in enumerate(used)}
        if used:
            idx = torch.tensor(used, device=inp.w1.device)
            w1 = np_of(inp.w1.index_select(0, idx))
            w3 = np_of(inp.w3.index_select(0, idx))
            w2 = np_of(inp.w2.index_select(0, idx))
            ids_c = np.vectorize(remap.get)(ids).astype(np.int32).reshape(ids.shape)
        else:
            w1 = w3 = np.zeros((1, w.M, w.d), np.uint16)
            w2 = np.zeros((1, w.d, w.M), np.uint16)
            ids_c = np.zeros((len(sel), w.k), np.int32)
    xs = x[sel]
    loc = np.arange(len(sel), dtype=np.int32)
    return oracle.layer_tokens(xs, ids_c, ref.routing.gates[sel], ref.disp.dropped[sel], w1, w3,
                               w2, np_of(inp.ws1), np_of(inp.ws3), np_of(inp.ws2), loc)


def assert_y_close(y_gpu: np.ndarray, y_ref: np.ndarray, what="y"):
    y_gpu = np.asarray(y_gpu, np.float64)
    assert y_gpu.shape == y_ref.shape
    den = np.linalg.norm(y_ref)
    num = np.linalg.norm(y_gpu - y_ref)
    mx = np.abs(y_ref).max() if y_ref.size else 0.0
    if den == 0.0:
        assert num == 0.0, f"{what}: expected exact zeros, got |y| = {num}"
        return
    assert num <= Y_REL_FRO * den, f"{what}: rel Frobenius {num / den:.3e} > {Y_REL_FRO}"
    err = np.abs(y_gpu - y_ref).max()
    assert err <= Y_MAX_ABS * mx, f"{what}: max abs {err:.3e} > {Y_MAX_ABS} * {mx:.3e}"


def rel_close(a: float, b: float, tol: float, what: str):
    scale = max(abs(b), 1e-30)
    assert abs(a - b) <= tol * scale, f"{what}: {a} vs {b} (rel {abs(a - b) / scale:.2e})"


def assert_routing_parity(g: GpuOut, ref: OracleRef, w: synth.Workload):
    if w.k > 0:
        np.testing.assert_array_equal(g.ids, ref.routing.ids)
        assert np.abs(g.gates - ref.routing.gates).max() <= GATE_ABS
    np.testing.assert_array_equal(g.counts, ref.disp.counts)
    np.testing.assert_array_equal(g.drop.astype(np.uint8), ref.disp.dropped)
    np.testing.assert_allclose(g.f, ref.loss.f, rtol=1e-6, atol=0)
    np.testing.assert_allclose(g.P, ref.loss.P, rtol=LOSS_REL, atol=1e-7)
    rel_close(g.bal, ref.loss.L_bal, LOSS_REL, "balance loss")
    rel_close(g.z, ref.loss.L_z, LOSS_REL, "z-loss")


def check_layer(inp: synth.Inputs, sel: Optional[np.ndarray] = None, layer=None,
                tuning: Optional[dict] = None):
    """Runs the GPU layer (with the given moe_tuning_t fields) and checks it
    against the oracle.  Returns (gpu, ref)."""
    g = run_layer(inp, layer, tuning)
    ref = oracle_routing(inp, g.ids, g.drop)
    assert_routing_parity(g, ref, inp.w)
    if sel is None:
        sel = np.arange(inp.w.T)
    if len(sel):
        y_ref = oracle_y(inp, ref, sel)
        assert_y_close(bf16_to_f64(g.y)[sel], y_ref)
    return g, ref


# --------------------------------------------------------------------------- #
# expert choice                                                                #
# --------------------------------------------------------------------------- #
@dataclass
class EcGpuOut:
    y: torch.Tensor
    row_token: np.ndarray
    row_gate: np.ndarray
    counts: np.ndarray
    f: np.ndarray
    P: np.ndarray
    bal: float
    z: float
    r: int


def run_ec_layer(inp: synth.Inputs, layer: Optional[moe.MoELayer] = None,
                 tuning: Optional[dict] = None) -> EcGpuOut:
    w = inp.w
    assert w.flags & moe.MOE_FLAG_EXPERT_CHOICE
    if layer is None:
        layer = guard_layer(moe.MoELayer(shape_of(w, **(tuning or {})), inp.wr, inp.w1, inp.w3,
                                         inp.w2, inp.ws1, inp.ws3, inp.ws2, inp.offset, None,
                                         device=inp.x.device))
    layer.forward(inp.x)
    torch.cuda.synchronize()
    assert moe.moe_check_status(layer.ws) == 0
    n = w.E * layer.r
    return EcGpuOut(layer.y.clone(), np_of(layer.row_token)[:n], np_of(layer.row_gate)[:n],
                    np_of(layer.counts), np_of(layer.f), np_of(layer.P), float(layer.losses[0]),
                    float(layer.losses[1]), layer.r)


@dataclass
class EcRef:
    routing: oracle.Routing
    ec: oracle.ExpertChoice
    loss: oracle.Losses
    forced: int      # near-cut (expert, token) entries decided by the GPU
    flipped: int     # rows where that differs from the oracle's own pick


def oracle_ec(inp: synth.Inputs, gpu_row_token: np.ndarray) -> EcRef:
    """Oracle expert-choice routing; near-cut (expert, token) picks take the
    GPU's decision after the validity checks of cut_force."""
    w = inp.w
    logits = oracle.router_logits(np_of(inp.x), np_of(inp.wr), np_of(inp.offset))
    r0 = oracle.route(logits, 0, None, flags=w.flags & oracle.SIGMOID)
    r = oracle.ec_capacity(float(np.float32(w.capacity_factor)), w.k, w.T, w.E)
    force = np.zeros((w.E, w.T), np.int8)
    for e in range(w.E):
        picked = np.zeros(w.T, bool)
        rows = gpu_row_token[e * r:(e + 1) * r]
        assert np.all(np.diff(rows) > 0), f"expert {e}: rows not in ascending token order"
        picked[rows] = True
        force[e] = cut_force(r0.p[:, e], r, picked, f"expert {e}")
    ec = oracle.expert_choice(r0.p, r, force=force)
    free = oracle.expert_choice(r0.p, r)
    ls = oracle.losses(np.full(w.E, r, np.int32), r0.p, r0.lse, w.k,
                       float(np.float32(w.balance_coef)), n_pairs=w.E * r)
    flipped = int(np.count_nonzero(ec.row_token != free.row_token))
    return EcRef(r0, ec, ls, int(np.count_nonzero(force)), flipped)


def oracle_ec_y(inp: synth.Inputs, ref: EcRef, sel: np.ndarray) -> np.ndarray:
    """Oracle expert-choice output for the tokens in ``sel``, copying to the
    host only the weights of the experts that picked them."""
    w = inp.w
    r = ref.ec.r
    sel = np.asarray(sel, np.int32)
    used = [e for e in range(w.E)
            if r > 0 and np.isin(ref.ec.row_token[e * r:(e + 1) * r], sel).any()]
    if used:
        idx = torch.tensor(used, device=inp.w1.device)
        w1 = np_of(inp.w1.index_select(0, idx))
        w3 = np_of(inp.w3.index_select(0, idx))
        w2 = np_of(inp.w2.index_select(0, idx))
        rows = np.concatenate([np.arange(e * r, (e + 1) * r) for e in used])
        sub = oracle.ExpertChoice(r, ref.ec.row_token[rows], ref.ec.row_gate[rows])
    else:
        w1 = w3 = np.zeros((1, w.M, w.d), np.uint16)
        w2 = np.zeros((1, w.d, w.M), np.uint16)
        sub = oracle.ExpertChoice(0, np.zeros(0, np.int32), np.zeros(0))
    return oracle.ec_layer_tokens(np_of(inp.x), sub, w1, w3, w2, np_of(inp.ws1),
                                  np_of(inp.ws3), np_of(inp.ws2), sel)


def check_ec_layer(inp: synth.Inputs, sel: Optional[np.ndarray] = None, layer=None,
                   tuning: Optional[dict] = None):
    """Runs the GPU expert-choice layer and checks it against the oracle."""
    w = inp.w
    g = run_ec_layer(inp, layer, tuning)
    ref = oracle_ec(inp, g.row_token)
    assert g.r == ref.ec.r
    np.testing.assert_array_equal(g.row_token, ref.ec.row_token)
    if g.r > 0:
        assert np.abs(g.row_gate - ref.ec.row_gate).max() <= GATE_ABS
    np.testing.assert_array_equal(g.counts, np.full(w.E, g.r))
    np.testing.assert_allclose(g.f, ref.loss.f, rtol=1e-6, atol=0)
    np.testing.assert_allclose(g.P, ref.loss.P, rtol=LOSS_REL, atol=1e-7)
    rel_close(g.bal, ref.loss.L_bal, LOSS_REL, "balance loss")
    rel_close(g.z, ref.loss.L_z, LOSS_REL, "z-loss")
    if sel is None:
        sel = np.arange(w.T)
    if len(sel):
        y_ref = oracle_ec_y(inp, ref, sel)
        assert_y_close(bf16_to_f64(g.y)[sel], y_ref)
    return g, ref

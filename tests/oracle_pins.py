"""Pins for the oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes an oracle library handle (``oracle.load()`` or a
mutated build) and raises AssertionError on mismatch.  The pins are:

* the hand-worked 2-token / 4-expert example in ``golden/hand_2tok_4exp.json``
  (closed-form values, worked out by hand);
* per-row experts (the reference of the grouped-FFN stage tests): a closed-form
  hand case and rows through different random experts against numpy;
* the second gating formula Softmax(TopK(W_g x, k)) of the aiattnstudio page
  (§2.2), which must give the same set and gates as softmax -> TopK ->
  renormalise when there is no selection bias;
* brute-force enumeration of every k-subset of experts on tiny inputs, with the
  expert FFNs recomputed by numpy matrix products;
* dispatch against numpy's stable argsort (the permutation of the CSDN note's
  moe_infer, with ties in token order) and a cumulative-count capacity cut;
* closed forms and invariants: gates sum to 1, sum f = 1, sum P = 1,
  sum n_e = kT, uniform logits give L_bal = lambda, L_z from scipy's logsumexp,
  k = 0 gives the shared-only output, c -> inf equals dropless, E = 1 / k = 1
  is the dense SwiGLU FFN, k = E is the dense soft mixture, token permutation
  equivariance;
* probability-priority capacity: a hand case from closed forms, a numpy
  lexsort cut, equal scores reduce to the token-order cut;
* expert-choice routing: a hand case from closed forms (ties, a token no
  expert picks, a shared expert), numpy lexsort picks with a numpy recompute
  of y, and r = T equal to the token-choice k = E soft mixture.
"""
from __future__ import annotations

import itertools
import json
import os

import numpy as np
from scipy.special import logsumexp

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# --------------------------------------------------------------------------- #
# helpers (numpy, independent of the oracle's C code)                          #
# --------------------------------------------------------------------------- #
def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float64 -> float32 -> bf16 (RNE) and return uint16 bits."""
    f = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    r = ((f >> 16) & 1) + 0x7FFF
    return ((f + r) >> 16).astype(np.uint16)


def bf16_val(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def np_swiglu(x, w1, w3, w2):
    """Dense SwiGLU with numpy matmuls: W2 (SiLU(W1 x) * (W3 x)), row-batched."""
    a = x @ w1.T
    b = x @ w3.T
    return ((a / (1.0 + np.exp(-a))) * b) @ w2.T


def rand_problem(rng, T, d, E, k, M, Ms=0, x_std=1.0, w_std=0.3):
    x = bf16_bits(rng.standard_normal((T, d)) * x_std)
    wr = bf16_bits(rng.standard_normal((E, d)) * w_std)
    w1 = bf16_bits(rng.standard_normal((E, M, d)) * w_std)
    w3 = bf16_bits(rng.standard_normal((E, M, d)) * w_std)
    w2 = bf16_bits(rng.standard_normal((E, d, M)) * w_std)
    sh = (None, None, None)
    if Ms:
        sh = (bf16_bits(rng.standard_normal((Ms, d)) * w_std),
              bf16_bits(rng.standard_normal((Ms, d)) * w_std),
              bf16_bits(rng.standard_normal((d, Ms)) * w_std))
    return x, wr, w1, w3, w2, sh


def _close(a, b, tol, what):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    err = np.max(np.abs(a - b)) if a.size else 0.0
    assert err <= tol, f"{what}: max abs err {err} > {tol}"


# --------------------------------------------------------------------------- #
# hand-worked example                                                          #
# --------------------------------------------------------------------------- #
def _hand():
    with open(os.path.join(GOLDEN, "hand_2tok_4exp.json")) as fh:
        return json.load(fh)


def _hand_weights():
    I = np.eye(4)
    w1 = np.stack([I] * 4)
    w3 = np.stack([I] * 4)
    w2 = np.stack([(e + 1) * I for e in range(4)])
    return bf16_bits(w1), bf16_bits(w3), bf16_bits(w2), bf16_bits(I)


def pin_hand_routing(lib):
    g = _hand()
    ex = g["expect"]
    x = bf16_bits(np.array(g["x"], np.float64))
    w1, w3, w2, I = _hand_weights()
    res = oracle.layer_forward(x, I, w1, w3, w2, g["k"], lam=g["lambda"], lib=lib)
    r = res.routing
    _close(r.p, ex["p"], 1e-14, "p")
    _close(r.lse, ex["lse"], 1e-14, "lse")
    assert r.ids.tolist() == ex["ids"], f"ids {r.ids.tolist()}"
    _close(r.gates, ex["gates"], 1e-14, "gates")
    assert res.disp.counts.tolist() == ex["counts"]
    _close(res.loss.f, ex["f"], 1e-15, "f")
    _close(res.loss.P, ex["P"], 1e-14, "P")
    _close(res.loss.L_bal, ex["L_bal"], 1e-15, "L_bal")
    _close(res.loss.L_z, ex["L_z"], 1e-13, "L_z")
    assert res.disp.offsets.tolist() == ex["dropless_offsets"]
    assert res.disp.slot_row.tolist() == ex["dropless_slot_row"]
    assert res.disp.row_token.tolist() == ex["dropless_row_token"]
    _close(res.y, ex["y_dropless"], 1e-10, "y dropless")


def pin_hand_capacity(lib):
    g = _hand()
    ex = g["expect"]
    x = bf16_bits(np.array(g["x"], np.float64))
    w1, w3, w2, I = _hand_weights()
    assert oracle.capacity(ex["capacity_c"], 2, 2, 4, lib=lib) == ex["capacity_C"]
    res = oracle.layer_forward(x, I, w1, w3, w2, g["k"], capacity_factor=ex["capacity_c"],
                               lib=lib)
    assert res.disp.dropped.tolist() == ex["capacity_dropped"]
    assert res.disp.offsets.tolist() == ex["capacity_offsets"]
    assert res.disp.slot_row.tolist() == ex["capacity_slot_row"]
    assert res.disp.row_token.tolist() == ex["capacity_row_token"]
    # f counts routing decisions, before the capacity cut
    assert res.disp.counts.tolist() == ex["counts"]
    _close(res.y, ex["y_capacity"], 1e-10, "y capacity")


def pin_hand_shared_k0(lib):
    g = _hand()
    ex = g["expect"]
    x = bf16_bits(np.array(g["x"], np.float64))
    w1, w3, w2, I = _hand_weights()
    res = oracle.layer_forward(x, I, w1, w3, w2, 0, ws1=I, ws3=I, ws2=I, lib=lib)
    _close(res.y, ex["y_shared_only_k0"], 1e-10, "y shared only")
    s = ex["silu"]
    for z in (1.0, 2.0, -1.0):
        xr = bf16_bits(np.array([z]))
        one = bf16_bits(np.ones((1, 1)))
        _close(oracle.swiglu_row(xr, one, one, one, lib=lib)[0], s[str(int(z))] * z, 1e-15,
               f"SiLU({z})*{z}")


# --------------------------------------------------------------------------- #
# independent formulas / brute force                                           #
# --------------------------------------------------------------------------- #
def pin_two_gating_formulas(lib):
    rng = np.random.default_rng(11)
    for (T, E, k) in [(50, 8, 2), (40, 16, 4), (30, 5, 5), (20, 64, 6)]:
        logits = rng.standard_normal((T, E)) * 2.0
        r = oracle.route(logits, k, lib=lib)
        for t in range(T):
            order = np.argsort(-logits[t], kind="stable")[:k]     # TopK on logits
            l_s = logits[t, order]
            gB = np.exp(l_s - l_s.max()) / np.exp(l_s - l_s.max()).sum()
            assert r.ids[t].tolist() == order.tolist(), (t, r.ids[t], order)
            _close(r.gates[t], gB, 1e-12, "Softmax(TopK(logits))")
            _close(r.gates[t].sum(), 1.0, 1e-12, "gate sum")


def pin_bruteforce_subsets(lib):
    rng = np.random.default_rng(5)
    for (T, d, E, k, M) in [(12, 8, 6, 2, 4), (10, 8, 8, 3, 4), (8, 16, 10, 4, 8),
                            (6, 8, 4, 4, 4), (9, 8, 7, 1, 4)]:
        x, wr, w1, w3, w2, _ = rand_problem(rng, T, d, E, k, M)
        bias = (rng.uniform(-0.05, 0.05, E)).astype(np.float32)
        # make two biases equal so bias ties are exercised
        bias[1] = bias[0]
        res = oracle.layer_forward(x, wr, w1, w3, w2, k, sel_bias=bias, lib=lib)
        xv = bf16_val(x)
        lg = xv @ bf16_val(wr).T
        p = np.exp(lg - lg.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        key = p + bias.astype(np.float64)
        for t in range(T):
            best, best_sum = None, -np.inf
            for comb in itertools.combinations(range(E), k):   # lexicographic order
                s = key[t, list(comb)].sum()
                if s > best_sum + 1e-15:
                    best, best_sum = comb, s
            assert sorted(res.routing.ids[t].tolist()) == list(best), (t, res.routing.ids[t],
                                                                      best)
            ks = key[t, res.routing.ids[t]]
            assert np.all(np.diff(ks) <= 1e-15), "ids not in descending key order"
            g = p[t, list(res.routing.ids[t])] / p[t, list(res.routing.ids[t])].sum()
            _close(res.routing.gates[t], g, 1e-12, "gates from unbiased p")
            y = np.zeros(d)
            for s, e in enumerate(res.routing.ids[t]):
                y += g[s] * np_swiglu(xv[t:t + 1], bf16_val(w1[e]), bf16_val(w3[e]),
                                      bf16_val(w2[e]))[0]
            _close(res.y[t], y, 1e-10 * max(1.0, np.abs(y).max()), "y brute force")


def pin_dispatch_argsort(lib):
    rng = np.random.default_rng(7)
    for (T, E, k, c) in [(100, 8, 2, 0.0), (257, 16, 3, 0.0), (300, 8, 2, 1.0),
                         (129, 4, 1, 1.3), (64, 32, 6, 0.5), (50, 5, 5, 0.7)]:
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
        for t in range(T // 3):        # skew: a third of the tokens pick expert 0 first
            ids[t] = np.concatenate([[0], rng.choice(np.arange(1, E), k - 1, replace=False)])
        C = oracle.capacity(c, k, T, E, lib=lib)
        disp = oracle.dispatch(ids, E, C, lib=lib)
        flat = ids.reshape(-1)
        assert disp.counts.tolist() == np.bincount(flat, minlength=E).tolist()
        # capacity: rank of each pair among earlier pairs (token-major) of its expert
        rank = np.zeros_like(flat)
        for e in range(E):
            pos = np.nonzero(flat == e)[0]
            rank[pos] = np.arange(len(pos))
        kept = (rank < C) if C >= 0 else np.ones_like(flat, bool)
        assert disp.dropped.reshape(-1).tolist() == (~kept).astype(np.uint8).tolist()
        # permutation: stable argsort by expert over the kept pairs
        kept_pairs = np.nonzero(kept)[0]
        order = kept_pairs[np.argsort(flat[kept_pairs], kind="stable")]
        assert disp.row_token.tolist() == (order // k).tolist()
        sr = np.full(T * k, -1)
        sr[order] = np.arange(len(order))
        assert disp.slot_row.reshape(-1).tolist() == sr.tolist()
        kc = np.bincount(flat[kept_pairs], minlength=E)
        assert disp.offsets.tolist() == [0] + np.cumsum(kc).tolist()
        if C >= 0:
            assert kc.max(initial=0) <= C and disp.offsets[-1] <= min(T * k, E * C)


def pin_capacity_formula(lib):
    # ceil(c k T / E), MoE：条件计算与路由 §3
    cases = [((1.0, 1, 3, 2), 2), ((1.25, 1, 32768, 128), 320), ((0.5, 2, 2, 4), 1),
             ((1.0, 2, 10, 4), 5), ((1.1, 1, 10, 4), 3), ((2.0, 6, 8192, 160), 615),
             ((0.0, 2, 10, 4), -1), ((-1.0, 1, 10, 4), -1)]
    for args, want in cases:
        assert oracle.capacity(*args, lib=lib) == want, (args, want)


# --------------------------------------------------------------------------- #
# closed forms and invariants                                                  #
# --------------------------------------------------------------------------- #
def pin_invariants(lib):
    rng = np.random.default_rng(3)
    T, d, E, k, M, Ms = 70, 16, 8, 3, 8, 16
    x, wr, w1, w3, w2, (s1, s3, s2) = rand_problem(rng, T, d, E, k, M, Ms)
    off = rng.standard_normal(E).astype(np.float32)
    res = oracle.layer_forward(x, wr, w1, w3, w2, k, offset=off, ws1=s1, ws3=s3, ws2=s2,
                               lib=lib)
    r, ls = res.routing, res.loss
    _close(r.gates.sum(1), np.ones(T), 1e-12, "gates sum to 1")
    _close(r.p.sum(1), np.ones(T), 1e-12, "softmax sums to 1")
    _close(ls.f.sum(), 1.0, 1e-12, "sum f")
    _close(ls.P.sum(), 1.0, 1e-12, "sum P")
    assert int(res.disp.counts.sum()) == k * T
    lg = bf16_val(x) @ bf16_val(wr).T + off.astype(np.float64)
    _close(r.lse, logsumexp(lg, axis=1), 1e-12, "lse")
    _close(ls.L_z, np.mean(logsumexp(lg, axis=1) ** 2), 1e-11, "L_z = mean lse^2")
    # L_bal against its definition with independently counted f and P
    f = np.bincount(r.ids.reshape(-1), minlength=E) / (k * T)
    P = np.exp(lg - logsumexp(lg, axis=1, keepdims=True)).mean(0)
    _close(ls.L_bal, 0.01 * E * float((f * P).sum()), 1e-14, "L_bal")

    # uniform logits (zero router) -> P = 1/E -> L_bal = lambda
    wr0 = np.zeros_like(wr)
    res0 = oracle.layer_forward(x, wr0, w1, w3, w2, k, lam=0.01, lib=lib)
    _close(res0.loss.L_bal, 0.01, 1e-15, "uniform routing L_bal = lambda")
    _close(res0.loss.L_z, np.log(E) ** 2, 1e-12, "uniform routing L_z = (ln E)^2")

    # k = 0: shared experts only, and zero without them
    resk0 = oracle.layer_forward(x, wr, w1, w3, w2, 0, ws1=s1, ws3=s3, ws2=s2, lib=lib)
    ys = np_swiglu(bf16_val(x), bf16_val(s1), bf16_val(s3), bf16_val(s2))
    _close(resk0.y, ys, 1e-10 * np.abs(ys).max(), "k=0 shared only")
    resk00 = oracle.layer_forward(x, wr, w1, w3, w2, 0, lib=lib)
    assert np.all(resk00.y == 0.0)

    # routed part + shared part
    res_ns = oracle.layer_forward(x, wr, w1, w3, w2, k, offset=off, lib=lib)
    _close(res.y, res_ns.y + ys, 1e-10 * np.abs(res.y).max(), "shared added with gate 1")

    # c -> infinity equals dropless
    resbig = oracle.layer_forward(x, wr, w1, w3, w2, k, offset=off, ws1=s1, ws3=s3, ws2=s2,
                                  capacity_factor=1e6, lib=lib)
    assert not resbig.disp.dropped.any()
    np.testing.assert_array_equal(resbig.y, res.y)

    # E = 1, k = 1: the dense SwiGLU FFN
    res1 = oracle.layer_forward(x, wr[:1], w1[:1], w3[:1], w2[:1], 1, lib=lib)
    yd = np_swiglu(bf16_val(x), bf16_val(w1[0]), bf16_val(w3[0]), bf16_val(w2[0]))
    _close(res1.y, yd, 1e-10 * np.abs(yd).max(), "E=1 dense FFN")
    _close(res1.routing.gates, np.ones((T, 1)), 0.0, "E=1 gate")

    # k = E: dense soft mixture sum_e p_e E_e(x)
    resE = oracle.layer_forward(x, wr, w1, w3, w2, E, offset=off, lib=lib)
    pd = np.exp(lg - logsumexp(lg, axis=1, keepdims=True))
    ymix = sum(pd[:, e:e + 1] * np_swiglu(bf16_val(x), bf16_val(w1[e]), bf16_val(w3[e]),
                                          bf16_val(w2[e])) for e in range(E))
    _close(resE.y, ymix, 1e-10 * np.abs(ymix).max(), "k=E soft mixture")

    # token permutation equivariance (dropless)
    perm = rng.permutation(T)
    resp = oracle.layer_forward(x[perm], wr, w1, w3, w2, k, offset=off, ws1=s1, ws3=s3,
                                ws2=s2, lib=lib)
    np.testing.assert_array_equal(resp.routing.ids, res.routing.ids[perm])
    _close(resp.y, res.y[perm], 1e-12 * np.abs(res.y).max(), "permutation equivariance")


def pin_determinism(lib):
    rng = np.random.default_rng(9)
    x, wr, w1, w3, w2, _ = rand_problem(rng, 40, 16, 8, 2, 8)
    a = oracle.layer_forward(x, wr, w1, w3, w2, 2, capacity_factor=0.8, lib=lib)
    b = oracle.layer_forward(x, wr, w1, w3, w2, 2, capacity_factor=0.8, lib=lib)
    np.testing.assert_array_equal(a.y, b.y)
    np.testing.assert_array_equal(a.routing.ids, b.routing.ids)
    np.testing.assert_array_equal(a.disp.slot_row, b.disp.slot_row)


def pin_gap_and_force(lib):
    """gap = key_k - key_{k+1}; forcing a token's ids recomputes its gates."""
    logits = np.array([[3.0, 1.0, 1.0 + 1e-9, 0.0], [0.0, 0.0, 0.0, 0.0]])
    r = oracle.route(logits, 2, lib=lib)
    pe = np.exp(logits[0] - logits[0].max())
    pe /= pe.sum()
    _close(r.gap[0], pe[2] - pe[1], 1e-15, "gap")
    assert r.ids[0].tolist() == [0, 2]
    assert r.gap[1] == 0.0 and r.ids[1].tolist() == [0, 1]
    f = oracle.route(logits, 2, force_ids=np.array([[0, 1], [3, 2]]),
                     force_mask=np.array([1, 0]), lib=lib)
    assert f.ids.tolist() == [[0, 1], [0, 1]]
    _close(f.gates[0], [pe[0] / (pe[0] + pe[1]), pe[1] / (pe[0] + pe[1])], 1e-15, "forced")


def pin_combine(lib):
    """The standalone combine against the layer's own composition and a
    hand-sized case: a dropped slot adds nothing, gates are not renormalised."""
    yp = bf16_bits(np.array([[1.0, 2.0], [3.0, -4.0], [0.5, 0.25]]))
    sr = np.array([[0, 1], [2, -1]], np.int32)
    g = np.array([[0.75, 0.25], [0.5, 0.5]])
    ys = bf16_bits(np.array([[10.0, 20.0], [30.0, 40.0]]))
    y = oracle.combine(yp, sr, g, ys, lib=lib)
    _close(y, [[0.75 * 1 + 0.25 * 3 + 10, 0.75 * 2 - 0.25 * 4 + 20], [0.25 + 30, 0.125 + 40]],
           1e-15, "combine")
    # the layer's y equals combine over the oracle's own expert rows
    rng = np.random.default_rng(13)
    T, d, E, k, M = 30, 8, 5, 2, 4
    x, wr, w1, w3, w2, _ = rand_problem(rng, T, d, E, k, M)
    res = oracle.layer_forward(x, wr, w1, w3, w2, k, capacity_factor=0.6, lib=lib)
    R = len(res.disp.row_token)
    exp_rows = np.zeros((R, d))
    for t in range(T):
        for s in range(k):
            r = res.disp.slot_row[t, s]
            if r >= 0:
                e = res.routing.ids[t, s]
                exp_rows[r] = np_swiglu(bf16_val(x[t:t + 1]), bf16_val(w1[e]), bf16_val(w3[e]),
                                        bf16_val(w2[e]))[0]
    # combine on exactly-representable rows: compare the two paths on bf16 rows
    rows_b = bf16_bits(exp_rows)
    yc = oracle.combine(rows_b, res.disp.slot_row, res.routing.gates, lib=lib)
    want = np.zeros((T, d))
    for t in range(T):
        for s in range(k):
            r = res.disp.slot_row[t, s]
            if r >= 0:
                want[t] += res.routing.gates[t, s] * bf16_val(rows_b[r])
    _close(yc, want, 1e-12, "combine vs explicit sum")
    _close(yc, res.y, 2e-2 * np.abs(res.y).max(), "combine vs layer")


def pin_routing_variants(lib):
    """Sigmoid scores and un-renormalised gates on a hand-worked token
    (CSDN note §9; "MoE：条件计算与路由" §7), with closed-form values."""
    sig2, sig1 = 0.8807970779778823, 0.7310585786300049
    logits = np.array([[2.0, 1.0, 0.0, -1.0]])
    r = oracle.route(logits, 2, flags=oracle.SIGMOID, lib=lib)
    assert r.ids.tolist() == [[0, 1]]
    _close(r.p[0], [sig2, sig1, 0.5, 1.0 - sig1], 1e-15, "sigmoid scores")
    _close(r.gates[0], [sig2 / (sig2 + sig1), sig1 / (sig2 + sig1)], 1e-15, "sigmoid renorm")
    r = oracle.route(logits, 2, flags=oracle.SIGMOID | oracle.NO_RENORM, lib=lib)
    _close(r.gates[0], [sig2, sig1], 1e-15, "sigmoid raw gates")
    r = oracle.route(logits, 2, flags=oracle.NO_RENORM, lib=lib)
    g = _hand()["expect"]["p"][0]
    _close(r.gates[0], g[:2], 1e-15, "softmax raw gates")
    _close(r.lse, oracle.route(logits, 2, lib=lib).lse, 0.0, "lse independent of the scores")
    # un-renormalised softmax gates with k = E: the same soft mixture (they sum to 1)
    rng = np.random.default_rng(21)
    x, wr, w1, w3, w2, _ = rand_problem(rng, 20, 8, 4, 4, 4)
    a = oracle.layer_forward(x, wr, w1, w3, w2, 4, lib=lib)
    b = oracle.layer_forward(x, wr, w1, w3, w2, 4, flags=oracle.NO_RENORM, lib=lib)
    _close(a.y, b.y, 1e-12 * np.abs(a.y).max(), "k=E renorm or not")
    # sigmoid routing selects the largest logits (sigmoid is increasing)
    lg = rng.standard_normal((30, 9))
    rs = oracle.route(lg, 3, flags=oracle.SIGMOID, lib=lib)
    assert rs.ids.tolist() == np.argsort(-lg, axis=1, kind="stable")[:, :3].tolist()


def pin_entropy_and_importance(lib):
    """Router entropy ("MoE：条件计算与路由" §9) and the importance CV^2 (CSDN
    note, balancing expert utilization) against closed forms and scipy."""
    from scipy.stats import entropy as sp_entropy
    r = oracle.route(np.array([[0.0, np.log(3.0)], [1.0, 1.0]]), 1, lib=lib)
    _close(r.entropy, [0.5623351446188083, np.log(2.0)], 1e-14, "entropy closed forms")
    rng = np.random.default_rng(22)
    lg = rng.standard_normal((25, 12)) * 2
    r = oracle.route(lg, 3, lib=lib)
    _close(r.entropy, sp_entropy(r.p, axis=1), 1e-12, "entropy vs scipy")
    rs = oracle.route(lg, 3, flags=oracle.SIGMOID, lib=lib)
    q = rs.p / rs.p.sum(1, keepdims=True)
    _close(rs.entropy, sp_entropy(q, axis=1), 1e-12, "sigmoid entropy vs scipy")
    imp, cv2 = oracle.importance(np.array([[0, 1], [2, 0]]), np.array([[0.75, 0.25], [0.5, 0.5]]),
                                 4, lib=lib)
    _close(imp, [1.25, 0.25, 0.5, 0.0], 1e-15, "importance")
    _close(cv2, 0.875, 1e-15, "importance CV^2")
    imp, cv2 = oracle.importance(np.array([[0, 1], [1, 0]]), np.full((2, 2), 0.5), 2, lib=lib)
    assert cv2 == 0.0


def pin_alf_bias_update(lib):
    """ALF-LB: overloaded experts' bias goes down, underloaded up, balanced
    unchanged (hand case); iterating the update on fixed logits with a strong
    skew reduces the load imbalance (a wrong sign makes it grow)."""
    b = oracle.alf_bias_update([5, 3, 4, 0], T=8, k=2, gamma=0.25,
                               bias=np.array([0.0, 0.5, -0.5, 1.0], np.float32), lib=lib)
    assert b.tolist() == [-0.25, 0.75, -0.5, 1.25]          # nbar = 4
    rng = np.random.default_rng(31)
    T, E, k = 512, 16, 2
    logits = rng.standard_normal((T, E)) + np.linspace(2.0, -2.0, E)[None, :]
    bias = np.zeros(E, np.float32)
    first = None
    for _ in range(300):
        r = oracle.route(logits, k, bias, lib=lib)
        n = np.bincount(r.ids.reshape(-1), minlength=E)
        spread = n.max() / (k * T / E)
        first = spread if first is None else first
        bias = oracle.alf_bias_update(n, T, k, 0.002, bias, lib=lib)
    assert first > 3.0 and spread < 1.5, (first, spread)


# --------------------------------------------------------------------------- #
# probability-priority capacity and expert-choice routing                      #
# --------------------------------------------------------------------------- #
def _sig(z):
    return 1.0 / (1.0 + np.exp(-z))


def pin_priority_capacity(lib):
    """Capacity that keeps each expert's highest-score pairs (aiattnstudio
    §4.2.2).  Hand case from closed forms: with W_r = I and x = [1,0,0,0],
    [3,0,0,0], [2,0,0,0] every token picks expert 0 with p = e^z/(e^z+3); C = 2
    keeps tokens 1 and 2 (token order would keep 0 and 1); their rows stay in
    token order.  Random cases against a numpy lexsort cut; equal scores reduce
    to the token-order dispatch; a capacity above every load is dropless."""
    w1, w3, w2, I = _hand_weights()
    x = bf16_bits(np.array([[1, 0, 0, 0], [3, 0, 0, 0], [2, 0, 0, 0]], np.float64))
    assert oracle.capacity(2.0, 1, 3, 4, lib=lib) == 2
    res = oracle.layer_forward(x, I, w1, w3, w2, 1, capacity_factor=2.0,
                               flags=oracle.PRIORITY, lib=lib)
    e = np.e
    _close(res.routing.p[:, 0], [e / (e + 3), e ** 3 / (e ** 3 + 3), e ** 2 / (e ** 2 + 3)],
           1e-14, "hand p")
    assert res.disp.dropped.reshape(-1).tolist() == [1, 0, 0]
    assert res.disp.slot_row.reshape(-1).tolist() == [-1, 0, 1]
    assert res.disp.row_token.tolist() == [1, 2]
    assert res.disp.counts.tolist() == [3, 0, 0, 0]
    # y: dropped token 0 gets nothing; E_0(x)_o = SiLU(x_o) x_o = x_o^2 sigmoid(x_o)
    _close(res.y, [[0, 0, 0, 0], [9 * _sig(3.0), 0, 0, 0], [4 * _sig(2.0), 0, 0, 0]], 1e-12,
           "hand y")
    tok = oracle.layer_forward(x, I, w1, w3, w2, 1, capacity_factor=2.0, lib=lib)
    assert tok.disp.dropped.reshape(-1).tolist() == [0, 0, 1]

    rng = np.random.default_rng(41)
    for (T, E, k, c) in [(200, 8, 2, 0.5), (129, 4, 1, 1.0), (300, 16, 4, 0.8),
                         (64, 32, 6, 0.3), (50, 5, 5, 0.7)]:
        lg = rng.standard_normal((T, E)) * 1.5
        lg[:, 0] += 1.0                                  # overload expert 0
        r = oracle.route(lg, k, lib=lib)
        C = oracle.capacity(c, k, T, E, lib=lib)
        disp = oracle.dispatch_priority(r.ids, r.p, E, C, lib=lib)
        flat = r.ids.reshape(-1)
        score = r.p[np.repeat(np.arange(T), k), flat]
        q = np.arange(T * k)
        kept = np.zeros(T * k, bool)
        for ee in range(E):
            pos = q[flat == ee]
            order = pos[np.lexsort((pos, -score[pos]))]  # score desc, then (t, s)
            kept[order[:C]] = True
            if len(pos) > C:
                assert score[order[:C]].min() >= score[order[C:]].max()
        assert disp.dropped.reshape(-1).tolist() == (~kept).astype(np.uint8).tolist()
        kp = q[kept]
        order = kp[np.argsort(flat[kp], kind="stable")]
        assert disp.row_token.tolist() == (order // k).tolist()
        sr = np.full(T * k, -1)
        sr[order] = np.arange(len(order))
        assert disp.slot_row.reshape(-1).tolist() == sr.tolist()
        assert disp.counts.tolist() == np.bincount(flat, minlength=E).tolist()
        assert disp.kept_counts.tolist() == np.minimum(disp.counts, C).tolist()
        # equal scores: the cut falls back to token order
        eq = oracle.dispatch_priority(r.ids, np.full((T, E), 0.25), E, C, lib=lib)
        ref = oracle.dispatch(r.ids, E, C, lib=lib)
        for f in ("dropped", "slot_row", "row_token", "offsets"):
            assert getattr(eq, f).tolist() == getattr(ref, f).tolist(), f
        # no cut when C covers every load
        big = oracle.dispatch_priority(r.ids, r.p, E, T * k, lib=lib)
        assert big.slot_row.tolist() == oracle.dispatch(r.ids, E, -1, lib=lib).slot_row.tolist()
        # forcing: zeros change nothing; +1 on expert 0's lowest-score pair keeps
        # it and drops the lowest of its kept pairs instead
        f0 = oracle.dispatch_priority(r.ids, r.p, E, C, force=np.zeros((T, k), np.int8), lib=lib)
        assert f0.slot_row.tolist() == disp.slot_row.tolist()
        pos = q[flat == 0]
        if len(pos) > C > 0:
            order = pos[np.lexsort((pos, -score[pos]))]
            force = np.zeros(T * k, np.int8)
            force[order[-1]] = 1
            fd = oracle.dispatch_priority(r.ids, r.p, E, C, force=force.reshape(T, k), lib=lib)
            fdr = fd.dropped.reshape(-1)
            assert fdr[order[-1]] == 0 and fdr[order[C - 1]] == 1
            assert fd.kept_counts[0] == C


def pin_expert_choice(lib):
    """Expert-choice routing (aiattnstudio §9.2; routing table of
    "MoE：条件计算与路由").  Hand case from closed forms (W_r = I, d = 2,
    x = [1,0], [0,1], [2,0], [1,0], k = 1, c = 1, so r = ceil(4/2) = 2): expert 0
    scores sigmoid(1), sigmoid(-1), sigmoid(2), sigmoid(1) and takes tokens 2
    and 0 (0 beats its duplicate 3 on the index); expert 1 takes 1 and 0; token
    3 gets nothing.  Random cases against a numpy lexsort; r = T is the dense
    soft mixture, the same output as token choice with k = E."""
    assert oracle.ec_capacity(1.0, 1, 4, 2, lib=lib) == 2
    assert oracle.ec_capacity(0.0, 1, 3, 2, lib=lib) == 2        # c <= 0 reads as c = 1
    assert oracle.ec_capacity(1.0, 2, 4096, 8, lib=lib) == 1024
    assert oracle.ec_capacity(5.0, 2, 10, 4, lib=lib) == 10      # at most T
    assert oracle.ec_capacity(1.25, 1, 32768, 128, lib=lib) == 320
    I2 = bf16_bits(np.eye(2))
    w1 = bf16_bits(np.stack([np.eye(2)] * 2))
    w2 = bf16_bits(np.stack([(e + 1) * np.eye(2) for e in range(2)]))
    x = bf16_bits(np.array([[1, 0], [0, 1], [2, 0], [1, 0]], np.float64))
    res = oracle.ec_layer_forward(x, I2, w1, w1, w2, 1, capacity_factor=1.0, lib=lib)
    s1, s2, sm1 = _sig(1.0), _sig(2.0), _sig(-1.0)
    assert res.ec.r == 2
    assert res.ec.row_token.tolist() == [0, 2, 0, 1]
    _close(res.ec.row_gate, [s1, s2, sm1, s1], 1e-14, "EC gates")
    # E_e(x)_o = (e+1) x_o^2 sigmoid(x_o)
    _close(res.y, [[s1 * s1 + sm1 * 2 * s1, 0], [0, s1 * 2 * s1], [s2 * 4 * s2, 0], [0, 0]],
           1e-12, "EC hand y")
    # one shared expert of width 2 (W1s = W3s = W2s = I) adds x_o^2 sigmoid(x_o) to
    # every token, also to token 3, which no expert picked
    sh = oracle.ec_layer_forward(x, I2, w1, w1, w2, 1, ws1=I2, ws3=I2, ws2=I2,
                                 capacity_factor=1.0, lib=lib)
    _close(sh.y - res.y, [[s1, 0], [0, s1], [4 * s2, 0], [s1, 0]], 1e-12, "EC shared expert")
    _close(res.loss.f, [0.5, 0.5], 1e-15, "EC f")
    _close(res.loss.L_bal, 0.01, 1e-15, "EC L_bal = lambda")

    rng = np.random.default_rng(43)
    for (T, d, E, k, M, c) in [(40, 8, 6, 2, 4, 1.0), (33, 8, 4, 1, 4, 0.5),
                               (25, 16, 8, 3, 8, 2.0)]:
        xx, wr, w1, w3, w2, _ = rand_problem(rng, T, d, E, k, M)
        res = oracle.ec_layer_forward(xx, wr, w1, w3, w2, k, capacity_factor=c, lib=lib)
        xv = bf16_val(xx)
        lg = xv @ bf16_val(wr).T
        p = np.exp(lg - lg.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        r = min(T, int(np.ceil(c * k * T / E)))
        assert res.ec.r == r
        y = np.zeros((T, d))
        for e in range(E):
            pick = np.sort(np.lexsort((np.arange(T), -p[:, e]))[:r])
            assert res.ec.row_token[e * r:(e + 1) * r].tolist() == pick.tolist()
            _close(res.ec.row_gate[e * r:(e + 1) * r], p[pick, e], 1e-12, "EC gate = p")
            y[pick] += p[pick, e][:, None] * np_swiglu(xv[pick], bf16_val(w1[e]),
                                                       bf16_val(w3[e]), bf16_val(w2[e]))
        _close(res.y, y, 1e-10 * max(1.0, np.abs(y).max()), "EC y vs numpy")
        # forcing expert 0's lowest-score token in swaps it for its r-th pick;
        # gates stay the scores
        if 0 < r < T:
            force = np.zeros((E, T), np.int8)
            low = int(np.lexsort((np.arange(T), -p[:, 0]))[-1])
            force[0, low] = 1
            fe = oracle.expert_choice(res.routing.p, r, force=force, lib=lib)
            pick = np.sort(np.lexsort((np.arange(T), -p[:, 0]))[:r - 1].tolist() + [low])
            assert fe.row_token[:r].tolist() == pick.tolist()
            _close(fe.row_gate[:r], p[pick, 0], 1e-12, "forced EC gate")
    # every expert takes every token: the dense soft mixture
    T, d, E, M = 12, 8, 4, 4
    xx, wr, w1, w3, w2, _ = rand_problem(rng, T, d, E, E, M)
    ec = oracle.ec_layer_forward(xx, wr, w1, w3, w2, E, capacity_factor=float(E), lib=lib)
    assert ec.ec.r == T
    tc = oracle.layer_forward(xx, wr, w1, w3, w2, E, lib=lib)
    _close(ec.y, tc.y, 1e-12, "EC with r = T vs token choice k = E")


def pin_expert_rows(lib):
    """oracle_expert_rows: each row goes through its own expert ("深入理解 MoE"
    §10.2, the SwiGLU expert W2 (SiLU(W1 x) * W3 x)).
    Hand case: W1 = W3 = I and W2_e = (e + 1) I give E_e(x)_i = (e + 1) x_i
    SiLU(x_i), with SiLU(1), SiLU(2), SiLU(-1) from the closed form; random
    case: experts with different weights, d != M, each row against a numpy
    SwiGLU with that row's expert."""
    w1, w3, w2, _ = _hand_weights()
    x = bf16_bits(np.array([[1.0, 2.0, -1.0, 0.0]] * 4))
    expert = np.array([2, 0, 3, 1], np.int32)
    got = oracle.expert_rows(x, expert, w1, w3, w2, lib=lib)
    s1, s2, sm1 = 1 / (1 + np.exp(-1.0)), 2 / (1 + np.exp(-2.0)), -1 / (1 + np.exp(1.0))
    base = np.array([1.0 * s1, 2.0 * s2, -1.0 * sm1, 0.0])
    _close(got, (expert[:, None] + 1.0) * base[None, :], 1e-12, "expert rows, hand case")
    rng = np.random.default_rng(77)
    n, d, M, E = 9, 12, 8, 4
    xr = bf16_bits(rng.standard_normal((n, d)))
    ww1 = bf16_bits(rng.standard_normal((E, M, d)) * 0.4)
    ww3 = bf16_bits(rng.standard_normal((E, M, d)) * 0.4)
    ww2 = bf16_bits(rng.standard_normal((E, d, M)) * 0.4)
    ex = np.array([3, 0, 1, 2, 2, 0, 3, 1, 3], np.int32)
    got = oracle.expert_rows(xr, ex, ww1, ww3, ww2, lib=lib)
    for r in range(n):
        e = ex[r]
        want = np_swiglu(bf16_val(xr[r:r + 1]), bf16_val(ww1[e]), bf16_val(ww3[e]),
                         bf16_val(ww2[e]))[0]
        _close(got[r], want, 1e-12 * max(1.0, np.abs(want).max()), f"expert row {r} (expert {e})")


ALL_PINS = [pin_expert_rows, pin_priority_capacity, pin_expert_choice, pin_alf_bias_update, pin_routing_variants, pin_entropy_and_importance, pin_combine, pin_hand_routing, pin_hand_capacity, pin_hand_shared_k0, pin_two_gating_formulas,
            pin_bruteforce_subsets, pin_dispatch_argsort, pin_capacity_formula, pin_invariants,
            pin_determinism, pin_gap_and_force]

"""Write the calibrated per-expert logit offsets of the Zipf-skewed workloads.

"Zipf(s)-skewed routing via logit offsets" is read as: the realised expert
loads n_e (routing decisions, before any capacity cut) follow Zipf(s) over a
seeded rank order of the experts.  Literal offsets -s ln(rank) concentrate
top-k routing far more than that, so the offsets are calibrated on the seeded
tokens of the workload:

  targets  t_r proportional to r^-s (r = rank of the expert), water-filled so
           that no expert exceeds T pairs, scaled to k T in total;
  start    o_e = -s ln(rank_e);
  repeat   300 times:  o_e += clip(0.1 (ln t_e - ln max(n_e, 0.5)), -0.05, 0.05),
           with n_e counted by the oracle's routing (softmax, selection bias,
           Top-k) of logits W_r x + o.  (A larger, unclipped gain oscillates.)

Where a selection bias is present (the DeepSeek-V2-shaped workload, b_e drawn
from U(-0.1, 0.1)) the bias dominates softmax probabilities spread over 160
experts, so the highest-bias experts are picked by almost every token whatever
their offset; Zipf loads are then out of reach and the stored vector is the
iteration's fixed point, whose loads are reported in the file header.

The result is stored as plain text (one fp32 value per line, expert order) and
read back by ``synth.zipf_offsets``; both sides of every check take it as an
input.  This script calls only the oracle and the input generator.

Usage:  python tests/golden/calibrate_zipf_offsets.py [workload ...]
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth   # noqa: E402


def water_filled_targets(rank: np.ndarray, s: float, total: float, cap: float) -> np.ndarray:
    w = rank.astype(np.float64) ** (-s)
    lo, hi = 0.0, total / w.min() + 1.0
    for _ in range(200):                      # bisection on the scale
        mid = 0.5 * (lo + hi)
        if np.minimum(mid * w, cap).sum() > total:
            hi = mid
        else:
            lo = mid
    return np.minimum(lo * w, cap)


def calibrate(name: str, iters: int = 300, verbose: bool = True):
    w = synth.WORKLOADS[name]
    x = synth.normal_bf16(w.seed, synth.TID_X, (w.T, w.d), w.x_std)
    wr = synth.normal_bf16(w.seed, synth.TID_WR, (w.E, w.d), w.w_std)
    bias = synth.make_sel_bias(w)
    bias_np = None if bias is None else bias.numpy()
    base = oracle.router_logits(synth.to_u16(x), synth.to_u16(wr), None)
    rank = synth.zipf_rank(w.seed, w.E).numpy()
    target = water_filled_targets(rank, w.zipf_s, float(w.k * w.T), float(w.T))
    off = -w.zipf_s * np.log(rank.astype(np.float64))
    for it in range(iters):
        r = oracle.route(base + off.astype(np.float32).astype(np.float64)[None, :], w.k,
                         bias_np)
        n = np.bincount(r.ids.reshape(-1), minlength=w.E).astype(np.float64)
        if it == iters - 1:
            break
        off = off + np.clip(0.1 * (np.log(target) - np.log(np.maximum(n, 0.5))), -0.05, 0.05)
        if verbose and it % 50 == 0:
            rel = np.abs(n - target).sum() / target.sum()
            print(f"{name} iter {it}: L1 load mismatch {rel:.4f}, max n {n.max():.0f}")
    rel = np.abs(n - target).sum() / target.sum()
    if verbose:
        print(f"{name} final: L1 load mismatch {rel:.4f}")
    return off.astype(np.float32), n, target, rel


def main(names):
    for name in names:
        off, n, target, rel = calibrate(name)
        path = synth.zipf_offsets_path(name)
        w = synth.WORKLOADS[name]
        top = ", ".join(str(int(v)) for v in np.sort(n)[::-1][:8])
        ttop = ", ".join(str(int(round(v))) for v in np.sort(target)[::-1][:8])
        with open(path, "w") as fh:
            fh.write(f"# calibrated logit offsets, workload {name}: Zipf(s={w.zipf_s}) "
                     f"realised loads, seed {w.seed}; written by calibrate_zipf_offsets.py\n")
            fh.write(f"# realised loads (largest 8): {top}; targets: {ttop}; "
                     f"L1 mismatch {rel:.4f}; empty experts {int((n == 0).sum())}\n")
            for v in off:
                fh.write(f"{float(v):.9g}\n")
        print("wrote", path)


if __name__ == "__main__":
    main(sys.argv[1:] or [n for n, w in synth.WORKLOADS.items() if w.offsets == "zipf"])

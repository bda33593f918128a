#!/usr/bin/env python
"""Benchmark of the MoE layer forward on B300 (tokens/s; grouped-FFN TFLOP/s
against the bf16 tensor roofline; memory stages against the HBM roofline).

One step = one whole layer forward (router, permute, grouped SwiGLU FFN with
shared experts, combine, losses) over one batch of seeded synthetic tokens,
through the C ABI (moe_layer_forward), each timed step replaying a CUDA graph
of that call (--no-graph: direct calls).  Default workload: the Mixtral-shaped
layer (T=4096, d=4096, E=8, k=2, M=14336, dropless).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle, timed on host cores

Under torchrun (N > 1) every rank runs an independent replica of the workload
(the layer shards by independent batches; there is no data-path exchange);
rank 0 prints one JSON line with the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer fwd tokens/s and grouped-FFN TFLOP/s (% bf16 roofline), 1×B300"
FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mixtral")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--clocks-dir", default=None,
                    help="keep the nvidia-smi clock samples as CSV in this directory")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0,
                    help="target seconds of oracle work for the CPU baseline sample")
    ap.add_argument("--routing", choices=["token", "priority", "expert-choice"],
                    default="token",
                    help="token: token-choice top-k (the headline); priority: capacity "
                         "keeps each expert's highest scores; expert-choice: every expert "
                         "takes its top-r tokens (secondary lines: no e2e or CPU leg)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the other workloads' lines (per_config)")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch every timed step directly instead of replaying CUDA graphs")
    ap.add_argument("--stage", choices=["layer", "router", "ffn", "ab", "dense"], default="layer",
                    help="router: time moe_route alone (no expert weights are drawn); "
                         "ffn: time moe_grouped_ffn on a slice of the workload's realised "
                         "expert loads (--experts of them); ab: two layers that differ only "
                         "in moe_tuning_t (--tune for A, --tune-b for B) called alternately "
                         "--steps times each; dense: the gate/up projection of one expert "
                         "holding --rows rows, on single-CTA and on CTA-pair tiles, called "
                         "alternately with torch's (cuBLAS) GEMM of the same shape; for "
                         "profiling, not the headline")
    ap.add_argument("--rows", type=int, default=8192,
                    help="--stage dense: rows of the one expert")
    ap.add_argument("--experts", type=int, default=0,
                    help="--stage ffn: experts in the slice (0: all)")
    ap.add_argument("--tune", action="append", default=[],
                    help="moe_tuning_t field=value for --stage ffn / ab (repeatable), "
                         "e.g. --tune gemm1_tile=256")
    ap.add_argument("--tune-b", action="append", default=[],
                    help="--stage ab: moe_tuning_t field=value of layer B (repeatable)")
    return ap.parse_args(argv)


def parse_tune(items):
    return {kv.split("=")[0]: int(kv.split("=")[1]) for kv in items}


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes (read + write) per launch of `kernel` from the committed ncu
    summary, or None when the kernel's sources changed since that capture."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
            rec = json.load(fh)[workload]
        if rec["kernel"] != kernel:
            return None
        h = hashlib.sha256()
        for f in rec["kernel_sources"]:
            with open(os.path.join(ROOT, f), "rb") as fh:
                h.update(fh.read())
        return rec["traffic_bytes"] if h.hexdigest() == rec["sources_sha256"] else None
    except Exception:
        return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured (MEASURED_PEAKS.json)"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------------------- #
# algorithmic work                                                             #
# --------------------------------------------------------------------------- #
ROUTING_FLAGS = {"token": 0, "priority": 4, "expert-choice": 8}  # MOE_FLAG_* bits


def algorithmic_work(w, R: int):
    """FLOPs of the two grouped projections and bytes of the memory stages.

    gemm_swiglu: 2 * (R * d * 2M + T * d * 2Ms)   gemm_down: 2 * (R * M * d + T * Ms * d)
    router  bytes: x (T d 2) + W_r (E d 2) + ids/gates (T k 8)
    scatter bytes: x read once (T d 2) + rows written (R d 2) + slot rows/drop mask (T k 5)
                   + row->token (R 4)
    combine bytes: rows read (R d 2) + shared rows (T d 2 if shared) + y (T d 2)
                   + slot rows/gates (T k 8)
    """
    T, d, M, E, k, Ms = w.T, w.d, w.M, w.E, w.k, w.Ms
    f1 = 2.0 * (R * d * 2 * M + T * d * 2 * Ms)
    f2 = 2.0 * (R * M * d + T * Ms * d)
    b_router = T * d * 2 + E * d * 2 + T * k * 8
    b_scatter = T * d * 2 + R * d * 2 + T * k * 5 + R * 4
    b_combine = R * d * 2 + (T * d * 2 if Ms else 0) + T * d * 2 + T * k * 8
    bytes_ = {"router": b_router, "scatter": b_scatter, "combine": b_combine}
    if w.flags & 8:
        # expert choice: the router also writes every score (E T 4); the cut
        # reads them and writes the (expert, token) row map (E T 4) and R rows
        # of token + gate (R 8); the gather reads and writes R rows; the
        # combine reads the row map instead of slot rows
        bytes_["router"] = T * d * 2 + E * d * 2 + E * T * 4
        bytes_["select"] = E * T * 4 + E * T * 4 + R * 8
        bytes_["gather"] = 2 * R * d * 2 + R * 4
        bytes_["combine"] = R * d * 2 + (T * d * 2 if Ms else 0) + T * d * 2 + E * T * 4 + R * 4
        del bytes_["scatter"]
    elif w.flags & 4 and w.capacity_factor > 0:
        # priority capacity: the scatter only stages (pair, score) per expert;
        # the cut reads them and writes slot rows / drop mask / row tokens;
        # the gather moves the kept rows
        bytes_["scatter"] = T * k * 4 + T * k * 16
        bytes_["select"] = T * k * 8 + T * k * 5 + R * 4
        bytes_["gather"] = 2 * R * d * 2 + R * 4
    return {"gemm_swiglu": f1, "gemm_down": f2}, bytes_


def kept_rows_per_expert(layer, w):
    """Rows each expert computed (after capacity), from the layer's outputs."""
    import torch
    if getattr(layer, "expert_choice", False):
        return [layer.r] * w.E
    if w.k == 0:
        return [0] * w.E
    ids = layer.ids.view(-1).long()
    keep = (layer.drop_mask.view(-1) == 0)
    return torch.bincount(ids[keep], minlength=w.E).tolist()


def attainable_ffn_ms(w, kept, peaks):
    """Attainable time of the two expert projections: every expert (and the
    shared group) takes max(its FLOPs at the bf16 peak, its weight bytes at the
    HBM bandwidth); the sum is the bound when experts run back to back."""
    peak = peaks["bf16_tflops"] * 1e12
    bw = peaks["hbm_gbs"] * 1e9
    wbytes = 3 * w.M * w.d * 2
    t = 0.0
    for n in kept:
        if n > 0:
            t += max(6.0 * n * w.d * w.M / peak, wbytes / bw)
    if w.n_shared:
        t += max(6.0 * w.T * w.d * w.Ms / peak, 3 * w.Ms * w.d * 2 / bw)
    return 1000.0 * t


def workload_desc(w):
    cap = f"capacity c={w.capacity_factor}" if w.capacity_factor > 0 else "dropless"
    sh = f", {w.n_shared} shared" if w.n_shared else ""
    rt = {4: ", probability-priority capacity", 8: ", expert-choice routing"}.get(w.flags & 12, "")
    return (f"{w.name}: T={w.T} d={w.d} E={w.E} k={w.k} M={w.M}{sh}, {cap}, "
            f"offsets={w.offsets}, sel_bias={w.sel_bias}{rt}")


# --------------------------------------------------------------------------- #
# clocks                                                                       #
# --------------------------------------------------------------------------- #
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class NvmlPoller:
    """SM clock and power every ~5 ms through NVML (read-only queries) on a
    host thread, so that a timed region of a few hundred ms still gets tens of
    samples; mark() brackets the region of interest."""

    def __init__(self, device_index: int, period_s: float = 0.005):
        import threading
        self.samples = []  # (host time, sm MHz, power W)
        self.window = None
        self.period = period_s
        self.stop = threading.Event()
        self.thread = None
        self.err = None
        self.nv = None
        try:
            # the driver's NVML library through ctypes (read-only queries)
            import ctypes
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit_v2 failed")
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(device_index),
                                                 ctypes.byref(h)) != 0:
                raise RuntimeError("nvmlDeviceGetHandleByIndex_v2 failed")
            self.nv, self.h = lib, h
        except Exception as e:  # reported in the summary
            self.err = f"{type(e).__name__}: {e}"

    def _run(self):
        import ctypes
        nv, h = self.nv, self.h
        clk, mw = ctypes.c_uint(), ctypes.c_uint()
        NVML_CLOCK_SM = 1
        while not self.stop.is_set():
            if (nv.nvmlDeviceGetClockInfo(h, NVML_CLOCK_SM, ctypes.byref(clk)) == 0 and
                    nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw)) == 0):
                self.samples.append((time.perf_counter(), float(clk.value), mw.value / 1000.0))
            else:
                self.err = "NVML query failed"
            time.sleep(self.period)

    def start(self):
        import threading
        if self.nv is not None:
            self.thread = threading.Thread(target=self._run, daemon=True)
            self.thread.start()

    def finish(self):
        self.stop.set()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def in_window(self):
        if not self.window:
            return []
        a, b = self.window
        return [s for s in self.samples if a <= s[0] <= b]


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples (CSV, every 100 ms) plus the
    NVML poller.  The CSV goes to `csv_dir` when given, else to a temporary
    file removed after the summary."""

    def __init__(self, device_index: int, enabled: bool = True, csv_dir=None):
        self.proc = None
        self.enabled = enabled
        self.idx = device_index
        self.path = None
        self.csv_dir = csv_dir
        self.poll = NvmlPoller(device_index) if enabled else None

    def mark_start(self):
        self.t0 = time.perf_counter()

    def mark_end(self):
        if self.poll is not None:
            self.poll.window = (getattr(self, "t0", 0.0), time.perf_counter())

    def __enter__(self):
        if not self.enabled:
            return self
        self.poll.start()
        if self.csv_dir:
            os.makedirs(self.csv_dir, exist_ok=True)
            self.path = os.path.join(self.csv_dir, f"clocks_rank{self.idx}.csv")
        else:
            import tempfile
            fd, self.path = tempfile.mkstemp(prefix="moe_clocks_", suffix=".csv")
            os.close(fd)
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.poll is not None:
            self.poll.finish()
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or self.path is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["not sampled"]}
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        if not self.csv_dir:
            os.remove(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].lower().startswith("active")})
        busy = [s for s in sm if s is not None]
        win = self.window_summary()
        region = win.get("sm_mhz_region_median")
        return {"sm_mhz": region if region is not None else
                (statistics.median(busy) if busy else None),
                "sm_mhz_smi_median": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "samples": len(rows), "reasons": reasons, **win}

    def window_summary(self):
        """Median SM clock and power over NVML samples taken inside the timed
        region only (the nvidia-smi median above also counts idle samples)."""
        if self.poll is None:
            return {}
        win = self.poll.in_window()
        if not win:
            return {"nvml_samples_in_region": 0, "nvml_samples": len(self.poll.samples),
                    "nvml_error": self.poll.err}
        return {"nvml_samples_in_region": len(win),
                "sm_mhz_region_median": statistics.median(s[1] for s in win),
                "sm_mhz_region_min": min(s[1] for s in win),
                "power_w_region_median": statistics.median(s[2] for s in win)}


# --------------------------------------------------------------------------- #
# oracle timing (CPU baseline and the reference arm)                           #
# --------------------------------------------------------------------------- #
def _host_inputs(inp):
    import synth
    u = synth.to_u16
    return dict(x=u(inp.x), wr=u(inp.wr), w1=u(inp.w1), w3=u(inp.w3), w2=u(inp.w2),
                ws1=u(inp.ws1), ws3=u(inp.ws3), ws2=u(inp.ws2),
                off=None if inp.offset is None else inp.offset.cpu().numpy(),
                bias=None if inp.sel_bias is None else inp.sel_bias.cpu().numpy())


def oracle_tokens(w, h, start: int, n: int):
    """The oracle's full layer on tokens [start, start+n) of the workload, as a
    batch of n tokens; returns wall seconds."""
    import oracle
    x = h["x"][start:start + n]
    t0 = time.perf_counter()
    oracle.layer_forward(x, h["wr"], h["w1"], h["w3"], h["w2"], w.k, offset=h["off"],
                         sel_bias=h["bias"], ws1=h["ws1"], ws3=h["ws3"], ws2=h["ws2"],
                         capacity_factor=w.capacity_factor, lam=w.balance_coef)
    return time.perf_counter() - t0


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(w, inp, budget_s: float):
    """Times the oracle as it stands on a bounded sample of the workload."""
    import oracle
    oracle.load()
    h = _host_inputs(inp)
    cores = cpu_cores()
    probe_n = min(w.T, cores)
    t_probe = oracle_tokens(w, h, 0, probe_n)             # also the warm-up
    per_round = max(t_probe, 1e-3)
    rounds = max(1, int(budget_s / per_round))
    n = min(w.T, probe_n * rounds)
    t = oracle_tokens(w, h, 0, n)
    threads = min(cores, n)
    return {"value": n / t, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"first {n} tokens of the workload run through the fp64 oracle layer "
                      f"as one batch of {n} (router, dispatch, experts, combine, losses); "
                      f"{t:.1f} s wall, OpenMP over tokens"}


def run_reference(args, w):
    """Reference arm: the oracle on host cores (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import torch

    import synth
    import oracle
    oracle.load()
    # inputs are drawn on the GPU when there is one (faster), then copied to the host
    inp = synth.make_inputs(w, "cuda" if torch.cuda.is_available() else "cpu")
    h = _host_inputs(inp)
    del inp
    cores = cpu_cores()
    t1 = oracle_tokens(w, h, 0, min(w.T, cores))
    per_tok_round = max(t1, 1e-3)
    budget = 150.0 / max(1, args.steps + args.warmup)     # whole run within a few minutes
    n = max(1, min(w.T, int(min(w.T, cores) * max(1.0, budget / per_tok_round))))
    if t1 > budget:
        n = max(1, min(cores, int(min(w.T, cores) * budget / t1)))
    for i in range(args.warmup):
        oracle_tokens(w, h, 0, n)
    times = [oracle_tokens(w, h, (i * n) % max(1, w.T - n + 1), n) for i in range(args.steps)]
    ms = 1000.0 * statistics.mean(times)
    value = n / (ms / 1000.0)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": workload_desc(w), "T": w.T, "d": w.d, "E": w.E, "k": w.k,
                       "M": w.M, "n_shared": w.n_shared,
                       "capacity_factor": w.capacity_factor,
                       "step": f"{n} tokens through the oracle layer"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": min(cores, n),
                             "kind": "oracle",
                             "sample": f"{n} tokens per step (fp64 oracle, OpenMP over tokens)"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- #
# replicas across ranks                                                        #
# --------------------------------------------------------------------------- #
def max_over_ranks(value: float, device) -> float:
    """The slowest rank's time: every rank runs its own replica of the
    workload (there is no data-path exchange), so the job's step time is the
    maximum over ranks.  A no-op without an initialised process group."""
    import torch
    import torch.distributed as dist
    if not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_rank: int, ms: float) -> float:
    """Whole-job throughput: every rank processes its own batch of tokens in
    the (max-over-ranks) step time."""
    return world * tokens_per_rank / (ms * 1e-3)


# --------------------------------------------------------------------------- #
# per-kernel stage times and the other workloads                               #
# --------------------------------------------------------------------------- #
WORKLOAD_ORDER = ["tiny", "mixtral", "deepseekmoe16b", "deepseekv2", "switch"]


def stage_pass(layer, inp, w, flush, dev, n: int, graph: bool = True):
    """Per-kernel device time of one layer forward, every kernel bracketed by
    events.  With ``graph`` the n forwards are captured as CUDA graphs first
    (the events become event nodes of the graphs) and replayed with an L2
    flush before each, so the brackets hold only device time, as in the timed
    loop; otherwise they are launched directly (host launch gaps included)."""
    import torch
    import top_routing_expert_lb_b300 as moe
    stream = torch.cuda.current_stream(dev)
    moe.moe_profile_collect()
    moe.moe_profile_enable(True)
    if graph:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        graphs = []
        with torch.cuda.stream(side):
            for _ in range(n):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=side):
                    layer.forward(inp.x)
                graphs.append(g)
        stream.wait_stream(side)
        torch.cuda.synchronize(dev)
        for g in graphs:
            flush.zero_()
            g.replay()
    else:
        for _ in range(n):
            flush.zero_()
            layer.forward(inp.x)
    torch.cuda.synchronize(dev)
    moe.moe_profile_enable(False)
    per_kernel = {}
    for name, t in moe.moe_profile_collect():
        per_kernel.setdefault(name, []).append(t)
    kern_ms = {k: sum(v) / n for k, v in per_kernel.items()}
    if layer.expert_choice:
        R = w.E * layer.r
    else:
        R = int(w.T * w.k - int(layer.drop_mask.sum().item())) if w.k else 0
    flops, bytes_ = algorithmic_work(w, R)
    peaks, _ = load_peaks()
    kept = kept_rows_per_expert(layer, w)
    ffn_ms = kern_ms.get("gemm_swiglu", 0.0) + kern_ms.get("gemm_down", 0.0)
    ffn_flops = flops["gemm_swiglu"] + flops["gemm_down"]
    return {"kernel_ms": kern_ms, "kernel_launches": {k: len(v) for k, v in per_kernel.items()},
            "rows": R, "kept": kept, "ffn_ms": ffn_ms,
            "ffn_tflops": ffn_flops / (ffn_ms * 1e-3) / 1e12 if ffn_ms > 0 else 0.0,
            "ffn_attainable_ms": attainable_ffn_ms(w, kept, peaks),
            "stage_gbs": {k: bytes_[k] / (kern_ms[k] * 1e-3) / 1e9
                          for k in bytes_ if k in kern_ms},
            "how": (f"{n} CUDA-graph replays of one forward, every kernel bracketed by event "
                    "nodes, L2 flushed before each" if graph else
                    f"{n} direct forwards, every launch bracketed by events, L2 flushed "
                    "before each")}


def st_summary(st, w, step_ms: float, peaks):
    """The per-workload figures of one stage pass and timed loop."""
    kept = st["kept"]
    tot = sum(kept)
    return {"workload": workload_desc(w), "tokens_per_s": w.T / (step_ms * 1e-3),
            "ms_per_step": step_ms, "ffn_ms": st["ffn_ms"], "ffn_tflops": st["ffn_tflops"],
            "ffn_frac_of_bf16_peak": st["ffn_tflops"] / peaks["bf16_tflops"],
            "ffn_attainable_ms": st["ffn_attainable_ms"],
            "ffn_frac_of_attainable": (st["ffn_attainable_ms"] / st["ffn_ms"]
                                       if st["ffn_ms"] > 0 else None),
            "kernel_ms": st["kernel_ms"],
            "stage_gbs": st["stage_gbs"],
            "stage_frac_of_hbm": {k: v / peaks["hbm_gbs"] for k, v in st["stage_gbs"].items()},
            "load": {"max_over_mean": float(max(kept) / (tot / len(kept))) if tot else None,
                     "empty_experts": int(sum(1 for v in kept if v == 0)),
                     "rows_computed": st["rows"],
                     "dropped_pairs": int(w.T * w.k - st["rows"])}}


def measure_other(w, args, dev, flush, steps: int = 20, warmup: int = 3):
    """One more workload in this process: graph-replayed timed steps (L2
    flushed before each) and a stage pass; inputs released afterwards."""
    import torch

    import synth
    import top_routing_expert_lb_b300 as moe
    inp = synth.make_inputs(w, dev)
    shape = moe.Shape.of(w.T, w.d, w.M, w.E, w.k, w.n_shared, w.capacity_factor,
                         w.balance_coef, w.flags)
    layer = moe.MoELayer(shape, inp.wr, inp.w1, inp.w3, inp.w2, inp.ws1, inp.ws3, inp.ws2,
                         inp.offset, inp.sel_bias, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        layer.forward(inp.x)
    torch.cuda.synchronize(dev)
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    graphs = []
    moe.moe_profile_collect()
    moe.moe_profile_enable(True, kernels=["gemm_swiglu", "gemm_down"])
    with torch.cuda.stream(side):
        for _ in range(steps):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                layer.forward(inp.x)
            graphs.append(g)
    stream.wait_stream(side)
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for g, (a, b) in zip(graphs, ev):
        flush.zero_()
        a.record(stream)
        g.replay()
        b.record(stream)
    torch.cuda.synchronize(dev)
    moe.moe_profile_enable(False)
    gemm = moe.moe_profile_collect()
    if moe.moe_check_status(layer.ws) != 0:
        raise RuntimeError(f"device wait timed out ({w.name})")
    step_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    st = stage_pass(layer, inp, w, flush, dev, 5)
    peaks, _ = load_peaks()
    if gemm:
        # the expert FFN as timed inside the timed replays
        R = st["rows"]
        flops, _ = algorithmic_work(w, R)
        st["ffn_ms"] = sum(t for _, t in gemm) / steps
        st["ffn_tflops"] = (flops["gemm_swiglu"] + flops["gemm_down"]) / (st["ffn_ms"] * 1e-3) / 1e12
    out = dict(st_summary(st, w, step_ms, peaks), steps=steps, warmup=warmup)
    del graphs, layer, inp
    torch.cuda.empty_cache()
    return out


# --------------------------------------------------------------------------- #
# our arm                                                                      #
# --------------------------------------------------------------------------- #
def run_ours(args, w):
    import torch
    import torch.distributed as dist

    import synth
    import top_routing_expert_lb_b300 as moe
    from top_routing_expert_lb_b300 import build as mbuild

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        mbuild.ensure_built()
    if world > 1:
        dist.barrier()

    inp = synth.make_inputs(w, dev)
    shape = moe.Shape.of(w.T, w.d, w.M, w.E, w.k, w.n_shared, w.capacity_factor,
                         w.balance_coef, w.flags)
    layer = moe.MoELayer(shape, inp.wr, inp.w1, inp.w3, inp.w2, inp.ws1, inp.ws3, inp.ws2,
                         inp.offset, inp.sel_bias, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        layer.forward(inp.x)
    torch.cuda.synchronize(dev)
    if moe.moe_check_status(layer.ws) != 0:
        raise RuntimeError("device wait timed out during warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    # Inside the headline loop only the dominant kernel is bracketed by events.
    # By default each timed step replays its own CUDA graph of one layer
    # forward (captured here, events included), which drops the host-side
    # launch work from the step; --no-graph launches every step directly.
    graphs = None
    per_forward = 0
    moe.moe_profile_enable(True, kernels=["gemm_swiglu", "gemm_down"])
    if not args.no_graph:
        graphs = []
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        c0 = moe.moe_launch_count()
        with torch.cuda.stream(side):
            for _ in range(args.steps):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=side):
                    layer.forward(inp.x)
                graphs.append(g)
        per_forward = (moe.moe_launch_count() - c0) // max(1, args.steps)
        stream.wait_stream(side)
        torch.cuda.synchronize(dev)
    launches0 = moe.moe_launch_count()
    with ClockSampler(local, enabled=not args.no_clocks, csv_dir=args.clocks_dir) as clk:
        clk.mark_start()
        for i in range(args.steps):
            flush.zero_()                                  # evict L2 between steps
            starts[i].record(stream)
            if graphs is None:
                layer.forward(inp.x)
            else:
                graphs[i].replay()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        clk.mark_end()
    moe.moe_profile_enable(False)
    prof = moe.moe_profile_collect()
    launches = moe.moe_launch_count() - launches0
    if graphs is not None:
        # each replay runs the kernels captured once (counted at capture)
        launches = per_forward * args.steps
    if world > 1:
        dist.barrier()
    if moe.moe_check_status(layer.ws) != 0:
        raise RuntimeError("device wait timed out during the timed steps")
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = max_over_ranks(statistics.mean(step_ms), dev)

    dom_times = [t for name, t in prof if name == "gemm_swiglu"]
    down_times = [t for name, t in prof if name == "gemm_down"]
    used_graph = graphs is not None
    expert_choice = layer.expert_choice
    st = stage_pass(layer, inp, w, flush, dev, max(3, min(args.steps, 10)),
                    graph=not args.no_graph)
    kern_ms, kern_n = st["kernel_ms"], st["kernel_launches"]
    R = st["rows"]
    flops, bytes_ = algorithmic_work(w, R)
    peaks, peak_src = load_peaks()
    kept = st["kept"]
    attainable_ms = st["ffn_attainable_ms"]
    # the expert FFN as timed inside the timed steps (event nodes around both
    # projections), not from the stage pass
    ffn_ms = (sum(dom_times) + sum(down_times)) / args.steps if dom_times else st["ffn_ms"]
    ffn_tflops = (flops["gemm_swiglu"] + flops["gemm_down"]) / (ffn_ms * 1e-3) / 1e12
    st["ffn_ms"], st["ffn_tflops"] = ffn_ms, ffn_tflops
    dom = "gemm_swiglu"
    # the gate/up projection may take two launches per step (pair tiles for
    # whole 256-row blocks, single-CTA tiles for the rest): time per step
    dom_per_step = len(dom_times) // max(1, args.steps)
    dom_ms = sum(dom_times) / args.steps if dom_times else kern_ms[dom]
    ach = flops[dom] / (dom_ms * 1e-3) / 1e12
    stage_gbs = st["stage_gbs"]

    # end to end: host tokens in, host output and losses out, through the C ABI.
    # Headline: a stream of batches through moe_layer_forward_host_batches
    # (copy-in of batch i+1 and copy-out of batch i-1 overlap the layer of
    # batch i); beside it one batch at a time through moe_layer_forward_host.
    e2e = None
    if not args.no_e2e and args.routing == "token":
        batch_bytes = w.T * w.d * 2
        weight_bytes = 2 * (3 * w.E * w.M * w.d + 3 * w.n_shared * w.M * w.d + w.E * w.d)
        n_b = max(3, min(16, (1 << 30) // max(1, batch_bytes)))
        x_host = inp.x.cpu().pin_memory()
        xs_host = x_host.unsqueeze(0).repeat(n_b, 1, 1).pin_memory()
        ys_host = torch.empty_like(xs_host).pin_memory()
        bl_host = torch.empty(n_b, 2, dtype=torch.float32).pin_memory()
        x_slots = torch.empty((2,) + tuple(inp.x.shape), dtype=inp.x.dtype, device=dev)
        y_slots = torch.empty_like(x_slots)
        loss_slots = torch.empty(2, 2, dtype=torch.float32, device=dev)
        h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def e2e_stream(n):
            moe.moe_layer_forward_host_batches(
                layer.shape, xs_host[:n], ys_host[:n], bl_host[:n], x_slots, y_slots,
                loss_slots, layer.w_router, layer.logit_offset, layer.sel_bias, layer.w13,
                layer.w2, layer.w13_shared, layer.w2_shared, layer.ids, layer.gates,
                layer.counts, layer.drop_mask, layer.f, layer.P, layer.ws, stream, h2d, d2h)
        e2e_stream(2)
        reps = 3
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)]
        for a, b in ev:
            a.record(h2d)          # h2d is idle: the first copy-in starts after this
            e2e_stream(n_b)        # returns once every stream has drained
            b.record(d2h)
        torch.cuda.synchronize(dev)
        stream_ms = max_over_ranks(
            statistics.mean(a.elapsed_time(b) for a, b in ev) / n_b, dev)

        y_host = torch.empty_like(x_host).pin_memory()
        losses_host = torch.empty(2, dtype=torch.float32).pin_memory()
        x_dev = torch.empty_like(inp.x)
        y_dev = torch.empty_like(inp.x)
        n_e2e = max(3, min(args.steps, 10))

        def e2e_step():
            moe.moe_layer_forward_host(layer.shape, x_host, x_dev, layer.w_router,
                                       layer.logit_offset, layer.sel_bias, layer.w13, layer.w2,
                                       layer.w13_shared, layer.w2_shared, y_dev, y_host,
                                       losses_host, layer.ids, layer.gates, layer.counts,
                                       layer.drop_mask, layer.f, layer.P, layer.losses[0:1],
                                       layer.losses[1:2], layer.ws)
        for _ in range(2):
            e2e_step()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n_e2e)]
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            e2e_step()
            b.record(stream)
        torch.cuda.synchronize(dev)
        single_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ev), dev)
        e2e = {"value": job_tokens_per_s(world, w.T, stream_ms), "unit": "tokens/s",
               "ms_per_step": stream_ms, "h2d_bytes_per_step": batch_bytes,
               "d2h_bytes_per_step": batch_bytes + 8,
               "path": f"moe_layer_forward_host_batches: {n_b} batches of T tokens from pinned "
                       "host memory, y and losses back to pinned host memory; copy-in, layer "
                       "and copy-out on three streams; timed from before the first copy-in to "
                       f"after the call returned, mean of {reps} calls",
               "l2": (f"not flushed: each batch streams {weight_bytes / 1e9:.2f} GB of weights, "
                      "more than the 126 MB L2" if weight_bytes > (126 << 20) else
                      f"not flushed; weights ({weight_bytes / 1e6:.1f} MB) stay in L2"),
               "single_batch": {"value": job_tokens_per_s(world, w.T, single_ms),
                                "ms_per_step": single_ms,
                                "path": "moe_layer_forward_host (copy in, layer, copy out, "
                                        "one stream, L2 flushed before each)"}}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline and args.routing == "token":
        cpu = cpu_baseline(w, inp, args.cpu_budget_s)

    per_config = None
    if not args.no_per_config and args.routing == "token" and world == 1:
        # every other workload of the layer, measured the same way in this
        # process (fewer steps; no e2e or CPU leg), after the headline's
        # graphs, inputs and layer are released
        graphs = None
        layer = inp = None
        torch.cuda.empty_cache()
        per_config = {w.name: dict(st_summary(st, w, ms, peaks), steps=args.steps,
                                   warmup=args.warmup)}
        for name in WORKLOAD_ORDER:
            if name == w.name:
                continue
            per_config[name] = measure_other(synth.WORKLOADS[name], args, dev, flush)
        per_config = {k: per_config[k] for k in WORKLOAD_ORDER if k in per_config}

    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": job_tokens_per_s(world, w.T, ms), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded N(0,1) tokens, random-init N(0,0.02) weights",
        "config": {"workload": workload_desc(w), "T": w.T, "d": w.d, "E": w.E, "k": w.k,
                   "M": w.M, "n_shared": w.n_shared, "capacity_factor": w.capacity_factor,
                   "rows_computed": R,
                   "l2": f"flushed: {FLUSH_BYTES >> 20} MiB written before every timed step",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "cuda_graph": used_graph},
        "ffn_tflops": ffn_tflops,
        "ffn_frac_of_bf16_peak": ffn_tflops / peaks["bf16_tflops"],
        "ffn_attainable_ms": attainable_ms,
        "ffn_frac_of_attainable": attainable_ms / ffn_ms if ffn_ms > 0 else None,
        "routing": args.routing,
        "load": {"max_over_mean": float(max(kept) / (sum(kept) / len(kept))) if sum(kept) else None,
                 "empty_experts": int(sum(1 for v in kept if v == 0)),
                 "dropped_pairs": int(w.T * w.k - R) if not expert_choice else None},
        "kernel_ms": kern_ms, "kernel_launches_stage_pass": kern_n,
        "stage_pass": st["how"],
        "stage_gbs": stage_gbs,
        "stage_frac_of_hbm": {k: v / peaks["hbm_gbs"] for k, v in stage_gbs.items()},
        "roofline": {"bound": "tensor", "kernel": dom, "achieved": ach,
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": ach / peaks["bf16_tflops"],
                     "traffic": recorded_traffic(w.name, dom),
                     "peak_source": f"bf16_tflops burst, {peak_src}",
                     "frac_of_sustained": ach / peaks["bf16_tflops_sustained"],
                     "algorithmic_flops_per_launch": flops[dom],
                     "step_ms": dom_ms, "launches_timed": len(dom_times),
                     "launches_per_step": dom_per_step,
                     "step_ms_first_last": [
                         sum(dom_times[:5 * dom_per_step]) / 5,
                         sum(dom_times[-5 * dom_per_step:]) / 5]
                     if len(dom_times) >= 5 * max(1, dom_per_step) else None},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "per_config": per_config,
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


def run_router_stage(args, w):
    """moe_route alone at the workload's shape: per-call device time and HBM
    fraction of its algorithmic bytes (one JSON line, not the headline)."""
    import torch

    import synth
    import top_routing_expert_lb_b300 as moe
    from top_routing_expert_lb_b300 import build as mbuild

    mbuild.ensure_built()
    dev = torch.device("cuda", 0)
    inp = synth.make_inputs(w, dev, experts=False)
    s = moe.Shape.of(w.T, w.d, w.M, w.E, w.k, w.n_shared, w.capacity_factor, w.balance_coef)
    ws = moe.alloc_workspace(s, dev)
    ids = torch.empty((w.T, w.k), dtype=torch.int32, device=dev)
    gates = torch.empty((w.T, w.k), dtype=torch.float32, device=dev)
    counts = torch.empty(w.E, dtype=torch.int32, device=dev)
    f = torch.empty(w.E, device=dev)
    P = torch.empty(w.E, device=dev)
    lb = torch.empty(1, device=dev)
    lz = torch.empty(1, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call():
        moe.moe_route(s, inp.x, inp.wr, inp.offset, inp.sel_bias, ids, gates, counts, f, P, lb,
                      lz, ws)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(dev)
    moe.moe_profile_enable(True)
    for _ in range(args.steps):
        flush.zero_()
        call()
    torch.cuda.synchronize(dev)
    moe.moe_profile_enable(False)
    per = {}
    for name, t in moe.moe_profile_collect():
        per.setdefault(name, []).append(t)
    kern = {k: statistics.mean(v) for k, v in per.items()}
    peaks, _ = load_peaks()
    b = algorithmic_work(w, 0)[1]["router"]
    print(json.dumps({"stage": "router", "workload": workload_desc(w), "kernel_ms": kern,
                      "router_gbs": b / (kern["router"] * 1e-3) / 1e9,
                      "router_frac_of_hbm": b / (kern["router"] * 1e-3) / 1e9 / peaks["hbm_gbs"]}),
          flush=True)
    return 0


def run_ffn_stage(args, w):
    """moe_grouped_ffn alone on a slice of the workload's realised loads: the
    router runs on the full workload (no expert weights), the experts are
    sorted by load and every (E / n)-th of them is kept in index order, and
    the shared group (if any) gets T n / E rows.  Device time per projection
    (L2 flushed before each call), FFN TFLOP/s and the attainable bound of the
    slice.  For profiling the expert GEMMs on small footprints."""
    import torch

    import synth
    import top_routing_expert_lb_b300 as moe
    from top_routing_expert_lb_b300 import build as mbuild

    mbuild.ensure_built()
    dev = torch.device("cuda", 0)
    inp = synth.make_inputs(w, dev, experts=False)
    s = moe.Shape.of(w.T, w.d, w.M, w.E, w.k, w.n_shared, w.capacity_factor, w.balance_coef)
    ws = moe.alloc_workspace(s, dev)
    ids = torch.empty((w.T, max(w.k, 1)), dtype=torch.int32, device=dev)
    gates = torch.empty((w.T, max(w.k, 1)), dtype=torch.float32, device=dev)
    counts = torch.empty(w.E, dtype=torch.int32, device=dev)
    f, P = torch.empty(w.E, device=dev), torch.empty(w.E, device=dev)
    lb, lz = torch.empty(1, device=dev), torch.empty(1, device=dev)
    moe.moe_route(s, inp.x, inp.wr, inp.offset, inp.sel_bias, ids, gates, counts, f, P, lb, lz, ws)
    C = moe.moe_capacity(s)
    n = counts.cpu().tolist()
    if C >= 0:
        n = [min(v, C) for v in n]
    del inp, ws, ids, gates
    n_sel = args.experts if 0 < args.experts < w.E else w.E
    order = sorted(range(w.E), key=lambda e: (-n[e], e))
    picked = sorted(order[int(i * w.E / n_sel)] for i in range(n_sel))
    rows = [n[e] for e in picked]
    R = sum(rows)
    T_sh = max(1, round(w.T * n_sel / w.E), -(-R // min(8, n_sel))) if w.n_shared else 0
    Tshape = T_sh if w.n_shared else max(R, 1)
    k = max(1, -(-R // Tshape))
    tune = parse_tune(args.tune)
    sf = moe.Shape.of(Tshape, w.d, w.M, n_sel, min(k, n_sel), w.n_shared, **tune)
    assert R <= moe.moe_max_rows(sf), "slice rows exceed the shape's row bound"
    x_perm = synth.normal_bf16(5, synth.TID_X, (max(R, 1), w.d), 1.0, dev)
    offsets = torch.tensor([0] + list(__import__("itertools").accumulate(rows)), dtype=torch.int32,
                           device=dev)
    w1 = synth.normal_bf16(5, synth.TID_W1, (n_sel, w.M, w.d), w.w_std, dev)
    w3 = synth.normal_bf16(5, synth.TID_W3, (n_sel, w.M, w.d), w.w_std, dev)
    w13 = moe.moe_pack_w13(w1, w3)
    del w1, w3
    w2 = synth.normal_bf16(5, synth.TID_W2, (n_sel, w.d, w.M), w.w_std, dev)
    y_perm = torch.empty((max(moe.moe_max_rows(sf), 1), w.d), dtype=torch.bfloat16, device=dev)
    xs = w13s = w2s = ys = None
    if w.n_shared:
        Ms = w.n_shared * w.M
        xs = synth.normal_bf16(6, synth.TID_X, (T_sh, w.d), 1.0, dev)
        w13s = moe.moe_pack_w13(synth.normal_bf16(5, synth.TID_WS1, (Ms, w.d), w.w_std, dev),
                                synth.normal_bf16(5, synth.TID_WS3, (Ms, w.d), w.w_std, dev))
        w2s = synth.normal_bf16(5, synth.TID_WS2, (w.d, Ms), w.w_std, dev)
        ys = torch.empty((T_sh, w.d), dtype=torch.bfloat16, device=dev)
    xp = torch.zeros((max(moe.moe_max_rows(sf), 1), w.d), dtype=torch.bfloat16, device=dev)
    xp[:R] = x_perm[:R]
    del x_perm
    ws = moe.alloc_workspace(sf, dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def call():
        moe.moe_grouped_ffn(sf, xp, offsets, w13, w2, y_perm, xs, w13s, w2s, ys, ws)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(dev)
    moe.moe_profile_collect()
    moe.moe_profile_enable(True)
    for _ in range(args.steps):
        flush.zero_()
        call()
    torch.cuda.synchronize(dev)
    moe.moe_profile_enable(False)
    if moe.moe_check_status(ws) != 0:
        raise RuntimeError("device wait timed out")
    per = {}
    for name, t in moe.moe_profile_collect():
        per.setdefault(name, []).append(t)
    kern = {k2: sum(v) / args.steps for k2, v in per.items()}
    peaks, _ = load_peaks()
    ws2 = w.replace(T=T_sh if w.n_shared else w.T, E=n_sel)
    flops, _ = algorithmic_work(ws2, R)
    ffn_ms = kern.get("gemm_swiglu", 0.0) + kern.get("gemm_down", 0.0)
    att = attainable_ffn_ms(ws2, rows, peaks)
    print(json.dumps({"stage": "ffn", "workload": workload_desc(w), "experts": n_sel, "tune": tune,
                      "rows": rows, "shared_rows": T_sh, "kernel_ms": kern,
                      "gemm_swiglu_tflops": flops["gemm_swiglu"] / (kern["gemm_swiglu"] * 1e-3) / 1e12,
                      "ffn_tflops": (flops["gemm_swiglu"] + flops["gemm_down"]) / (ffn_ms * 1e-3) / 1e12,
                      "ffn_attainable_ms": att, "ffn_frac_of_attainable": att / ffn_ms,
                      "weight_bytes": 2 * 3 * w.M * w.d * (n_sel + w.n_shared)}), flush=True)
    return 0


def run_ab_stage(args, w):
    """Two layers of the workload that differ only in their moe_tuning_t
    fields, built once and called alternately (A B B A ...), the L2 flushed
    before every call and each call bracketed by events, and with every
    kernel bracketed too.  Prints the medians of both and of the paired
    differences: the power cap makes separate runs drift by several percent,
    while alternating calls see the same clock."""
    import statistics

    import torch

    import synth
    import top_routing_expert_lb_b300 as moe
    from top_routing_expert_lb_b300 import build as mbuild

    mbuild.ensure_built()
    dev = torch.device("cuda", 0)
    inp = synth.make_inputs(w, dev)
    tunes = (parse_tune(args.tune), parse_tune(args.tune_b))
    layers = [moe.MoELayer(moe.Shape.of(w.T, w.d, w.M, w.E, w.k, w.n_shared, w.capacity_factor,
                                        w.balance_coef, w.flags, **t),
                           inp.wr, inp.w1, inp.w3, inp.w2, inp.ws1, inp.ws3, inp.ws2, inp.offset,
                           inp.sel_bias, device=dev) for t in tunes]
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(max(args.warmup, 1)):
        for L in layers:
            L.forward(inp.x)
    torch.cuda.synchronize(dev)
    times = ([], [])
    kern = ({}, {})
    moe.moe_profile_collect()
    moe.moe_profile_enable(True)
    for i in range(args.steps):
        for v in ((0, 1) if i % 2 == 0 else (1, 0)):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            layers[v].forward(inp.x)
            b.record()
            torch.cuda.synchronize(dev)
            times[v].append(a.elapsed_time(b))
            for name, ms in moe.moe_profile_collect():
                kern[v].setdefault(name, []).append(ms)
    moe.moe_profile_enable(False)
    for L in layers:
        if moe.moe_check_status(L.ws) != 0:
            raise RuntimeError("device wait timed out")
    med = lambda xs: statistics.median(xs)
    print(json.dumps({
        "stage": "ab", "workload": workload_desc(w), "calls_each": args.steps,
        "A": tunes[0], "B": tunes[1],
        "layer_ms": [med(times[0]), med(times[1])],
        "median_diff_a_minus_b_us": 1000.0 * med([x - y for x, y in zip(*times)]),
        "kernel_us": [{k: 1000.0 * med(v) for k, v in kern[0].items()},
                      {k: 1000.0 * med(v) for k, v in kern[1].items()}],
        "same_y": bool(torch.equal(layers[0].y.view(torch.int16), layers[1].y.view(torch.int16))),
    }), flush=True)
    return 0


def run_dense_stage(args, w):
    """The gate/up projection of one expert holding all --rows rows (a dense
    rows x d x 2M GEMM with the SwiGLU epilogue) through moe_grouped_ffn on
    single-CTA and on CTA-pair tiles, called alternately with torch.matmul of
    the same operands (cuBLAS, no epilogue), the L2 flushed before every call.
    Prints the median gate/up kernel time of each (events around the kernel)."""
    import statistics

    import torch

    import synth
    import top_routing_expert_lb_b300 as moe
    from top_routing_expert_lb_b300 import build as mbuild

    mbuild.ensure_built()
    dev = torch.device("cuda", 0)
    rows, d, M = args.rows, w.d, w.M
    x = synth.normal_bf16(5, synth.TID_X, (rows, d), 1.0, dev)
    w13 = moe.moe_pack_w13(synth.normal_bf16(5, synth.TID_W1, (1, M, d), w.w_std, dev),
                           synth.normal_bf16(5, synth.TID_W3, (1, M, d), w.w_std, dev))
    w2 = synth.normal_bf16(5, synth.TID_W2, (1, d, M), w.w_std, dev)
    w13_t = w13.view(2 * M, d).t()
    offsets = torch.tensor([0, rows], dtype=torch.int32, device=dev)
    # the down projection follows the gate/up tiles where d allows 256-wide tiles
    pair = dict(gemm1_tile=256, **({"gemm2_tile": 256} if d % 256 == 0 else {}))
    tiles = {"single_cta": dict(gemm1_tile=128), "cta_pair": pair}
    runs = {}
    for name, tu in tiles.items():
        s = moe.Shape.of(rows, d, M, 1, 1, 0, **tu)
        xp = torch.zeros((moe.moe_max_rows(s), d), dtype=torch.bfloat16, device=dev)
        xp[:rows] = x
        y = torch.empty((moe.moe_max_rows(s), d), dtype=torch.bfloat16, device=dev)
        ws = moe.alloc_workspace(s, dev)
        runs[name] = (lambda s=s, xp=xp, y=y, ws=ws:
                      moe.moe_grouped_ffn(s, xp, offsets, w13, w2, y, None, None, None, None, ws))
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(max(args.warmup, 1)):
        for f in runs.values():
            f()
        x @ w13_t
    torch.cuda.synchronize(dev)
    times = {k: [] for k in list(runs) + ["cublas"]}
    moe.moe_profile_collect()
    moe.moe_profile_enable(True)
    order = list(runs) + ["cublas"]
    for i in range(args.steps):
        for name in (order if i % 2 == 0 else order[::-1]):
            flush.zero_()
            torch.cuda.synchronize(dev)
            if name == "cublas":
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                x @ w13_t
                b.record()
                torch.cuda.synchronize(dev)
                times[name].append(a.elapsed_time(b))
            else:
                runs[name]()
                torch.cuda.synchronize(dev)
                times[name] += [ms for k, ms in moe.moe_profile_collect() if k == "gemm_swiglu"]
    moe.moe_profile_enable(False)
    flops = 2.0 * rows * d * 2 * M
    med = {k: statistics.median(v) for k, v in times.items()}
    print(json.dumps({
        "stage": "dense", "shape": {"rows": rows, "d": d, "two_M": 2 * M}, "calls_each": args.steps,
        "gate_up_ms": med, "tflops": {k: flops / v / 1e9 for k, v in med.items()},
        "vs_cublas": {k: med[k] / med["cublas"] for k in runs},
    }), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    import synth
    w = synth.WORKLOADS[args.workload]
    if args.routing != "token":
        w = w.replace(flags=w.flags | ROUTING_FLAGS[args.routing])
        if args.routing == "expert-choice":
            w = w.replace(sel_bias="none")      # a selection bias has no role there
    if args.impl == "reference":
        if args.routing != "token":
            print(json.dumps({"impl": "reference", "unavailable": "the CPU leg times the "
                              "token-choice layer only"}), flush=True)
            return 0
        return run_reference(args, w)
    if args.stage == "router":
        return run_router_stage(args, w)
    if args.stage == "ffn":
        return run_ffn_stage(args, w)
    if args.stage == "ab":
        return run_ab_stage(args, w)
    if args.stage == "dense":
        return run_dense_stage(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())

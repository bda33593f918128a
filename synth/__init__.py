"""Seeded synthetic inputs for the MoE layer: tokens, router and expert weights,
per-expert logit offsets and selection biases.

This module is shared by both sides of every parity check (the oracle and the
CUDA library receive the very same bf16 bits) and holds none of the layer's
arithmetic: it only draws numbers.

Generator (counter-based, so any slice can be drawn independently):
  * splitmix64 (Steele, Lea & Flood 2014; Vigna's reference constants): the
    i-th output of the stream that starts at state s0 is mix(s0 + (i+1)*GAMMA),
    with mix the published 30/27/31 xor-shift-multiply finaliser.
  * s0 = mix(seed * GAMMA2 xor tensor_id), one stream per tensor.
  * uniform u_i = (out_i >> 11) * 2^-53 in [0, 1).
  * normal n_i = sqrt(-2 ln(1 - u_{2i})) * cos(2 pi u_{2i+1})  (Box-Muller),
    computed in float64, scaled by the standard deviation, then rounded to
    float32 and from there to bf16, both round-to-nearest-even.

Tensor ids: x=1, W_r=2, W1=3, W3=4, W2=5, W1s=6, W3s=7, W2s=8, logit offsets=9,
selection bias=10, Zipf rank permutation=12.  Seed 0 for every workload.

Zipf-skewed workloads carry a per-expert logit offset vector that was calibrated
once so that the realised loads follow Zipf(s) (a stored input, see
``zipf_offsets``); it is read from ``tests/golden/``, where the script that wrote
it lives.
"""
from __future__ import annotations

import math
import os
from dataclasses import dataclass, field
from typing import Dict, Optional

import torch

GAMMA = 0x9E3779B97F4A7C15
GAMMA2 = 0xD1B54A32D192ED03
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB
_M64 = (1 << 64) - 1

TID_X, TID_WR, TID_W1, TID_W3, TID_W2, TID_WS1, TID_WS3, TID_WS2 = 1, 2, 3, 4, 5, 6, 7, 8
TID_OFFSET, TID_BIAS, TID_ZIPF_RANK = 9, 10, 12

_REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN_DIR = os.path.join(_REPO, "tests", "golden")


def _s64(v: int) -> int:
    """Two's-complement view of a 64-bit unsigned constant (torch has int64)."""
    v &= _M64
    return v - (1 << 64) if v >> 63 else v


def _mix_int(z: int) -> int:
    z &= _M64
    z = ((z ^ (z >> 30)) * MIX1) & _M64
    z = ((z ^ (z >> 27)) * MIX2) & _M64
    return z ^ (z >> 31)


def _srl(z: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 lanes holding uint64 bit patterns."""
    return (z >> s) & ((1 << (64 - s)) - 1)


def _mix(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _srl(z, 30)) * _s64(MIX1)
    z = (z ^ _srl(z, 27)) * _s64(MIX2)
    return z ^ _srl(z, 31)


def stream_start(seed: int, tid: int) -> int:
    return _mix_int(((seed * GAMMA2) & _M64) ^ tid)


def raw64(seed: int, tid: int, start: int, n: int, device="cpu") -> torch.Tensor:
    """Outputs start .. start+n-1 of the (seed, tid) splitmix64 stream (int64 bits)."""
    s0 = stream_start(seed, tid)
    i = torch.arange(start + 1, start + n + 1, dtype=torch.int64, device=device)
    z = i * _s64(GAMMA) + _s64(s0)
    return _mix(z)


def uniform(seed: int, tid: int, start: int, n: int, device="cpu") -> torch.Tensor:
    """float64 uniforms in [0,1) from the top 53 bits of each output."""
    return _srl(raw64(seed, tid, start, n, device), 11).to(torch.float64) * (2.0 ** -53)


_CHUNK = 1 << 24


def normal_f64(seed: int, tid: int, n: int, std: float = 1.0, device="cpu") -> torch.Tensor:
    out = torch.empty(n, dtype=torch.float64, device=device)
    for b in range(0, n, _CHUNK):
        m = min(_CHUNK, n - b)
        u = uniform(seed, tid, 2 * b, 2 * m, device).view(m, 2)
        r = torch.sqrt(-2.0 * torch.log1p(-u[:, 0]))
        out[b:b + m] = r * torch.cos((2.0 * math.pi) * u[:, 1]) * std
    return out


def normal_bf16(seed: int, tid: int, shape, std: float = 1.0, device="cpu") -> torch.Tensor:
    """N(0, std^2) draws rounded f64 -> f32 -> bf16 (RNE each), as a bf16 tensor."""
    n = 1
    for s in shape:
        n *= s
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    for b in range(0, n, _CHUNK):
        m = min(_CHUNK, n - b)
        u = uniform(seed, tid, 2 * b, 2 * m, device).view(m, 2)
        r = torch.sqrt(-2.0 * torch.log1p(-u[:, 0]))
        v = r * torch.cos((2.0 * math.pi) * u[:, 1]) * std
        out[b:b + m] = v.to(torch.float32).to(torch.bfloat16)
    return out.view(*shape)


def uniform_f32(seed: int, tid: int, n: int, lo: float, hi: float, device="cpu"):
    return (lo + (hi - lo) * uniform(seed, tid, 0, n, device)).to(torch.float32)


def zipf_rank(seed: int, E: int) -> torch.Tensor:
    """A seeded permutation: rank_of[e] in 1..E (1 = hottest expert)."""
    u = uniform(seed, TID_ZIPF_RANK, 0, E)
    order = torch.argsort(u)            # expert order[0] gets rank 1, ...
    rank = torch.empty(E, dtype=torch.int64)
    rank[order] = torch.arange(1, E + 1)
    return rank


# --------------------------------------------------------------------------- #
# Workloads                                                                    #
# --------------------------------------------------------------------------- #
@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    E: int
    k: int
    M: int
    n_shared: int = 0
    capacity_factor: float = 0.0      # <= 0: dropless
    offsets: str = "none"             # none | normal | zipf
    zipf_s: float = 0.0
    sel_bias: str = "none"            # none | uniform
    bias_range: float = 0.1
    x_std: float = 1.0
    w_std: float = 0.02
    balance_coef: float = 0.01
    seed: int = 0
    flags: int = 0                    # routing variant bits (sigmoid scores, no renorm)

    @property
    def Ms(self) -> int:
        return self.n_shared * self.M

    def replace(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", T=64, d=64, E=8, k=2, M=128),
    "mixtral": Workload("mixtral", T=4096, d=4096, E=8, k=2, M=14336),
    "deepseekmoe16b": Workload("deepseekmoe16b", T=8192, d=2048, E=64, k=6, M=1408,
                               n_shared=2, offsets="normal"),
    "deepseekv2": Workload("deepseekv2", T=8192, d=5120, E=160, k=6, M=1536, n_shared=2,
                           offsets="zipf", zipf_s=1.1, sel_bias="uniform"),
    "switch": Workload("switch", T=32768, d=1024, E=128, k=1, M=4096, capacity_factor=1.25,
                       offsets="zipf", zipf_s=1.2),
}


def zipf_offsets_path(name: str) -> str:
    return os.path.join(GOLDEN_DIR, f"zipf_offsets_{name}.txt")


def zipf_offsets(w: Workload) -> torch.Tensor:
    """The stored, calibrated logit-offset vector of a Zipf-skewed workload."""
    path = zipf_offsets_path(w.name)
    vals = []
    with open(path) as fh:
        for line in fh:
            line = line.strip()
            if line and not line.startswith("#"):
                vals.append(float(line))
    if len(vals) != w.E:
        raise ValueError(f"{path}: {len(vals)} values, expected {w.E}")
    return torch.tensor(vals, dtype=torch.float32)


@dataclass
class Inputs:
    w: Workload
    x: torch.Tensor                       # [T,d] bf16
    wr: torch.Tensor                      # [E,d] bf16
    w1: torch.Tensor                      # [E,M,d] bf16
    w3: torch.Tensor                      # [E,M,d] bf16
    w2: torch.Tensor                      # [E,d,M] bf16
    ws1: Optional[torch.Tensor] = None    # [Ms,d] bf16
    ws3: Optional[torch.Tensor] = None    # [Ms,d] bf16
    ws2: Optional[torch.Tensor] = None    # [d,Ms] bf16
    offset: Optional[torch.Tensor] = None  # [E] fp32
    sel_bias: Optional[torch.Tensor] = None  # [E] fp32
    extra: dict = field(default_factory=dict)


def make_offsets(w: Workload, device="cpu") -> Optional[torch.Tensor]:
    if w.offsets == "none":
        return None
    if w.offsets == "normal":
        return normal_f64(w.seed, TID_OFFSET, w.E, 1.0, device).to(torch.float32)
    if w.offsets == "zipf":
        return zipf_offsets(w).to(device)
    raise ValueError(w.offsets)


def make_sel_bias(w: Workload, device="cpu") -> Optional[torch.Tensor]:
    if w.sel_bias == "none":
        return None
    if w.sel_bias == "uniform":
        return uniform_f32(w.seed, TID_BIAS, w.E, -w.bias_range, w.bias_range, device)
    raise ValueError(w.sel_bias)


def make_inputs(w: Workload, device="cpu", experts: bool = True) -> Inputs:
    """Draw every input of workload ``w`` on ``device``."""
    s = w.seed
    x = normal_bf16(s, TID_X, (w.T, w.d), w.x_std, device)
    wr = normal_bf16(s, TID_WR, (w.E, w.d), w.w_std, device)
    if experts:
        w1 = normal_bf16(s, TID_W1, (w.E, w.M, w.d), w.w_std, device)
        w3 = normal_bf16(s, TID_W3, (w.E, w.M, w.d), w.w_std, device)
        w2 = normal_bf16(s, TID_W2, (w.E, w.d, w.M), w.w_std, device)
    else:
        w1 = w3 = w2 = None
    ws1 = ws3 = ws2 = None
    if w.n_shared > 0 and experts:
        ws1 = normal_bf16(s, TID_WS1, (w.Ms, w.d), w.w_std, device)
        ws3 = normal_bf16(s, TID_WS3, (w.Ms, w.d), w.w_std, device)
        ws2 = normal_bf16(s, TID_WS2, (w.d, w.Ms), w.w_std, device)
    return Inputs(w, x, wr, w1, w3, w2, ws1, ws3, ws2, make_offsets(w, device),
                  make_sel_bias(w, device))


def to_u16(t: Optional[torch.Tensor]):
    """bf16 torch tensor -> numpy uint16 bit patterns (host copy)."""
    if t is None:
        return None
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")

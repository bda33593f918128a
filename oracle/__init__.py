"""Oracle for one top-k routed Mixture-of-Experts FFN layer forward.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use this package; the CUDA library never does.

This module is a thin ctypes wrapper around ``moe_oracle.c`` (plain fp64 C).  It
builds that file with gcc on first use (``build()``), marshals numpy arrays in and
out, and adds the one loop-free composition the tests need
(``layer_forward``).  All of the method's arithmetic lives in the C file; each
function there cites the page passage it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")
_lib = None


def build(src: str = _SRC, out: str = _LIB, extra_flags=()) -> str:
    """Compile the oracle with gcc (fp64, no fast-math) into a shared library."""
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99", *extra_flags,
           src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    if out == _LIB:
        with open(_LIB + ".srchash", "w") as fh:
            fh.write(_src_hash() + "\n")
    return out


def _src_hash() -> str:
    import hashlib
    with open(_SRC, "rb") as fh:
        return hashlib.sha256(fh.read()).hexdigest()


def _needs_build() -> bool:
    if not os.path.exists(_LIB) or not os.path.exists(_LIB + ".srchash"):
        return True
    with open(_LIB + ".srchash") as fh:
        return fh.read().strip() != _src_hash()


_P = ctypes.c_void_p


def load(path: Optional[str] = None):
    """Load (building if stale) the oracle library; ``path`` loads another build."""
    global _lib
    if path is None:
        if _lib is not None:
            return _lib
        if _needs_build():
            build()
        path = _LIB
    lib = ctypes.CDLL(path)
    i32, f64 = ctypes.c_int, ctypes.c_double
    lib.oracle_router_logits.argtypes = [i32, i32, i32, _P, _P, _P, _P]
    lib.oracle_route.argtypes = [i32, i32, i32, i32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]
    lib.oracle_capacity.argtypes = [f64, i32, i32, i32]
    lib.oracle_capacity.restype = ctypes.c_int64
    lib.oracle_dispatch.argtypes = [i32, i32, i32, _P, ctypes.c_int64, _P, _P, _P, _P, _P, _P]
    lib.oracle_swiglu_row.argtypes = [i32, i32, _P, _P, _P, _P, _P]
    lib.oracle_expert_rows.argtypes = [i32, i32, i32, _P, _P, _P, _P, _P, _P]
    lib.oracle_layer_tokens.argtypes = [i32] * 6 + [_P] * 10 + [i32, _P, _P]
    lib.oracle_losses.argtypes = [i32, i32, i32, _P, _P, _P, f64, _P, _P, _P, _P]
    lib.oracle_combine.argtypes = [i32, i32, i32, _P, _P, _P, _P, _P]
    lib.oracle_importance.argtypes = [i32, i32, i32, _P, _P, _P, _P]
    lib.oracle_alf_bias_update.argtypes = [i32, i32, i32, _P, ctypes.c_float, _P, _P]
    i64 = ctypes.c_int64
    lib.oracle_dispatch_priority.argtypes = [i32, i32, i32, _P, _P, _P, i64, _P, _P, _P, _P, _P,
                                             _P]
    lib.oracle_ec_capacity.argtypes = [f64, i32, i32, i32]
    lib.oracle_ec_capacity.restype = i64
    lib.oracle_expert_choice.argtypes = [i32, i32, i64, _P, _P, _P, _P]
    lib.oracle_ec_layer_tokens.argtypes = [i32, i32, i32, i32, i64, i32] + [_P] * 9 + [i32, _P, _P]
    lib.oracle_losses_n.argtypes = [i32, i32, f64, _P, _P, _P, f64, _P, _P, _P, _P]
    if path == _LIB:
        _lib = lib
    return lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, "bf16 tensors are passed as uint16 bit patterns"
    return a


def _f32(a) -> Optional[np.ndarray]:
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


# --------------------------------------------------------------------------- #
# Thin wrappers, one per C entry point                                         #
# --------------------------------------------------------------------------- #
def router_logits(x, wr, offset=None, lib=None) -> np.ndarray:
    lib = lib or load()
    x, wr = _u16(x), _u16(wr)
    T, d = x.shape
    E = wr.shape[0]
    off = _f32(offset)
    out = np.empty((T, E), np.float64)
    lib.oracle_router_logits(T, d, E, _ptr(x), _ptr(wr), _ptr(off), _ptr(out))
    return out


SIGMOID = 1     # sigmoid scores instead of the softmax
NO_RENORM = 2   # gates = selected scores, not renormalised
PRIORITY = 4    # capacity keeps each expert's highest-score pairs


@dataclass
class Routing:
    p: np.ndarray        # [T,E] router scores (softmax probabilities, or sigmoids)
    lse: np.ndarray      # [T]   log-sum-exp of the logits
    ids: np.ndarray      # [T,k] selected experts, descending key
    gates: np.ndarray    # [T,k] gates (renormalised unless NO_RENORM)
    gap: np.ndarray      # [T]   key_k - key_{k+1}
    entropy: np.ndarray  # [T]   entropy of the router distribution


def route(logits, k, sel_bias=None, force_ids=None, force_mask=None, flags=0,
          lib=None) -> Routing:
    lib = lib or load()
    logits = np.ascontiguousarray(logits, np.float64)
    T, E = logits.shape
    p = np.empty((T, E), np.float64)
    lse = np.empty(T, np.float64)
    ids = np.empty((T, k), np.int32)
    gates = np.empty((T, k), np.float64)
    gap = np.empty(T, np.float64)
    ent = np.empty(T, np.float64)
    fi = None if force_ids is None else np.ascontiguousarray(force_ids, np.int32)
    fm = None if force_mask is None else np.ascontiguousarray(force_mask, np.uint8)
    lib.oracle_route(T, E, k, int(flags), _ptr(logits), _ptr(_f32(sel_bias)), _ptr(fi),
                     _ptr(fm), _ptr(p), _ptr(lse), _ptr(ids), _ptr(gates), _ptr(gap), _ptr(ent))
    return Routing(p, lse, ids, gates, gap, ent)


def importance(ids, gates, E: int, lib=None):
    """(importance [E], CV^2) of the sparse gates, before any capacity cut."""
    lib = lib or load()
    ids = np.ascontiguousarray(ids, np.int32)
    g = np.ascontiguousarray(gates, np.float64)
    T, k = ids.shape
    imp = np.empty(E, np.float64)
    cv2 = ctypes.c_double()
    lib.oracle_importance(T, E, k, _ptr(ids), _ptr(g), _ptr(imp), ctypes.byref(cv2))
    return imp, cv2.value


def capacity(c: float, k: int, T: int, E: int, lib=None) -> int:
    lib = lib or load()
    return int(lib.oracle_capacity(float(c), k, T, E))


@dataclass
class Dispatch:
    counts: np.ndarray       # [E]   n_e before capacity
    kept_counts: np.ndarray  # [E]   pairs kept per expert
    offsets: np.ndarray      # [E+1] exclusive scan of kept_counts
    slot_row: np.ndarray     # [T,k] row of each pair, -1 if dropped
    row_token: np.ndarray    # [R]   token of each row
    dropped: np.ndarray      # [T,k] 1 where the pair was dropped


def dispatch(ids, E: int, C: int, lib=None) -> Dispatch:
    lib = lib or load()
    ids = np.ascontiguousarray(ids, np.int32)
    T, k = ids.shape
    counts = np.empty(E, np.int32)
    kept = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    slot_row = np.empty((T, k), np.int32)
    row_token = np.full(max(T * k, 1), -1, np.int32)
    dropped = np.empty((T, k), np.uint8)
    lib.oracle_dispatch(T, E, k, _ptr(ids), int(C), _ptr(counts), _ptr(kept), _ptr(offsets),
                        _ptr(slot_row), _ptr(row_token), _ptr(dropped))
    R = int(offsets[E])
    return Dispatch(counts, kept, offsets, slot_row, row_token[:R].copy(), dropped)


def dispatch_priority(ids, p, E: int, C: int, force=None, lib=None) -> Dispatch:
    """Dispatch whose capacity cut keeps each expert's C highest-score pairs.
    ``force`` [T,k] int8: +1 / -1 place a pair above / below every score."""
    lib = lib or load()
    ids = np.ascontiguousarray(ids, np.int32)
    p = np.ascontiguousarray(p, np.float64)
    fo = None if force is None else np.ascontiguousarray(force, np.int8)
    T, k = ids.shape
    assert p.shape == (T, E)
    counts = np.empty(E, np.int32)
    kept = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    slot_row = np.empty((T, k), np.int32)
    row_token = np.full(max(T * k, 1), -1, np.int32)
    dropped = np.empty((T, k), np.uint8)
    lib.oracle_dispatch_priority(T, E, k, _ptr(ids), _ptr(p), _ptr(fo), int(C), _ptr(counts),
                                 _ptr(kept), _ptr(offsets), _ptr(slot_row), _ptr(row_token),
                                 _ptr(dropped))
    R = int(offsets[E])
    return Dispatch(counts, kept, offsets, slot_row, row_token[:R].copy(), dropped)


def ec_capacity(c: float, k: int, T: int, E: int, lib=None) -> int:
    """Tokens each expert takes under expert-choice routing."""
    lib = lib or load()
    return int(lib.oracle_ec_capacity(float(c), k, T, E))


@dataclass
class ExpertChoice:
    r: int
    row_token: np.ndarray  # [E*r] token of each row; expert e owns rows e*r .. e*r+r-1
    row_gate: np.ndarray   # [E*r] gate (the router score) of each row


def expert_choice(p, r: int, force=None, lib=None) -> ExpertChoice:
    """Each expert's r highest-score tokens.  ``force`` [E,T] int8: +1 / -1
    place (e, t) above / below every score for the pick."""
    lib = lib or load()
    p = np.ascontiguousarray(p, np.float64)
    T, E = p.shape
    fo = None if force is None else np.ascontiguousarray(force, np.int8)
    rt = np.empty(max(E * r, 1), np.int32)
    rg = np.empty(max(E * r, 1), np.float64)
    lib.oracle_expert_choice(T, E, int(r), _ptr(p), _ptr(fo), _ptr(rt), _ptr(rg))
    return ExpertChoice(int(r), rt[:E * r].copy(), rg[:E * r].copy())


def swiglu_row(xrow, w1, w3, w2, lib=None) -> np.ndarray:
    lib = lib or load()
    xrow, w1, w3, w2 = map(_u16, (xrow, w1, w3, w2))
    Mw, d = w1.shape
    out = np.empty(d, np.float64)
    lib.oracle_swiglu_row(d, Mw, _ptr(xrow), _ptr(w1), _ptr(w3), _ptr(w2), _ptr(out))
    return out


def expert_rows(x_rows, expert, w1, w3, w2, lib=None) -> np.ndarray:
    """E_{expert[r]}(x_rows[r]) for each row; w1/w3 [E][M][d], w2 [E][d][M]."""
    lib = lib or load()
    x_rows, w1, w3, w2 = map(_u16, (x_rows, w1, w3, w2))
    n, d = x_rows.shape
    M = w1.shape[1]
    expert = np.ascontiguousarray(expert, np.int32)
    out = np.empty((n, d), np.float64)
    lib.oracle_expert_rows(n, d, M, _ptr(x_rows), _ptr(expert), _ptr(w1), _ptr(w3), _ptr(w2),
                           _ptr(out))
    return out


def layer_tokens(x, routing_ids, gates, dropped, w1, w3, w2, ws1=None, ws3=None, ws2=None,
                 sel=None, lib=None) -> np.ndarray:
    lib = lib or load()
    x, w1, w3, w2 = map(_u16, (x, w1, w3, w2))
    T, d = x.shape
    E, M = w1.shape[0], w1.shape[1]
    k = routing_ids.shape[1]
    Ms = 0 if ws1 is None else ws1.shape[0]
    if ws1 is not None:
        ws1, ws3, ws2 = map(_u16, (ws1, ws3, ws2))
    sel = np.arange(T, dtype=np.int32) if sel is None else np.ascontiguousarray(sel, np.int32)
    ids = np.ascontiguousarray(routing_ids, np.int32)
    g = np.ascontiguousarray(gates, np.float64)
    dr = np.ascontiguousarray(dropped, np.uint8)
    y = np.empty((len(sel), d), np.float64)
    lib.oracle_layer_tokens(T, d, M, E, k, Ms, _ptr(x), _ptr(ids), _ptr(g), _ptr(dr),
                            _ptr(w1), _ptr(w3), _ptr(w2), _ptr(ws1), _ptr(ws3), _ptr(ws2),
                            len(sel), _ptr(sel), _ptr(y))
    return y


def ec_layer_tokens(x, ec: ExpertChoice, w1, w3, w2, ws1=None, ws3=None, ws2=None, sel=None,
                    lib=None) -> np.ndarray:
    lib = lib or load()
    x, w1, w3, w2 = map(_u16, (x, w1, w3, w2))
    T, d = x.shape
    E, M = w1.shape[0], w1.shape[1]
    Ms = 0 if ws1 is None else ws1.shape[0]
    if ws1 is not None:
        ws1, ws3, ws2 = map(_u16, (ws1, ws3, ws2))
    sel = np.arange(T, dtype=np.int32) if sel is None else np.ascontiguousarray(sel, np.int32)
    rt = np.ascontiguousarray(ec.row_token, np.int32)
    rg = np.ascontiguousarray(ec.row_gate, np.float64)
    y = np.empty((len(sel), d), np.float64)
    lib.oracle_ec_layer_tokens(T, d, M, E, ec.r, Ms, _ptr(x), _ptr(rt), _ptr(rg), _ptr(w1),
                               _ptr(w3), _ptr(w2), _ptr(ws1), _ptr(ws3), _ptr(ws2), len(sel),
                               _ptr(sel), _ptr(y))
    return y


def combine(y_perm, slot_row, gates, y_shared=None, lib=None) -> np.ndarray:
    """y[t] = sum over kept slots of gates * y_perm[slot_row] (+ y_shared[t])."""
    lib = lib or load()
    y_perm = _u16(y_perm)
    slot_row = np.ascontiguousarray(slot_row, np.int32)
    T, k = slot_row.shape
    d = y_perm.shape[1]
    g = np.ascontiguousarray(gates, np.float64)
    ys = None if y_shared is None else _u16(y_shared)
    y = np.empty((T, d), np.float64)
    lib.oracle_combine(T, d, k, _ptr(y_perm), _ptr(slot_row), _ptr(g), _ptr(ys), _ptr(y))
    return y


def alf_bias_update(counts, T: int, k: int, gamma: float, bias, lib=None) -> np.ndarray:
    """ALF-LB step: b + gamma * sign(kT/E - n_e), fp32."""
    lib = lib or load()
    counts = np.ascontiguousarray(counts, np.int32)
    E = counts.shape[0]
    b = np.ascontiguousarray(bias, np.float32)
    out = np.empty(E, np.float32)
    lib.oracle_alf_bias_update(E, T, k, _ptr(counts), float(gamma), _ptr(b), _ptr(out))
    return out


@dataclass
class Losses:
    f: np.ndarray
    P: np.ndarray
    L_bal: float
    L_z: float


def losses(counts, p, lse, k: int, lam: float = 0.01, lib=None, n_pairs=None) -> Losses:
    """f, P, L_bal, L_z; f_e = n_e / (k T), or n_e / n_pairs when given."""
    lib = lib or load()
    p = np.ascontiguousarray(p, np.float64)
    T, E = p.shape
    counts = np.ascontiguousarray(counts, np.int32)
    lse = np.ascontiguousarray(lse, np.float64)
    f = np.empty(E, np.float64)
    P = np.empty(E, np.float64)
    lb = ctypes.c_double()
    lz = ctypes.c_double()
    if n_pairs is None:
        lib.oracle_losses(T, E, k, _ptr(counts), _ptr(p), _ptr(lse), float(lam), _ptr(f),
                          _ptr(P), ctypes.byref(lb), ctypes.byref(lz))
    else:
        lib.oracle_losses_n(T, E, float(n_pairs), _ptr(counts), _ptr(p), _ptr(lse), float(lam),
                            _ptr(f), _ptr(P), ctypes.byref(lb), ctypes.byref(lz))
    return Losses(f, P, lb.value, lz.value)


# --------------------------------------------------------------------------- #
# Composition: the whole layer (routing -> dispatch -> experts -> combine).    #
# --------------------------------------------------------------------------- #
@dataclass
class LayerResult:
    routing: Routing
    disp: Dispatch
    C: int
    loss: Losses
    y: Optional[np.ndarray]      # [n_sel, d] fp64 (None if no tokens requested)
    sel: np.ndarray


def layer_forward(x, wr, w1, w3, w2, k, offset=None, sel_bias=None, ws1=None, ws3=None,
                  ws2=None, capacity_factor=0.0, lam=0.01, force_ids=None, force_mask=None,
                  sel=None, flags=0, lib=None) -> LayerResult:
    """Full oracle forward.  ``sel`` picks the tokens whose output y is computed
    (all by default; routing, dispatch and losses always cover every token)."""
    lib = lib or load()
    T = x.shape[0]
    E = wr.shape[0]
    logits = router_logits(x, wr, offset, lib=lib)
    r = route(logits, k, sel_bias, force_ids, force_mask, flags=flags & 3, lib=lib)
    C = capacity(capacity_factor, k, T, E, lib=lib)
    if flags & PRIORITY:
        disp = dispatch_priority(r.ids, r.p, E, C, lib=lib)
    else:
        disp = dispatch(r.ids, E, C, lib=lib)
    ls = losses(disp.counts, r.p, r.lse, k, lam, lib=lib)
    if sel is None:
        sel = np.arange(T, dtype=np.int32)
    y = None
    if len(sel) > 0:
        y = layer_tokens(x, r.ids, r.gates, disp.dropped, w1, w3, w2, ws1, ws3, ws2, sel,
                         lib=lib)
    return LayerResult(r, disp, C, ls, y, np.asarray(sel, np.int32))


@dataclass
class ECLayerResult:
    routing: Routing             # p, lse, entropy (ids/gates unused: k = 0 selection)
    ec: ExpertChoice
    loss: Losses
    y: Optional[np.ndarray]
    sel: np.ndarray


def ec_layer_forward(x, wr, w1, w3, w2, k, offset=None, ws1=None, ws3=None, ws2=None,
                     capacity_factor=0.0, lam=0.01, sel=None, flags=0, lib=None) -> ECLayerResult:
    """Expert-choice forward: each expert takes its r highest-score tokens."""
    lib = lib or load()
    T = x.shape[0]
    E = wr.shape[0]
    logits = router_logits(x, wr, offset, lib=lib)
    r0 = route(logits, 0, None, flags=flags & SIGMOID, lib=lib)
    r = ec_capacity(capacity_factor, k, T, E, lib=lib)
    ec = expert_choice(r0.p, r, lib=lib)
    counts = np.full(E, r, np.int32)
    ls = losses(counts, r0.p, r0.lse, k, lam, lib=lib, n_pairs=E * r)
    if sel is None:
        sel = np.arange(T, dtype=np.int32)
    y = None
    if len(sel) > 0:
        y = ec_layer_tokens(x, ec, w1, w3, w2, ws1, ws3, ws2, sel, lib=lib)
    return ECLayerResult(r0, ec, ls, y, np.asarray(sel, np.int32))

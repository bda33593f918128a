"""ctypes binding of libmoe_b300.so: one Python function per C entry point, same
names, arguments marshalled from torch tensors (device pointers, the current
CUDA stream).  No computation happens here; every step runs in the library's
kernels.  Errors from the library raise ``MoeError``."""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from .build import LIB

_P = ctypes.c_void_p
_lib = None

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_CUDA = -3
MOE_ERR_TIMEOUT = -4
MOE_ERR_WORKSPACE = -5
MOE_ERR_BOUNDS = -6


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {moe_error_string(code)} ({code})")


MOE_FLAG_SIGMOID = 1
MOE_FLAG_NO_RENORM = 2
MOE_FLAG_PRIORITY_CAPACITY = 4
MOE_FLAG_EXPERT_CHOICE = 8


class RouteOut(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("ids", "gates", "counts", "f", "P", "bal_loss",
                                                "z_loss", "importance", "importance_cv2",
                                                "entropy_mean")]


MOE_TUNE_NO_HALF_TILES = 1
MOE_TUNE_GEMM1_SPLIT = 2
MOE_TUNE_FUSED_GATHER = 4
MOE_TUNE_GATE_IN_EPILOGUE = 8
MOE_TUNE_SWAP_ALL_TAILS = 16
MOE_TUNE_TWO_CTAS_PER_SM = 32
MOE_TUNE_NO_PDL = 64


def _check_tuning_names(tuning):
    # ctypes would store an unknown keyword as a plain attribute and pass
    # nothing to the library
    known = {name for name, _ in Tuning._fields_}
    unknown = sorted(set(tuning) - known)
    if unknown:
        raise TypeError(f"unknown moe_tuning_t fields {unknown}; known: {sorted(known)}")


class Tuning(ctypes.Structure):
    """moe_tuning_t: scheduling choices of the expert GEMMs (all zero: the
    measured defaults)."""
    _fields_ = [("gemm1_tile", ctypes.c_int32), ("gemm2_tile", ctypes.c_int32),
                ("tile_order", ctypes.c_int32), ("tail_max_n", ctypes.c_int32),
                ("n_block", ctypes.c_int32), ("block_min_rows", ctypes.c_int32),
                ("options", ctypes.c_uint32), ("reserved", ctypes.c_uint32),
                ("wait_timeout_ns", ctypes.c_uint64)]


class Shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("M", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("n_shared", ctypes.c_int32),
                ("capacity_factor", ctypes.c_float), ("balance_coef", ctypes.c_float),
                ("flags", ctypes.c_uint32), ("reserved", ctypes.c_uint32),
                ("tuning", Tuning)]

    @classmethod
    def of(cls, T, d, M, E, k, n_shared=0, capacity_factor=0.0, balance_coef=0.01, flags=0,
           **tuning):
        """Shape with the default tuning; keyword arguments set moe_tuning_t
        fields (e.g. gemm1_tile=256, options=MOE_TUNE_FUSED_GATHER)."""
        _check_tuning_names(tuning)
        return cls(T, d, M, E, k, n_shared, capacity_factor, balance_coef, flags, 0,
                   Tuning(**tuning))

    def tuned(self, **tuning) -> "Shape":
        """A copy of this shape with the given moe_tuning_t fields changed."""
        _check_tuning_names(tuning)
        t = Tuning()
        ctypes.pointer(t)[0] = self.tuning
        for key, v in tuning.items():
            setattr(t, key, v)
        return Shape(self.T, self.d, self.M, self.E, self.k, self.n_shared, self.capacity_factor,
                     self.balance_coef, self.flags, 0, t)

    @property
    def Ms(self) -> int:
        return self.n_shared * self.M


def lib():
    """Loads libmoe_b300.so (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB):
        raise RuntimeError(f"{LIB} is missing: build it with top_routing_expert_lb_b300.build")
    L = ctypes.CDLL(LIB)
    S = ctypes.POINTER(Shape)
    i32, u64 = ctypes.c_int32, ctypes.c_uint64
    sz = ctypes.c_size_t
    L.moe_error_string.argtypes = [ctypes.c_int]
    L.moe_error_string.restype = ctypes.c_char_p
    L.moe_workspace_size.argtypes = [S, ctypes.POINTER(sz)]
    L.moe_capacity.argtypes = [S, ctypes.POINTER(ctypes.c_int64)]
    L.moe_max_rows.argtypes = [S, ctypes.POINTER(ctypes.c_int64)]
    L.moe_pack_w13.argtypes = [i32, i32, i32, _P, _P, _P, _P]
    L.moe_route.argtypes = [S] + [_P] * 11 + [_P, sz, _P]
    L.moe_permute.argtypes = [S] + [_P] * 7 + [_P, sz, _P]
    L.moe_grouped_ffn.argtypes = [S] + [_P] * 9 + [_P, sz, _P]
    L.moe_combine.argtypes = [S] + [_P] * 5 + [_P]
    L.moe_layer_forward.argtypes = [S] + [_P] * 17 + [_P, sz, _P]
    L.moe_layer_forward_host.argtypes = [S] + [_P] * 20 + [_P, sz, _P]
    L.moe_layer_forward_host_batches.argtypes = [S, ctypes.c_int32] + [_P] * 20 + [sz] + [_P] * 3
    L.moe_check_status.argtypes = [_P, ctypes.POINTER(ctypes.c_int), _P]
    L.moe_set_wait_timeout_ns.argtypes = [u64]
    L.moe_debug_timeout_probe.argtypes = [_P, sz, _P]
    L.moe_profile_enable.argtypes = [ctypes.c_int]
    L.moe_profile_collect.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int), _P, _P]
    L.moe_launch_count.argtypes = [ctypes.POINTER(ctypes.c_uint64)]
    L.moe_route_noalloc.argtypes = [S] + [_P] * 11 + [_P]
    L.moe_route_ex.argtypes = [S, _P, _P, _P, _P, ctypes.POINTER(RouteOut), _P, sz, _P]
    L.moe_alf_bias_update.argtypes = [S, _P, ctypes.c_float, _P, _P]
    L.moe_ec_capacity.argtypes = [S, ctypes.POINTER(ctypes.c_int64)]
    L.moe_ec_route.argtypes = [S] + [_P] * 10 + [_P, sz, _P]
    L.moe_ec_layer_forward.argtypes = [S] + [_P] * 15 + [_P, sz, _P]
    for name in ("moe_workspace_size", "moe_capacity", "moe_max_rows", "moe_pack_w13",
                 "moe_route", "moe_permute", "moe_grouped_ffn", "moe_combine",
                 "moe_layer_forward", "moe_layer_forward_host", "moe_layer_forward_host_batches", "moe_check_status",
                 "moe_set_wait_timeout_ns", "moe_debug_timeout_probe", "moe_profile_enable",
                 "moe_profile_collect", "moe_launch_count", "moe_route_noalloc",
                 "moe_route_ex", "moe_alf_bias_update"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if t.device.type == "cuda" and not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc: int, where: str):
    if rc != MOE_OK:
        raise MoeError(rc, where)


def moe_error_string(code: int) -> str:
    return lib().moe_error_string(code).decode()


def moe_workspace_size(shape: Shape) -> int:
    v = ctypes.c_size_t()
    _check(lib().moe_workspace_size(ctypes.byref(shape), ctypes.byref(v)), "moe_workspace_size")
    return v.value


def moe_capacity(shape: Shape) -> int:
    v = ctypes.c_int64()
    _check(lib().moe_capacity(ctypes.byref(shape), ctypes.byref(v)), "moe_capacity")
    return v.value


def moe_max_rows(shape: Shape) -> int:
    v = ctypes.c_int64()
    _check(lib().moe_max_rows(ctypes.byref(shape), ctypes.byref(v)), "moe_max_rows")
    return v.value


def alloc_workspace(shape: Shape, device="cuda") -> torch.Tensor:
    """Zero-initialised workspace (the status word must start at 0)."""
    return torch.zeros(max(moe_workspace_size(shape), 256), dtype=torch.uint8, device=device)


def moe_pack_w13(w1: torch.Tensor, w3: torch.Tensor, out: Optional[torch.Tensor] = None,
                 stream=None) -> torch.Tensor:
    """w1, w3: [G][Mw][d] (or [Mw][d]) bf16 -> packed [G][2Mw][d]."""
    squeeze = w1.dim() == 2
    if squeeze:
        w1, w3 = w1.unsqueeze(0), w3.unsqueeze(0)
    G, Mw, d = w1.shape
    if out is None:
        out = torch.empty((G, 2 * Mw, d), dtype=w1.dtype, device=w1.device)
    _check(lib().moe_pack_w13(G, Mw, d, _ptr(w1), _ptr(w3), _ptr(out), _stream(stream)),
           "moe_pack_w13")
    return out[0] if squeeze else out


def moe_route(shape, x, w_router, logit_offset, sel_bias, ids, gates, counts, f, P, bal_loss,
              z_loss, ws, stream=None):
    _check(lib().moe_route(ctypes.byref(shape), _ptr(x), _ptr(w_router), _ptr(logit_offset),
                           _ptr(sel_bias), _ptr(ids), _ptr(gates), _ptr(counts), _ptr(f),
                           _ptr(P), _ptr(bal_loss), _ptr(z_loss), _ptr(ws), ws.numel(),
                           _stream(stream)), "moe_route")


def moe_route_ex(shape, x, w_router, logit_offset, sel_bias, ws, ids=None, gates=None,
                 counts=None, f=None, P=None, bal_loss=None, z_loss=None, importance=None,
                 importance_cv2=None, entropy_mean=None, stream=None):
    """moe_route with the optional side outputs (importance, its CV^2, mean
    router entropy); every output is a device tensor or None."""
    out = RouteOut(*[None if t is None else t.data_ptr() for t in (
        ids, gates, counts, f, P, bal_loss, z_loss, importance, importance_cv2, entropy_mean)])
    _check(lib().moe_route_ex(ctypes.byref(shape), _ptr(x), _ptr(w_router), _ptr(logit_offset),
                              _ptr(sel_bias), ctypes.byref(out), _ptr(ws), ws.numel(),
                              _stream(stream)), "moe_route_ex")


def moe_alf_bias_update(shape, counts, gamma, sel_bias, stream=None):
    """In place: sel_bias += gamma * sign(k T / E - counts) (device tensors)."""
    _check(lib().moe_alf_bias_update(ctypes.byref(shape), _ptr(counts), float(gamma),
                                     _ptr(sel_bias), _stream(stream)), "moe_alf_bias_update")


def moe_route_noalloc(shape, x, w_router, logit_offset, sel_bias, ids, gates, counts, f, P,
                      bal_loss, z_loss, stream=None):
    """moe_route without a workspace, for callers that cannot allocate device
    memory: the library keeps the scratch in a static device array (T up to
    65536 tokens).  Calls sharing a device must not overlap on the GPU."""
    _check(lib().moe_route_noalloc(ctypes.byref(shape), _ptr(x), _ptr(w_router),
                                   _ptr(logit_offset), _ptr(sel_bias), _ptr(ids), _ptr(gates),
                                   _ptr(counts), _ptr(f), _ptr(P), _ptr(bal_loss), _ptr(z_loss),
                                   _stream(stream)), "moe_route_noalloc")


def moe_permute(shape, x, ids, offsets, slot_row, row_token, drop_mask, x_perm, ws,
                stream=None):
    _check(lib().moe_permute(ctypes.byref(shape), _ptr(x), _ptr(ids), _ptr(offsets),
                             _ptr(slot_row), _ptr(row_token), _ptr(drop_mask), _ptr(x_perm),
                             _ptr(ws), ws.numel(), _stream(stream)), "moe_permute")


def moe_grouped_ffn(shape, x_perm, offsets, w13, w2, y_perm, x, w13_shared, w2_shared,
                    y_shared, ws, stream=None):
    _check(lib().moe_grouped_ffn(ctypes.byref(shape), _ptr(x_perm), _ptr(offsets), _ptr(w13),
                                 _ptr(w2), _ptr(y_perm), _ptr(x), _ptr(w13_shared),
                                 _ptr(w2_shared), _ptr(y_shared), _ptr(ws), ws.numel(),
                                 _stream(stream)), "moe_grouped_ffn")


def moe_combine(shape, y_perm, slot_row, gates, y_shared, y, stream=None):
    _check(lib().moe_combine(ctypes.byref(shape), _ptr(y_perm), _ptr(slot_row), _ptr(gates),
                             _ptr(y_shared), _ptr(y), _stream(stream)), "moe_combine")


def moe_layer_forward(shape, x, w_router, logit_offset, sel_bias, w13, w2, w13_shared,
                      w2_shared, y, ids, gates, counts, drop_mask, f, P, bal_loss, z_loss, ws,
                      stream=None):
    _check(lib().moe_layer_forward(ctypes.byref(shape), _ptr(x), _ptr(w_router),
                                   _ptr(logit_offset), _ptr(sel_bias), _ptr(w13), _ptr(w2),
                                   _ptr(w13_shared), _ptr(w2_shared), _ptr(y), _ptr(ids),
                                   _ptr(gates), _ptr(counts), _ptr(drop_mask), _ptr(f), _ptr(P),
                                   _ptr(bal_loss), _ptr(z_loss), _ptr(ws), ws.numel(),
                                   _stream(stream)), "moe_layer_forward")


def moe_layer_forward_host(shape, x_host, x_dev, w_router, logit_offset, sel_bias, w13, w2,
                           w13_shared, w2_shared, y_dev, y_host, losses_host, ids, gates, counts,
                           drop_mask, f, P, bal_loss, z_loss, ws, stream=None):
    _check(lib().moe_layer_forward_host(
        ctypes.byref(shape), ctypes.c_void_p(x_host.data_ptr()), _ptr(x_dev), _ptr(w_router),
        _ptr(logit_offset), _ptr(sel_bias), _ptr(w13), _ptr(w2), _ptr(w13_shared),
        _ptr(w2_shared), _ptr(y_dev), ctypes.c_void_p(y_host.data_ptr()),
        ctypes.c_void_p(losses_host.data_ptr()), _ptr(ids), _ptr(gates), _ptr(counts),
        _ptr(drop_mask), _ptr(f), _ptr(P), _ptr(bal_loss), _ptr(z_loss), _ptr(ws), ws.numel(),
        _stream(stream)), "moe_layer_forward_host")


def moe_layer_forward_host_batches(shape, x_host, y_host, losses_host, x_dev, y_dev, loss_dev,
                                   w_router, logit_offset, sel_bias, w13, w2, w13_shared,
                                   w2_shared, ids, gates, counts, drop_mask, f, P, ws, stream=None,
                                   h2d_stream=None, d2h_stream=None):
    """x_host / y_host: [n][T][d] bf16 host tensors (pinned for overlap);
    losses_host [n][2] fp32 host; x_dev / y_dev [2][T][d], loss_dev [2][2]."""
    n = x_host.shape[0] if x_host.dim() == 3 else 0
    if y_host.shape != x_host.shape or losses_host.numel() < 2 * n:
        raise ValueError("moe_layer_forward_host_batches: host buffer shapes")
    _check(lib().moe_layer_forward_host_batches(
        ctypes.byref(shape), n, ctypes.c_void_p(x_host.data_ptr()),
        ctypes.c_void_p(y_host.data_ptr()), ctypes.c_void_p(losses_host.data_ptr()), _ptr(x_dev),
        _ptr(y_dev), _ptr(loss_dev), _ptr(w_router), _ptr(logit_offset), _ptr(sel_bias),
        _ptr(w13), _ptr(w2), _ptr(w13_shared), _ptr(w2_shared), _ptr(ids), _ptr(gates),
        _ptr(counts), _ptr(drop_mask), _ptr(f), _ptr(P), _ptr(ws), ws.numel(), _stream(stream),
        _stream(h2d_stream), _stream(d2h_stream)), "moe_layer_forward_host_batches")


def moe_ec_capacity(shape: Shape) -> int:
    v = ctypes.c_int64()
    _check(lib().moe_ec_capacity(ctypes.byref(shape), ctypes.byref(v)), "moe_ec_capacity")
    return v.value


def moe_ec_route(shape, x, w_router, logit_offset, row_token, row_gate, counts, f, P, bal_loss,
                 z_loss, ws, stream=None):
    _check(lib().moe_ec_route(ctypes.byref(shape), _ptr(x), _ptr(w_router), _ptr(logit_offset),
                              _ptr(row_token), _ptr(row_gate), _ptr(counts), _ptr(f), _ptr(P),
                              _ptr(bal_loss), _ptr(z_loss), _ptr(ws), ws.numel(),
                              _stream(stream)), "moe_ec_route")


def moe_ec_layer_forward(shape, x, w_router, logit_offset, w13, w2, w13_shared, w2_shared, y,
                         row_token, row_gate, counts, f, P, bal_loss, z_loss, ws, stream=None):
    _check(lib().moe_ec_layer_forward(
        ctypes.byref(shape), _ptr(x), _ptr(w_router), _ptr(logit_offset), _ptr(w13), _ptr(w2),
        _ptr(w13_shared), _ptr(w2_shared), _ptr(y), _ptr(row_token), _ptr(row_gate),
        _ptr(counts), _ptr(f), _ptr(P), _ptr(bal_loss), _ptr(z_loss), _ptr(ws), ws.numel(),
        _stream(stream)), "moe_ec_layer_forward")


def moe_check_status(ws, stream=None) -> int:
    v = ctypes.c_int()
    _check(lib().moe_check_status(_ptr(ws), ctypes.byref(v), _stream(stream)),
           "moe_check_status")
    return v.value


def moe_set_wait_timeout_ns(ns: int):
    _check(lib().moe_set_wait_timeout_ns(int(ns)), "moe_set_wait_timeout_ns")


def moe_debug_timeout_probe(ws, stream=None):
    _check(lib().moe_debug_timeout_probe(_ptr(ws), ws.numel(), _stream(stream)),
           "moe_debug_timeout_probe")


KERNEL_NAMES = {1: "router", 2: "finalize", 3: "tile_hist", 4: "scatter", 5: "gemm_swiglu",
                6: "gemm_down", 7: "combine", 8: "other", 9: "select", 10: "gather"}


KERNEL_IDS = {v: k for k, v in KERNEL_NAMES.items()}


def moe_profile_enable(on=True, kernels=None):
    """Bracket kernel launches with CUDA events: all of them, or only the
    named kernels (e.g. ["gemm_swiglu"])."""
    if not on:
        mask = 0
    elif kernels is None:
        mask = 1
    else:
        mask = 0
        for name in kernels:
            mask |= 1 << KERNEL_IDS[name]
    _check(lib().moe_profile_enable(mask), "moe_profile_enable")


def moe_profile_collect(cap: int = 1 << 16):
    """[(kernel name, ms), ...] in launch order since the last collect."""
    import numpy as np
    ids = np.zeros(cap, np.int32)
    ms = np.zeros(cap, np.float32)
    n = ctypes.c_int()
    _check(lib().moe_profile_collect(cap, ctypes.byref(n), ids.ctypes.data_as(_P),
                                     ms.ctypes.data_as(_P)), "moe_profile_collect")
    return [(KERNEL_NAMES.get(int(i), str(int(i))), float(t)) for i, t in
            zip(ids[:n.value], ms[:n.value])]


def moe_launch_count() -> int:
    v = ctypes.c_uint64()
    _check(lib().moe_launch_count(ctypes.byref(v)), "moe_launch_count")
    return v.value


class MoELayer:
    """Owns packed weights, outputs and the workspace of one layer shape and
    runs ``moe_layer_forward`` (``moe_ec_layer_forward`` when the shape has
    MOE_FLAG_EXPERT_CHOICE).  Weights are given in canonical form:
    w1, w3 [E][M][d], w2 [E][d][M], optional shared ws1, ws3 [Ms][d], ws2 [d][Ms]."""

    def __init__(self, shape: Shape, w_router, w1, w3, w2, ws1=None, ws3=None, ws2=None,
                 logit_offset=None, sel_bias=None, device="cuda"):
        self.shape = shape
        self.w_router = w_router.contiguous()
        self.w13 = moe_pack_w13(w1.contiguous(), w3.contiguous())
        self.w2 = w2.contiguous()
        self.w13_shared = None
        self.w2_shared = None
        if shape.n_shared > 0:
            self.w13_shared = moe_pack_w13(ws1.contiguous(), ws3.contiguous())
            self.w2_shared = ws2.contiguous()
        self.logit_offset = logit_offset
        self.sel_bias = sel_bias
        T, d, E, k = shape.T, shape.d, shape.E, shape.k
        dev = torch.device(device)
        self.ws = alloc_workspace(shape, dev)
        self.y = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
        self.ids = torch.empty((T, k), dtype=torch.int32, device=dev)
        self.gates = torch.empty((T, k), dtype=torch.float32, device=dev)
        self.drop_mask = torch.empty((T, k), dtype=torch.uint8, device=dev)
        self.counts = torch.empty(E, dtype=torch.int32, device=dev)
        self.f = torch.empty(E, dtype=torch.float32, device=dev)
        self.P = torch.empty(E, dtype=torch.float32, device=dev)
        self.losses = torch.empty(2, dtype=torch.float32, device=dev)
        self.expert_choice = bool(shape.flags & MOE_FLAG_EXPERT_CHOICE)
        if self.expert_choice:
            r = moe_ec_capacity(shape)
            self.r = r
            self.row_token = torch.empty(max(E * r, 1), dtype=torch.int32, device=dev)
            self.row_gate = torch.empty(max(E * r, 1), dtype=torch.float32, device=dev)

    def forward(self, x, stream=None):
        if self.expert_choice:
            moe_ec_layer_forward(self.shape, x, self.w_router, self.logit_offset, self.w13,
                                 self.w2, self.w13_shared, self.w2_shared, self.y, self.row_token,
                                 self.row_gate, self.counts, self.f, self.P, self.losses[0:1],
                                 self.losses[1:2], self.ws, stream)
            return self.y
        moe_layer_forward(self.shape, x, self.w_router, self.logit_offset, self.sel_bias,
                          self.w13, self.w2, self.w13_shared, self.w2_shared, self.y, self.ids,
                          self.gates, self.counts, self.drop_mask, self.f, self.P,
                          self.losses[0:1], self.losses[1:2], self.ws, stream)
        return self.y

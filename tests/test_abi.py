"""The C-ABI library builds, loads and exports every declared entry point; host
argument checks and host-side size logic behave as documented.  No compute
call is made (CPU only)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from top_routing_expert_lb_b300 import _binding as B
from top_routing_expert_lb_b300 import build as mbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "moe.h")


@pytest.fixture(scope="module")
def lib():
    mbuild.ensure_built()
    return B.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("moe_route", "moe_permute", "moe_grouped_ffn", "moe_combine", "moe_layer_forward",
              "moe_workspace_size", "moe_pack_w13"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_library_reads_no_environment():
    """Every scheduling choice comes through moe_shape_t.tuning: the sources
    read no environment variable."""
    csrc = os.path.join(os.path.dirname(HEADER), "..", "top_routing_expert_lb_b300", "csrc")
    for fn in os.listdir(csrc):
        if fn.endswith((".cu", ".cuh", ".h")):
            assert "getenv" not in open(os.path.join(csrc, fn)).read(), fn


def test_shape_struct_layout_matches_the_header():
    """moe_shape_t / moe_tuning_t as ctypes sees them: 80 and 40 bytes, the
    tuning block after the flags word and its padding word."""
    assert ctypes.sizeof(B.Tuning) == 40
    assert ctypes.sizeof(B.Shape) == 80
    assert B.Shape.tuning.offset == 40


@pytest.mark.parametrize("tune,code", [
    (dict(gemm1_tile=64), B.MOE_ERR_INVALID_ARG),
    (dict(gemm2_tile=192), B.MOE_ERR_INVALID_ARG),
    (dict(tile_order=3), B.MOE_ERR_INVALID_ARG),
    (dict(tail_max_n=8), B.MOE_ERR_INVALID_ARG),
    (dict(tail_max_n=129), B.MOE_ERR_INVALID_ARG),
    (dict(n_block=-1), B.MOE_ERR_INVALID_ARG),
    (dict(block_min_rows=-5), B.MOE_ERR_INVALID_ARG),
    (dict(options=128), B.MOE_ERR_INVALID_ARG),
    (dict(reserved=1), B.MOE_ERR_INVALID_ARG),
    (dict(options=B.MOE_TUNE_FUSED_GATHER, gemm1_tile=256), B.MOE_ERR_INVALID_ARG),
    (dict(gemm2_tile=256), B.MOE_ERR_UNSUPPORTED),   # d = 64 is not a multiple of 256
])
def test_tuning_fields_are_checked(lib, tune, code):
    s = B.Shape.of(64, 64, 128, 8, 2, **tune)
    v = ctypes.c_size_t()
    assert lib.moe_workspace_size(ctypes.byref(s), ctypes.byref(v)) == code


@pytest.mark.parametrize("tune", [dict(), dict(gemm1_tile=128, gemm2_tile=128, tile_order=1,
                                               tail_max_n=-1, n_block=1, block_min_rows=1,
                                               options=127, wait_timeout_ns=10**9)])
def test_valid_tuning_leaves_the_workspace_size_unchanged(lib, tune):
    base = B.Shape.of(4096, 256, 512, 8, 2, 1)
    assert B.moe_workspace_size(base.tuned(**tune)) == B.moe_workspace_size(base)


def test_error_strings(lib):
    for code in (0, -1, -2, -3, -4, -5):
        assert B.moe_error_string(code)
    assert B.moe_error_string(-99) == "unknown error"


def shape(**kw):
    base = dict(T=64, d=64, M=128, E=8, k=2, n_shared=0, capacity_factor=0.0,
                balance_coef=0.01, flags=0)
    base.update(kw)
    return B.Shape.of(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(k=9, E=8), B.MOE_ERR_INVALID_ARG),         # k > E
    (dict(k=-1), B.MOE_ERR_INVALID_ARG),
    (dict(T=-1), B.MOE_ERR_INVALID_ARG),
    (dict(d=100), B.MOE_ERR_UNSUPPORTED),            # d % 64
    (dict(d=0), B.MOE_ERR_INVALID_ARG),
    (dict(M=200), B.MOE_ERR_UNSUPPORTED),            # M % 128
    (dict(E=300, k=2), B.MOE_ERR_UNSUPPORTED),
    (dict(E=16, k=9), B.MOE_ERR_UNSUPPORTED),        # k > 8
    (dict(flags=16), B.MOE_ERR_UNSUPPORTED),
    (dict(flags=B.MOE_FLAG_PRIORITY_CAPACITY | B.MOE_FLAG_EXPERT_CHOICE), B.MOE_ERR_UNSUPPORTED),
    (dict(n_shared=9), B.MOE_ERR_UNSUPPORTED),
    (dict(capacity_factor=float("nan")), B.MOE_ERR_INVALID_ARG),
])
def test_shape_validation(lib, kw, code):
    s = shape(**kw)
    v = ctypes.c_size_t()
    assert lib.moe_workspace_size(ctypes.byref(s), ctypes.byref(v)) == code


def test_workspace_and_pointer_checks(lib):
    s = shape()
    need = B.moe_workspace_size(s)
    assert need > 0
    buf = (ctypes.c_uint8 * (need + 512))()
    base = (ctypes.addressof(buf) + 255) // 256 * 256
    fake = ctypes.c_void_p(base)                      # never dereferenced: checks fail first
    outs = [fake] * 9
    # no workspace
    assert lib.moe_route(ctypes.byref(s), fake, fake, None, None, *outs[:7], None, need,
                         None) == B.MOE_ERR_INVALID_ARG
    # workspace too small
    assert lib.moe_route(ctypes.byref(s), fake, fake, None, None, *outs[:7], fake, need - 1,
                         None) == B.MOE_ERR_WORKSPACE
    # misaligned workspace
    assert lib.moe_route(ctypes.byref(s), fake, fake, None, None, *outs[:7],
                         ctypes.c_void_p(base + 8), need, None) == B.MOE_ERR_INVALID_ARG
    # misaligned token pointer
    assert lib.moe_route(ctypes.byref(s), ctypes.c_void_p(base + 2), fake, None, None,
                         *outs[:7], fake, need, None) == B.MOE_ERR_INVALID_ARG
    # missing outputs of the layer
    assert lib.moe_layer_forward(ctypes.byref(s), fake, fake, None, None, fake, fake, None, None,
                                 fake, fake, fake, None, fake, fake, fake, fake, fake, fake,
                                 need, None) == B.MOE_ERR_INVALID_ARG
    # shared experts requested without their weights
    s2 = shape(n_shared=1)
    need2 = B.moe_workspace_size(s2)
    buf2 = (ctypes.c_uint8 * (need2 + 512))()
    base2 = ctypes.c_void_p((ctypes.addressof(buf2) + 255) // 256 * 256)
    assert lib.moe_grouped_ffn(ctypes.byref(s2), base2, base2, base2, base2, base2, base2, None,
                               None, base2, base2, need2, None) == B.MOE_ERR_INVALID_ARG
    # the batched host stream: argument checks come before anything is enqueued
    fwd_b = lib.moe_layer_forward_host_batches
    tail = [fake] * 13 + [fake, need, None, None, None]   # weights .. P, ws, ws_bytes, streams
    assert fwd_b(ctypes.byref(s), -1, fake, fake, fake, fake, fake, fake,
                 *tail) == B.MOE_ERR_INVALID_ARG            # negative batch count
    assert fwd_b(ctypes.byref(s), 2, fake, fake, None, fake, fake, fake,
                 *tail) == B.MOE_ERR_INVALID_ARG            # no host losses buffer
    assert fwd_b(ctypes.byref(s), 2, None, fake, fake, fake, fake, fake,
                 *tail) == B.MOE_ERR_INVALID_ARG            # no host tokens
    assert fwd_b(ctypes.byref(s), 2, fake, fake, fake, fake, fake, fake,
                 *tail[:13], fake, need - 1, None, None, None) == B.MOE_ERR_WORKSPACE
    assert fwd_b(ctypes.byref(s), 0, fake, fake, fake, fake, fake, fake, *tail) == B.MOE_OK
    ec = shape(flags=B.MOE_FLAG_EXPERT_CHOICE)
    assert fwd_b(ctypes.byref(ec), 1, fake, fake, fake, fake, fake, fake,
                 *tail) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_pack_w13(1, 100, 64, fake, fake, fake, None) == B.MOE_ERR_UNSUPPORTED
    assert lib.moe_set_wait_timeout_ns(0) == B.MOE_ERR_INVALID_ARG


def test_capacity_matches_oracle(lib):
    rng = np.random.default_rng(0)
    cases = [(1.25, 1, 32768, 128), (0.5, 2, 2, 4), (1.0, 1, 3, 2), (0.0, 2, 10, 4),
             (2.0, 6, 8192, 160)]
    for _ in range(200):
        cases.append((float(np.float32(rng.uniform(0.1, 3.0))), int(rng.integers(1, 9)),
                      int(rng.integers(1, 70000)), int(rng.integers(8, 257))))
    for c, k, T, E in cases:
        k = min(k, E)
        s = shape(T=T, E=E, k=k, capacity_factor=c)
        c32 = float(np.float32(c))
        assert B.moe_capacity(s) == oracle.capacity(c32, k, T, E), (c, k, T, E)
        C = oracle.capacity(c32, k, T, E)
        assert B.moe_max_rows(s) == (T * k if C < 0 else min(T * k, E * C))


def test_workspace_grows_with_shape(lib):
    a = B.moe_workspace_size(shape(T=4096, d=4096, M=14336, E=8, k=2))
    b = B.moe_workspace_size(shape(T=4096, d=4096, M=14336, E=8, k=2, capacity_factor=0.5))
    assert b < a
    # intermediate rows: x_perm, h, y_perm for 8192 rows at least
    assert a >= 8192 * (4096 * 2 * 2 + 14336 * 2)


def test_expert_choice_sizes_match_oracle(lib):
    rng = np.random.default_rng(3)
    cases = [(1.0, 2, 4096, 8), (0.0, 1, 3, 2), (5.0, 2, 10, 4), (1.25, 1, 32768, 128),
             (1.0, 6, 8192, 160), (0.5, 0, 100, 8)]
    for _ in range(100):
        cases.append((float(np.float32(rng.uniform(0.1, 4.0))), int(rng.integers(0, 9)),
                      int(rng.integers(0, 50000)), int(rng.integers(8, 257))))
    for c, k, T, E in cases:
        k = min(k, E)
        s = shape(T=T, E=E, k=k, capacity_factor=c, flags=B.MOE_FLAG_EXPERT_CHOICE)
        r = oracle.ec_capacity(float(np.float32(c)), k, T, E)
        assert B.moe_ec_capacity(s) == r, (c, k, T, E)
        assert B.moe_max_rows(s) == E * r
    # the expert-choice count needs the flag
    with pytest.raises(B.MoeError):
        B.moe_ec_capacity(shape())


def test_entry_points_check_the_routing_mode(lib):
    """Token-choice entry points refuse an expert-choice shape and the other
    way round; moe_permute cannot run the priority cut (it gets no scores).
    Every call here is refused by the host checks, so nothing is enqueued (the
    pointers are host addresses that are never dereferenced)."""
    ec = shape(flags=B.MOE_FLAG_EXPERT_CHOICE)
    tc = shape()
    prio = shape(capacity_factor=1.0, flags=B.MOE_FLAG_PRIORITY_CAPACITY)
    bufs = []

    def ws_for(s):
        need = B.moe_workspace_size(s)
        buf = (ctypes.c_uint8 * (need + 512))()
        bufs.append(buf)
        return ctypes.c_void_p((ctypes.addressof(buf) + 255) // 256 * 256), need

    base, need = ws_for(ec)
    fake = base
    assert lib.moe_route(ctypes.byref(ec), fake, fake, None, None, *([fake] * 7), base, need,
                         None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_permute(ctypes.byref(ec), fake, fake, fake, fake, fake, fake, fake, base,
                           need, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_combine(ctypes.byref(ec), fake, fake, fake, None, fake,
                           None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_forward(ctypes.byref(ec), *([fake] * 17), base, need,
                                 None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_route_noalloc(ctypes.byref(ec), *([None] * 12)) == B.MOE_ERR_INVALID_ARG
    for s in (tc, prio):
        base, need = ws_for(s)
        assert lib.moe_ec_route(ctypes.byref(s), base, base, None, base, base, base, base, base,
                                base, base, base, need, None) == B.MOE_ERR_INVALID_ARG
        assert lib.moe_ec_layer_forward(ctypes.byref(s), *([base] * 15), base, need,
                                        None) == B.MOE_ERR_INVALID_ARG
    base, need = ws_for(prio)
    assert lib.moe_permute(ctypes.byref(prio), base, base, base, base, base, base, base, base,
                           need, None) == B.MOE_ERR_UNSUPPORTED
    # the extra scratch is sized only when a mode needs it
    assert B.moe_workspace_size(shape(capacity_factor=1.0)) < B.moe_workspace_size(prio)


def test_bounds_checked_build_compiles(tmp_path):
    """The debug build with every data-dependent device index range-checked
    (-DMOE_BOUNDS_CHECK) compiles and exports the same entry points."""
    out = str(tmp_path / "libmoe_bounds.so")
    mbuild.build(extra=("-DMOE_BOUNDS_CHECK",), out=out)
    L = ctypes.CDLL(out)
    for name in declared_functions():
        assert hasattr(L, name), name
    assert L.moe_error_string.restype is not None

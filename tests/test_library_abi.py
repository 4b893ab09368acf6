"""The C-ABI library builds, loads without a GPU, and exports every entry point
declared in include/moe.h.  Only host-side calls are made here."""

import ctypes
import os
import re

import pytest

from mxfp4_mixture_experts_router_gb300 import binding as B
from mxfp4_mixture_experts_router_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.lib()


def _declared():
    txt = open(os.path.join(ROOT, "include", "moe.h")).read()
    return re.findall(r"MOE_API\s+[\w\s\*]+?\b(\w+)\s*\(", txt)


def test_header_declares_the_abi():
    names = _declared()
    for fn in ("moe_route", "moe_expert_block", "moe_combine", "q8_0_block_matmul", "moe_workspace_size",
               "moe_get_error"):
        assert fn in names
    assert sorted(names) == sorted(B.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_host_only_queries(lib):
    kimi = B.desc(7168, 1536, 896, 16)
    assert B.moe_slab_bytes(kimi, B.MOE_FMT_MXFP4) == 17547264
    assert B.moe_slab_bytes(kimi, B.MOE_FMT_Q8_0) == 35094528
    a = B.moe_workspace_size(kimi, 1, 2)
    b = B.moe_workspace_size(kimi, 16, 2)
    assert 0 < a < b and b % 256 == 0
    o = B.moe_workspace_offsets(kimi, 16, 2)
    assert o.error_word == 0 and 0 < o.uexp < o.off < o.pair < o.h < o.shared_y < b
    assert B.q8_0_workspace_size(16, 7168, 3072) > 16 * 7168 * 6


def test_argument_errors_are_reported_before_any_launch(lib):
    kimi = B.desc(7168, 1536, 896, 16)
    bad_group = B.desc(7168, 1536, 896, 16, group=16)
    L = lib
    # NULL outputs / workspace -> invalid argument, nothing enqueued
    assert L.moe_route(ctypes.byref(kimi), 1, None, None, None, None, None, None, None, 16, 2, None) == \
        B.MOE_ERR_INVALID_ARG
    assert L.moe_route(ctypes.byref(bad_group), 1, 16, 16, None, None, 16, 16, 256, 16, 2, None) == \
        B.MOE_ERR_UNSUPPORTED
    # more rows than the workspace holds
    assert L.moe_route(ctypes.byref(kimi), 17, 16, 16, None, None, 16, 16, 256, 16, 2, None) == \
        B.MOE_ERR_UNSUPPORTED
    assert L.moe_combine(ctypes.byref(kimi), 1, None, None, None, None, 0, None, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_expert_block(ctypes.byref(kimi), 1, 0, None, None, None, None, 0, None, 16, None, None) == \
        B.MOE_ERR_INVALID_ARG
    # decode mode is limited to 16 rows
    pool = B.pool(256, 17547264 + 256 - 17547264 % 256, 1, B.MOE_FMT_MXFP4)
    assert L.moe_expert_block(ctypes.byref(kimi), 17, 0, ctypes.byref(pool), 256, None, None, 0, 256, 32, 256,
                              None) == B.MOE_ERR_UNSUPPORTED
    # MOE_MODE_AFTER_SHARED only with MOE_MODE_ROUTED_ONLY
    assert L.moe_expert_block(ctypes.byref(kimi), 1, B.MOE_MODE_AFTER_SHARED, ctypes.byref(pool), 256, None, None, 0,
                              256, 16, 256, None) == B.MOE_ERR_INVALID_ARG
    # q8_0: SwiGLU needs the up matrix; K must be a multiple of 256
    assert L.q8_0_block_matmul(1, 7168, 64, 256, 0, 256, 256, None, None, B.MOE_EPI_SWIGLU, 256, 256, None) == \
        B.MOE_ERR_INVALID_ARG
    assert L.q8_0_block_matmul(1, 100, 64, 256, 0, 256, 256, None, None, B.MOE_EPI_NONE, 256, 256, None) == \
        B.MOE_ERR_UNSUPPORTED

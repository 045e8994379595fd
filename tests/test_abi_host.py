"""CPU checks of the C-ABI library: it loads, exports every symbol the header
declares, and its host-side validation returns the documented status without
launching anything (no GPU needed: these paths return before any CUDA call)."""
import ctypes
import os
import re

import pytest

from mixture_experts_routing_router_gb300 import build as B
from mixture_experts_routing_router_gb300 import native as N

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    B.build()
    return N.lib()


def header_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    return sorted(set(re.findall(r"^MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_binding_exports():
    assert header_functions() == sorted(N.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in header_functions():
        assert hasattr(L, name), name


def test_nm_shows_only_the_abi(L):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", N.LIB_PATH], capture_output=True, text=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if " T " in line}
    moe = {s for s in syms if s.startswith("moe_")}
    assert moe == set(header_functions())


def shape(**kw):
    base = dict(tokens=64, hidden=256, experts=16, top_k=2, inter=512)
    base.update(kw)
    return N.make_shape(**base)


def test_workspace_size_is_host_only_and_grows_with_tokens(L):
    a = N.moe_workspace_size(shape())
    b = N.moe_workspace_size(shape(tokens=128))
    assert 0 < a < b
    # the whole-layer workspace holds x_perm, h and y_perm at least
    R = 64 * 2
    assert a >= R * 256 * 2 * 2 + R * 512 * 2


@pytest.mark.parametrize("bad", [
    dict(tokens=0), dict(hidden=12), dict(hidden=0), dict(experts=0), dict(experts=1025),
    dict(top_k=0), dict(top_k=17), dict(experts=64, top_k=33), dict(inter=20), dict(capacity=-1),
    dict(act=2), dict(shared=1, shared_inter=0), dict(shared=1, shared_inter=12),
])
def test_bad_shapes_are_rejected(L, bad):
    s = shape(**bad)
    if "capacity" in bad:
        s.capacity = bad["capacity"]
    n = ctypes.c_size_t(0)
    assert L.moe_workspace_size(ctypes.byref(s), ctypes.byref(n)) == N.MOE_ERR_INVALID_ARG


def test_null_and_misaligned_pointers_are_rejected_before_launch(L):
    s = shape()
    n = N.moe_workspace_size(s)
    fake_ws = ctypes.c_void_p(1 << 20)          # never dereferenced: validation fails first
    # null logits
    assert L.moe_route(ctypes.byref(s), None, ctypes.c_void_p(4096), ctypes.c_void_p(8192), fake_ws, n, None) \
        == N.MOE_ERR_INVALID_ARG
    # misaligned ids
    assert L.moe_route(ctypes.byref(s), ctypes.c_void_p(4096), ctypes.c_void_p(4100), ctypes.c_void_p(8192),
                       fake_ws, n, None) == N.MOE_ERR_INVALID_ARG
    # workspace too small
    assert L.moe_layer(ctypes.byref(s), ctypes.c_void_p(4096), None, None, ctypes.c_void_p(4096),
                       ctypes.c_void_p(4096), ctypes.c_void_p(4096), None, None, None, ctypes.c_void_p(4096),
                       fake_ws, n - 1, None) == N.MOE_ERR_INVALID_ARG
    # misaligned residual
    assert L.moe_combine(ctypes.byref(s), ctypes.c_void_p(4096), ctypes.c_void_p(4096), ctypes.c_void_p(4096),
                         None, ctypes.c_void_p(4100), ctypes.c_void_p(4096), fake_ws, n, None) \
        == N.MOE_ERR_INVALID_ARG
    # misaligned workspace
    assert L.moe_combine(ctypes.byref(s), ctypes.c_void_p(4096), ctypes.c_void_p(4096), ctypes.c_void_p(4096),
                         None, None, ctypes.c_void_p(4096), ctypes.c_void_p((1 << 20) + 16), n, None) \
        == N.MOE_ERR_INVALID_ARG
    # preselected path without weights
    assert L.moe_layer(ctypes.byref(s), None, ctypes.c_void_p(4096), None, ctypes.c_void_p(4096),
                       ctypes.c_void_p(4096), ctypes.c_void_p(4096), None, None, None, ctypes.c_void_p(4096),
                       fake_ws, n, None) == N.MOE_ERR_INVALID_ARG
    # shared experts without their weights
    s2 = shape(shared=2, shared_inter=64)
    n2 = N.moe_workspace_size(s2)
    assert L.moe_expert_up(ctypes.byref(s2), ctypes.c_void_p(4096), ctypes.c_void_p(4096), ctypes.c_void_p(4096),
                           None, None, ctypes.c_void_p(4096), fake_ws, n2, None) == N.MOE_ERR_INVALID_ARG


def test_status_strings(L):
    for code in range(9):
        assert len(N.status_string(code)) > 0
    assert N.status_string(3).startswith("an expert")


def test_nvfp4_entry_points_validate_on_the_host(L):
    fake = ctypes.c_void_p(4096)
    ws = ctypes.c_void_p(1 << 20)
    s = shape(shared=1, shared_inter=64)
    n = N.moe_workspace_size(s)
    assert L.moe_expert_up_nvfp4(ctypes.byref(s), fake, fake, fake, fake, fake, fake, ws, n,
                                 None) == N.MOE_ERR_UNSUPPORTED
    # two codes per byte: TMA-loaded rows need hidden and inter multiples of 32
    s = shape(hidden=272)
    n = N.moe_workspace_size(s)
    assert L.moe_layer_nvfp4(ctypes.byref(s), fake, None, None, fake, fake, fake, fake, fake, fake, fake, None, fake,
                             ws, n, None) == N.MOE_ERR_INVALID_ARG
    s = shape(inter=528)
    n = N.moe_workspace_size(s)
    assert L.moe_expert_down_nvfp4(ctypes.byref(s), fake, fake, fake, fake, fake, fake, ws, n,
                                   None) == N.MOE_ERR_INVALID_ARG
    # misaligned or missing block scales
    s = shape()
    n = N.moe_workspace_size(s)
    assert L.moe_expert_up_nvfp4(ctypes.byref(s), fake, fake, fake, ctypes.c_void_p(4100), fake, fake, ws, n,
                                 None) == N.MOE_ERR_INVALID_ARG
    assert L.moe_expert_down_nvfp4(ctypes.byref(s), fake, fake, fake, None, fake, fake, ws, n,
                                   None) == N.MOE_ERR_INVALID_ARG


def test_fp8_entry_points_validate_on_the_host(L):
    fake = ctypes.c_void_p(4096)
    # shared experts are not part of the FP8 entry points
    s = shape(shared=1, shared_inter=64)
    n = N.moe_workspace_size(s)
    ws = ctypes.c_void_p(1 << 20)
    assert L.moe_expert_up_fp8(ctypes.byref(s), fake, fake, fake, fake, fake, ws, n, None) == N.MOE_ERR_UNSUPPORTED
    # TMA-loaded FP8 rows need hidden and inter to be multiples of 16
    s = shape(hidden=264)
    n = N.moe_workspace_size(s)
    assert L.moe_layer_fp8(ctypes.byref(s), fake, None, None, fake, fake, fake, fake, fake, None, fake, ws, n,
                           None) == N.MOE_ERR_INVALID_ARG
    s = shape(inter=520)
    n = N.moe_workspace_size(s)
    assert L.moe_expert_down_fp8(ctypes.byref(s), fake, fake, fake, fake, fake, ws, n, None) == N.MOE_ERR_INVALID_ARG
    # misaligned scale pointer
    s = shape()
    n = N.moe_workspace_size(s)
    assert L.moe_expert_up_fp8(ctypes.byref(s), fake, fake, fake, ctypes.c_void_p(4100), fake, ws, n,
                               None) == N.MOE_ERR_INVALID_ARG

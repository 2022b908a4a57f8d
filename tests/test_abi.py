"""Host-side checks of the C ABI that need no GPU: the library loads, exports every
function its headers declare, sizes its workspace and rejects bad arguments before
touching the device."""
import ctypes
import os
import re

import pytest

import __graft_entry__
from conftest import ROOT

INCLUDE = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def L():
    __graft_entry__.build()
    from routed_moe_decode_gb300 import _lib
    return _lib


def _declared_functions():
    names = set()
    for h in ("moe.h", "moe_selftest.h"):
        text = open(os.path.join(INCLUDE, h)).read()
        names.update(re.findall(r"^MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text, flags=re.M))
    return names


def test_every_declared_function_is_exported(L):
    names = _declared_functions()
    assert len(names) >= 16
    lib = ctypes.CDLL(L.LIB_PATH)
    for n in sorted(names):
        assert hasattr(lib, n), n
    # the binding's table covers the public header
    public = set(re.findall(r"^MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(",
                            open(os.path.join(INCLUDE, "moe.h")).read(), flags=re.M))
    assert public <= set(L.SIGNATURES)


def test_status_strings(L):
    for rc in (0, -1, -2, -3, -4, -5):
        assert L.lib().moe_status_string(rc).decode().startswith("MOE_")
    assert L.lib().moe_status_string(7).decode() == "unknown moe_status"


def test_workspace_size_and_shape_checks(L):
    b1 = L.shape_of(4, 2048, 512, 512, 10)
    n = L.workspace_bytes(b1)
    assert n > 0 and n % 256 == 0
    # the per-route down outputs dominate and grow with T
    big = L.workspace_bytes(L.shape_of(8192, 2048, 512, 512, 10))
    assert big > 8192 * 10 * 2048 * 4
    assert L.check_shape(L.shape_of(4, 2048, 512, 512, 10)) == 0
    assert L.check_shape(L.shape_of(4, 2048, 512, 8, 10)) == L.MOE_ERR_INVALID_ARG  # k > E
    assert L.check_shape(L.shape_of(4, 2000, 512, 512, 10)) == L.MOE_ERR_UNSUPPORTED  # d % 128
    assert L.check_shape(L.shape_of(4, 2048, 512, 2048, 10)) == L.MOE_ERR_UNSUPPORTED  # E > 1024
    assert L.check_shape(L.shape_of(4, 2048, 512, 512, 40)) == L.MOE_ERR_UNSUPPORTED  # k > 32
    assert L.check_shape(L.shape_of(-1, 2048, 512, 512, 10)) == L.MOE_ERR_INVALID_ARG
    assert L.workspace_bytes(L.shape_of(4, 2000, 512, 512, 10)) == 0


def test_auto_algo_selection(L):
    # the wide kernel for >= 32 routed rows per expert on average; else the decode kernel for d
    # and ffn powers of two from 256 to 2048; the tcgen05 kernel otherwise
    assert L.auto_algo(L.shape_of(4, 2048, 512, 512, 10)) == L.ALGO_MMA
    assert L.auto_algo(L.shape_of(8192, 256, 2048, 64, 8)) == L.ALGO_WIDE  # 1024 rows per expert
    assert L.auto_algo(L.shape_of(8192, 2048, 512, 512, 10)) == L.ALGO_WIDE  # prefill chunk: 160
    assert L.auto_algo(L.shape_of(256, 2048, 512, 512, 10)) == L.ALGO_MMA  # decode batch: 5
    assert L.auto_algo(L.shape_of(1637, 2048, 512, 512, 10)) == L.ALGO_MMA  # just below 32 rows
    assert L.auto_algo(L.shape_of(1639, 2048, 512, 512, 10)) == L.ALGO_WIDE
    assert L.auto_algo(L.shape_of(4, 768, 512, 64, 8)) == L.ALGO_TCGEN05
    assert L.auto_algo(L.shape_of(4, 2048, 128, 64, 8)) == L.ALGO_TCGEN05
    assert L.auto_algo(L.shape_of(4, 4096, 512, 64, 8)) == L.ALGO_TCGEN05
    with pytest.raises(L.MoeError):
        L.auto_algo(L.shape_of(4, 2000, 512, 512, 10))


def test_unroute_fused_selection(L):
    # the decode kernel runs the un-route itself for T <= 8; other kernels never do
    assert L.unroute_fused(L.shape_of(4, 2048, 512, 512, 10))
    assert L.unroute_fused(L.shape_of(8, 2048, 512, 512, 10), L.ALGO_MMA)
    assert not L.unroute_fused(L.shape_of(9, 2048, 512, 512, 10))
    assert not L.unroute_fused(L.shape_of(32, 2048, 512, 512, 10))
    assert not L.unroute_fused(L.shape_of(257, 2048, 512, 512, 10))
    assert not L.unroute_fused(L.shape_of(4, 2048, 512, 512, 10), L.ALGO_TCGEN05)
    assert not L.unroute_fused(L.shape_of(4, 2048, 512, 512, 10), L.ALGO_SIMT)
    assert not L.unroute_fused(L.shape_of(4, 768, 512, 64, 8))
    with pytest.raises(L.MoeError):
        L.unroute_fused(L.shape_of(4, 2048, 512, 512, 10), 7)


def test_bad_arguments_rejected_on_host(L):
    lib = L.lib()
    s = L.shape_of(4, 256, 128, 16, 2)
    sp = ctypes.byref(s)
    assert lib.moe_route_topk(sp, None, None, None, None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_plan(sp, None, None, None, 0, None) == L.MOE_ERR_INVALID_ARG
    fake = ctypes.c_void_p(0x100000)
    assert lib.moe_plan(sp, fake, fake, None, 0, None) == L.MOE_ERR_WORKSPACE
    assert lib.moe_plan(sp, fake, fake, ctypes.c_void_p(0x100010), 1 << 30, None) == L.MOE_ERR_WORKSPACE
    assert lib.moe_plan(sp, fake, fake, fake, 16, None) == L.MOE_ERR_WORKSPACE
    # misaligned hidden, unknown algorithm
    args = [sp, ctypes.c_void_p(0x100002), fake, fake, 1.0, fake, fake, 1.0, None, fake, fake, 1 << 30]
    assert lib.moe_forward_algo(*args, 0, None) == L.MOE_ERR_INVALID_ARG
    args[1] = fake
    assert lib.moe_forward_algo(*args, 9, None) == L.MOE_ERR_INVALID_ARG
    # T = 0 is an empty, valid call that enqueues nothing
    z = L.shape_of(0, 256, 128, 16, 2)
    assert lib.moe_route_topk(ctypes.byref(z), None, None, None, None) == 0
    # the two-part expert entry takes part 0 or 1 only, and checks the shape first
    part_args = [fake, fake, 1.0, fake, fake, 1.0, fake, 1 << 30, 0]
    for part in (-1, 2):
        assert lib.moe_selftest_expert_part(sp, *part_args, part, None) == L.MOE_ERR_INVALID_ARG
    bad = L.shape_of(4, 200, 128, 16, 2)
    assert lib.moe_selftest_expert_part(ctypes.byref(bad), *part_args, 0, None) == L.MOE_ERR_UNSUPPORTED


def test_expert_range_bounds_rejected_on_host(L):
    """moe_layer_expert_range checks its expert block before touching anything."""
    lib = L.lib()
    s = L.shape_of(4, 256, 128, 16, 2)
    sp = ctypes.byref(s)
    rest = [None] * 2 + [None, None, 1.0, None, None, 1.0, None, None, None, None, None, 0, None]
    for e0, e1 in ((-1, 4), (4, 4), (9, 3), (8, 17)):
        assert lib.moe_layer_expert_range(sp, e0, e1, *rest) == L.MOE_ERR_INVALID_ARG
    bad = L.shape_of(4, 200, 128, 16, 2)  # d not a multiple of 128
    assert lib.moe_layer_expert_range(ctypes.byref(bad), 0, 8, *rest) == L.MOE_ERR_UNSUPPORTED
    # a valid block with missing weights fails on the host as moe_layer does
    assert lib.moe_layer_expert_range(sp, 0, 8, *rest) == L.MOE_ERR_INVALID_ARG


def test_layer_launch_counts(L):
    # one launch for a layer of at most eight tokens on the warp-MMA path; otherwise the
    # front, the expert kernel(s) and the un-route kernel
    cases = [((4, 2048, 512, 512, 10), 1),     # one-launch layer
             ((1, 256, 256, 16, 1), 1),
             ((8, 2048, 512, 512, 32), 1),     # 256 routes: the own front's limit
             ((8, 2048, 512, 2048 // 2, 33 - 1), 1),
             ((4, 256, 128, 16, 2), 3),        # ffn below the warp-MMA range: front, tcgen05, un-route
             ((32, 2048, 512, 512, 10), 3),    # front, decode kernel (8-row passes derived in the kernel), un-route
             ((256, 2048, 512, 512, 10), 3),   # the same up to 256 tokens
             ((512, 2048, 512, 512, 10), 3),   # front, warp-MMA batch kernel, un-route
             ((8192, 2048, 512, 512, 10), 9),  # router, 3-launch plan, staging, gather, task table, wide, un-route
             ((0, 2048, 512, 512, 10), 0)]
    for dims, n in cases:
        assert L.layer_launches(L.shape_of(*dims)) == n, dims
    with pytest.raises(L.MoeError):
        L.layer_launches(L.shape_of(4, 2048, 512, 512, 600))

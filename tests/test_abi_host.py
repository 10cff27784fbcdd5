"""Host-side checks of the C ABI (no GPU): the library loads and exports every
function include/*.h declares, and argument errors come back as the
documented status codes before anything touches a device."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from top_routing_grouped_moe_gb300 import _binding
    return _binding


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        names.update(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 17
    raw = ctypes.CDLL(lib.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n
    # and the binding covers every compute entry point
    for n in names:
        if n not in ("moe_version", "moe_status_string", "moe_last_cuda_error", "moe_device_status",
                     "moe_workspace_size", "moe_timing_begin", "moe_timing_end", "moe_timing_name",
                     "moe_timing_record",
                     "moe_mxfp8_rows", "moe_mxfp8_scales_bytes"):
            assert n in lib.SIGNATURES, n


def test_status_strings(lib):
    for code in range(0, 8):
        s = lib.status_string(code)
        assert isinstance(s, str) and s
    assert lib.moe_version() >> 16 >= 1


def test_workspace_size(lib):
    a = lib.moe_workspace_size(8192, 2048, 64, 4, 1024, 1024)
    b = lib.moe_workspace_size(16384, 2048, 64, 4, 1024, 1024)
    assert 0 < a < b
    with pytest.raises(lib.MoEError) as e:
        lib.moe_workspace_size(8192, 2048, 63, 4, 1024, 1024)   # E % 8 != 0
    assert e.value.status == lib.MOE_ERR_UNSUPPORTED
    with pytest.raises(lib.MoEError) as e:
        lib.moe_workspace_size(8192, 2048, 64, 4, 1000, 0)      # H % 128 != 0
    assert e.value.status == lib.MOE_ERR_UNSUPPORTED


P = 1 << 12  # stand-in device addresses (16-byte aligned); never dereferenced


@pytest.mark.parametrize("call,expect", [
    # k > 8
    (lambda L: L.moe_route_topk(None, None, None, P, 16, 0, 64, 9, None, P, P, None, 0, 0), 2),
    # missing outputs
    (lambda L: L.moe_route_topk(None, None, None, P, 16, 0, 64, 4, None, None, P, None, 0, 0), 1),
    # learned routing without logits buffer
    (lambda L: L.moe_route_topk(P, P, None, None, 16, 256, 64, 4, None, P, P, None, 0, 0), 1),
    # d not a multiple of 64
    (lambda L: L.moe_permute(P, P, 16, 100, 64, 4, 0, P, P, P, P, P, P, P, 1 << 20, 0), 2),
    # workspace too small
    (lambda L: L.moe_permute(P, P, 16, 128, 64, 4, 0, P, P, P, P, P, P, P, 16, 0), 3),
    # misaligned x
    (lambda L: L.moe_permute(P + 2, P, 16, 128, 64, 4, 0, P, P, P, P, P, P, P, 1 << 20, 0), 1),
    # E > 256
    (lambda L: L.moe_permute_static(P, P, 16, 128, 264, 4, 0, P, P, P, P, P, P, 0), 2),
    # shared expert without its buffers
    (lambda L: L.moe_grouped_swiglu(P, P, None, 16, 128, 8, 2, 128, 128, P, P, P, None, None, None,
                                    P, P, P, None, None, None, None, 0, 0), 1),
    # recompute: no a|u output
    (lambda L: L.moe_grouped_swiglu_recompute(P, P, None, 16, 128, 8, 2, 128, 0, P, P, None, None, None, None, 0),
     1),
    # recompute: shared expert without its a|u output
    (lambda L: L.moe_grouped_swiglu_recompute(P, P, P, 16, 128, 8, 2, 128, 128, P, P, P, P, P, None, 0), 1),
    # recompute: hidden width not a multiple of 128
    (lambda L: L.moe_grouped_swiglu_recompute(P, P, None, 16, 128, 8, 2, 96, 0, P, P, None, None, P, None, 0), 2),
    # failure self-check: limit out of range
    (lambda L: L.moe_selftest_wait_timeout(0, 0), 1),
    (lambda L: L.moe_selftest_wait_timeout(3_000_000, 0), 1),
    # combine: null y
    (lambda L: L.moe_unpermute_combine(P, None, P, P, 16, 128, 2, None, 0), 1),
    # backward workspace too small
    (lambda L: L.moe_grouped_swiglu_bwd(P, P, P, P, P, P, P, P, P, P, 16, 128, 8, 2, 128, 128, P, P, P, P, P, P,
                                        P, P, P, P, P, P, P, P, P, P, 64, 0), 3),
    # router backward: x without dW_r
    (lambda L: L.moe_route_topk_bwd(P, P, P, P, 16, 128, 8, 2, P, None, P, 1 << 20, 0), 1),
    # permute backward: dlogits without W_r
    (lambda L: L.moe_permute_bwd(P, None, P, P, None, 16, 128, 8, 2, P, P, 1 << 20, 0), 1),
    # balance loss: no loss output
    (lambda L: L.moe_router_balance_loss(P, P, 16, 8, 2, 0.02, None, None, None, P, 1 << 20, 0), 1),
    # balance loss: E not a multiple of 8
    (lambda L: L.moe_router_balance_loss(P, P, 16, 12, 2, 0.02, P, None, None, P, 1 << 20, 0), 2),
    # balance loss: workspace too small
    (lambda L: L.moe_router_balance_loss(P, P, 4096, 64, 2, 0.02, P, None, None, P, 16, 0), 3),
    # fused forward: no x to gather from
    (lambda L: L.moe_grouped_swiglu_fused(None, P, P, P, P, 16, 128, 8, 2, 128, 128, P, P, P, P, P, P, None, P, P,
                                          None, P, P, 0), 1),
    # fused forward: shared expert without its hidden buffer
    (lambda L: L.moe_grouped_swiglu_fused(P, P, P, P, P, 16, 128, 8, 2, 128, 128, P, P, P, P, P, P, None, P, P,
                                          None, None, P, 0), 1),
    # fused forward: misaligned expert-output buffer
    (lambda L: L.moe_grouped_swiglu_fused(P, P, P, P, P, 16, 128, 8, 2, 128, 0, P, P, P, None, None, None, None,
                                          P, P + 4, None, None, P, 0), 1),
    # fused forward: hidden width not a multiple of 128
    (lambda L: L.moe_grouped_swiglu_fused(P, P, P, P, P, 16, 128, 8, 2, 96, 0, P, P, P, None, None, None, None,
                                          P, P, None, None, P, 0), 2),
    # fused recompute: no slot map
    (lambda L: L.moe_grouped_swiglu_recompute_fused(P, None, P, 16, 128, 8, 2, 128, 0, P, P, None, None, P, None,
                                                    0), 1),
    # backward: x_perm given, dY_perm not (neither the copied nor the gather form)
    (lambda L: L.moe_grouped_swiglu_bwd(None, P, P, P, P, P, P, P, P, P, 16, 128, 8, 2, 128, 128, P, P, P, P, P, P,
                                        P, P, P, P, P, P, P, P, P, P, 1 << 30, 0), 1),
    # backward, gather form: no dY to gather from
    (lambda L: L.moe_grouped_swiglu_bwd(None, None, P, P, P, P, None, P, P, P, 16, 128, 8, 2, 128, 0, P, P, P,
                                        None, None, None, P, None, P, P, P, None, None, None, P, P, 1 << 30, 0), 1),
    # backward: a scale word without the dY it is taken from (Hs = 0 allows dY = NULL)
    (lambda L: L.moe_grouped_swiglu_bwd(P, None, P, P, P, P, P, None, P, None, 16, 128, 8, 2, 128, 0, P, P, P,
                                        None, None, None, P, None, P, P, P, None, None, None, P, P, 1 << 30, 0,
                                        dx_scale=P), 1),
    # permute, maps only: still needs its maps
    (lambda L: L.moe_permute(None, P, 16, 128, 64, 4, 0, P, P, P, None, P, None, P, 1 << 20, 0), 1),
])
def test_argument_errors_are_reported_on_the_host(lib, call, expect):
    with pytest.raises(lib.MoEError) as e:
        call(lib)
    assert e.value.status == expect


def test_launch_timing_host_side(lib):
    """The timing hook's host-side contract (no launch is made): argument
    errors, end without begin, an empty session, names out of range."""
    L = lib._lib
    assert L.moe_timing_begin(None, 4) == lib.MOE_ERR_INVALID_ARG
    assert L.moe_timing_begin(None, -1) == lib.MOE_ERR_INVALID_ARG
    arr = (ctypes.c_void_p * 2)(None, None)
    assert L.moe_timing_begin(arr, 2) == lib.MOE_ERR_INVALID_ARG  # NULL event handles
    n = ctypes.c_int(-1)
    assert L.moe_timing_end(ctypes.byref(n)) == lib.MOE_ERR_INVALID_ARG  # no session open
    assert L.moe_timing_begin(None, 0) == lib.MOE_OK
    assert L.moe_timing_end(ctypes.byref(n)) == lib.MOE_OK and n.value == 0
    assert L.moe_timing_name(0) == b"" and L.moe_timing_name(-1) == b""
    assert L.moe_timing_record(None, None) == lib.MOE_ERR_INVALID_ARG

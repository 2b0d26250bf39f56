"""The C ABI without a GPU: the library builds for sm_103a, loads, exports
every function the header declares, and rejects bad arguments on the host
before enqueuing anything."""
import ctypes
import os
import re

import pytest

from grouped_gemm_moe_gb300 import binding as B
from grouped_gemm_moe_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_gb300.h")


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_hot_path():
    names = declared_functions()
    for n in ["moe_route_topk", "moe_build_permutation", "moe_ep_layout", "moe_dispatch",
              "moe_grouped_ffn", "moe_combine", "moe_combine_backward", "moe_grouped_ffn_backward",
              "moe_dispatch_backward", "moe_route_topk_backward", "moe_workspace_size"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n
        assert n in B.SIGNATURES, n


def test_library_has_no_cpu_compute_symbols(lib):
    # the binding's only entry into compute is the C ABI; nothing else is exported under moe_
    out = os.popen(f"nm -D --defined-only {B.LIB_PATH}").read()
    exported = sorted(set(re.findall(r"\bT (moe_[a-z_0-9]+)", out)))
    assert exported == declared_functions()


def test_status_strings_and_version(lib):
    assert lib.moe_status_string(0) == b"ok"
    assert b"workspace" in lib.moe_status_string(3)
    assert lib.moe_version() >= 200


FAKE = ctypes.c_void_p(0x10000)          # aligned, never dereferenced
MIS = ctypes.c_void_p(0x10004)           # misaligned


def test_argument_validation_route(lib):
    f = lib.moe_route_topk
    assert f(FAKE, 16, 8, 9, 1, FAKE, FAKE, None) == B.MOE_ERR_INVALID_ARG        # K > E
    assert f(FAKE, 16, 64, 33, 1, FAKE, FAKE, None) == B.MOE_ERR_INVALID_ARG      # K > 32
    assert f(FAKE, 16, 2048, 2, 1, FAKE, FAKE, None) == B.MOE_ERR_INVALID_ARG     # E > 1024
    assert f(None, 16, 8, 2, 1, FAKE, FAKE, None) == B.MOE_ERR_INVALID_ARG
    assert f(MIS, 16, 8, 2, 1, FAKE, FAKE, None) == B.MOE_ERR_MISALIGNED
    assert f(None, 0, 8, 2, 1, None, None, None) == B.MOE_OK                      # empty batch
    g = lib.moe_route_topk_backward
    assert g(None, FAKE, FAKE, FAKE, 4, 8, 2, 0, FAKE, None) == B.MOE_ERR_INVALID_ARG  # renorm=0 needs logits


def test_argument_validation_permutation(lib):
    f = lib.moe_build_permutation
    assert f(FAKE, 16, 8, 2, FAKE, FAKE, FAKE, FAKE, FAKE, 0, None) == B.MOE_ERR_WORKSPACE
    assert f(FAKE, 16, 8, 2, FAKE, FAKE, FAKE, MIS, FAKE, 1 << 20, None) == B.MOE_ERR_MISALIGNED
    assert f(FAKE, 16, 2000, 2, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == B.MOE_ERR_INVALID_ARG
    g = lib.moe_ep_layout
    args = (FAKE, FAKE, FAKE, FAKE, None, FAKE, 1 << 20, None)
    assert g(FAKE, 16, 8, 2, 3, *args) == B.MOE_ERR_INVALID_ARG   # R does not divide E
    assert g(FAKE, 18, 8, 2, 4, *args) == B.MOE_ERR_INVALID_ARG   # R does not divide T
    assert g(FAKE, 16, 8, 2, 2, FAKE, FAKE, FAKE, FAKE, None, FAKE, 16, None) == B.MOE_ERR_WORKSPACE


def test_argument_validation_rows_and_gemm(lib):
    assert lib.moe_dispatch(FAKE, 16, 12, 2, FAKE, FAKE, None) == B.MOE_ERR_INVALID_ARG   # d % 8
    assert lib.moe_dispatch(FAKE, 16, 16, 2, FAKE, MIS, None) == B.MOE_ERR_MISALIGNED
    assert lib.moe_dispatch_scatter(FAKE, 16, 12, 2, FAKE, FAKE, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch_scatter(FAKE, 16, 16, 0, FAKE, FAKE, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch_scatter(FAKE, 16, 16, 33, FAKE, FAKE, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch_scatter(FAKE, 16, 16, 2, None, FAKE, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch_scatter(FAKE, 16, 16, 2, MIS, FAKE, None) == B.MOE_ERR_MISALIGNED
    assert lib.moe_dispatch_scatter(FAKE, 0, 16, 2, None, None, None) == B.MOE_OK
    assert lib.moe_combine(FAKE, FAKE, FAKE, 16, 2, 16, MIS, FAKE, None) == B.MOE_ERR_MISALIGNED
    assert lib.moe_dispatch_backward(FAKE, FAKE, 16, 0, 16, None, FAKE, None) == B.MOE_ERR_INVALID_ARG
    f = lib.moe_grouped_ffn
    ok = (FAKE, FAKE, 4, 256, 128, 256, FAKE, FAKE, FAKE, FAKE, FAKE, None)
    assert f(*ok, FAKE, 0, None) == B.MOE_ERR_WORKSPACE
    assert f(FAKE, FAKE, 4, 256, 128, 204, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 256,
             None) == B.MOE_ERR_INVALID_ARG                                           # I % 8
    assert f(FAKE, FAKE, 4, 256, 136, 200, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 0,
             None) == B.MOE_ERR_WORKSPACE                                  # d, I % 8: accepted
    f8 = lib.moe_grouped_ffn_fp8
    assert f8(FAKE, FAKE, 4, 256, 136, 256, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 1 << 20,
              None) == B.MOE_ERR_UNSUPPORTED                                     # MXFP8: d % 128
    assert f(FAKE, FAKE, 4, 256, 100, 256, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 256,
             None) == B.MOE_ERR_INVALID_ARG                                           # d % 8
    assert f(FAKE, FAKE, 4, 256, 128, 256, FAKE, FAKE, FAKE, MIS, FAKE, None, FAKE, 256,
             None) == B.MOE_ERR_MISALIGNED
    g = lib.moe_grouped_ffn_backward
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 256, 132, 256, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
             FAKE, FAKE, 1 << 30, None) == B.MOE_ERR_INVALID_ARG                       # d % 8
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 256, 128, 256, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
             FAKE, FAKE, 256, None) == B.MOE_ERR_WORKSPACE
    gd = lib.moe_grouped_ffn_backward_data
    assert gd(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 256, 128, 256, FAKE, FAKE, FAKE, FAKE, FAKE, 256,
              None) == B.MOE_ERR_WORKSPACE
    assert gd(FAKE, FAKE, None, FAKE, FAKE, 4, 256, 128, 256, FAKE, FAKE, FAKE, FAKE, FAKE, 256,
              None) == B.MOE_ERR_INVALID_ARG                                          # gu
    assert gd(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 256, 128, 256, None, FAKE, FAKE, FAKE, FAKE, 256,
              None) == B.MOE_ERR_INVALID_ARG                                          # w_gate
    assert gd(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 256, 136, 200, FAKE, FAKE, FAKE, FAKE, FAKE, 256,
              None) == B.MOE_ERR_WORKSPACE                                   # d, I % 8: accepted
    assert gd(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 256, 136, 204, FAKE, FAKE, FAKE, FAKE, FAKE, 256,
              None) == B.MOE_ERR_INVALID_ARG                                          # I % 8
    gw = lib.moe_grouped_ffn_backward_weights
    assert gw(FAKE, FAKE, FAKE, FAKE, 4, 256, 128, 256, FAKE, FAKE, FAKE, FAKE, 256,
              None) == B.MOE_ERR_WORKSPACE
    assert gw(FAKE, FAKE, FAKE, FAKE, 4, 256, 8, 8, FAKE, FAKE, FAKE, FAKE, 256,
              None) == B.MOE_ERR_WORKSPACE                                   # d, I = 8: accepted
    assert gw(FAKE, FAKE, FAKE, FAKE, 4, 256, 12, 8, FAKE, FAKE, FAKE, FAKE, 1 << 30,
              None) == B.MOE_ERR_INVALID_ARG                                          # d % 8
    assert gw(FAKE, FAKE, FAKE, FAKE, 4, 256, 128, 256, FAKE, None, FAKE, FAKE, 256,
              None) == B.MOE_ERR_INVALID_ARG                                          # dw_up
    assert gw(FAKE, FAKE, FAKE, FAKE, 4, 256, 128, 256, FAKE, MIS, FAKE, FAKE, 1 << 30,
              None) == B.MOE_ERR_MISALIGNED


def test_debug_wait_argument_checks(lib):
    assert lib.moe_debug_wait_timeout(None, 1000, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_debug_wait_timeout(FAKE, 0, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_debug_wait_timeout(FAKE, 20000000, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_debug_wait_timeout(MIS, 1000, None) == B.MOE_ERR_INVALID_ARG


def test_argument_validation_load_balance(lib):
    f = lib.moe_load_balance
    assert f(FAKE, FAKE, 16, 8, 2, FAKE, FAKE, FAKE, FAKE, 0, None) == B.MOE_ERR_WORKSPACE
    assert f(FAKE, FAKE, 0, 8, 2, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == B.MOE_ERR_INVALID_ARG
    assert f(FAKE, FAKE, 16, 8, 9, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == B.MOE_ERR_INVALID_ARG
    assert f(MIS, FAKE, 16, 8, 2, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == B.MOE_ERR_MISALIGNED
    g = lib.moe_load_balance_backward
    assert g(FAKE, FAKE, 16, 2048, 1.0, 1, FAKE, None) == B.MOE_ERR_INVALID_ARG
    assert g(None, FAKE, 16, 8, 1.0, 1, FAKE, None) == B.MOE_ERR_INVALID_ARG
    assert g(FAKE, FAKE, 0, 8, 1.0, 1, FAKE, None) == B.MOE_OK
    assert B.workspace_size(B.MOE_OP_LOAD_BALANCE, 8192, 128, 8) == B.WORKSPACE_HEADER + 256 * 128 * 4


def test_workspace_sizes(lib):
    hdr = B.WORKSPACE_HEADER
    assert B.workspace_size(B.MOE_OP_GROUPED_FFN, 8192, 128, 8, 1, 2048, 768) == hdr
    assert B.workspace_size(B.MOE_OP_GROUPED_FFN_BACKWARD, 8192, 128, 8, 1, 2048, 768) == \
        hdr + 8192 * 8 * 2 * 768 * 2 + 128 * 16 * (2048 + 768) * 2
    n = B.workspace_size(B.MOE_OP_BUILD_PERMUTATION, 8192, 128, 8)
    assert n >= hdr + 16 * 128 * 4
    assert B.workspace_size(B.MOE_OP_EP_LAYOUT, 8192, 128, 8, 3) == 0
    assert B.workspace_size(99, 8192, 128, 8) == 0

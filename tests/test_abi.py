"""The C ABI library: it builds, loads and exports every entry point that
include/moe.h declares; host-side argument checks return their status codes
before touching a device.  CPU only."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def libmoe():
    from token_dispatch_gb300 import build
    build.build()
    from token_dispatch_gb300 import _lib
    return _lib


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    return set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(\w+)\s*\(", text))


def test_header_declares_the_seven_calls():
    names = declared_symbols()
    for n in ("moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_route_bwd",
              "moe_permute_bwd", "mod_select"):
        assert n in names


def test_library_exports_every_declared_symbol(libmoe):
    lib = ctypes.CDLL(libmoe.LIB_PATH)
    for n in declared_symbols():
        assert hasattr(lib, n), n
    assert set(libmoe.EXPORTS) == declared_symbols()


def test_status_strings_and_version(libmoe):
    assert libmoe.moe_status_str(0) == "MOE_OK"
    assert libmoe.moe_status_str(libmoe.MOE_ERR_WORKSPACE) == "MOE_ERR_WORKSPACE"
    assert libmoe.moe_status_str(99) == "MOE_ERR_UNKNOWN"
    assert libmoe.moe_version() >= 100


def test_workspace_sizes(libmoe):
    L = libmoe
    # router: 8 or 16 experts stream in one launch without workspace; on the
    # GEMM path 64 token tiles of 128 leave SMs idle -> partial sums over slices of H
    assert L.moe_workspace_bytes(L.MOE_OP_ROUTE, 8192, 4096, 8, 2, 14336) == 0
    r = L.moe_workspace_bytes(L.MOE_OP_ROUTE, 8192, 4096, 32, 2, 14336)
    assert r >= 2 * 8192 * 32 * 4 and r % 256 == 0
    assert L.moe_workspace_bytes(L.MOE_OP_ROUTE, 16384, 2048, 64, 6, 1408) == 0
    # optional tail-split workspace of the bf16 expert FFN: independent of the sizes
    n_ffn = L.moe_workspace_bytes(L.MOE_OP_EXPERT_FFN, 8192, 4096, 8, 2, 14336)
    assert n_ffn > 0 and n_ffn == L.moe_workspace_bytes(L.MOE_OP_EXPERT_FFN, 16, 64, 2, 1, 64)
    d = L.moe_workspace_bytes(L.MOE_OP_DISPATCH, 8192, 4096, 8, 2, 14336)
    assert d >= (8192 // 256) * 8 * 4 and d % 256 == 0
    assert L.moe_workspace_bytes(L.MOE_OP_ROUTE_BWD, 8192, 4096, 8, 2, 0) >= 4096 * 8 * 4
    assert L.moe_workspace_bytes(L.MOE_OP_DISPATCH, -1, 1, 1, 1, 1) == 0


def test_argument_errors_are_reported_before_launch(libmoe):
    L = libmoe
    raw = L.lib()
    A = 1 << 20  # a fake, 16-byte aligned address: never dereferenced on these paths
    # K > E
    assert raw.moe_route(A, A, None, 4, 64, 4, 5, L.MOE_F32, A, A, A, None, 0, None) == L.MOE_ERR_INVALID_ARG
    # bad dtype
    assert raw.moe_route(A, A, None, 4, 64, 8, 2, 7, A, A, A, None, 0, None) == L.MOE_ERR_INVALID_ARG
    # misaligned pointer
    assert raw.moe_route(A + 4, A, None, 4, 64, 8, 2, L.MOE_F32, A, A, A, None, 0, None) == L.MOE_ERR_MISALIGNED
    # E not a multiple of 4
    assert raw.moe_route(A, A, None, 4, 64, 6, 2, L.MOE_F32, A, A, A, None, 0, None) == L.MOE_ERR_UNSUPPORTED
    # bf16 router with idle SMs needs its partial-sum workspace
    assert raw.moe_route(A, A, None, 1024, 2048, 32, 2, L.MOE_BF16, A, A, A, None, 0, None) == L.MOE_ERR_WORKSPACE
    # unknown route flags; renormalised-gate backward of the linear score
    assert raw.moe_route_ex(A, A, None, 4, 64, 8, 2, L.MOE_F32, 4, A, A, A, None, 0, None) == L.MOE_ERR_INVALID_ARG
    assert raw.moe_route_bwd(L.MOE_ROUTE_MOD_LINEAR | L.MOE_ROUTE_GATE_RENORM, A, None, None, A, A, 4, 64, 1, 1,
                             L.MOE_F32, None, A, None, A, 1 << 30, None) == L.MOE_ERR_INVALID_ARG
    # failure-detection probe: wait limit out of range
    assert raw.moe_check_wait_timeout(0, None) == L.MOE_ERR_INVALID_ARG
    assert raw.moe_check_wait_timeout((1 << 31) + 1, None) == L.MOE_ERR_INVALID_ARG
    # workspace too small
    need = L.moe_workspace_bytes(L.MOE_OP_DISPATCH, 1000, 64, 8, 2, 0)
    assert raw.moe_dispatch(A, A, 1000, 64, 8, 2, L.MOE_F32, A, A, A, A, A, need - 256, None) == L.MOE_ERR_WORKSPACE
    assert raw.moe_dispatch(A, A, 1000, 64, 8, 2, L.MOE_F32, A, A, A, A, None, need, None) == L.MOE_ERR_WORKSPACE
    # null required output
    assert raw.moe_combine(A, A, A, None, None, None, 4, 64, 2, L.MOE_F32, None, None) == L.MOE_ERR_INVALID_ARG
    # dx without dxs
    assert raw.moe_permute_bwd(A, A, A, A, None, None, None, 4, 64, 2, L.MOE_F32, None, None, None, A,
                               None) == L.MOE_ERR_INVALID_ARG
    # linear mode requires E = K = 1
    assert raw.moe_route_bwd(L.MOE_ROUTE_MOD_LINEAR, A, None, None, A, A, 4, 64, 4, 1, L.MOE_F32, None, A,
                             None, A, 1 << 30, None) == L.MOE_ERR_INVALID_ARG
    # capacity above the sequence length
    assert raw.mod_select(A, A, 2, 16, 64, 17, L.MOE_F32, A, A, None, A, None, None, None, 0,
                          None) == L.MOE_ERR_INVALID_ARG
    # expert backward: bf16 only; needs its [dg | du] workspace; g/u output needs bf16
    assert raw.moe_expert_ffn_bwd(A, A, 8, A, A, A, 2, 64, 64, L.MOE_F32, A, A, A, A, A, A, A, A, 1 << 20,
                                  None) == L.MOE_ERR_UNSUPPORTED
    assert raw.moe_expert_ffn_bwd(A, A, 8, A, A, A, 2, 64, 64, L.MOE_BF16, A, A, A, A, A, A, A, None, 0,
                                  None) == L.MOE_ERR_WORKSPACE
    assert raw.moe_expert_ffn_ex(A, A, 8, A, A, A, 2, 64, 64, L.MOE_F32, A, A, A, None, 0,
                                 None) == L.MOE_ERR_UNSUPPORTED
    assert L.moe_workspace_bytes(L.MOE_OP_EXPERT_FFN_BWD, 8192, 4096, 8, 2, 14336) >= 16384 * 2 * 14336 * 2
    # H not a multiple of the 16-byte vector
    assert raw.moe_expert_ffn(A, A, 8, A, A, A, 2, 60, 64, L.MOE_BF16, A, A, None, 0, None) == L.MOE_ERR_UNSUPPORTED


def test_product_package_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "token_dispatch_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f

"""The C ABI on the CPU: libdsc.so loads, exports every entry point that
include/dsc.h declares, and rejects bad arguments on the host before any
CUDA call (no GPU is touched: every case below returns during validation;
the non-null pointers are never dereferenced).
"""
import ctypes
import os
import re

import pytest

from lm_local_sequence_causal_b300 import dsc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsc.h")

P = ctypes.c_void_p
A = P(0x10000)          # 16-byte aligned stand-in address (never dereferenced)
A2 = P(0x20000)
A3 = P(0x30000)
A4 = P(0x40000)
A5 = P(0x50000)
MIS = P(0x10002)        # misaligned stand-in address


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dsc_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    return dsc.load()


def test_header_declares_the_four_kernels_and_helpers():
    names = declared_functions()
    for n in ("dsc_headwise_fwd", "dsc_headwise_bwd", "dsc_lowrank_fwd", "dsc_lowrank_bwd",
              "dsc_lowrank_bwd_workspace_size", "dsc_status_string", "dsc_abi_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libdsc.so does not export {name}"


def test_status_strings(lib):
    assert dsc.status_string(dsc.DSC_OK) == "DSC_OK"
    assert dsc.status_string(dsc.DSC_ERR_WORKSPACE) == "DSC_ERR_WORKSPACE"
    assert dsc.abi_version() == 1


BF16, F32 = dsc.DSC_BF16, dsc.DSC_F32


@pytest.mark.parametrize("args,expect", [
    # (x, w, y, B, T, C, H, W, residual, dtype)
    ((A, A2, A3, 2, 8, 64, 1, 0, 1, BF16), dsc.DSC_ERR_INVALID_ARG),   # W = 0
    ((A, A2, A3, 2, 8, 64, 1, 5, 1, BF16), dsc.DSC_ERR_UNSUPPORTED),   # W > 4
    ((A, A2, A3, 2, 8, 64, 3, 4, 1, BF16), dsc.DSC_ERR_INVALID_ARG),   # C % H != 0
    ((A, A2, A3, 2, 8, 12, 1, 4, 1, BF16), dsc.DSC_ERR_ALIGNMENT),     # C % 8 != 0 (bf16)
    ((None, None, None, 0, 8, 12, 1, 4, 1, F32), dsc.DSC_OK),          # C % 4 == 0 is enough for fp32
    ((A, A2, A3, -1, 8, 64, 1, 4, 1, BF16), dsc.DSC_ERR_INVALID_ARG),  # B < 0
    ((None, A2, A3, 2, 8, 64, 1, 4, 1, BF16), dsc.DSC_ERR_INVALID_ARG),  # null x
    ((MIS, A2, A3, 2, 8, 64, 1, 4, 1, BF16), dsc.DSC_ERR_ALIGNMENT),   # misaligned x
    ((A, A, A, 2, 8, 64, 1, 4, 1, BF16), dsc.DSC_ERR_INVALID_ARG),     # y aliases x
    ((A, A2, A3, 2, 8, 64, 1, 4, 1, 7), dsc.DSC_ERR_INVALID_ARG),      # bad dtype
    ((None, None, None, 0, 8, 64, 1, 4, 1, BF16), dsc.DSC_OK),         # empty: no-op
    ((None, None, None, 3, 0, 64, 1, 4, 1, BF16), dsc.DSC_OK),         # empty: no-op
])
def test_headwise_fwd_validation(lib, args, expect):
    x, w, y, B, T, C, H, W, res, dt = args
    rc = lib.dsc_headwise_fwd(x, w, y, B, T, C, H, W, res, dt, None)
    assert rc == expect, dsc.status_string(rc)


def test_headwise_bwd_validation(lib):
    f = lib.dsc_headwise_bwd
    assert f(A, A2, A3, A4, A5, 2, 8, 64, 1, 9, 1, BF16, None) == dsc.DSC_ERR_UNSUPPORTED
    assert f(A, A2, A3, None, A5, 2, 8, 64, 1, 4, 1, BF16, None) == dsc.DSC_ERR_INVALID_ARG
    assert f(A, A2, A3, A4, MIS, 2, 8, 64, 1, 4, 1, BF16, None) == dsc.DSC_ERR_ALIGNMENT
    assert f(A, A2, A3, A, A5, 2, 8, 64, 1, 4, 1, BF16, None) == dsc.DSC_ERR_INVALID_ARG
    assert f(A, A2, A3, A4, A4, 2, 8, 64, 1, 4, 1, BF16, None) == dsc.DSC_ERR_INVALID_ARG
    assert f(None, None, None, None, None, 0, 5, 64, 1, 4, 1, F32, None) == dsc.DSC_OK


def test_lowrank_validation_and_workspace(lib):
    f = lib.dsc_lowrank_fwd
    # R out of range / H not built
    assert f(A, A2, A3, A4, 2, 8, 64, 1, 4, 0, 1, BF16, None) == dsc.DSC_ERR_INVALID_ARG
    assert f(A, A2, A3, A4, 2, 8, 64, 1, 4, 33, 1, BF16, None) == dsc.DSC_ERR_UNSUPPORTED
    assert f(A, A2, A3, A4, 2, 8, 96, 3, 4, 16, 1, BF16, None) == dsc.DSC_ERR_UNSUPPORTED
    assert f(A, MIS, A3, A4, 2, 8, 64, 1, 4, 16, 1, BF16, None) == dsc.DSC_ERR_ALIGNMENT
    ws = lib.dsc_lowrank_bwd_workspace_size
    n = ws(8, 2048, 6144, 1, 4, 16, BF16)
    assert n > 0 and n % 256 == 0
    assert ws(8, 2048, 6144, 1, 4, 40, BF16) == 0      # unsupported R
    assert ws(0, 2048, 6144, 1, 4, 16, BF16) == 0      # empty
    g = lib.dsc_lowrank_bwd
    # workspace missing or too small: rejected before launch
    assert g(A, A2, A3, A4, A5, P(0x60000), P(0x70000), None, 0,
             8, 2048, 6144, 1, 4, 16, 1, BF16, None) == dsc.DSC_ERR_WORKSPACE
    assert g(A, A2, A3, A4, A5, P(0x60000), P(0x70000), P(0x80000), n - 16,
             8, 2048, 6144, 1, 4, 16, 1, BF16, None) == dsc.DSC_ERR_WORKSPACE
    assert g(A, A2, A3, A4, A5, P(0x60000), P(0x70000), P(0x80008), n,
             8, 2048, 6144, 1, 4, 16, 1, BF16, None) == dsc.DSC_ERR_ALIGNMENT
    # dx aliasing x
    assert g(A, A2, A3, A4, A, P(0x60000), P(0x70000), P(0x80000), n,
             8, 2048, 6144, 1, 4, 16, 1, BF16, None) == dsc.DSC_ERR_INVALID_ARG


def test_binding_rejects_cpu_tensors():
    import torch
    x = torch.zeros(1, 4, 8)
    w = torch.zeros(1, 4, 8, 4)
    with pytest.raises(ValueError):
        dsc.headwise_fwd(x, w, 1)


def test_lowrank_path_query():
    q = dsc.dsc_lowrank_uses_tensor_cores
    import torch
    bf, f32 = torch.bfloat16, torch.float32
    # the headline low-rank workload and the sweep / linear-RNN shapes run on
    # tcgen05 forward (bit 0) and backward (bit 1)
    assert q(8, 2048, 6144, 1, 4, 16, bf) == 3
    assert q(32, 512, 5632, 1, 3, 16, bf) == 3
    assert q(2, 16384, 4096, 1, 4, 16, bf) == 3
    for R in (8, 24, 32):                              # ranks padded to 16 or 32 on chip
        assert q(2, 100, 256, 1, 2, R, bf) == 3
    # everything else takes the CUDA-core kernels
    assert q(8, 2048, 6144, 1, 4, 16, f32) == 0        # fp32 keeps exact fp32 filters
    for H in (2, 4, 8, 16, 32):                        # tied filters
        assert q(8, 2048, 6144, H, 4, 16, bf) == 3
    assert q(2, 100, 6144, 32, 3, 16, bf) == 2         # (64/H)*W = 6: U offsets off 16 B
    assert q(2, 100, 200, 8, 4, 16, bf) == 2           # rows of U (G*W = 100) off 16 B
    assert q(8, 2048, 6144, 1, 4, 12, bf) == 0         # R not a multiple of 8
    # invalid or unbuilt arguments
    assert q(8, 2048, 6144, 1, 4, 0, bf) == -1
    assert q(8, 2048, 6144, 1, 5, 16, bf) == -1
    assert q(8, 2048, 6144, 3, 4, 16, bf) == -1


def test_static_validation_and_workspace(lib):
    f = lib.dsc_static_fwd
    assert f(A, A2, A3, 2, 8, 60, 4, 1, BF16, None) == dsc.DSC_ERR_ALIGNMENT   # C % 8
    assert f(A, A2, A3, 2, 8, 64, 5, 1, BF16, None) == dsc.DSC_ERR_UNSUPPORTED  # W > 4
    assert f(A, A2, A, 2, 8, 64, 4, 1, BF16, None) == dsc.DSC_ERR_INVALID_ARG   # y aliases x
    assert f(A, MIS, A3, 2, 8, 64, 4, 1, BF16, None) == dsc.DSC_ERR_ALIGNMENT
    assert f(None, None, None, 0, 8, 64, 4, 1, BF16, None) == dsc.DSC_OK       # empty
    ws = lib.dsc_static_bwd_workspace_size
    n = ws(8, 2048, 6144, 4, BF16)
    # one fp32 partial per token range, channel and tap; a function of the shape only
    assert n > 0 and n % (6144 * 4 * 4) == 0 and n == ws(8, 2048, 6144, 4, BF16)
    assert ws(0, 2048, 6144, 4, BF16) == 0
    assert ws(8, 2048, 6144, 5, BF16) == 0
    g = lib.dsc_static_bwd
    assert g(A, A2, A3, A4, A5, None, 0, 8, 2048, 6144, 4, 1, BF16, None) == dsc.DSC_ERR_WORKSPACE
    assert g(A, A2, A3, A4, A5, P(0x60000), n - 16, 8, 2048, 6144, 4, 1, BF16,
             None) == dsc.DSC_ERR_WORKSPACE
    assert g(A, A2, A3, A4, A5, P(0x60008), n, 8, 2048, 6144, 4, 1, BF16,
             None) == dsc.DSC_ERR_ALIGNMENT
    assert g(A, A2, A3, A, A5, P(0x60000), n, 8, 2048, 6144, 4, 1, BF16,
             None) == dsc.DSC_ERR_INVALID_ARG                                   # dx aliases x
    assert g(A, A2, A3, A4, None, None, 0, 0, 8, 64, 4, 1, BF16,
             None) == dsc.DSC_ERR_INVALID_ARG                                   # empty, no dw


def test_selftest_entry_points_validate_on_the_host(lib):
    f = lib.dsc_lowrank_fwd_selftest_timeout
    u64 = ctypes.c_uint64
    ok_limit = u64(2_000_000)
    # limit out of range, empty problem: rejected before any CUDA call
    for lim in (0, 999, 2_000_000_000):
        assert f(A, A2, A3, A4, 2, 256, 128, 1, 4, 16, 1, BF16, u64(lim), None) == \
            dsc.DSC_ERR_INVALID_ARG
    assert f(A, A2, A3, A4, 0, 256, 128, 1, 4, 16, 1, BF16, ok_limit, None) == \
        dsc.DSC_ERR_INVALID_ARG
    # fp32 and R = 3 take the CUDA-core kernels, which have no self-test
    assert f(A, A2, A3, A4, 2, 256, 128, 1, 4, 16, 1, F32, ok_limit, None) == \
        dsc.DSC_ERR_UNSUPPORTED
    assert f(A, A2, A3, A4, 2, 256, 128, 1, 4, 3, 1, BF16, ok_limit, None) == \
        dsc.DSC_ERR_UNSUPPORTED
    assert f(A, MIS, A3, A4, 2, 256, 128, 1, 4, 16, 1, BF16, ok_limit, None) == \
        dsc.DSC_ERR_ALIGNMENT
    g = lib.dsc_lowrank_bwd_selftest_timeout
    assert g(A, A2, A3, A4, A5, P(0x60000), P(0x70000), None, 0, 2, 256, 128, 1, 4, 16, 1,
             BF16, ok_limit, None) == dsc.DSC_ERR_WORKSPACE
    assert g(A, A2, A3, A4, A5, P(0x60000), P(0x70000), P(0x80000), 1 << 30, 2, 256, 128, 1, 4,
             16, 1, BF16, u64(10), None) == dsc.DSC_ERR_INVALID_ARG


def test_proj_decode_selftest_validates_on_the_host(lib):
    # (h, Wp, w, state, y, B, D, C, H, W, residual, dtype, limit)
    f = lib.dsc_headwise_proj_decode_selftest_timeout
    u64 = ctypes.c_uint64
    ok_limit = u64(2_000_000)
    for lim in (0, 999, 2_000_000_000):
        assert f(A, A2, A3, A4, A5, 24, 1024, 1024, 16, 4, 1, BF16, u64(lim), None) == \
            dsc.DSC_ERR_INVALID_ARG
    assert f(A, A2, A3, A4, A5, 0, 1024, 1024, 16, 4, 1, BF16, ok_limit, None) == \
        dsc.DSC_ERR_INVALID_ARG
    # fewer than 17 sequences, or fp32: not the tcgen05 kernel
    assert f(A, A2, A3, A4, A5, 16, 1024, 1024, 16, 4, 1, BF16, ok_limit, None) == \
        dsc.DSC_ERR_UNSUPPORTED
    assert f(A, A2, A3, A4, A5, 24, 1024, 1024, 16, 4, 1, F32, ok_limit, None) == \
        dsc.DSC_ERR_UNSUPPORTED
    assert f(A, MIS, A3, A4, A5, 24, 1024, 1024, 16, 4, 1, BF16, ok_limit, None) == \
        dsc.DSC_ERR_ALIGNMENT
    assert f(A, A2, A3, A4, A, 24, 1024, 1024, 16, 4, 1, BF16, ok_limit, None) == \
        dsc.DSC_ERR_INVALID_ARG                                               # y aliases h


def test_proj_decode_validation(lib):
    # (h, Wp, w, state, y, B, D, C, H, W, residual, dtype)
    f = lib.dsc_headwise_proj_decode
    assert f(A, A2, A3, A4, A5, 8, 2044, 6144, 16, 4, 1, BF16, None) == dsc.DSC_ERR_ALIGNMENT
    assert f(A, A2, A3, A4, A5, 8, 2046, 6144, 16, 4, 1, F32, None) == dsc.DSC_ERR_ALIGNMENT
    assert f(A, A2, A3, A4, A5, 8, 0, 6144, 16, 4, 1, BF16, None) == dsc.DSC_ERR_INVALID_ARG
    assert f(A, A2, A3, A4, A5, 8, 2048, 6144, 16, 5, 1, BF16, None) == dsc.DSC_ERR_UNSUPPORTED
    assert f(A, A2, A3, A4, A5, 8, 2048, 6008, 16, 4, 1, BF16, None) == dsc.DSC_ERR_INVALID_ARG
    assert f(A, A2, A3, A4, A, 8, 2048, 6144, 16, 4, 1, BF16, None) == dsc.DSC_ERR_INVALID_ARG
    assert f(A, A2, A3, A5, A5, 8, 2048, 6144, 16, 4, 1, BF16, None) == dsc.DSC_ERR_INVALID_ARG
    assert f(A, A2, A3, A2, A5, 8, 2048, 6144, 16, 4, 1, BF16, None) == dsc.DSC_ERR_INVALID_ARG
    assert f(A, A2, A3, None, A5, 8, 2048, 6144, 16, 4, 1, BF16, None) == dsc.DSC_ERR_INVALID_ARG
    assert f(MIS, A2, A3, A4, A5, 8, 2048, 6144, 16, 4, 1, BF16, None) == dsc.DSC_ERR_ALIGNMENT
    assert f(None, None, None, None, None, 0, 2048, 6144, 16, 4, 1, BF16, None) == dsc.DSC_OK
    g = lib.dsc_lowrank_proj_decode
    # (h, Wp, z, U, state, y, B, D, C, H, W, R, residual, dtype)
    assert g(A, A2, A3, A4, A5, P(0x60000), 8, 2048, 6144, 1, 4, 33, 1, BF16,
             None) == dsc.DSC_ERR_UNSUPPORTED
    assert g(A, A2, A3, A4, A5, P(0x60000), 8, 2048, 6144, 1, 4, 0, 1, BF16,
             None) == dsc.DSC_ERR_INVALID_ARG
    assert g(A, A2, A3, None, A5, P(0x60000), 8, 2048, 6144, 1, 4, 16, 1, BF16,
             None) == dsc.DSC_ERR_INVALID_ARG
    assert g(A, A2, A3, A4, A5, P(0x60000), 8, 12, 6144, 1, 4, 16, 1, BF16,
             None) == dsc.DSC_ERR_ALIGNMENT

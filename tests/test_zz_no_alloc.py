"""dsc_lowrank_bwd_noalloc: the low-rank backward for callers that cannot
allocate device memory.

Some users of this library cannot call cudaMalloc -- a plugin inside a host
program that owns all device memory, a service that forbids allocation after
start-up, a latency-critical path that cannot afford the synchronisation an
allocation may cause.  They cannot provide the workspace dsc_lowrank_bwd
asks for, so this entry point takes its scratch from a fixed array inside
the library.  These tests call it through the C ABI (the ctypes binding)
and check that:
  - it gives bit for bit what the workspace-taking entry point gives (both
    run the same deterministic kernels and fixed-order reductions), on
    several calls in a row whose shapes, and so whose partial-sum layouts,
    differ: each call finds the previous call's leftovers in the shared
    array;
  - one call near the array's capacity (the QKV placement) also matches the
    fp64 oracle;
  - a problem too large for the array is refused before any work is
    enqueued;
  - no bounded wait in the kernels gave up.

The file is named so that pytest collects it last.
"""
import pytest
import torch

import oracle as orc
from lm_local_sequence_causal_b300 import dsc, synthetic as syn
from _parity import assert_grad

pytestmark = pytest.mark.gpu

MAX_BYTES = 32 << 20     # DSC_LOWRANK_BWD_NOALLOC_MAX_BYTES in include/dsc.h


@pytest.fixture(autouse=True)
def no_device_error():
    dsc.dsc_device_error(reset=True)
    yield
    torch.cuda.synchronize()
    assert dsc.dsc_device_error() == 0, "a bounded wait in the tensor-core kernels gave up"


def need_bytes(wl):
    return dsc.dsc_lowrank_bwd_workspace_size(wl.B, wl.T, wl.C, wl.H, wl.W, wl.R, wl.dtype)


def noalloc_and_reference(wl, seed):
    """(inputs, no-alloc outputs, workspace-entry-point outputs)."""
    inp = syn.make_inputs(wl, seed, device="cuda")
    x, z, U, dy = inp["x"], inp["z"], inp["U"], inp["dy"]
    dx, dz, dU = torch.empty_like(x), torch.empty_like(z), torch.empty_like(U)
    dsc.dsc_lowrank_bwd_noalloc(x, z, U, dy, dx, dz, dU, wl.H, wl.W, wl.residual)
    torch.cuda.synchronize()
    ref = dsc.lowrank_bwd(x, z, U, dy, wl.H, wl.W, wl.residual)
    torch.cuda.synchronize()
    return inp, (dx, dz, dU), ref


def assert_bitwise_equal(got, want):
    for g, w, name in zip(got, want, ("dx", "dz", "dU")):
        assert torch.equal(g, w), f"{name}: no-alloc result differs from dsc_lowrank_bwd"


# A call near the array's capacity, then smaller ones with other partial-sum
# layouts (tied filters, padded rank 32, another token split), each after
# the previous call's leftovers.
SEQUENCE = [
    syn.qkv_lowrank(),
    syn.Workload("noalloc_tied", B=2, T=512, C=1024, W=4, H=4, R=16),
    syn.Workload("noalloc_r32", B=3, T=333, C=768, W=3, H=1, R=32, zu_std=32 ** -0.5),
    syn.Workload("noalloc_small", B=2, T=512, C=1024, W=4, H=1, R=16),
]


def test_noalloc_matches_the_workspace_entry_point_on_calls_in_a_row():
    needs = [need_bytes(wl) for wl in SEQUENCE]
    assert all(0 < n <= MAX_BYTES for n in needs)
    assert needs[0] > 0.9 * MAX_BYTES          # the QKV call fills most of the array
    for i, wl in enumerate(SEQUENCE):
        inp, got, want = noalloc_and_reference(wl, seed=11 + i)
        assert_bitwise_equal(got, want)
        if i == 0:
            # and against the fp64 oracle: dz and dU in full, dx on sampled rows
            x, z, U, dy = inp["x"], inp["z"], inp["U"], inp["dy"]
            assert_grad(got[1], orc.lowrank_dz(x, z, U, dy, wl.H, wl.W), wl.dtype, "dz")
            assert_grad(got[2], orc.lowrank_dU(x, z, dy, wl.H, wl.W), wl.dtype, "dU")
            rows = syn.sample_rows(wl.B, wl.T, wl.W, 1024, 11)
            rdx, _ = orc.lowrank_bwd_rows(x, z, U, dy, wl.H, wl.W, wl.residual, rows=rows)
            flat = got[0].reshape(wl.B * wl.T, wl.C)[rows.cuda()]
            assert_grad(flat, rdx, wl.dtype, "dx")


def test_noalloc_twice_on_the_same_shape():
    wl = SEQUENCE[-1]
    a = noalloc_and_reference(wl, seed=21)
    b = noalloc_and_reference(wl, seed=22)
    assert_bitwise_equal(a[1], a[2])
    assert_bitwise_equal(b[1], b[2])


def test_noalloc_refuses_a_problem_larger_than_its_scratch():
    lib = dsc.load()
    B, T, C, H, W, R = 32, 2048, 6144, 1, 4, 16       # 64 Ki tokens at the QKV width
    need = dsc.dsc_lowrank_bwd_workspace_size(B, T, C, H, W, R, torch.bfloat16)
    assert need > MAX_BYTES
    # Refused during the size check, before any pointer is used or work enqueued.
    import ctypes
    fake = [ctypes.c_void_p(0x100000 * (i + 1)) for i in range(7)]
    rc = lib.dsc_lowrank_bwd_noalloc(*fake, B, T, C, H, W, R, 1, dsc.DSC_BF16, None)
    assert rc == dsc.DSC_ERR_WORKSPACE

"""dsc_lowrank_bwd_noalloc: the low-rank backward for callers that cannot
allocate device memory.

Some users of this library cannot call cudaMalloc -- a plugin inside a host
program that owns all device memory, a service that forbids allocation after
start-up, a latency-critical path that cannot afford the synchronisation an
allocation may cause.  They cannot provide the workspace dsc_lowrank_bwd
asks for, so this entry point takes its scratch from a fixed array inside
the library.  These tests call it through the C ABI and check that it gives
what the workspace-taking entry point gives, on two calls in a row (the
second call finds the first call's leftovers in the shared array), and that
a problem too large for the array is refused before any work is enqueued.

The file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

from lm_local_sequence_causal_b300 import dsc, synthetic as syn
from _parity import assert_grad

pytestmark = pytest.mark.gpu

MAX_BYTES = 32 << 20     # DSC_LOWRANK_BWD_NOALLOC_MAX_BYTES in include/dsc.h


def noalloc_entry():
    lib = dsc.load()
    f = lib.dsc_lowrank_bwd_noalloc
    P, I64, INT = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    f.argtypes = [P] * 7 + [I64] * 6 + [INT, INT, P]
    f.restype = INT
    return f


def ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_matches_the_workspace_entry_point_on_two_calls_in_a_row():
    f = noalloc_entry()
    wl = syn.Workload("noalloc", B=2, T=512, C=1024, W=4, H=1, R=16)
    need = dsc.dsc_lowrank_bwd_workspace_size(wl.B, wl.T, wl.C, wl.H, wl.W, wl.R, wl.dtype)
    assert 0 < need <= MAX_BYTES
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for seed in (11, 12):
        inp = syn.make_inputs(wl, seed, device="cuda")
        x, z, U, dy = inp["x"], inp["z"], inp["U"], inp["dy"]
        ref = dsc.lowrank_bwd(x, z, U, dy, wl.H, wl.W, True)
        dx, dz, dU = torch.empty_like(x), torch.empty_like(z), torch.empty_like(U)
        rc = f(ptr(x), ptr(z), ptr(U), ptr(dy), ptr(dx), ptr(dz), ptr(dU), wl.B, wl.T, wl.C,
               wl.H, wl.W, wl.R, 1, dsc.DSC_BF16, stream)
        assert rc == dsc.DSC_OK, dsc.status_string(rc)
        torch.cuda.synchronize()
        for got, want, name in zip((dx, dz, dU), ref, ("dx", "dz", "dU")):
            assert_grad(got, want.double().cpu(), wl.dtype, name)


def test_noalloc_refuses_a_problem_larger_than_its_scratch():
    f = noalloc_entry()
    B, T, C, H, W, R = 32, 2048, 6144, 1, 4, 16       # 64 Ki tokens at the QKV width
    need = dsc.dsc_lowrank_bwd_workspace_size(B, T, C, H, W, R, torch.bfloat16)
    assert need > MAX_BYTES
    # Refused during the size check, before any pointer is used or work enqueued.
    fake = [ctypes.c_void_p(0x100000 * (i + 1)) for i in range(7)]
    rc = f(*fake, B, T, C, H, W, R, 1, dsc.DSC_BF16, None)
    assert rc == dsc.DSC_ERR_WORKSPACE

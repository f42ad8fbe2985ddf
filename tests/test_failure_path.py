"""Failure path of the tensor-core low-rank kernels and of the tcgen05
merged decode kernel, exercised without a GPU fault.

Every wait of those kernels on an mbarrier is bounded: when it runs out the
waiting role records a code in the device error word, raises the CTA's abort
flag, lets the copies and MMAs it issued finish, and the CTA frees its TMEM
and returns.  The self-test entry points run the real forward and backward
with a short limit (2 ms here; 1 s in normal use) and a producer that issues
no loads, so the other roles' waits run out.  The tests check that the
kernels return, that dsc_device_error reports a wait code, and that the next
normal call on the same device runs and matches the fp64 oracle (which it
could not if a CTA had kept its TMEM or left the device in a bad state).
Nothing traps, faults or hangs: the waits simply expire.
"""
import time

import pytest
import torch

import oracle as orc
from lm_local_sequence_causal_b300 import dsc, synthetic as syn
from _parity import assert_fwd, assert_grad

pytestmark = pytest.mark.gpu

LIMIT_NS = 2_000_000
WAIT_CODES = {2, 3, 5}       # MMA issuer, epilogue, second MMA issuer (include/dsc.h)


def workload():
    return syn.Workload("selftest", B=2, T=512, C=1024, W=4, H=1, R=16)


def check_normal_call_after(wl, inp):
    """A normal forward and backward right after the failed call."""
    x, z, U, dy = inp["x"], inp["z"], inp["U"], inp["dy"]
    y = dsc.lowrank_fwd(x, z, U, wl.H, wl.W, wl.residual)
    dx, dz, dU = dsc.lowrank_bwd(x, z, U, dy, wl.H, wl.W, wl.residual)
    torch.cuda.synchronize()
    assert dsc.dsc_device_error() == 0
    assert_fwd(y, orc.lowrank_fwd(x, z, U, wl.H, wl.W, wl.residual), wl.dtype)
    rdx, rdz, rdU = orc.lowrank_bwd(x, z, U, dy, wl.H, wl.W, wl.residual)
    assert_grad(dx, rdx, wl.dtype, "dx")
    assert_grad(dz, rdz, wl.dtype, "dz")
    assert_grad(dU, rdU, wl.dtype, "dU")


def test_forward_wait_timeout_is_reported_and_the_device_recovers():
    wl = workload()
    assert dsc.dsc_lowrank_uses_tensor_cores(wl.B, wl.T, wl.C, wl.H, wl.W, wl.R, wl.dtype) & 1
    inp = syn.make_inputs(wl, 3, device="cuda")
    y = torch.empty_like(inp["x"])
    torch.cuda.synchronize()
    dsc.dsc_device_error(reset=True)
    t0 = time.perf_counter()
    dsc.dsc_lowrank_fwd_selftest_timeout(inp["x"], inp["z"], inp["U"], y, wl.H, wl.W, LIMIT_NS)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    code = dsc.dsc_device_error(reset=True)
    assert code in WAIT_CODES, f"error word {code}"
    assert elapsed < 5.0, f"the kernel took {elapsed:.2f} s to give up"
    assert dsc.dsc_device_error() == 0
    check_normal_call_after(wl, inp)


def test_backward_wait_timeout_is_reported_and_the_device_recovers():
    wl = workload()
    assert dsc.dsc_lowrank_uses_tensor_cores(wl.B, wl.T, wl.C, wl.H, wl.W, wl.R, wl.dtype) & 2
    inp = syn.make_inputs(wl, 4, device="cuda")
    x, z, U, dy = inp["x"], inp["z"], inp["U"], inp["dy"]
    dx, dz, dU = torch.empty_like(x), torch.empty_like(z), torch.empty_like(U)
    ws = dsc.lowrank_workspace(x, z, wl.H, wl.W)
    torch.cuda.synchronize()
    dsc.dsc_device_error(reset=True)
    t0 = time.perf_counter()
    dsc.dsc_lowrank_bwd_selftest_timeout(x, z, U, dy, dx, dz, dU, ws, wl.H, wl.W, LIMIT_NS)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    code = dsc.dsc_device_error(reset=True)
    assert code in WAIT_CODES, f"error word {code}"
    assert elapsed < 5.0, f"the kernels took {elapsed:.2f} s to give up"
    check_normal_call_after(wl, inp)


def test_merged_decode_cluster_kernel_times_out_and_the_device_recovers():
    # the tcgen05 merged decode: CTAs in clusters of 2 to 8 that meet at two
    # cluster barriers; with no loads issued the MMA issuer's wait runs out,
    # and every CTA must still pass both barriers and free its TMEM
    B, D, C, H, W = 24, 1024, 1024, 16, 4
    inp = syn.proj_decode_inputs(B, D, C, H, W, 0, torch.bfloat16, seed=6, device="cuda")
    y = torch.empty(B, C, dtype=torch.bfloat16, device="cuda")
    st = inp["state"].clone()
    torch.cuda.synchronize()
    dsc.dsc_device_error(reset=True)
    t0 = time.perf_counter()
    dsc.dsc_headwise_proj_decode_selftest_timeout(inp["h"], inp["Wp"], inp["w"], st, y, H,
                                                  LIMIT_NS)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    code = dsc.dsc_device_error(reset=True)
    assert code in WAIT_CODES, f"error word {code}"
    assert elapsed < 5.0, f"the kernel took {elapsed:.2f} s to give up"
    # a normal call on the same device afterwards
    st0 = inp["state"].clone()
    ry, rstate, _ = orc.headwise_proj_decode(inp["h"], inp["Wp"], inp["w"], st0, H, True)
    st = inp["state"].clone()
    dsc.dsc_headwise_proj_decode(inp["h"], inp["Wp"], inp["w"], st, y, H, True)
    torch.cuda.synchronize()
    assert dsc.dsc_device_error() == 0
    assert_fwd(y, ry, torch.bfloat16)
    assert torch.equal(st[:, 1:].double().cpu(), rstate[:, 1:])
    # shapes that do not take the tcgen05 kernel have no self-test
    with pytest.raises(dsc.DSCError) as e:
        dsc.dsc_headwise_proj_decode_selftest_timeout(inp["h"][:8], inp["Wp"], inp["w"][:8],
                                                      st[:8], y[:8], H, LIMIT_NS)
    assert e.value.status == dsc.DSC_ERR_UNSUPPORTED


def test_selftest_rejects_bad_limits_and_non_tensor_core_shapes():
    wl = workload()
    inp = syn.make_inputs(wl, 5, device="cuda")
    y = torch.empty_like(inp["x"])
    for bad in (0, 999, 2_000_000_000):
        with pytest.raises(dsc.DSCError) as e:
            dsc.dsc_lowrank_fwd_selftest_timeout(inp["x"], inp["z"], inp["U"], y, wl.H, wl.W, bad)
        assert e.value.status == dsc.DSC_ERR_INVALID_ARG
    f32 = {k: v.float() for k, v in inp.items()}          # fp32 runs on the CUDA cores
    with pytest.raises(dsc.DSCError) as e:
        dsc.dsc_lowrank_fwd_selftest_timeout(f32["x"], f32["z"], f32["U"], y.float(), wl.H, wl.W,
                                             LIMIT_NS)
    assert e.value.status == dsc.DSC_ERR_UNSUPPORTED

"""GPU parity of the tensor-core (tcgen05) low-rank kernels against the fp64
oracle, on shapes chosen for that path: bf16, per-channel filters (H = 1),
R = 16 or 32, every W, several 64-channel chunks and 128-token tiles with
ragged tails, sequences shorter than the causal window, and channel counts
that are not a multiple of the 64-channel chunk.  Each case first checks
that the library does route it to the tensor cores, and every test checks
that no bounded wait in those kernels gave up.
"""
import pytest
import torch

import oracle as orc
from lm_local_sequence_causal_b300 import dsc, synthetic as syn
from _parity import Guarded, assert_fwd, assert_grad

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def no_device_error():
    dsc.dsc_device_error(reset=True)
    yield
    torch.cuda.synchronize()
    assert dsc.dsc_device_error() == 0, "a bounded wait in the tensor-core kernels gave up"


def run_fwd(wl, seed):
    assert dsc.dsc_lowrank_uses_tensor_cores(wl.B, wl.T, wl.C, wl.H, wl.W, wl.R, wl.dtype) == 1
    inp = syn.make_inputs(wl, seed, device="cuda")
    y = Guarded(inp["x"].shape, wl.dtype)
    dsc.dsc_lowrank_fwd(inp["x"], inp["z"], inp["U"], y.t, wl.H, wl.W, wl.residual)
    torch.cuda.synchronize()
    assert y.guards_intact(), "y: write outside the tensor"
    ry = orc.lowrank_fwd(inp["x"], inp["z"], inp["U"], wl.H, wl.W, wl.residual)
    return y.t, ry


@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("R", [16, 32])
def test_fwd_every_width_both_ranks(W, R):
    wl = syn.Workload("tc_fwd", B=2, T=300, C=320, W=W, H=1, R=R, residual=True,
                      zu_std=R ** -0.5)
    y, ry = run_fwd(wl, seed=10 * W + R)
    assert_fwd(y, ry, wl.dtype)


@pytest.mark.parametrize("residual", [False, True])
def test_fwd_residual_flag(residual):
    wl = syn.Workload("tc_fwd_res", B=3, T=257, C=192, W=4, H=1, R=16, residual=residual)
    y, ry = run_fwd(wl, seed=3)
    assert_fwd(y, ry, wl.dtype)


@pytest.mark.parametrize("T", [1, 2, 3, 4, 127, 128, 129, 131])
def test_fwd_short_and_ragged_sequences(T):
    wl = syn.Workload("tc_fwd_T", B=3, T=T, C=128, W=4, H=1, R=16)
    y, ry = run_fwd(wl, seed=T)
    assert_fwd(y, ry, wl.dtype)


@pytest.mark.parametrize("C", [8, 24, 72, 136, 200])
def test_fwd_channels_not_a_multiple_of_the_chunk(C):
    wl = syn.Workload("tc_fwd_C", B=2, T=150, C=C, W=4, H=1, R=16)
    y, ry = run_fwd(wl, seed=C)
    assert_fwd(y, ry, wl.dtype)


def test_fwd_many_chunks_and_tiles_per_cta():
    # 4096 items over the SMs: every CTA crosses at least one chunk boundary
    wl = syn.Workload("tc_fwd_big", B=4, T=1024, C=2048, W=4, H=1, R=16)
    y, ry = run_fwd(wl, seed=77)
    assert_fwd(y, ry, wl.dtype)


def test_fwd_repeated_calls_are_identical():
    wl = syn.Workload("tc_fwd_det", B=2, T=640, C=1024, W=4, H=1, R=16)
    inp = syn.make_inputs(wl, 5, device="cuda")
    a = dsc.lowrank_fwd(inp["x"], inp["z"], inp["U"], 1, 4, True)
    b = dsc.lowrank_fwd(inp["x"], inp["z"], inp["U"], 1, 4, True)
    assert torch.equal(a, b)

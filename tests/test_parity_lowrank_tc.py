"""GPU parity of the tensor-core (tcgen05) low-rank kernels against the fp64
oracle, on shapes chosen for that path: bf16, per-channel filters (H = 1)
and filters tied over H channels, R in {8, 16, 24, 32} (ranks below a multiple of 16 padded with zeros on
chip), every W, several 64-channel chunks and 128-token tiles with
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
    assert dsc.dsc_lowrank_uses_tensor_cores(wl.B, wl.T, wl.C, wl.H, wl.W, wl.R, wl.dtype) & 1
    inp = syn.make_inputs(wl, seed, device="cuda")
    y = Guarded(inp["x"].shape, wl.dtype)
    dsc.dsc_lowrank_fwd(inp["x"], inp["z"], inp["U"], y.t, wl.H, wl.W, wl.residual)
    torch.cuda.synchronize()
    assert y.guards_intact(), "y: write outside the tensor"
    ry = orc.lowrank_fwd(inp["x"], inp["z"], inp["U"], wl.H, wl.W, wl.residual)
    return y.t, ry


@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("R", [8, 16, 24, 32])
def test_fwd_every_width_every_rank(W, R):
    wl = syn.Workload("tc_fwd", B=2, T=300, C=320, W=W, H=1, R=R, residual=True,
                      zu_std=R ** -0.5)
    y, ry = run_fwd(wl, seed=10 * W + R)
    assert_fwd(y, ry, wl.dtype)


@pytest.mark.parametrize("residual", [False, True])
@pytest.mark.parametrize("W,R", [(4, 16), (1, 16), (3, 16), (4, 32)])
def test_fwd_residual_flag(residual, W, R):
    # the residual flag is compiled into the forward too
    wl = syn.Workload("tc_fwd_res", B=3, T=257, C=192, W=W, H=1, R=R, residual=residual,
                      zu_std=R ** -0.5)
    y, ry = run_fwd(wl, seed=3 + W + R)
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


def run_bwd(wl, seed):
    assert dsc.dsc_lowrank_uses_tensor_cores(wl.B, wl.T, wl.C, wl.H, wl.W, wl.R, wl.dtype) & 2
    inp = syn.make_inputs(wl, seed, device="cuda")
    x, z, U, dy = inp["x"], inp["z"], inp["U"], inp["dy"]
    dx, dz, dU = Guarded(x.shape, wl.dtype), Guarded(z.shape, wl.dtype), Guarded(U.shape, wl.dtype)
    ws = dsc.lowrank_workspace(x, z, wl.H, wl.W)
    ws.fill_(0x5A)                      # workspace contents on entry must not matter
    dsc.dsc_lowrank_bwd(x, z, U, dy, dx.t, dz.t, dU.t, ws, wl.H, wl.W, wl.residual)
    torch.cuda.synchronize()
    for o, n in ((dx, "dx"), (dz, "dz"), (dU, "dU")):
        assert o.guards_intact(), f"{n}: write outside the tensor"
    rdx, rdz, rdU = orc.lowrank_bwd(x, z, U, dy, wl.H, wl.W, wl.residual)
    assert_grad(dx.t, rdx, wl.dtype, "dx")
    assert_grad(dz.t, rdz, wl.dtype, "dz")
    assert_grad(dU.t, rdU, wl.dtype, "dU")


@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("R", [8, 16, 24, 32])
def test_bwd_every_width_every_rank(W, R):
    wl = syn.Workload("tc_bwd", B=2, T=300, C=320, W=W, H=1, R=R, residual=True,
                      zu_std=R ** -0.5)
    run_bwd(wl, seed=20 + W + R)


@pytest.mark.parametrize("R", [8, 32])
def test_bwd_other_ranks_many_chunks_and_tiles(R):
    # R = 32 holds at most 4 token tiles per split in TMEM: many splits
    wl = syn.Workload("tc_bwd_big_r", B=4, T=1024, C=2048, W=4, H=1, R=R, zu_std=R ** -0.5)
    run_bwd(wl, seed=90 + R)


@pytest.mark.parametrize("residual", [False, True])
@pytest.mark.parametrize("W,R", [(4, 16), (1, 16), (2, 16), (3, 16), (4, 32), (2, 32)])
def test_bwd_residual_flag(residual, W, R):
    # the residual flag is compiled into the backward: each (W, rank step)
    # has a kernel with and one without it
    wl = syn.Workload("tc_bwd_res", B=3, T=257, C=192, W=W, H=1, R=R, residual=residual,
                      zu_std=R ** -0.5)
    run_bwd(wl, seed=4 + W + R)


@pytest.mark.parametrize("T", [1, 3, 4, 127, 128, 129, 131])
def test_bwd_short_and_ragged_sequences(T):
    wl = syn.Workload("tc_bwd_T", B=3, T=T, C=128, W=4, H=1, R=16)
    run_bwd(wl, seed=100 + T)


@pytest.mark.parametrize("C", [8, 24, 72, 136, 200])
def test_bwd_channels_not_a_multiple_of_the_chunk(C):
    wl = syn.Workload("tc_bwd_C", B=2, T=150, C=C, W=4, H=1, R=16)
    run_bwd(wl, seed=200 + C)


def test_bwd_many_chunks_per_cta_and_many_tiles_per_split():
    # several channel chunks per CTA (dU accumulators handed over between
    # chunks) and several token tiles per split (dz accumulators per tile)
    wl = syn.Workload("tc_bwd_big", B=4, T=1024, C=4096, W=4, H=1, R=16)
    run_bwd(wl, seed=88)


def test_bwd_repeated_calls_are_identical():
    wl = syn.Workload("tc_bwd_det", B=2, T=640, C=1024, W=4, H=1, R=16)
    inp = syn.make_inputs(wl, 6, device="cuda")
    a = dsc.lowrank_bwd(inp["x"], inp["z"], inp["U"], inp["dy"], 1, 4, True)
    b = dsc.lowrank_bwd(inp["x"], inp["z"], inp["U"], inp["dy"], 1, 4, True)
    for p, q in zip(a, b):
        assert torch.equal(p, q)


# Tied filters (H > 1): the forward reads the chunk's (64/H)*W U columns and
# each channel picks its group's taps; the backward sees per-channel filters
# equal within a group and adds the group's H channels for dU.
@pytest.mark.parametrize("H", [2, 4, 8, 16, 32])
@pytest.mark.parametrize("W", [2, 3, 4])
def test_tied_fwd_and_bwd(H, W):
    wl = syn.Workload("tc_tied", B=2, T=300, C=320, W=W, H=H, R=16, residual=True)
    q = dsc.dsc_lowrank_uses_tensor_cores(wl.B, wl.T, wl.C, H, W, 16, wl.dtype)
    assert q & 2
    if q & 1:
        y, ry = run_fwd(wl, seed=40 + H + W)
        assert_fwd(y, ry, wl.dtype)
    run_bwd(wl, seed=50 + H + W)


@pytest.mark.parametrize("R", [8, 32])
def test_tied_other_ranks_and_a_ragged_chunk(R):
    # C = 200: the last chunk holds 8 channels; G*W = 100 keeps the forward
    # off the tensor cores, the backward stays on them
    wl = syn.Workload("tc_tied_r", B=2, T=257, C=200, W=4, H=8, R=R, zu_std=R ** -0.5)
    run_bwd(wl, seed=60 + R)
    wl2 = syn.Workload("tc_tied_r2", B=2, T=257, C=448, W=4, H=8, R=R, zu_std=R ** -0.5)
    y, ry = run_fwd(wl2, seed=61 + R)
    assert_fwd(y, ry, wl2.dtype)
    run_bwd(wl2, seed=62 + R)


def test_tied_qkv_size_sampled():
    # the QKV shape with head-wise tying H = 16 on the low-rank path
    wl = syn.Workload("tc_tied_qkv", B=8, T=2048, C=6144, W=4, H=16, R=16)
    assert dsc.dsc_lowrank_uses_tensor_cores(8, 2048, 6144, 16, 4, 16, wl.dtype) == 3
    inp = syn.make_inputs(wl, 9, device="cuda")
    y = dsc.lowrank_fwd(inp["x"], inp["z"], inp["U"], 16, 4, True)
    dx, dz, dU = dsc.lowrank_bwd(inp["x"], inp["z"], inp["U"], inp["dy"], 16, 4, True)
    torch.cuda.synchronize()
    rows = syn.sample_rows(8, 2048, 4, 1024, seed=5)
    from _parity import rows_of
    ry = orc.lowrank_fwd(inp["x"], inp["z"], inp["U"], 16, 4, True, rows=rows)
    assert_fwd(rows_of(y, rows), ry, wl.dtype)
    rdx, rdz = orc.lowrank_bwd_rows(inp["x"], inp["z"], inp["U"], inp["dy"], 16, 4, True, rows=rows)
    assert_grad(rows_of(dx, rows), rdx, wl.dtype, "dx")
    assert_grad(rows_of(dz, rows), rdz, wl.dtype, "dz")
    rdU = orc.lowrank_dU(inp["x"], inp["z"], inp["dy"], 16, 4)
    assert_grad(dU, rdU, wl.dtype, "dU")

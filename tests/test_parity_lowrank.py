"""GPU parity of the low-rank fused DSC kernels against the fp64 oracle.

The oracle forms each token's filters z_t U in fp64 and runs the plain
definition; the kernels generate the filters on-chip.  dU is a reduction
over every token and dz one over every channel, so both are compared in
full at every shape; y and dx are compared in full on small shapes and on a
seeded sample of at least 4096 token rows at full size.
"""
import pytest
import torch

import oracle as orc
from lm_local_sequence_causal_b300 import dsc, synthetic as syn
from _parity import Guarded, assert_by_channel_set, assert_fwd, assert_grad, rows_of

pytestmark = pytest.mark.gpu


def run_lowrank(x, z, U, dy, H, W, residual):
    y = Guarded(x.shape, x.dtype)
    dx = Guarded(x.shape, x.dtype)
    dz = Guarded(z.shape, z.dtype)
    dU = Guarded(U.shape, U.dtype)
    ws = dsc.lowrank_workspace(x, z, H, W)
    ws.fill_(0xA5)                      # workspace contents on entry must not matter
    dsc.dsc_lowrank_fwd(x, z, U, y.t, H, W, residual)
    dsc.dsc_lowrank_bwd(x, z, U, dy, dx.t, dz.t, dU.t, ws, H, W, residual)
    torch.cuda.synchronize()
    for o, n in ((y, "y"), (dx, "dx"), (dz, "dz"), (dU, "dU")):
        assert o.guards_intact(), f"{n}: write outside the tensor"
    return y.t, dx.t, dz.t, dU.t


def check_full(wl, seed=0):
    inp = syn.make_inputs(wl, seed, device="cuda")
    x, z, U, dy = inp["x"], inp["z"], inp["U"], inp["dy"]
    y, dx, dz, dU = run_lowrank(x, z, U, dy, wl.H, wl.W, wl.residual)
    ry = orc.lowrank_fwd(x, z, U, wl.H, wl.W, wl.residual)
    rdx, rdz, rdU = orc.lowrank_bwd(x, z, U, dy, wl.H, wl.W, wl.residual)
    assert_fwd(y, ry, wl.dtype)
    assert_grad(dx, rdx, wl.dtype, "dx")
    assert_grad(dz, rdz, wl.dtype, "dz")
    assert_grad(dU, rdU, wl.dtype, "dU")


def check_sampled(wl, seed=0, nrows=4096):
    """y and dx on a seeded sample of >= nrows token rows (sequence edges
    and tile seams included); dz on every row; dU in full."""
    inp = syn.make_inputs(wl, seed, device="cuda")
    x, z, U, dy = inp["x"], inp["z"], inp["U"], inp["dy"]
    y, dx, dz, dU = run_lowrank(x, z, U, dy, wl.H, wl.W, wl.residual)
    rows = syn.sample_rows(wl.B, wl.T, wl.W, nrows, seed)
    assert len(rows) >= nrows
    ry = orc.lowrank_fwd(x, z, U, wl.H, wl.W, wl.residual, rows=rows)
    rdx, _ = orc.lowrank_bwd_rows(x, z, U, dy, wl.H, wl.W, wl.residual, rows=rows)
    assert_fwd(rows_of(y, rows), ry, wl.dtype)
    assert_grad(rows_of(dx, rows), rdx, wl.dtype, "dx")
    assert_grad(dz, orc.lowrank_dz(x, z, U, dy, wl.H, wl.W), wl.dtype, "dz")
    assert_grad(dU, orc.lowrank_dU(x, z, dy, wl.H, wl.W), wl.dtype, "dU")
    if wl.hot_frac > 0:
        hot = syn.hot_channels(wl.C, wl.hot_frac, seed)
        assert_by_channel_set(rows_of(y, rows), ry, hot, wl.dtype, "y", grad=False)
        assert_by_channel_set(rows_of(dx, rows), rdx, hot, wl.dtype, "dx", grad=True)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("residual", [False, True])
def test_small_full_compare(dtype, residual):
    wl = syn.Workload("lr_small", B=2, T=203, C=256, W=4, H=1, R=16, dtype=dtype,
                      residual=residual, zu_std=0.25)
    check_full(wl, seed=1)


def test_qkv_placement_full_size():
    check_sampled(syn.qkv_lowrank())


def test_linear_rnn_long_sequence():
    check_sampled(syn.linear_rnn_lowrank())


@pytest.mark.parametrize("wl", [w for w in syn.all_linear_sweep() if w.lowrank],
                         ids=lambda w: w.name)
def test_all_linear_sweep(wl):
    check_sampled(wl)


@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("R", [1, 3, 8, 16, 17, 32])
def test_every_width_and_rank(W, R):
    wl = syn.Workload("wr", B=2, T=150, C=256, W=W, H=1, R=R, dtype=torch.float32,
                      residual=True, zu_std=0.25)
    check_full(wl, seed=W * 100 + R)


@pytest.mark.parametrize("H", [2, 4, 8, 32])
def test_lowrank_with_headwise_tying(H):
    wl = syn.Workload("lr_tied", B=2, T=150, C=512, W=4, H=H, R=16, residual=True)
    check_full(wl, seed=H)


@pytest.mark.parametrize("T", [1, 2, 3, 5, 64, 65])
def test_short_and_ragged_sequences(T):
    wl = syn.Workload("lr_ragged", B=3, T=T, C=128, W=4, H=1, R=16, residual=True)
    check_full(wl, seed=T)


@pytest.mark.parametrize("C", [8, 24, 136])
def test_odd_channel_counts(C):
    wl = syn.Workload("lr_odd_c", B=2, T=99, C=C, W=4, H=1, R=16, residual=True)
    check_full(wl, seed=C)


def test_results_are_deterministic():
    wl = syn.Workload("lr_det", B=4, T=512, C=1024, W=4, H=1, R=16)
    inp = syn.make_inputs(wl, 5, device="cuda")
    a = run_lowrank(inp["x"], inp["z"], inp["U"], inp["dy"], 1, 4, True)
    b = run_lowrank(inp["x"], inp["z"], inp["U"], inp["dy"], 1, 4, True)
    for p, q in zip(a, b):
        assert torch.equal(p, q)

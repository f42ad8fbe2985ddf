"""GPU parity of the head-wise DSC kernels against the fp64 oracle.

Small and medium shapes compare every element; the full-size workloads
(the QKV placement B=8 T=2048 C=6144 H=16, the all-linear sweep, the
linear-RNN shape) compare a seeded sample of token rows that always holds
the sequence edges and the tile seams.  The kernels are called through the
C ABI (ctypes binding), in the same launch configuration the benchmark
times.
"""
import pytest
import torch

import oracle as orc
from lm_local_sequence_causal_b300 import dsc, synthetic as syn
from _parity import Guarded, assert_by_channel_set, assert_fwd, assert_grad, rows_of

pytestmark = pytest.mark.gpu


def run_headwise(x, w, dy, H, residual):
    B, T, C = x.shape
    y = Guarded(x.shape, x.dtype)
    dx = Guarded(x.shape, x.dtype)
    dw = Guarded(w.shape, w.dtype)
    dsc.dsc_headwise_fwd(x, w, y.t, H, residual)
    dsc.dsc_headwise_bwd(x, w, dy, dx.t, dw.t, H, residual)
    torch.cuda.synchronize()
    for o, n in ((y, "y"), (dx, "dx"), (dw, "dw")):
        assert o.guards_intact(), f"{n}: write outside the tensor"
    return y.t, dx.t, dw.t


def check_full(wl, seed=0):
    inp = syn.make_inputs(wl, seed, device="cuda")
    x, w, dy = inp["x"], inp["w"], inp["dy"]
    y, dx, dw = run_headwise(x, w, dy, wl.H, wl.residual)
    ry = orc.headwise_fwd(x, w, wl.H, wl.residual)
    rdx, rdw = orc.headwise_bwd(x, w, dy, wl.H, wl.residual)
    assert_fwd(y, ry, wl.dtype)
    assert_grad(dx, rdx, wl.dtype, "dx")
    assert_grad(dw, rdw, wl.dtype, "dw")


def check_sampled(wl, seed=0, nrows=4096):
    inp = syn.make_inputs(wl, seed, device="cuda")
    x, w, dy = inp["x"], inp["w"], inp["dy"]
    y, dx, dw = run_headwise(x, w, dy, wl.H, wl.residual)
    rows = syn.sample_rows(wl.B, wl.T, wl.W, nrows, seed)
    ry = orc.headwise_fwd(x, w, wl.H, wl.residual, rows=rows)
    rdx, rdw = orc.headwise_bwd(x, w, dy, wl.H, wl.residual, rows=rows)
    assert len(rows) >= nrows
    assert_fwd(rows_of(y, rows), ry, wl.dtype)
    assert_grad(rows_of(dx, rows), rdx, wl.dtype, "dx")
    assert_grad(rows_of(dw, rows), rdw.reshape(len(rows), -1), wl.dtype, "dw")
    if wl.hot_frac > 0:
        hot = syn.hot_channels(wl.C, wl.hot_frac, seed)
        assert_by_channel_set(rows_of(y, rows), ry, hot, wl.dtype, "y", grad=False)
        assert_by_channel_set(rows_of(dx, rows), rdx, hot, wl.dtype, "dx", grad=True)


@pytest.mark.parametrize("residual", [False, True])
def test_tiny_fp32_per_channel(residual):
    check_full(syn.tiny_fp32(residual))


def test_qkv_placement_full_size():
    check_sampled(syn.qkv_headwise())


def test_linear_rnn_long_sequence():
    check_sampled(syn.linear_rnn_headwise(), nrows=4096)


@pytest.mark.parametrize("wl", [w for w in syn.all_linear_sweep() if not w.lowrank],
                         ids=lambda w: w.name)
def test_all_linear_sweep(wl):
    check_sampled(wl, nrows=4096)


# Every H path (vector-split groups, shuffle-reduced groups, generic), every
# W, both dtypes, with ragged T that crosses several tiles.
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("H", [1, 2, 4, 8, 16, 32, 64, 128, 256, 3, 24])
@pytest.mark.parametrize("W", [1, 2, 3, 4])
def test_every_group_size_and_width(dtype, H, W):
    C = 768 if H in (3, 24) else 512
    if dtype == torch.float32 and H == 256:
        C = 1024
    wl = syn.Workload("grid", B=2, T=203, C=C, W=W, H=H, dtype=dtype, residual=(W % 2 == 0))
    check_full(wl, seed=H * 10 + W)


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 63, 64, 65, 129])
def test_short_and_ragged_sequences(T):
    wl = syn.Workload("ragged", B=3, T=T, C=256, W=4, H=16, residual=True)
    check_full(wl, seed=T)


@pytest.mark.parametrize("C", [8, 16, 24, 40, 1032])
def test_odd_channel_counts(C):
    wl = syn.Workload("odd_c", B=2, T=77, C=C, W=4, H=8, residual=True)
    check_full(wl, seed=C)
    wl = syn.Workload("odd_c1", B=2, T=77, C=C, W=3, H=1, residual=False)
    check_full(wl, seed=C + 1)


def test_empty_batch_is_a_no_op():
    x = torch.empty(0, 16, 64, dtype=torch.bfloat16, device="cuda")
    w = torch.empty(0, 16, 4, 4, dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    dsc.dsc_headwise_fwd(x, w, y, 16, True)


def test_results_are_deterministic():
    wl = syn.Workload("det", B=2, T=300, C=1024, W=4, H=16)
    inp = syn.make_inputs(wl, 3, device="cuda")
    a = run_headwise(inp["x"], inp["w"], inp["dy"], wl.H, True)
    b = run_headwise(inp["x"], inp["w"], inp["dy"], wl.H, True)
    for p, q in zip(a, b):
        assert torch.equal(p, q)

"""GPU parity of the static short convolution (w [C, W], the same filter at
every token) against the fp64 oracle: forward, dx and the token-summed dw,
both element types, every W, ragged channel blocks and token ranges, the
degenerate sequence lengths, and bitwise reproducibility of dw."""
import pytest
import torch

import oracle as orc
from lm_local_sequence_causal_b300 import dsc, synthetic as syn
from _parity import Guarded, assert_fwd, assert_grad, rows_of

pytestmark = pytest.mark.gpu


def _inputs(B, T, C, W, dtype, seed):
    wl = syn.Workload("static", B=B, T=T, C=C, W=W, H=1, dtype=dtype)
    inp = syn.make_inputs(wl, seed=seed, device="cuda", need_grad_inputs=False)
    x = inp["x"]
    dy = syn.draw((B, T, C), 1.0, seed, syn.SLOT_DY, dtype, "cuda")
    w = syn.static_filters(C, W, 0.5, seed, dtype, "cuda")
    return x, w, dy


def _run(x, w, dy, residual):
    B, T, C = x.shape
    W = w.shape[-1]
    dtype = x.dtype
    y = Guarded((B, T, C), dtype)
    dx = Guarded((B, T, C), dtype)
    dw = Guarded((C, W), dtype)
    dsc.dsc_static_fwd(x, w, y.t, residual)
    n = dsc.dsc_static_bwd_workspace_size(B, T, C, W, dtype)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")
    dsc.dsc_static_bwd(x, w, dy, dx.t, dw.t, ws, residual)
    torch.cuda.synchronize()
    assert y.guards_intact() and dx.guards_intact() and dw.guards_intact()
    return y.t, dx.t, dw.t


# C = 2088: three channel blocks of 128 vectors (bf16), the last one ragged;
# five for fp32.  T = 37 and T < W make token ranges and sequences ragged.
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("B,T,C", [(3, 37, 2088), (2, 200, 512), (4, 2, 256), (1, 1, 64)])
@pytest.mark.parametrize("residual", [False, True])
def test_static_matches_the_oracle(dtype, W, B, T, C, residual):
    x, w, dy = _inputs(B, T, C, W, dtype, seed=W * 10 + T)
    y, dx, dw = _run(x, w, dy, residual)
    ry = orc.static_fwd(x, w, residual)
    rdx, rdw = orc.static_bwd(x, w, dy, residual)
    assert_fwd(y, ry, dtype)
    assert_grad(dx, rdx, dtype, "dx")
    assert_grad(dw, rdw, dtype, "dw")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_static_large_sampled(dtype):
    # many token ranges per channel block: dw sums about a hundred partials
    B, T, C, W = 2, 2048, 2048, 4
    x, w, dy = _inputs(B, T, C, W, dtype, seed=11)
    y, dx, dw = _run(x, w, dy, True)
    rows = syn.sample_rows(B, T, W, 512, seed=3)
    assert_fwd(rows_of(y, rows), orc.static_fwd(x, w, True, rows=rows), dtype)
    assert_grad(rows_of(dx, rows), orc.static_dx_rows(w, dy, True, T, rows), dtype, "dx")
    _, rdw = orc.static_bwd(x, w, dy, True)
    assert_grad(dw, rdw, dtype, "dw")


# bf16 with C a multiple of 64 takes the TMA-staged kernels: one CTA per
# (64-channel chunk, part of the chunk's 128-token tiles).  (3, 300, 384):
# 9 tiles (a partial one per sequence), one tile per CTA, so the second
# epilogue group of every CTA has no tile and contributes zeros; (2, 2048,
# 640): 32 tiles over 11 parts, both groups busy.
@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("B,T,C", [(3, 300, 384), (2, 2048, 640)])
@pytest.mark.parametrize("residual", [False, True])
def test_static_tma_kernels(W, B, T, C, residual):
    x, w, dy = _inputs(B, T, C, W, torch.bfloat16, seed=W + T + C)
    y, dx, dw = _run(x, w, dy, residual)
    assert_fwd(y, orc.static_fwd(x, w, residual), torch.bfloat16)
    rdx, rdw = orc.static_bwd(x, w, dy, residual)
    assert_grad(dx, rdx, torch.bfloat16, "dx")
    assert_grad(dw, rdw, torch.bfloat16, "dw")


def test_static_tma_kernels_qkv_size():
    # the benchmark's shape: 96 chunks x 3 parts, y and dx on 4096 sampled
    # rows, all of dw
    B, T, C, W = 8, 2048, 6144, 4
    x, w, dy = _inputs(B, T, C, W, torch.bfloat16, seed=21)
    y, dx, dw = _run(x, w, dy, True)
    rows = syn.sample_rows(B, T, W, 4096, seed=5)
    assert_fwd(rows_of(y, rows), orc.static_fwd(x, w, True, rows=rows), torch.bfloat16)
    assert_grad(rows_of(dx, rows), orc.static_dx_rows(w, dy, True, T, rows), torch.bfloat16, "dx")
    _, rdw = orc.static_bwd(x, w, dy, True)
    assert_grad(dw, rdw, torch.bfloat16, "dw")
    assert dsc.dsc_device_error() == 0


def test_static_dw_is_bitwise_reproducible():
    x, w, dy = _inputs(4, 1024, 1024, 4, torch.bfloat16, seed=2)
    _, _, dw1 = _run(x, w, dy, True)
    _, _, dw2 = _run(x, w, dy, True)
    assert torch.equal(dw1, dw2)


def test_static_equals_headwise_with_broadcast_filters():
    # the static kernels and the head-wise kernels with w repeated at every
    # token compute the same definition; compare both against each other
    B, T, C, W = 2, 96, 1024, 4
    x, w, dy = _inputs(B, T, C, W, torch.float32, seed=5)
    y, dx, dw = _run(x, w, dy, True)
    wb = w.reshape(1, 1, C, W).expand(B, T, C, W).contiguous()
    yh = dsc.headwise_fwd(x, wb, 1, True)
    dxh, dwh = dsc.headwise_bwd(x, wb, dy, 1, True)
    torch.cuda.synchronize()
    assert torch.allclose(y, yh, rtol=1e-6, atol=1e-6)
    assert torch.allclose(dx, dxh, rtol=1e-6, atol=1e-6)
    assert torch.allclose(dw, dwh.double().sum((0, 1)).float(), rtol=1e-4, atol=1e-4)


def test_static_empty_batch_zeroes_dw_and_small_workspace_is_refused():
    dw = torch.full((64, 4), 7.0, device="cuda")
    dsc.load().dsc_static_bwd(None, None, None, None, dw.data_ptr(), None, 0, 0, 5, 64, 4, 1,
                              dsc.DSC_F32, None)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dw).item() == 0
    x, w, dy = _inputs(2, 64, 256, 4, torch.float32, seed=1)
    n = dsc.dsc_static_bwd_workspace_size(2, 64, 256, 4, torch.float32)
    assert n > 0
    ws = torch.empty(n - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(dsc.DSCError) as e:
        dsc.dsc_static_bwd(x, w, dy, torch.empty_like(x), torch.empty_like(w), ws, True)
    assert e.value.status == dsc.DSC_ERR_WORKSPACE

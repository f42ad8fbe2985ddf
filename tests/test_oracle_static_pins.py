"""Pins of the oracle's static short convolution (w [C, W], the same filter
at every token) against an independent library routine: PyTorch's CPU
depthwise ``conv1d`` in fp64 with left zero padding and the taps reversed
(conv1d correlates, so its last tap multiplies the current token), and its
autograd for dx and dw.  Also a hand-worked case and the row-sampled forms
against the full ones."""
import pytest
import torch
import torch.nn.functional as F

import oracle as orc


def _conv1d_static(x, w, residual):
    B, T, C = x.shape
    W = w.shape[-1]
    xc = x.permute(0, 2, 1)
    y = F.conv1d(F.pad(xc, (W - 1, 0)), w.flip(-1).reshape(C, 1, W), groups=C)
    y = y.permute(0, 2, 1)
    return y + x if residual else y


@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("residual", [False, True])
@pytest.mark.parametrize("T", [1, 3, 11])
def test_static_matches_conv1d_and_its_autograd(W, residual, T):
    g = torch.Generator().manual_seed(100 * W + T + int(residual))
    B, C = 3, 8
    x = torch.randn(B, T, C, generator=g, dtype=torch.float64, requires_grad=True)
    w = torch.randn(C, W, generator=g, dtype=torch.float64, requires_grad=True)
    dy = torch.randn(B, T, C, generator=g, dtype=torch.float64)
    y_ref = _conv1d_static(x, w, residual)
    dx_ref, dw_ref = torch.autograd.grad(y_ref, (x, w), dy)
    y = orc.static_fwd(x.detach(), w.detach(), residual)
    dx, dw = orc.static_bwd(x.detach(), w.detach(), dy, residual)
    assert torch.allclose(y, y_ref.detach(), rtol=0, atol=1e-12)
    assert torch.allclose(dx, dx_ref, rtol=0, atol=1e-12)
    assert torch.allclose(dw, dw_ref, rtol=0, atol=1e-11)


def test_static_hand_worked():
    # One channel, W = 2, T = 3: y_t = w0 x_t + w1 x_{t-1}.
    x = torch.tensor([[[1.0], [2.0], [4.0]]], dtype=torch.float64)
    w = torch.tensor([[3.0, -1.0]], dtype=torch.float64)
    y = orc.static_fwd(x, w, False).reshape(-1).tolist()
    assert y == [3.0, 6.0 - 1.0, 12.0 - 2.0]
    dy = torch.tensor([[[1.0], [0.0], [2.0]]], dtype=torch.float64)
    dx, dw = orc.static_bwd(x, w, dy, False)
    # dx_s = w0 dy_s + w1 dy_{s+1}; dw0 = sum dy_t x_t, dw1 = sum dy_t x_{t-1}
    assert dx.reshape(-1).tolist() == [3.0, -2.0, 6.0]
    assert dw.reshape(-1).tolist() == [1.0 + 8.0, 2.0 * 2.0]


@pytest.mark.parametrize("W", [1, 4])
def test_static_row_forms_match_the_full_ones(W):
    g = torch.Generator().manual_seed(7 + W)
    B, T, C = 2, 13, 16
    x = torch.randn(B, T, C, generator=g, dtype=torch.float64)
    w = torch.randn(C, W, generator=g, dtype=torch.float64)
    dy = torch.randn(B, T, C, generator=g, dtype=torch.float64)
    rows = torch.tensor([0, 1, 2, 5, 12, 13, 14, 20, 25])
    for res in (False, True):
        y = orc.static_fwd(x, w, res)
        dx, _ = orc.static_bwd(x, w, dy, res)
        assert torch.equal(orc.static_fwd(x, w, res, rows=rows), y.reshape(B * T, C)[rows])
        assert torch.equal(orc.static_dx_rows(w, dy, res, T, rows), dx.reshape(B * T, C)[rows])

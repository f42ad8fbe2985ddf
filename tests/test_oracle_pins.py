"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Each test ties the oracle to something the pages or plain mathematics fix:
  * hand-worked integer examples (tests/golden/),
  * a static filter reduces to an ordinary causal depthwise convolution,
    checked against torch's conv1d (a library routine, not a retyped formula),
  * W = 1 reduces to an elementwise product,
  * a unit impulse returns the filter taps shifted causally,
  * the low-rank filter equals an einsum over U reshaped to [R, G, W],
  * every gradient equals a brute-force central finite difference,
  * adjoint (bilinearity) identities, causality, linearity in dy,
  * H = C equals per-channel filters broadcast over channels,
  * T < W and T = 1 truncate the sum,
  * bf16 / fp32 inputs are decoded exactly.
A plausible slip anywhere in the oracle (a dropped term, a flipped tap, a
wrong group index, a transposed U) breaks at least one of these.
"""
import json
import os

import pytest
import torch
import torch.nn.functional as F

import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
f64 = torch.float64


def rnd(*shape, seed=0, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=f64) * std


# ---------------------------------------------------------------- golden ----

def _golden():
    with open(os.path.join(GOLDEN, "hand_worked_T4_C2_W2.json")) as fh:
        return json.load(fh)


def test_golden_headwise_and_lowrank_hand_worked():
    gd = _golden()
    T, C, W = gd["shape"]["T"], gd["shape"]["C"], gd["shape"]["W"]
    x = torch.tensor(gd["x"], dtype=f64).view(1, T, C)
    dy = torch.tensor(gd["dy"], dtype=f64).view(1, T, C)
    for case in gd["cases"]:
        H = case["H"]
        G = C // H
        if "R" in case:
            R = case["R"]
            z = torch.tensor(case["z"], dtype=f64).view(1, T, R)
            U = torch.tensor(case["U"], dtype=f64)
            wm = orc.lowrank_filters(z, U, C, H, W)
            assert torch.equal(wm.view(T, G, W),
                               torch.tensor(case["w_materialised"], dtype=f64))
            y = orc.lowrank_fwd(x, z, U, H, W, residual=False)
            dx, dz, dU = orc.lowrank_bwd(x, z, U, dy, H, W, residual=False)
            assert torch.equal(dz.view(T, R), torch.tensor(case["dz"], dtype=f64))
            assert torch.equal(dU, torch.tensor(case["dU"], dtype=f64))
        else:
            w = torch.tensor(case["w"], dtype=f64).view(1, T, G, W)
            y = orc.headwise_fwd(x, w, H, residual=False)
            dx, dw = orc.headwise_bwd(x, w, dy, H, residual=False)
            assert torch.equal(dw.view(T, G, W), torch.tensor(case["dw"], dtype=f64))
            if "y_residual" in case:
                yr = orc.headwise_fwd(x, w, H, residual=True)
                assert torch.equal(yr.view(T, C),
                                   torch.tensor(case["y_residual"], dtype=f64))
                dxr, _ = orc.headwise_bwd(x, w, dy, H, residual=True)
                assert torch.equal(dxr.view(T, C),
                                   torch.tensor(case["dx_residual"], dtype=f64))
        assert torch.equal(y.view(T, C), torch.tensor(case["y"], dtype=f64)), case["name"]
        assert torch.equal(dx.view(T, C), torch.tensor(case["dx"], dtype=f64)), case["name"]


# ------------------------------------------------- static filter (conv1d) ----

@pytest.mark.parametrize("H", [1, 2, 4])
@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("residual", [False, True])
def test_static_filter_is_causal_depthwise_conv(H, W, residual):
    B, T, C = 2, 13, 8
    G = C // H
    x = rnd(B, T, C, seed=1)
    taps = rnd(G, W, seed=2)                       # one static filter per group
    w = taps.view(1, 1, G, W).expand(B, T, G, W).contiguous()
    y = orc.headwise_fwd(x, w, H, residual)
    # conv1d computes cross-correlation: out[t] = sum_i k[i] in[t + i - pad].
    # With pad = W-1 and k[i] = taps[W-1-i], out[t] = sum_k taps[k] in[t-k].
    kern = taps.repeat_interleave(H, dim=0).flip(-1).unsqueeze(1)   # [C,1,W]
    ref = F.conv1d(x.transpose(1, 2), kern, padding=W - 1, groups=C)[..., :T]
    ref = ref.transpose(1, 2)
    if residual:
        ref = ref + x
    assert torch.allclose(y, ref, rtol=0, atol=1e-12)


def test_static_filter_numpy_convolve_single_channel():
    import numpy as np
    T, W = 20, 4
    x = rnd(1, T, 1, seed=3)
    taps = rnd(1, W, seed=4)
    w = taps.view(1, 1, 1, W).expand(1, T, 1, W).contiguous()
    y = orc.headwise_fwd(x, w, 1, False).view(T).numpy()
    ref = np.convolve(x.view(T).numpy(), taps.view(W).numpy())[:T]
    assert np.allclose(y, ref, rtol=0, atol=1e-12)


# ------------------------------------------------------- special cases ------

@pytest.mark.parametrize("residual", [False, True])
def test_width_one_is_elementwise(residual):
    B, T, C, H = 2, 9, 8, 2
    x = rnd(B, T, C, seed=5)
    w = rnd(B, T, C // H, 1, seed=6)
    y = orc.headwise_fwd(x, w, H, residual)
    ref = w[..., 0].repeat_interleave(H, dim=-1) * x + (x if residual else 0)
    assert torch.allclose(y, ref, rtol=0, atol=1e-14)


@pytest.mark.parametrize("H", [1, 4])
def test_unit_impulse_returns_shifted_taps(H):
    B, T, C, W = 3, 11, 8, 4
    b0, t0, c0 = 1, 5, 6
    x = torch.zeros(B, T, C, dtype=f64)
    x[b0, t0, c0] = 1.0
    w = rnd(B, T, C // H, W, seed=7)
    y = orc.headwise_fwd(x, w, H, residual=False)
    ref = torch.zeros_like(y)
    for k in range(W):
        if t0 + k < T:
            ref[b0, t0 + k, c0] = w[b0, t0 + k, c0 // H, k]
    assert torch.equal(y, ref)


def test_unit_impulse_near_sequence_end_truncates():
    B, T, C, W = 2, 6, 8, 4
    x = torch.zeros(B, T, C, dtype=f64)
    x[0, T - 2, 3] = 1.0
    w = rnd(B, T, C, W, seed=8)
    y = orc.headwise_fwd(x, w, 1, False)
    assert y[1].abs().sum() == 0            # nothing leaks into the next sequence
    assert y[0, T - 2, 3] == w[0, T - 2, 3, 0]
    assert y[0, T - 1, 3] == w[0, T - 1, 3, 1]
    assert (y != 0).sum() == 2


def test_one_filter_per_token_equals_broadcast_per_channel():
    B, T, C, W = 2, 10, 8, 3
    x = rnd(B, T, C, seed=9)
    w1 = rnd(B, T, 1, W, seed=10)                  # H = C: one filter per token
    wc = w1.expand(B, T, C, W).contiguous()        # same filter in every channel
    assert torch.equal(orc.headwise_fwd(x, w1, C, True),
                       orc.headwise_fwd(x, wc, 1, True))
    dy = rnd(B, T, C, seed=11)
    dx1, dw1 = orc.headwise_bwd(x, w1, dy, C, True)
    dxc, dwc = orc.headwise_bwd(x, wc, dy, 1, True)
    assert torch.allclose(dx1, dxc, rtol=0, atol=1e-13)
    assert torch.allclose(dw1[..., 0, :], dwc.sum(dim=2), rtol=0, atol=1e-12)


@pytest.mark.parametrize("T", [1, 2, 3])
def test_short_sequences_truncate_the_sum(T):
    B, C, W, H = 2, 8, 4, 2
    x = rnd(B, T, C, seed=12)
    w = rnd(B, T, C // H, W, seed=13)
    y = orc.headwise_fwd(x, w, H, False)
    ref = torch.zeros_like(y)
    wc = w.repeat_interleave(H, dim=2)             # [B,T,C,W]
    for t in range(T):
        for k in range(min(W, t + 1)):
            ref[:, t] += wc[:, t, :, k] * x[:, t - k]
    assert torch.allclose(y, ref, rtol=0, atol=1e-13)


# ----------------------------------------------------- low-rank filter ------

@pytest.mark.parametrize("H", [1, 2])
def test_lowrank_filter_matches_einsum_and_headwise(H):
    B, T, C, W, R = 2, 7, 8, 3, 5
    G = C // H
    z = rnd(B, T, R, seed=14)
    U = rnd(R, G * W, seed=15)
    wm = orc.lowrank_filters(z, U, C, H, W)
    ref = torch.einsum("btr,rgk->btgk", z, U.view(R, G, W))
    assert torch.allclose(wm, ref, rtol=0, atol=1e-13)
    x = rnd(B, T, C, seed=16)
    dy = rnd(B, T, C, seed=17)
    for res in (False, True):
        assert torch.allclose(orc.lowrank_fwd(x, z, U, H, W, res),
                              orc.headwise_fwd(x, wm, H, res), rtol=0, atol=1e-12)
        dx_l, dz, dU = orc.lowrank_bwd(x, z, U, dy, H, W, res)
        dx_h, dw_h = orc.headwise_bwd(x, wm, dy, H, res)
        assert torch.allclose(dx_l, dx_h, rtol=0, atol=1e-12)
        # dz and dU through the chain rule of w = zU, written with einsum
        assert torch.allclose(dz, torch.einsum("btgk,rgk->btr", dw_h, U.view(R, G, W)),
                              rtol=0, atol=1e-11)
        assert torch.allclose(dU.view(R, G, W), torch.einsum("btr,btgk->rgk", z, dw_h),
                              rtol=0, atol=1e-11)


def test_lowrank_column_order_is_group_major_tap_minor():
    """Only U[0, g*W+k] for one (g, k) is nonzero: exactly filter (g, k) fires."""
    B, T, C, W, R, H = 1, 6, 8, 4, 2, 1
    g0, k0 = 5, 2
    U = torch.zeros(R, C * W, dtype=f64)
    U[0, g0 * W + k0] = 1.0
    z = torch.ones(B, T, R, dtype=f64)
    wm = orc.lowrank_filters(z, U, C, H, W)
    nz = (wm != 0).nonzero().tolist()
    assert nz == [[0, t, g0, k0] for t in range(T)]


# ------------------------------------------------ finite differences --------

def _loss_hw(x, w, dy, H, res):
    return float((orc.headwise_fwd(x, w, H, res) * dy).sum())


def _loss_lr(x, z, U, dy, H, W, res):
    return float((orc.lowrank_fwd(x, z, U, H, W, res) * dy).sum())


def _fd(fun, t, h=0.5):
    g = torch.zeros_like(t)
    flat, gf = t.view(-1), g.view(-1)
    for i in range(flat.numel()):
        v = float(flat[i])
        flat[i] = v + h
        lp = fun()
        flat[i] = v - h
        lm = fun()
        flat[i] = v
        gf[i] = (lp - lm) / (2 * h)
    return g


@pytest.mark.parametrize("H,W", [(1, 1), (1, 4), (2, 3), (4, 2), (8, 4)])
@pytest.mark.parametrize("res", [False, True])
def test_headwise_gradients_match_finite_differences(H, W, res):
    B, T, C = 2, 7, 8
    x = rnd(B, T, C, seed=20)
    w = rnd(B, T, C // H, W, seed=21)
    dy = rnd(B, T, C, seed=22)
    dx, dw = orc.headwise_bwd(x, w, dy, H, res)
    assert torch.allclose(dx, _fd(lambda: _loss_hw(x, w, dy, H, res), x),
                          rtol=1e-10, atol=1e-10)
    assert torch.allclose(dw, _fd(lambda: _loss_hw(x, w, dy, H, res), w),
                          rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("H,W,R", [(1, 1, 1), (1, 4, 3), (2, 3, 1), (4, 2, 3)])
@pytest.mark.parametrize("res", [False, True])
def test_lowrank_gradients_match_finite_differences(H, W, R, res):
    B, T, C = 2, 7, 8
    x = rnd(B, T, C, seed=23)
    z = rnd(B, T, R, seed=24)
    U = rnd(R, (C // H) * W, seed=25)
    dy = rnd(B, T, C, seed=26)
    dx, dz, dU = orc.lowrank_bwd(x, z, U, dy, H, W, res)
    L = lambda: _loss_lr(x, z, U, dy, H, W, res)  # noqa: E731
    assert torch.allclose(dx, _fd(L, x), rtol=1e-10, atol=1e-10)
    assert torch.allclose(dz, _fd(L, z), rtol=1e-10, atol=1e-10)
    assert torch.allclose(dU, _fd(L, U), rtol=1e-10, atol=1e-10)
    # dz on its own (the row-local backward with dx skipped) is the same dz
    assert torch.allclose(orc.lowrank_dz(x, z, U, dy, H, W), _fd(L, z), rtol=1e-10, atol=1e-10)


# ---------------------------------------------- algebraic identities --------

def test_adjoint_identities_headwise():
    B, T, C, W, H = 3, 17, 16, 4, 4
    x, w, dy = rnd(B, T, C, seed=30), rnd(B, T, C // H, W, seed=31), rnd(B, T, C, seed=32)
    y = orc.headwise_fwd(x, w, H, False)
    dx, dw = orc.headwise_bwd(x, w, dy, H, False)
    lhs = float((dy * y).sum())
    assert abs(lhs - float((dx * x).sum())) < 1e-10 * max(1, abs(lhs))   # linear in x
    assert abs(lhs - float((dw * w).sum())) < 1e-10 * max(1, abs(lhs))   # linear in w


def test_adjoint_identities_lowrank():
    B, T, C, W, H, R = 2, 15, 16, 4, 1, 6
    x, z = rnd(B, T, C, seed=33), rnd(B, T, R, seed=34)
    U, dy = rnd(R, C * W, seed=35), rnd(B, T, C, seed=36)
    y = orc.lowrank_fwd(x, z, U, H, W, False)
    dx, dz, dU = orc.lowrank_bwd(x, z, U, dy, H, W, False)
    lhs = float((dy * y).sum())
    for other in ((dx * x).sum(), (dz * z).sum(), (dU * U).sum()):
        assert abs(lhs - float(other)) < 1e-10 * max(1, abs(lhs))


def test_causality_forward_and_backward():
    B, T, C, W, H = 2, 20, 8, 4, 2
    x, w, dy = rnd(B, T, C, seed=40), rnd(B, T, C // H, W, seed=41), rnd(B, T, C, seed=42)
    ts = 9
    x2 = x.clone()
    x2[1, ts] += 1.0
    d = (orc.headwise_fwd(x2, w, H, False) - orc.headwise_fwd(x, w, H, False)).abs().sum(-1)
    changed = set((d[1] != 0).nonzero().view(-1).tolist())
    assert changed <= set(range(ts, ts + W)) and ts in changed
    assert d[0].sum() == 0
    dy2 = dy.clone()
    dy2[1, ts] += 1.0
    dd = (orc.headwise_bwd(x, w, dy2, H, False)[0] - orc.headwise_bwd(x, w, dy, H, False)[0])
    rows = set((dd[1].abs().sum(-1) != 0).nonzero().view(-1).tolist())
    assert rows <= set(range(ts - W + 1, ts + 1)) and ts in rows
    assert dd[0].abs().sum() == 0


def test_gradients_are_linear_in_dy():
    B, T, C, W, H, R = 2, 9, 8, 3, 1, 2
    x, z, U = rnd(B, T, C, seed=50), rnd(B, T, R, seed=51), rnd(R, C * W, seed=52)
    d1, d2 = rnd(B, T, C, seed=53), rnd(B, T, C, seed=54)
    a, b = 0.75, -2.5
    g1 = orc.lowrank_bwd(x, z, U, d1, H, W, False)
    g2 = orc.lowrank_bwd(x, z, U, d2, H, W, False)
    g12 = orc.lowrank_bwd(x, z, U, a * d1 + b * d2, H, W, False)
    for p, q, r in zip(g1, g2, g12):
        assert torch.allclose(r, a * p + b * q, rtol=1e-12, atol=1e-12)


# ------------------------------------------- rows / dtypes / threads --------

def test_row_subsets_equal_full_outputs():
    B, T, C, W, H, R = 2, 12, 16, 4, 1, 3
    x, w, dy = rnd(B, T, C, seed=60), rnd(B, T, C, W, seed=61), rnd(B, T, C, seed=62)
    z, U = rnd(B, T, R, seed=63), rnd(R, C * W, seed=64)
    rows = torch.tensor([0, 3, 11, 12, 13, 23])
    y = orc.headwise_fwd(x, w, H, True)
    assert torch.equal(orc.headwise_fwd(x, w, H, True, rows=rows), y.view(-1, C)[rows])
    dx, dw = orc.headwise_bwd(x, w, dy, H, True)
    dxr, dwr = orc.headwise_bwd(x, w, dy, H, True, rows=rows)
    assert torch.equal(dxr, dx.view(-1, C)[rows])
    assert torch.equal(dwr, dw.view(-1, C, W)[rows])
    dxl, dzl = orc.lowrank_bwd_rows(x, z, U, dy, H, W, True)
    dxs, dzs = orc.lowrank_bwd_rows(x, z, U, dy, H, W, True, rows=rows)
    assert torch.equal(dxs, dxl.view(-1, C)[rows])
    assert torch.equal(dzs, dzl.view(-1, R)[rows])
    assert torch.equal(orc.lowrank_dz(x, z, U, dy, H, W), dzl)
    assert torch.equal(orc.lowrank_dz(x, z, U, dy, H, W, rows=rows), dzl.view(-1, R)[rows])
    yl = orc.lowrank_fwd(x, z, U, H, W, True)
    assert torch.equal(orc.lowrank_fwd(x, z, U, H, W, True, rows=rows), yl.view(-1, C)[rows])


def test_low_precision_inputs_are_decoded_exactly():
    B, T, C, W, H = 2, 8, 16, 4, 4
    x = rnd(B, T, C, seed=70).to(torch.bfloat16)
    w = rnd(B, T, C // H, W, seed=71).to(torch.float32)
    y_mixed = orc.headwise_fwd(x, w, H, True)
    y_f64 = orc.headwise_fwd(x.double(), w.double(), H, True)
    assert torch.equal(y_mixed, y_f64)


def test_results_do_not_depend_on_thread_count():
    B, T, C, W, R = 2, 33, 64, 4, 4
    x, z = rnd(B, T, C, seed=80), rnd(B, T, R, seed=81)
    U, dy = rnd(R, C * W, seed=82), rnd(B, T, C, seed=83)
    n0 = orc.num_threads()
    try:
        orc.set_num_threads(1)
        a = orc.lowrank_bwd(x, z, U, dy, 1, W, True)
        orc.set_num_threads(max(2, n0))
        b = orc.lowrank_bwd(x, z, U, dy, 1, W, True)
    finally:
        orc.set_num_threads(n0)
    for p, q in zip(a, b):
        assert torch.equal(p, q)

"""Pins of the oracle's decode step merged with its projection
(x_t = h_t Wp^T, rounded once to the I/O type, then the decode step).

The projection is pinned by cases whose result is known without a matmul:
the identity and a permutation (a transposed Wp gives another permutation
and fails), a power-of-two scaling (exact), and brute-force Python loops on
tiny inputs.  The rounding is pinned against torch's float32 -> bfloat16
conversion on float32 values and on hand-made ties.  The decode step after
it is the one pinned in test_oracle_decode_pins.py."""
import numpy as np
import pytest
import torch

import oracle as orc


def _bf16(shape, gen, scale=1.0):
    return (torch.randn(shape, generator=gen, dtype=torch.float64) * scale).to(torch.bfloat16)


def test_round_to_bf16_matches_torch_on_fp32_values():
    gen = torch.Generator().manual_seed(11)
    v = torch.randn(20000, generator=gen, dtype=torch.float32) * 37.0
    got = orc.round_to(v.double(), torch.bfloat16)
    assert torch.equal(got, v.to(torch.bfloat16))


def test_round_to_bf16_ties_go_to_even():
    # spacing of bf16 in [1, 2) is 2^-7; 1 + 2^-8 is halfway between 1 (even)
    # and 1 + 2^-7 (odd); 1 + 3*2^-8 is halfway between 1 + 2^-7 (odd) and
    # 1 + 2^-6 (even); just past a tie rounds up
    v = torch.tensor([1 + 2.0**-8, 1 + 3 * 2.0**-8, -(1 + 2.0**-8), 1 + 2.0**-8 + 2.0**-30,
                      3 * 2.0**-8 * 2.0**5], dtype=torch.float64)
    got = orc.round_to(v, torch.bfloat16).double()
    want = torch.tensor([1.0, 1 + 2.0**-6, -1.0, 1 + 2.0**-7, 3 * 2.0**-3],
                        dtype=torch.float64)
    assert torch.equal(got, want)


def test_round_to_fp32_ties_go_to_even():
    v = torch.tensor([1 + 2.0**-24, 1 + 3 * 2.0**-24], dtype=torch.float64)
    got = orc.round_to(v, torch.float32).double()
    assert torch.equal(got, torch.tensor([1.0, 1 + 2.0**-22], dtype=torch.float64))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("H", [1, 4])
def test_identity_projection_is_the_decode_step(dtype, W, H):
    gen = torch.Generator().manual_seed(W * 10 + H)
    B, C = 3, 16
    h = _bf16((B, C), gen).to(dtype)
    Wp = torch.eye(C, dtype=dtype)
    w = _bf16((B, C // H, W), gen, 0.5).to(dtype)
    state = _bf16((B, W - 1, C), gen).to(dtype)
    y, st, x = orc.headwise_proj_decode(h, Wp, w, state, H, True)
    y0, st0 = orc.headwise_decode(h, w, state, H, True)
    assert torch.equal(x, h)
    assert torch.equal(y, y0) and torch.equal(st, st0)


def test_permutation_projection_permutes_channels():
    gen = torch.Generator().manual_seed(3)
    B, C = 2, 12
    perm = torch.randperm(C, generator=gen)
    Wp = torch.zeros(C, C, dtype=torch.bfloat16)
    Wp[torch.arange(C), perm] = 1.0                 # x[:, c] = h[:, perm[c]]
    h = _bf16((B, C), gen)
    x = orc.project(h, Wp, torch.bfloat16)
    assert torch.equal(x, h[:, perm])
    assert not torch.equal(orc.project(h, Wp.T.contiguous(), torch.bfloat16), h[:, perm])


def test_power_of_two_projection_is_exact():
    gen = torch.Generator().manual_seed(4)
    h = _bf16((4, 8), gen)
    x = orc.project(h, 4.0 * torch.eye(8, dtype=torch.bfloat16), torch.bfloat16)
    assert torch.equal(x.double(), 4.0 * h.double())


@pytest.mark.parametrize("W,H", [(4, 1), (3, 2), (2, 8)])
def test_brute_force_projection_and_step(W, H):
    gen = torch.Generator().manual_seed(W + 5 * H)
    B, D, C = 2, 5, 8
    h = _bf16((B, D), gen)
    Wp = _bf16((C, D), gen, 0.5)
    w = _bf16((B, C // H, W), gen, 0.5)
    state = _bf16((B, W - 1, C), gen)
    hl, wl = h.double().tolist(), Wp.double().tolist()
    x_loop = torch.tensor([[sum(hl[b][d] * wl[c][d] for d in range(D)) for c in range(C)]
                           for b in range(B)], dtype=torch.float64)
    x_ref = orc.round_to(x_loop, torch.bfloat16)
    y, st, x = orc.headwise_proj_decode(h, Wp, w, state, H, False)
    assert torch.equal(x, x_ref)
    # the step by hand: y = w0 x + sum_{k>=1} w_k state[k-1] (residual off)
    xs, ws, ss = x_ref.double(), w.double(), state.double()
    for b in range(B):
        for c in range(C):
            g = c // H
            want = ws[b, g, 0] * xs[b, c] + sum(ws[b, g, k] * ss[b, k - 1, c]
                                                for k in range(1, W))
            assert abs(float(y[b, c]) - float(want)) <= 1e-12 * (1 + abs(float(want)))
    if W > 1:
        assert torch.equal(st[:, 0], xs)
        assert torch.equal(st[:, 1:], ss[:, :W - 2])


def test_lowrank_identity_projection_is_the_lowrank_step():
    gen = torch.Generator().manual_seed(9)
    B, C, W, R = 2, 16, 4, 3
    h = _bf16((B, C), gen)
    z = _bf16((B, R), gen, 0.5)
    U = _bf16((R, C * W), gen, 0.5)
    state = _bf16((B, W - 1, C), gen)
    y, st, x = orc.lowrank_proj_decode(h, torch.eye(C, dtype=torch.bfloat16), z, U, state,
                                       1, W, True)
    y0, st0 = orc.lowrank_decode(h, z, U, state, 1, W, True)
    assert torch.equal(x, h) and torch.equal(y, y0) and torch.equal(st, st0)


def test_round_to_rejects_other_types():
    with pytest.raises(ValueError):
        orc.round_to(torch.zeros(2, dtype=torch.float64), torch.float16)
    assert np.isfinite(orc.round_to(torch.ones(2, dtype=torch.float64), torch.bfloat16)
                       .double().numpy()).all()

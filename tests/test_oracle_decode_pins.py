"""Pins of the oracle's decode step (one token with a carried state) against
the pinned full-sequence oracle: replaying a sequence token by token from a
zero state must give every row of the full forward, and the state must hold
the last W-1 inputs, newest first."""
import pytest
import torch

import oracle as orc
from lm_local_sequence_causal_b300 import synthetic as syn


@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("H", [1, 2, 4])
@pytest.mark.parametrize("residual", [False, True])
def test_headwise_decode_replays_the_forward(W, H, residual):
    wl = syn.Workload("dec", B=2, T=9, C=8, W=W, H=H, dtype=torch.float32,
                      residual=residual, w_std=0.5)
    inp = syn.make_inputs(wl, seed=W * 7 + H, need_grad_inputs=False)
    x, w = inp["x"].double(), inp["w"].double()
    full = orc.headwise_fwd(x, w, H, residual)
    state = torch.zeros(wl.B, W - 1, wl.C, dtype=torch.float64)
    for t in range(wl.T):
        y, state = orc.headwise_decode(x[:, t], w[:, t], state, H, residual)
        assert torch.allclose(y, full[:, t], rtol=0, atol=1e-12), t
        for j in range(W - 1):
            want = x[:, t - j] if t - j >= 0 else torch.zeros(wl.B, wl.C, dtype=torch.float64)
            assert torch.equal(state[:, j], want)


def test_lowrank_decode_replays_the_forward():
    wl = syn.Workload("dec_lr", B=2, T=7, C=16, W=4, H=1, R=3, dtype=torch.float32,
                      residual=True, zu_std=0.5)
    inp = syn.make_inputs(wl, seed=5, need_grad_inputs=False)
    x, z, U = inp["x"].double(), inp["z"].double(), inp["U"].double()
    full = orc.lowrank_fwd(x, z, U, 1, 4, True)
    state = torch.zeros(wl.B, 3, wl.C, dtype=torch.float64)
    for t in range(wl.T):
        y, state = orc.lowrank_decode(x[:, t], z[:, t], U, state, 1, 4, True)
        assert torch.allclose(y, full[:, t], rtol=0, atol=1e-12), t


def test_decode_hand_worked():
    # C = 1, H = 1, W = 3: y = res*x + w0*x + w1*s0 + w2*s1, state -> [x, s0]
    x = torch.tensor([[2.0]])
    w = torch.tensor([[[0.5, -1.0, 3.0]]])
    s = torch.tensor([[[4.0], [-1.0]]])
    y, ns = orc.headwise_decode(x, w, s, 1, True)
    assert y.item() == 2.0 + 0.5 * 2.0 - 1.0 * 4.0 + 3.0 * -1.0
    assert ns.reshape(-1).tolist() == [2.0, 4.0]

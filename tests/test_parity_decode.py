"""GPU parity of the decode step (one token with a carried state) against the
fp64 oracle, and a token-by-token replay of a sequence that must reproduce
the full-sequence forward kernels (the decode step is the forward at one new
position).  Both parameterisations, both element types, every W."""
import pytest
import torch

import oracle as orc
from lm_local_sequence_causal_b300 import dsc, synthetic as syn
from _parity import TOL, Guarded, assert_fwd

pytestmark = pytest.mark.gpu


def _state(B, W, C, dtype, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.randn(B, max(W - 1, 0), C, generator=g, device="cuda").to(dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("H", [1, 16, 24])
def test_headwise_decode_step(dtype, W, H):
    B, C = 5, 768
    wl = syn.Workload("dec", B=B, T=1, C=C, W=W, H=H, dtype=dtype, w_std=0.5)
    inp = syn.make_inputs(wl, seed=W + H, device="cuda", need_grad_inputs=False)
    x, w = inp["x"][:, 0].contiguous(), inp["w"][:, 0].contiguous()
    state = _state(B, W, C, dtype, 3)
    ry, rstate = orc.headwise_decode(x, w, state, H, True)
    y = Guarded((B, C), dtype)
    dsc.dsc_headwise_decode(x, w, state, y.t, H, True)
    torch.cuda.synchronize()
    assert y.guards_intact()
    assert_fwd(y.t, ry, dtype)
    assert torch.equal(state.double().cpu(), rstate)     # exact copies of the inputs


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("W", [1, 2, 4])
@pytest.mark.parametrize("R,H", [(16, 1), (3, 1), (16, 4), (32, 1)])
def test_lowrank_decode_step(dtype, W, R, H):
    B, C = 3, 512
    wl = syn.Workload("dec_lr", B=B, T=1, C=C, W=W, H=H, R=R, dtype=dtype, zu_std=R ** -0.5)
    inp = syn.make_inputs(wl, seed=R + W, device="cuda", need_grad_inputs=False)
    x, z = inp["x"][:, 0].contiguous(), inp["z"][:, 0].contiguous()
    state = _state(B, W, C, dtype, 4)
    ry, rstate = orc.lowrank_decode(x, z, inp["U"], state, H, W, False)
    y = torch.empty(B, C, dtype=dtype, device="cuda")
    dsc.dsc_lowrank_decode(x, z, inp["U"], state, y, H, W, False)
    torch.cuda.synchronize()
    assert_fwd(y, ry, dtype)
    assert torch.equal(state.double().cpu(), rstate)


@pytest.mark.parametrize("dtype,B,C,H,W,R", [
    # several passes of 32 (bf16) or 16 (fp32) sequences over one staged U
    # slice; a partial last slice of 32 channels; H = 3 splits groups across
    # slices, so some slices' columns start off a 16-byte boundary (element
    # copies) and others on one (16-byte copies)
    (torch.bfloat16, 40, 528, 3, 4, 16),
    # U rows of 99 elements: every slice takes element copies
    (torch.bfloat16, 70, 528, 16, 3, 7),
    (torch.float32, 37, 36, 3, 4, 32),
    (torch.float32, 5, 520, 1, 2, 16),
    (torch.bfloat16, 33, 1048, 8, 4, 5),
    (torch.bfloat16, 1, 6144, 1, 4, 16),
    (torch.bfloat16, 8, 6144, 1, 4, 16),
    (torch.bfloat16, 64, 6144, 1, 1, 32),
])
def test_lowrank_decode_blocks(dtype, B, C, H, W, R):
    wl = syn.Workload("dec_lr_blk", B=B, T=1, C=C, W=W, H=H, R=R, dtype=dtype,
                      zu_std=R ** -0.5)
    inp = syn.make_inputs(wl, seed=B + C + R, device="cuda", need_grad_inputs=False)
    x, z = inp["x"][:, 0].contiguous(), inp["z"][:, 0].contiguous()
    st = Guarded((B, W - 1, C), dtype) if W > 1 else None
    state = _state(B, W, C, dtype, 5)                  # [B, 0, C] when W = 1
    if st is not None:
        st.t.copy_(state)
        state = st.t
    ry, rstate = orc.lowrank_decode(x, z, inp["U"], state, H, W, True)
    y = Guarded((B, C), dtype)
    dsc.dsc_lowrank_decode(x, z, inp["U"], state, y.t, H, W, True)
    torch.cuda.synchronize()
    assert y.guards_intact()
    assert_fwd(y.t, ry, dtype)
    if st is not None:
        assert st.guards_intact()
        assert torch.equal(state.double().cpu(), rstate)


def test_replay_matches_the_full_sequence_kernels():
    # head-wise QKV-like shape and low-rank, decoded token by token from a
    # zero state, against one call of the forward over the whole sequence
    hw = syn.Workload("rep_hw", B=2, T=40, C=1024, W=4, H=16)
    a = syn.make_inputs(hw, 1, device="cuda", need_grad_inputs=False)
    yfull = dsc.headwise_fwd(a["x"], a["w"], 16, True)
    state = torch.zeros(2, 3, 1024, dtype=torch.bfloat16, device="cuda")
    ys = torch.empty(2, 1024, dtype=torch.bfloat16, device="cuda")
    for t in range(hw.T):
        dsc.dsc_headwise_decode(a["x"][:, t].contiguous(), a["w"][:, t].contiguous(), state, ys,
                                16, True)
        assert torch.equal(ys, yfull[:, t]), t          # same fp32 sum, same rounding
    lr = syn.Workload("rep_lr", B=2, T=30, C=512, W=4, H=1, R=16)
    b = syn.make_inputs(lr, 2, device="cuda", need_grad_inputs=False)
    yfull = dsc.lowrank_fwd(b["x"], b["z"], b["U"], 1, 4, True)
    state = torch.zeros(2, 3, 512, dtype=torch.bfloat16, device="cuda")
    ys = torch.empty(2, 512, dtype=torch.bfloat16, device="cuda")
    err = 0.0
    for t in range(lr.T):
        dsc.dsc_lowrank_decode(b["x"][:, t].contiguous(), b["z"][:, t].contiguous(), b["U"], state,
                               ys, 1, 4, True)
        d = (ys.double() - yfull[:, t].double()).abs().max().item()
        err = max(err, d / yfull[:, t].double().abs().max().item())
    # the tensor-core forward and the CUDA-core decode sum the filters in a
    # different order; both are fp32 from exact bf16 products
    assert err <= TOL[torch.bfloat16]["fwd"]


def test_decode_rejects_aliasing_and_bad_widths():
    x = torch.zeros(2, 64, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(2, 4, 4, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(2, 3, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dsc.DSCError):
        dsc.dsc_headwise_decode(x, w, st, x, 16, True)           # y aliases x
    w5 = torch.zeros(2, 4, 5, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dsc.DSCError):
        dsc.dsc_headwise_decode(x, w5, st, torch.empty_like(x), 16, True)

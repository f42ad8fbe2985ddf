"""GPU parity of the TMA-staged head-wise kernels against the fp64 oracle.

These shapes take the TMA path (bf16, C a multiple of 64, (H, W) with a
legal filter box); each case first checks that the library routes it there,
and every test checks that no bounded wait in those kernels gave up.  The
wider grid of H and W in test_parity_headwise.py also runs through this path
for the same (H, W) pairs.
"""
import pytest
import torch

import oracle as orc
from lm_local_sequence_causal_b300 import dsc, synthetic as syn
from _parity import Guarded, assert_fwd, assert_grad

pytestmark = pytest.mark.gpu

# (H, W, item width in channels)
TMA_PAIRS = [(8, 1, 64), (8, 2, 64), (8, 3, 64), (8, 4, 64), (16, 2, 64), (16, 4, 64),
             (32, 4, 64), (16, 1, 128), (32, 2, 128), (64, 4, 128)]


@pytest.fixture(autouse=True)
def no_device_error():
    dsc.dsc_device_error(reset=True)
    yield
    torch.cuda.synchronize()
    assert dsc.dsc_device_error() == 0, "a bounded wait in the TMA kernels gave up"


def check(wl, seed, paths=3):
    assert dsc.dsc_headwise_uses_tma(wl.B, wl.T, wl.C, wl.H, wl.W, wl.dtype) == paths
    inp = syn.make_inputs(wl, seed, device="cuda")
    x, w, dy = inp["x"], inp["w"], inp["dy"]
    y, dx, dw = Guarded(x.shape, wl.dtype), Guarded(x.shape, wl.dtype), Guarded(w.shape, wl.dtype)
    dsc.dsc_headwise_fwd(x, w, y.t, wl.H, wl.residual)
    dsc.dsc_headwise_bwd(x, w, dy, dx.t, dw.t, wl.H, wl.residual)
    torch.cuda.synchronize()
    for o, n in ((y, "y"), (dx, "dx"), (dw, "dw")):
        assert o.guards_intact(), f"{n}: write outside the tensor"
    ry = orc.headwise_fwd(x, w, wl.H, wl.residual)
    rdx, rdw = orc.headwise_bwd(x, w, dy, wl.H, wl.residual)
    assert_fwd(y.t, ry, wl.dtype)
    assert_grad(dx.t, rdx, wl.dtype, "dx")
    assert_grad(dw.t, rdw, wl.dtype, "dw")


@pytest.mark.parametrize("H,W,CW", TMA_PAIRS)
@pytest.mark.parametrize("residual", [False, True])
def test_every_legal_group_size_and_width(H, W, CW, residual):
    wl = syn.Workload("hw_tma", B=2, T=300, C=5 * CW, W=W, H=H, residual=residual)
    check(wl, seed=H * 10 + W + 100 * residual)


def test_w3_h16_on_tma():
    # the all-linear sweep's H = 16, W = 3: forward on 128-channel items,
    # backward on 64-channel items with the padded filter box (24-byte
    # filter rows: the taps start 0 or 4 elements into the loaded box, on
    # alternate chunks) and dw written from registers
    wl = syn.Workload("hw_tma_w3", B=2, T=300, C=640, W=3, H=16)
    check(wl, seed=33, paths=3)


@pytest.mark.parametrize("T", [1, 2, 3, 127, 129, 300])
@pytest.mark.parametrize("residual", [False, True])
def test_w3_h16_short_ragged_and_three_wide_chunks(T, residual):
    # six 64-channel backward chunks (both tap offsets, 0 and 4), three
    # 128-channel forward chunks, short and ragged sequences
    wl = syn.Workload("hw_tma_w3_T", B=3, T=T, C=384, W=3, H=16, residual=residual)
    check(wl, seed=T + 7 * residual, paths=3)


def test_w3_h16_backward_many_items_per_cta():
    wl = syn.Workload("hw_tma_w3_multi", B=4, T=2048, C=1024, W=3, H=16, residual=True)
    check(wl, seed=3, paths=3)


@pytest.mark.parametrize("T", [1, 2, 129, 300])
@pytest.mark.parametrize("residual", [False, True])
def test_h64_backward_two_lanes_per_token(T, residual):
    # H = 64 backward on 64-channel items: one filter group per item, its dw
    # summed over two adjacent lanes of a token; six chunks give both filter
    # box offsets (0 and 4 elements)
    wl = syn.Workload("hw_tma_h64", B=3, T=T, C=384, W=4, H=64, residual=residual)
    check(wl, seed=T + 11 * residual, paths=3)


def test_linear_rnn_shape_on_tma():
    wl = syn.Workload("hw_tma_rnn", B=1, T=1100, C=512, W=4, H=64, hot_frac=0.05)
    check(wl, seed=64)


@pytest.mark.parametrize("T", [1, 3, 4, 127, 128, 129, 131, 257])
def test_short_and_ragged_sequences(T):
    wl = syn.Workload("hw_tma_T", B=3, T=T, C=192, W=4, H=16)
    check(wl, seed=T)


def test_many_items_per_cta_qkv_pair():
    wl = syn.Workload("hw_tma_big", B=4, T=1024, C=2048, W=4, H=16)
    check(wl, seed=5)


def test_routing():
    q = dsc.dsc_headwise_uses_tma
    bf = torch.bfloat16
    assert q(8, 2048, 6144, 16, 4, bf) == 3           # the QKV placement
    assert q(8, 2048, 6144, 16, 3, bf) == 3           # fwd 128-ch items, bwd padded box
    assert q(8, 2048, 6080, 16, 3, bf) == 0           # C % 128 != 0: filter rows 3C/16
    assert q(8, 2048, 320, 16, 3, bf) == 0            # elements, not 16-byte multiples
    assert q(2, 16384, 4096, 64, 4, bf) == 3          # linear-RNN shape (128-channel items)
    assert q(8, 2048, 6144, 64, 3, bf) == 0           # 6-tap rows: no legal box
    assert q(8, 2048, 6144, 16, 4, torch.float32) == 0
    assert q(8, 2048, 6120, 8, 4, bf) == 0            # C not a multiple of 64
    assert q(8, 2048, 6144, 16, 5, bf) == -1



@pytest.mark.parametrize("H,W,CW", TMA_PAIRS)
def test_many_items_per_cta(H, W, CW):
    # 4 x 16 tiles x 16 chunks: every CTA takes about seven items, so each
    # epilogue group reuses the pipeline stages (the forward with 128-channel
    # items included)
    wl = syn.Workload("hw_tma_multi", B=4, T=2048, C=16 * CW, W=W, H=H, residual=True)
    check(wl, seed=H * 7 + W)


@pytest.mark.parametrize("H,W", [(8, 1), (16, 2), (32, 4)])
def test_wide_forward_items_of_narrow_pairs(H, W):
    # C a multiple of 128: these forwards take 128-channel items (64-channel
    # items when C is only a multiple of 64, as in the cases above)
    wl = syn.Workload("hw_tma_wide", B=4, T=1024, C=2048, W=W, H=H, residual=True)
    check(wl, seed=H * 5 + W)

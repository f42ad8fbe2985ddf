"""GPU parity of the decode step merged with its projection
(dsc_headwise_proj_decode, dsc_lowrank_proj_decode) against the fp64 oracle.

y is checked with the forward measure; the updated state must hold exact
copies of the old rows 0..W-3 in rows 1..W-2, and row 0 must hold x rounded
to the I/O type (forward measure: the kernel sums x in fp32, the oracle in
fp64, so a value next to a rounding boundary may land on the neighbouring
bf16).  Every output sits in guard bands.  Also: a token-by-token replay
against the full-sequence oracle, agreement with the unmerged pair
(cuBLAS projection, then dsc_headwise_decode), the batch-block edges, the
QKV decode shape, the tcgen05 kernel's tiles, clusters and launches, and
B = 0."""
import pytest
import torch

import oracle as orc
from lm_local_sequence_causal_b300 import dsc, synthetic as syn
from _parity import Guarded, assert_fwd

pytestmark = pytest.mark.gpu


def _run(dtype, B, D, C, H, W, R=0, residual=True, seed=0):
    inp = syn.proj_decode_inputs(B, D, C, H, W, R, dtype, seed, device="cuda")
    st0 = inp["state"].clone()
    if R:
        ry, rstate, rx = orc.lowrank_proj_decode(inp["h"], inp["Wp"], inp["z"], inp["U"], st0,
                                                 H, W, residual)
    else:
        ry, rstate, rx = orc.headwise_proj_decode(inp["h"], inp["Wp"], inp["w"], st0, H, residual)
    y = Guarded((B, C), dtype)
    st = Guarded((B, max(W - 1, 1), C), dtype) if W > 1 else None
    state = None
    if st is not None:
        state = st.t
        state.copy_(inp["state"])
    if R:
        dsc.dsc_lowrank_proj_decode(inp["h"], inp["Wp"], inp["z"], inp["U"], state, y.t, H, W,
                                    residual)
    else:
        dsc.dsc_headwise_proj_decode(inp["h"], inp["Wp"], inp["w"], state, y.t, H, residual)
    torch.cuda.synchronize()
    assert y.guards_intact()
    e = assert_fwd(y.t, ry, dtype)
    if W > 1:
        assert st.guards_intact()
        assert torch.equal(state[:, 1:].double().cpu(), rstate[:, 1:])
        assert_fwd(state[:, 0], rx, dtype, "x (state row 0)")
    return e


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("H", [1, 16])
def test_headwise_step(dtype, W, H):
    _run(dtype, B=5, D=200, C=768, H=H, W=W, seed=W + H)


@pytest.mark.parametrize("B", [1, 2, 3, 4, 5, 7, 8, 9, 16, 17, 31, 33, 64, 70])
def test_batch_blocks(B):
    # the CUDA-core kernel (1, 2 or 4 sequences per block; bf16 up to 4), the
    # warp-MMA one (16 per pass, up to 16 sequences) and the tcgen05 one
    # (from 17), partial blocks and passes
    _run(torch.bfloat16, B=B, D=512, C=256, H=16, W=4, seed=B)


@pytest.mark.parametrize("D", [8, 24, 256, 264, 1000, 3072, 3080, 4096, 6144, 6152])
@pytest.mark.parametrize("B", [3, 9])
def test_hidden_sizes(D, B):
    # one piece per row, fewer pieces than lanes, pieces not a multiple of the
    # lanes x pieces in flight, and long rows; both kernels (B = 3 and 9)
    _run(torch.bfloat16, B=B, D=D, C=128, H=8, W=3, seed=D + B)


@pytest.mark.parametrize("B", [9, 40])
def test_fp32_batches(B):
    # fp32 always takes the CUDA-core kernel: blocks of 8 sequences, passes
    _run(torch.float32, B=B, D=200, C=264, H=8, W=4, seed=B)


@pytest.mark.parametrize("residual", [False, True])
def test_residual_switch(residual):
    _run(torch.bfloat16, B=4, D=128, C=64, H=1, W=4, residual=residual, seed=7)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("W", [2, 4])
@pytest.mark.parametrize("R,H", [(16, 1), (3, 1), (16, 4), (32, 1)])
@pytest.mark.parametrize("B", [3, 20, 40])
def test_lowrank_step(dtype, W, R, H, B):
    _run(dtype, B=B, D=256, C=512, H=H, W=W, R=R, seed=R + W + B)


@pytest.mark.parametrize("B", [1, 8])
def test_qkv_decode_shape(B):
    # the QKV placement's decode step: D = 2048 hidden, C = 6144 = q, k, v
    _run(torch.bfloat16, B=B, D=2048, C=6144, H=16, W=4, seed=1)


@pytest.mark.parametrize("B,D,C,H,W,R", [
    (17, 512, 256, 16, 4, 0),      # the smallest batch on the tcgen05 kernel
    (24, 512, 256, 16, 4, 0),
    (24, 8, 136, 8, 3, 0),         # D of one short block; a partial 128-channel tile
    (25, 1000, 1024, 1, 2, 0),     # a ragged last block of D; 8 tiles, wide clusters
    (40, 6152, 128, 4, 1, 0),      # one tile, clusters of 8; W = 1
    (256, 256, 384, 16, 4, 0),     # one full launch (N = 256)
    (300, 128, 256, 2, 4, 0),      # two launches (256 + 44 sequences)
    (24, 512, 256, 1, 4, 16),
    (33, 1000, 520, 4, 3, 5),
    (64, 2048, 6144, 16, 4, 0),    # the QKV decode shape
    (64, 2048, 6144, 1, 4, 16),
    (20, 256, 384, 3, 4, 0),       # groups of 3 straddle the 128-channel tiles
    (18, 136, 264, 3, 2, 7),       # the same for tied low-rank filters; partial tile
])
def test_tensor_core_kernel(B, D, C, H, W, R):
    # batches from 17 sequences take the tcgen05 kernel (D split over a
    # cluster, partial sums added through distributed shared memory)
    _run(torch.bfloat16, B=B, D=D, C=C, H=H, W=W, R=R, seed=B + D + W)


def test_qkv_decode_shape_lowrank():
    _run(torch.bfloat16, B=8, D=2048, C=6144, H=1, W=4, R=16, seed=2)


def test_replay_matches_the_full_sequence_oracle():
    # a sequence decoded token by token from a zero state against the
    # full-sequence forward of the oracle on the projected inputs
    B, T, D, C, H, W = 2, 12, 256, 128, 16, 4
    g = [syn.proj_decode_inputs(B, D, C, H, W, 0, torch.bfloat16, seed=100 + t, device="cuda")
         for t in range(T)]
    Wp = g[0]["Wp"]
    hs = torch.stack([gi["h"] for gi in g], 1)                 # [B, T, D]
    ws = torch.stack([gi["w"] for gi in g], 1)                 # [B, T, G, W]
    x_seq = orc.project(hs.reshape(B * T, D), Wp, torch.bfloat16).reshape(B, T, C)
    yfull = orc.headwise_fwd(x_seq, ws, H, True)
    state = torch.zeros(B, W - 1, C, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(B, C, dtype=torch.bfloat16, device="cuda")
    for t in range(T):
        dsc.dsc_headwise_proj_decode(hs[:, t].contiguous(), Wp, ws[:, t].contiguous(), state, y,
                                     H, True)
        torch.cuda.synchronize()
        assert_fwd(y, yfull[:, t], torch.bfloat16, f"y at t={t}")
        assert_fwd(state[:, 0], x_seq[:, t], torch.bfloat16, f"x at t={t}")


@pytest.mark.parametrize("B", [4, 12])
def test_agrees_with_the_unmerged_pair(B):
    # cuBLAS projection (bf16 output), then the decode step, on the same inputs
    D, C, H, W = 2048, 1024, 16, 4
    inp = syn.proj_decode_inputs(B, D, C, H, W, 0, torch.bfloat16, seed=5, device="cuda")
    s1, s2 = inp["state"].clone(), inp["state"].clone()
    y1 = torch.empty(B, C, dtype=torch.bfloat16, device="cuda")
    y2 = torch.empty_like(y1)
    dsc.dsc_headwise_proj_decode(inp["h"], inp["Wp"], inp["w"], s1, y1, H, True)
    x = inp["h"] @ inp["Wp"].T
    dsc.dsc_headwise_decode(x, inp["w"], s2, y2, H, True)
    torch.cuda.synchronize()
    assert_fwd(y1, y2.double().cpu(), torch.bfloat16, "y vs unmerged")
    assert torch.equal(s1[:, 1:], s2[:, 1:])
    assert_fwd(s1[:, 0], x.double().cpu(), torch.bfloat16, "x vs unmerged")


def test_empty_batch_is_a_no_op():
    inp = syn.proj_decode_inputs(1, 64, 64, 1, 4, 0, torch.bfloat16, seed=3, device="cuda")
    y = torch.full((1, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    dsc.dsc_headwise_proj_decode(inp["h"][:0], inp["Wp"], inp["w"][:0], inp["state"][:0], y[:0],
                                 1, True)
    torch.cuda.synchronize()
    assert (y == 7.0).all()


def test_convenience_functions_match_the_entry_points():
    B, D, C, H, W, R = 3, 128, 64, 8, 4, 16
    a = syn.proj_decode_inputs(B, D, C, H, W, 0, torch.bfloat16, seed=21, device="cuda")
    b = syn.proj_decode_inputs(B, D, C, 1, W, R, torch.bfloat16, seed=22, device="cuda")
    s1, s2 = a["state"].clone(), a["state"].clone()
    y1 = dsc.headwise_proj_decode(a["h"], a["Wp"], a["w"], s1, H, True)
    y2 = torch.empty_like(y1)
    dsc.dsc_headwise_proj_decode(a["h"], a["Wp"], a["w"], s2, y2, H, True)
    t1, t2 = b["state"].clone(), b["state"].clone()
    z1 = dsc.lowrank_proj_decode(b["h"], b["Wp"], b["z"], b["U"], t1, 1, W, True)
    z2 = torch.empty_like(z1)
    dsc.dsc_lowrank_proj_decode(b["h"], b["Wp"], b["z"], b["U"], t2, z2, 1, W, True)
    x = torch.randn(B, C, device="cuda").to(torch.bfloat16)
    u1, u2 = a["state"].clone(), a["state"].clone()
    d1 = dsc.headwise_decode(x, a["w"], u1, H, True)
    d2 = torch.empty_like(d1)
    dsc.dsc_headwise_decode(x, a["w"], u2, d2, H, True)
    v1, v2 = b["state"].clone(), b["state"].clone()
    e1 = dsc.lowrank_decode(x, b["z"], b["U"], v1, 1, W, True)
    e2 = torch.empty_like(e1)
    dsc.dsc_lowrank_decode(x, b["z"], b["U"], v2, e2, 1, W, True)
    torch.cuda.synchronize()
    for p, q in ((y1, y2), (s1, s2), (z1, z2), (t1, t2), (d1, d2), (u1, u2), (e1, e2), (v1, v2)):
        assert torch.equal(p, q)

"""Seeded synthetic inputs for the DSC kernels.

This module is the one piece the CUDA path and the fp64 oracle both use: it
draws random tensors and nothing else.  It holds none of the method's
arithmetic (no convolution, no filter generation, no gradient).

Each tensor is drawn from a torch generator seeded with ``seed * 16 + slot``
(slot 0 = x, 1 = w, 2 = dy, 3 = z, 4 = U, 5 = the hot-channel permutation,
6 = h, 7 = Wp, 8 = a decode state), as
fp32 N(0, 1) scaled by its standard deviation, then rounded once to the I/O
dtype.  Both sides consume the rounded tensor, so they see identical values.
Draws on a CUDA device use torch's CUDA generator (fast for the full-size
shapes); the values then differ from a CPU draw with the same seed, but every
test feeds one draw to both sides.

Workload recipes (the standard deviations read "N(0, a)" as mean 0, standard
deviation a):
  tiny_fp32       B=1 T=256 C=64 H=1 W=4 fp32; x, dy ~ N(0,1); w std 1/W.
  qkv_headwise    B=8 T=2048 C=6144 H=16 W=4 bf16, residual; x, dy ~ N(0,1);
                  w std 0.5 -- DSC on the concatenated q,k,v of a 2B-scale LM.
  qkv_lowrank     same x; R=16, H=1; z and U std 1/sqrt(R).
  all-linear sweep C in {2048, 6144, 5632} x T in {512, 2048, 8192} with
                  B = 16384 / T, W in {2, 3, 4}; head-wise H=16, low-rank R=16.
  static conv     the head-wise shapes with H=1 and one filter per channel,
                  w [C, W] std 0.5 (``static_filters``).
  linear_rnn      B=2 T=16384 C=4096 W=4; head-wise H=64, low-rank R=16;
                  x ~ N(0,1) with round(0.05 C) channels (a seeded random
                  choice) scaled by 8 to stress accumulation.
  decode with its projection (``proj_decode_inputs``): hidden states
                  h [B,D] ~ N(0,1) (slot 6), projection weight Wp [C,D] std
                  1/sqrt(D) (slot 7, so x = h Wp^T is about N(0,1)), state
                  [B,W-1,C] ~ N(0,1) (slot 8), and w [B,G,W] std 0.5 or z
                  [B,R], U [R,G*W] std 1/sqrt(R) for the filters; the decode
                  shape of the QKV placement is B=8, D=2048, C=6144, H=16, W=4.
"""
from dataclasses import dataclass, replace
import math

import torch

SLOT_X, SLOT_W, SLOT_DY, SLOT_Z, SLOT_U, SLOT_HOT, SLOT_H, SLOT_WP, SLOT_STATE = range(9)


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    C: int
    W: int
    H: int = 1
    R: int = 0                # 0 = head-wise parameterisation
    dtype: torch.dtype = torch.bfloat16
    residual: bool = True
    w_std: float = 0.5
    zu_std: float = 0.25
    hot_frac: float = 0.0     # fraction of channels of x scaled by hot_scale
    hot_scale: float = 8.0

    @property
    def lowrank(self) -> bool:
        return self.R > 0

    @property
    def G(self) -> int:
        return self.C // self.H

    @property
    def tokens(self) -> int:
        return self.B * self.T

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def tiny_fp32(residual: bool = False) -> Workload:
    return Workload("tiny_fp32", B=1, T=256, C=64, W=4, H=1,
                    dtype=torch.float32, residual=residual, w_std=1.0 / 4)


def qkv_headwise() -> Workload:
    return Workload("qkv_headwise", B=8, T=2048, C=6144, W=4, H=16, w_std=0.5)


def qkv_lowrank() -> Workload:
    return Workload("qkv_lowrank", B=8, T=2048, C=6144, W=4, H=1, R=16,
                    zu_std=1.0 / math.sqrt(16))


def all_linear_sweep():
    """The 27 shapes x 2 parameterisations of the all-linear placement."""
    out = []
    for C in (2048, 6144, 5632):
        for T in (512, 2048, 8192):
            for W in (2, 3, 4):
                B = 16384 // T
                out.append(Workload(f"all_linear_hw_C{C}_T{T}_W{W}", B=B, T=T,
                                    C=C, W=W, H=16, w_std=0.5))
                out.append(Workload(f"all_linear_lr_C{C}_T{T}_W{W}", B=B, T=T,
                                    C=C, W=W, H=1, R=16, zu_std=0.25))
    return out


def linear_rnn_headwise() -> Workload:
    return Workload("linear_rnn_headwise", B=2, T=16384, C=4096, W=4, H=64,
                    w_std=0.5, hot_frac=0.05)


def linear_rnn_lowrank() -> Workload:
    return Workload("linear_rnn_lowrank", B=2, T=16384, C=4096, W=4, H=1,
                    R=16, zu_std=0.25, hot_frac=0.05)


def _gen(seed: int, slot: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 16 + slot)
    return g


def draw(shape, std: float, seed: int, slot: int, dtype, device="cpu"):
    """N(0, std^2) draw in fp32, rounded once to `dtype`."""
    t = torch.randn(shape, generator=_gen(seed, slot, device), device=device,
                    dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def hot_channels(C: int, frac: float, seed: int) -> torch.Tensor:
    """The seeded set of round(frac*C) channels that get scaled."""
    n = int(round(frac * C))
    perm = torch.randperm(C, generator=_gen(seed, SLOT_HOT, "cpu"))
    return perm[:n].sort().values


def make_inputs(wl: Workload, seed: int = 0, device="cpu", need_grad_inputs=True):
    """Dict of input tensors for a workload.

    Head-wise: x [B,T,C], w [B,T,G,W], dy [B,T,C].
    Low-rank:  x [B,T,C], z [B,T,R], U [R,G*W], dy [B,T,C].
    """
    B, T, C, W = wl.B, wl.T, wl.C, wl.W
    out = {}
    x = draw((B, T, C), 1.0, seed, SLOT_X, torch.float32, device)
    if wl.hot_frac > 0:
        idx = hot_channels(C, wl.hot_frac, seed).to(x.device)
        x[..., idx] *= wl.hot_scale
    out["x"] = x.to(wl.dtype)
    if wl.lowrank:
        out["z"] = draw((B, T, wl.R), wl.zu_std, seed, SLOT_Z, wl.dtype, device)
        out["U"] = draw((wl.R, wl.G * W), wl.zu_std, seed, SLOT_U, wl.dtype, device)
    else:
        out["w"] = draw((B, T, wl.G, W), wl.w_std, seed, SLOT_W, wl.dtype, device)
    if need_grad_inputs:
        out["dy"] = draw((B, T, C), 1.0, seed, SLOT_DY, wl.dtype, device)
    return out


def proj_decode_inputs(B, D, C, H, W, R=0, dtype=torch.bfloat16, seed=0, device="cpu"):
    """Inputs of one decode step merged with its projection: h [B,D],
    Wp [C,D], state [B,W-1,C], and w [B,C/H,W] (R = 0) or z [B,R], U [R,(C/H)*W]."""
    out = {
        "h": draw((B, D), 1.0, seed, SLOT_H, dtype, device),
        "Wp": draw((C, D), 1.0 / math.sqrt(D), seed, SLOT_WP, dtype, device),
        "state": draw((B, max(W - 1, 0), C), 1.0, seed, SLOT_STATE, dtype, device),
    }
    if R:
        out["z"] = draw((B, R), 1.0 / math.sqrt(R), seed, SLOT_Z, dtype, device)
        out["U"] = draw((R, (C // H) * W), 1.0 / math.sqrt(R), seed, SLOT_U, dtype, device)
    else:
        out["w"] = draw((B, C // H, W), 0.5, seed, SLOT_W, dtype, device)
    return out


def static_filters(C: int, W: int, std: float, seed: int, dtype, device="cpu"):
    """Filters w [C, W] of the static short convolution (one per channel)."""
    return draw((C, W), std, seed, SLOT_W, dtype, device)


def sample_rows(B: int, T: int, W: int, n: int, seed: int = 0, tile: int = 64):
    """A seeded subset of token rows b*T+t for full-size spot checks.

    It always holds the first W and last W tokens of every sequence and the
    tokens on either side of every `tile`-th position (where kernels switch
    tiles), topped up with uniformly drawn distinct rows to at least
    min(n, B*T) rows in total.
    """
    must = set()
    for b in range(B):
        base = b * T
        for t in list(range(min(W, T))) + list(range(max(0, T - W), T)):
            must.add(base + t)
    # tile seams of the first and last sequence only (keeps the set small)
    for b in {0, B - 1}:
        for t0 in range(tile, T, tile):
            for d in (-1, 0):
                must.add(b * T + t0 + d)
    g = _gen(seed, 7, "cpu")
    extra = min(max(0, n - len(must)), B * T - len(must))
    if extra:
        # the first `extra` rows of a seeded permutation that are not yet in
        # the set, so the result holds min(n, B*T) distinct rows (or more, if
        # the edges and seams alone exceed n)
        for r in torch.randperm(B * T, generator=g).tolist():
            if r not in must:
                must.add(r)
                extra -= 1
                if extra == 0:
                    break
    return torch.tensor(sorted(must), dtype=torch.int64)

"""fp64 CPU oracle for Dynamic Short Convolutions (DSC) -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product library (the CUDA kernels behind
the C ABI) never touches it, and it shares no code with them.

The arithmetic lives in ``dsc_oracle.c`` (plain fp64 loops, one function per
definition; see the comment block at its top for the passages each follows).
This module marshals torch CPU tensors into it and returns fp64 torch
tensors; the decode step, the decode step merged with its projection and
the static convolution at the end are compositions of those functions (a
W-token window through the forward; one fp64 matmul and a rounding before
that; the filter repeated at every token, its gradient summed over tokens
in fp64).  Inputs may be float64, float32 or bfloat16; the C side decodes
them exactly, so the oracle sees the values the GPU sees.

Every function takes an optional ``rows`` (int64 tensor of token indices
b*T + t); the outputs then hold only those rows, in that order.
"""
import ctypes

import numpy as np
import torch

from .build import LIB, build_oracle

_DT = {torch.float64: 0, torch.float32: 1, torch.bfloat16: 2}
_lib = None


def _load():
    global _lib
    if _lib is None:
        build_oracle()
        lib = ctypes.CDLL(LIB)
        P, I64, INT = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.orc_headwise_fwd.argtypes = [P, INT, P, INT, P, I64, I64, I64, I64,
                                         I64, INT, P, I64]
        lib.orc_lowrank_fwd.argtypes = [P, INT, P, INT, P, INT, P, I64, I64,
                                        I64, I64, I64, I64, INT, P, I64]
        lib.orc_lowrank_filters.argtypes = [P, INT, P, INT, P, I64, I64, I64,
                                            I64, I64, I64]
        lib.orc_headwise_bwd.argtypes = [P, INT, P, INT, P, INT, P, P, I64, I64,
                                         I64, I64, I64, INT, P, I64]
        lib.orc_lowrank_bwd_rows.argtypes = [P, INT, P, INT, P, INT, P, INT, P,
                                             P, P, I64, I64, I64, I64, I64,
                                             I64, INT, P, I64]
        lib.orc_lowrank_dU.argtypes = [P, INT, P, INT, P, INT, P, I64, I64,
                                       I64, I64, I64, I64]
        for f in ("orc_headwise_fwd", "orc_lowrank_fwd", "orc_lowrank_filters",
                  "orc_headwise_bwd", "orc_lowrank_bwd_rows", "orc_lowrank_dU"):
            getattr(lib, f).restype = INT
        lib.orc_num_threads.restype = INT
        lib.orc_set_num_threads.argtypes = [INT]
        _lib = lib
    return _lib


def _in(t):
    t = t.detach()
    if t.device.type != "cpu":
        t = t.cpu()
    t = t.contiguous()
    if t.dtype not in _DT:
        raise TypeError(f"oracle input dtype {t.dtype} not supported")
    return t, ctypes.c_void_p(t.data_ptr()), _DT[t.dtype]


def _rows(rows, n_all):
    if rows is None:
        return None, None, n_all
    r = torch.as_tensor(rows, dtype=torch.int64).contiguous()
    return r, ctypes.c_void_p(r.data_ptr()), r.numel()


def _out(*shape):
    return torch.empty(shape, dtype=torch.float64)


def _check(rc, name):
    if rc != 0:
        raise RuntimeError(f"oracle {name} failed (bad argument or out of memory)")


def num_threads() -> int:
    return _load().orc_num_threads()


def set_num_threads(n: int) -> None:
    _load().orc_set_num_threads(int(n))


def headwise_fwd(x, w, H, residual, rows=None):
    """y [B,T,C] (or [len(rows),C]) of the head-wise DSC forward."""
    lib = _load()
    B, T, C = x.shape
    W = w.shape[-1]
    xk, xp, xd = _in(x)
    wk, wp, wd = _in(w)
    rk, rp, n = _rows(rows, B * T)
    y = _out(n, C)
    _check(lib.orc_headwise_fwd(xp, xd, wp, wd, ctypes.c_void_p(y.data_ptr()),
                                B, T, C, H, W, int(residual), rp, n), "headwise_fwd")
    return y.view(B, T, C) if rows is None else y


def headwise_bwd(x, w, dy, H, residual, rows=None):
    """(dx, dw) of the head-wise DSC backward, full or for the listed rows."""
    lib = _load()
    B, T, C = x.shape
    W = w.shape[-1]
    G = C // H
    xk, xp, xd = _in(x)
    wk, wp, wd = _in(w)
    gk, gp, gd = _in(dy)
    rk, rp, n = _rows(rows, B * T)
    dx = _out(n, C)
    dw = _out(n, G, W)
    _check(lib.orc_headwise_bwd(xp, xd, wp, wd, gp, gd,
                                ctypes.c_void_p(dx.data_ptr()),
                                ctypes.c_void_p(dw.data_ptr()),
                                B, T, C, H, W, int(residual), rp, n), "headwise_bwd")
    if rows is None:
        return dx.view(B, T, C), dw.view(B, T, G, W)
    return dx, dw


def lowrank_filters(z, U, C, H, W):
    """Materialised w [B,T,G,W] = z U (fp64), the naive low-rank path."""
    lib = _load()
    B, T, R = z.shape
    G = C // H
    zk, zp, zd = _in(z)
    uk, up, ud = _in(U)
    w = _out(B, T, G, W)
    _check(lib.orc_lowrank_filters(zp, zd, up, ud, ctypes.c_void_p(w.data_ptr()),
                                   B, T, C, H, W, R), "lowrank_filters")
    return w


def lowrank_fwd(x, z, U, H, W, residual, rows=None):
    """y of the low-rank DSC forward (filters z_t U formed in fp64)."""
    lib = _load()
    B, T, C = x.shape
    R = z.shape[-1]
    xk, xp, xd = _in(x)
    zk, zp, zd = _in(z)
    uk, up, ud = _in(U)
    rk, rp, n = _rows(rows, B * T)
    y = _out(n, C)
    _check(lib.orc_lowrank_fwd(xp, xd, zp, zd, up, ud,
                               ctypes.c_void_p(y.data_ptr()), B, T, C, H, W, R,
                               int(residual), rp, n), "lowrank_fwd")
    return y.view(B, T, C) if rows is None else y


def lowrank_bwd_rows(x, z, U, dy, H, W, residual, rows=None, want_dw=False):
    """(dx, dz[, dw]) of the low-rank backward, full or for the listed rows."""
    lib = _load()
    B, T, C = x.shape
    R = z.shape[-1]
    G = C // H
    xk, xp, xd = _in(x)
    zk, zp, zd = _in(z)
    uk, up, ud = _in(U)
    gk, gp, gd = _in(dy)
    rk, rp, n = _rows(rows, B * T)
    dx = _out(n, C)
    dz = _out(n, R)
    dw = _out(n, G, W) if want_dw else None
    _check(lib.orc_lowrank_bwd_rows(
        xp, xd, zp, zd, up, ud, gp, gd, ctypes.c_void_p(dx.data_ptr()),
        ctypes.c_void_p(dz.data_ptr()),
        ctypes.c_void_p(dw.data_ptr()) if want_dw else None,
        B, T, C, H, W, R, int(residual), rp, n), "lowrank_bwd_rows")
    if rows is None:
        dx, dz = dx.view(B, T, C), dz.view(B, T, R)
        dw = dw.view(B, T, G, W) if want_dw else None
    return (dx, dz, dw) if want_dw else (dx, dz)


def lowrank_dz(x, z, U, dy, H, W, rows=None):
    """dz [B,T,R] (or [len(rows),R]) alone: the row-local low-rank backward
    with the dx rows skipped (dz does not depend on them)."""
    lib = _load()
    B, T, C = x.shape
    R = z.shape[-1]
    xk, xp, xd = _in(x)
    zk, zp, zd = _in(z)
    uk, up, ud = _in(U)
    gk, gp, gd = _in(dy)
    rk, rp, n = _rows(rows, B * T)
    dz = _out(n, R)
    _check(lib.orc_lowrank_bwd_rows(
        xp, xd, zp, zd, up, ud, gp, gd, None, ctypes.c_void_p(dz.data_ptr()), None,
        B, T, C, H, W, R, 0, rp, n), "lowrank_dz")
    return dz.view(B, T, R) if rows is None else dz


def lowrank_dU(x, z, dy, H, W):
    """dU [R, G*W] = sum over all tokens of z_t^T dw_t, in token order."""
    lib = _load()
    B, T, C = x.shape
    R = z.shape[-1]
    G = C // H
    xk, xp, xd = _in(x)
    zk, zp, zd = _in(z)
    gk, gp, gd = _in(dy)
    dU = _out(R, G * W)
    _check(lib.orc_lowrank_dU(xp, xd, zp, zd, gp, gd,
                              ctypes.c_void_p(dU.data_ptr()), B, T, C, H, W, R),
           "lowrank_dU")
    return dU


def lowrank_bwd(x, z, U, dy, H, W, residual):
    """(dx, dz, dU) of the low-rank backward over the whole batch."""
    dx, dz = lowrank_bwd_rows(x, z, U, dy, H, W, residual)
    return dx, dz, lowrank_dU(x, z, dy, H, W)


__all__ = ["headwise_fwd", "headwise_bwd", "lowrank_filters", "lowrank_fwd",
           "lowrank_bwd_rows", "lowrank_dz", "lowrank_dU", "lowrank_bwd", "num_threads",
           "set_num_threads", "LIB", "build_oracle"]


# ------------------------------------------------------------ decode step ----
# One new token per sequence with a carried state of the last W-1 inputs
# (state[b, j] = x at time t-1-j; zeros before the sequence start).  The
# pages leave inference to future engineering; the plainest reading is the
# forward definition evaluated at the one new position, with the state as
# its history.  Written here as exactly that: the W-token window [state
# reversed, x_t] run through the full-sequence oracle, whose last row is y_t.

def headwise_decode(x_t, w_t, state, H, residual):
    """(y_t [B, C], new_state [B, W-1, C]) in fp64.  x_t [B, C], w_t [B, G, W],
    state [B, W-1, C]."""
    B, C = x_t.shape
    W = w_t.shape[-1]
    xs = x_t.double().cpu().reshape(B, 1, C)
    st = state.double().cpu().reshape(B, W - 1, C)
    window = torch.cat([st.flip(1), xs], dim=1)                  # times t-W+1 .. t
    wwin = torch.zeros(B, W, w_t.shape[1], W, dtype=torch.float64)
    wwin[:, W - 1] = w_t.double().cpu()
    y = headwise_fwd(window, wwin, H, residual).reshape(B, W, C)[:, W - 1]
    new_state = torch.cat([xs, st[:, :W - 2]], dim=1) if W > 1 else st
    return y, new_state


def lowrank_decode(x_t, z_t, U, state, H, W, residual):
    """The low-rank decode step: filters z_t U, then the head-wise step."""
    B, C = x_t.shape
    w_t = lowrank_filters(z_t.reshape(B, 1, -1), U, C, H, W).reshape(B, C // H, W)
    return headwise_decode(x_t, w_t, state, H, residual)


# ------------------------------------ decode step merged with its projection --
# "Dynamic Short Convolutions: The 'Locality Bias' Transformers Were
# Missing", Limitations: for inference the convolution is to be merged into
# the matmul that precedes it.  In a decode step that matmul is the
# projection of the new token's hidden state, x_t = h_t Wp^T, with Wp [C, D]
# stored as a linear layer stores its weight.  The merged step computes what
# the two separate steps compute: the projection, its result rounded once to
# the I/O type (the unmerged pair stores x_t in that type), then the decode
# step above on that x_t.  The projection is one fp64 matmul; the rounding is
# round-to-nearest-even from the fp64 value.

def round_to(v, dtype):
    """fp64 tensor rounded to nearest-even `dtype` (torch.bfloat16 or
    torch.float32), returned in that dtype.  bf16 keeps 8 significant bits:
    v = m 2^e with 0.5 <= |m| < 1 becomes round_half_even(m 2^8) 2^(e-8)
    (normal range; the tests' values are far from under- and overflow)."""
    a = v.detach().double().cpu().numpy()
    if dtype == torch.float32:
        return torch.from_numpy(a.astype(np.float32))
    if dtype != torch.bfloat16:
        raise ValueError("round_to: bf16 or fp32")
    m, e = np.frexp(a)
    q = np.ldexp(np.round(m * 256.0), e - 8)       # np.round: half to even
    return torch.from_numpy(q).to(torch.bfloat16)   # exact: q is a bf16 value


def project(h, Wp, dtype):
    """x_t [B, C] = h [B, D] Wp[C, D]^T in fp64, rounded to `dtype`."""
    x64 = h.detach().double().cpu() @ Wp.detach().double().cpu().T
    return round_to(x64, dtype)


def headwise_proj_decode(h, Wp, w_t, state, H, residual):
    """(y_t, new_state, x_t): the projection, then the head-wise decode step."""
    x_t = project(h, Wp, h.dtype)
    y, new_state = headwise_decode(x_t, w_t, state, H, residual)
    return y, new_state, x_t


def lowrank_proj_decode(h, Wp, z_t, U, state, H, W, residual):
    """(y_t, new_state, x_t): the projection, then the low-rank decode step."""
    x_t = project(h, Wp, h.dtype)
    y, new_state = lowrank_decode(x_t, z_t, U, state, H, W, residual)
    return y, new_state, x_t


# -------------------------------------------------- static short conv ------
# "Dynamic Short Convolutions: The 'Locality Bias' Transformers Were
# Missing", Methodology: Adaptive Filtering at Scale, 1. Mathematical
# Intuition: the standard (static) convolution has one filter per channel,
# the same at every token.  It is the head-wise definition with H = 1 and
# w[b,t] = w for all b, t; its filter gradient is the head-wise dw summed
# over every token.  Written here as exactly that composition.

def _broadcast_w(w, B, T):
    C, W = w.shape
    return w.double().cpu().reshape(1, 1, C, W).expand(B, T, C, W).contiguous()


def static_fwd(x, w, residual, rows=None):
    """y of the static short conv, w [C, W]; full or for the listed rows.

    For rows, each listed token is evaluated on its own W-token causal
    window (zeros before the sequence start, as the definition pads)."""
    B, T, C = x.shape
    W = w.shape[-1]
    if rows is None:
        return headwise_fwd(x, _broadcast_w(w, B, T), 1, residual)
    rows = rows.to(torch.int64).cpu()
    xd = x.double().cpu().reshape(B * T, C)
    n = rows.numel()
    win = torch.zeros(n, W, C, dtype=torch.float64)
    t = rows % T
    for j in range(W):                      # window slot j holds time t-(W-1)+j
        back = W - 1 - j
        ok = t >= back
        win[ok, j] = xd[rows[ok] - back]
    return headwise_fwd(win, _broadcast_w(w, n, W), 1, residual)[:, W - 1]


def static_bwd(x, w, dy, residual):
    """(dx [B,T,C], dw [C,W]) of the static short conv over the whole batch."""
    B, T, C = x.shape
    dx, dw_tok = headwise_bwd(x, _broadcast_w(w, B, T), dy, 1, residual)
    return dx, dw_tok.sum(dim=(0, 1)).reshape(C, -1)


def static_dx_rows(w, dy, residual, T, rows):
    """dx of the static short conv for the listed token rows (dy [B,T,C]).

    dx at time s depends on dy at s..s+W-1 of the same sequence only; each
    row is evaluated on that forward window (zeros past the sequence end)."""
    B, _, C = dy.shape
    W = w.shape[-1]
    rows = rows.to(torch.int64).cpu()
    gd = dy.double().cpu().reshape(B * T, C)
    n = rows.numel()
    win = torch.zeros(n, W, C, dtype=torch.float64)
    s = rows % T
    for j in range(W):                      # window slot j holds time s+j
        ok = s + j < T
        win[ok, j] = gd[rows[ok] + j]
    dx, _ = headwise_bwd(torch.zeros(n, W, C, dtype=torch.float64), _broadcast_w(w, n, W),
                         win, 1, residual)
    return dx[:, 0]

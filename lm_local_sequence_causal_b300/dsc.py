"""Thin ctypes binding to libdsc.so (the C ABI of include/dsc.h).

The functions named like the C entry points (``dsc_headwise_fwd`` ...) take
torch CUDA tensors for the pointer arguments and only marshal them: check
dtype, contiguity and device, pass ``data_ptr()`` and the current CUDA
stream, and raise ``DSCError`` on any status other than DSC_OK.  All the
arithmetic runs in the CUDA kernels; there is no CPU or PyTorch fallback.
If the library is missing the first call raises.

``headwise_fwd`` and friends are conveniences that allocate the outputs
with torch and call the entry points.

``bind(entry, *args, **kw)`` marshals the arguments of one entry point once
and returns a ``BoundCall``: calling it re-issues the same C call with the
same pointers, sizes and stream, with no per-call Python checks.  It is for
loops that launch the same call on the same buffers many times, where the
marshalling would otherwise cost more host time than the kernel takes.
"""
import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdsc.so")

DSC_OK, DSC_ERR_INVALID_ARG, DSC_ERR_ALIGNMENT = 0, 1, 2
DSC_ERR_UNSUPPORTED, DSC_ERR_WORKSPACE, DSC_ERR_CUDA = 3, 4, 5
DSC_F32, DSC_BF16 = 0, 1
_DTYPES = {torch.float32: DSC_F32, torch.bfloat16: DSC_BF16}

_lib = None


class DSCError(RuntimeError):
    def __init__(self, status, name):
        self.status = status
        super().__init__(f"{name} failed: {status_string(status)} ({status})")


def load():
    """Load libdsc.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libdsc.so not found at {LIB_PATH}; build it with "
                           "`python -m lm_local_sequence_causal_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I64, INT, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    lib.dsc_abi_version.restype = INT
    lib.dsc_status_string.argtypes = [INT]
    lib.dsc_status_string.restype = ctypes.c_char_p
    lib.dsc_headwise_fwd.argtypes = [P, P, P, I64, I64, I64, I64, I64, INT, INT, P]
    lib.dsc_headwise_bwd.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I64, INT, INT, P]
    lib.dsc_lowrank_fwd.argtypes = [P, P, P, P, I64, I64, I64, I64, I64, I64, INT, INT, P]
    lib.dsc_lowrank_bwd_workspace_size.argtypes = [I64, I64, I64, I64, I64, I64, INT]
    lib.dsc_lowrank_bwd_workspace_size.restype = SZ
    lib.dsc_lowrank_bwd.argtypes = [P, P, P, P, P, P, P, P, SZ, I64, I64, I64, I64, I64,
                                    I64, INT, INT, P]
    lib.dsc_headwise_decode.argtypes = [P, P, P, P, I64, I64, I64, I64, INT, INT, P]
    lib.dsc_lowrank_decode.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I64, INT, INT, P]
    lib.dsc_headwise_decode.restype = INT
    lib.dsc_static_fwd.argtypes = [P, P, P, I64, I64, I64, I64, INT, INT, P]
    lib.dsc_static_fwd.restype = INT
    lib.dsc_static_bwd_workspace_size.argtypes = [I64, I64, I64, I64, INT]
    lib.dsc_static_bwd_workspace_size.restype = SZ
    lib.dsc_static_bwd.argtypes = [P, P, P, P, P, P, SZ, I64, I64, I64, I64, INT, INT, P]
    lib.dsc_static_bwd.restype = INT
    lib.dsc_lowrank_decode.restype = INT
    lib.dsc_headwise_proj_decode.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I64, INT,
                                             INT, P]
    lib.dsc_headwise_proj_decode.restype = INT
    lib.dsc_lowrank_proj_decode.argtypes = [P, P, P, P, P, P, I64, I64, I64, I64, I64, I64,
                                            INT, INT, P]
    lib.dsc_lowrank_proj_decode.restype = INT
    lib.dsc_headwise_proj_decode_selftest_timeout.argtypes = [P, P, P, P, P, I64, I64, I64, I64,
                                                              I64, INT, INT, ctypes.c_uint64, P]
    lib.dsc_headwise_proj_decode_selftest_timeout.restype = INT
    lib.dsc_lowrank_uses_tensor_cores.argtypes = [I64, I64, I64, I64, I64, I64, INT]
    lib.dsc_lowrank_uses_tensor_cores.restype = INT
    lib.dsc_headwise_uses_tma.argtypes = [I64, I64, I64, I64, I64, INT]
    lib.dsc_headwise_uses_tma.restype = INT
    lib.dsc_lowrank_bwd_noalloc.argtypes = [P, P, P, P, P, P, P, I64, I64, I64, I64, I64,
                                            I64, INT, INT, P]
    lib.dsc_lowrank_bwd_noalloc.restype = INT
    U64 = ctypes.c_uint64
    lib.dsc_lowrank_fwd_selftest_timeout.argtypes = [P, P, P, P, I64, I64, I64, I64, I64, I64,
                                                     INT, INT, U64, P]
    lib.dsc_lowrank_fwd_selftest_timeout.restype = INT
    lib.dsc_lowrank_bwd_selftest_timeout.argtypes = [P, P, P, P, P, P, P, P, SZ, I64, I64, I64,
                                                     I64, I64, I64, INT, INT, U64, P]
    lib.dsc_lowrank_bwd_selftest_timeout.restype = INT
    lib.dsc_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint), INT]
    lib.dsc_device_error.restype = INT
    for f in ("dsc_headwise_fwd", "dsc_headwise_bwd", "dsc_lowrank_fwd", "dsc_lowrank_bwd"):
        getattr(lib, f).restype = INT
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().dsc_status_string(int(status)).decode()


def abi_version() -> int:
    return load().dsc_abi_version()


def dsc_lowrank_uses_tensor_cores(B, T, C, H, W, R, dtype) -> int:
    """Bit 0: forward on the tensor cores, bit 1: backward; -1: invalid/unsupported."""
    return int(load().dsc_lowrank_uses_tensor_cores(B, T, C, H, W, R, _DTYPES[dtype]))


def dsc_headwise_uses_tma(B, T, C, H, W, dtype) -> int:
    """Bit 0: forward on the TMA-staged kernel, bit 1: backward; -1: invalid."""
    return int(load().dsc_headwise_uses_tma(B, T, C, H, W, _DTYPES[dtype]))


def dsc_device_error(reset=False) -> int:
    """Error word of the tensor-core kernels on the current device (0 = none)."""
    code = ctypes.c_uint(0)
    _check(load().dsc_device_error(ctypes.byref(code), int(bool(reset))), "dsc_device_error")
    return int(code.value)


# ------------------------------------------------------------ marshalling ----

def _ptr(t, dtype, name):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _dtype_code(t):
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype}; use float32 or bfloat16")
    return _DTYPES[t.dtype]


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(rc, name):
    if rc != DSC_OK:
        raise DSCError(rc, name)


def _bt_c(x):
    if x.dim() != 3:
        raise ValueError("x must be [B, T, C]")
    return x.shape


# --------------------------------------------------- the C entry points ------
# Each _m_<entry> returns the ctypes argument tuple of that C entry point.

def _m_dsc_headwise_fwd(x, w, y, H, residual=True, stream=None):
    B, T, C = _bt_c(x)
    W = w.shape[-1]
    dt = x.dtype
    return (_ptr(x, dt, "x"), _ptr(w, dt, "w"), _ptr(y, dt, "y"), B, T, C, H, W,
            int(bool(residual)), _dtype_code(x), _stream(stream))


def _m_dsc_headwise_bwd(x, w, dy, dx, dw, H, residual=True, stream=None):
    B, T, C = _bt_c(x)
    W = w.shape[-1]
    dt = x.dtype
    return (_ptr(x, dt, "x"), _ptr(w, dt, "w"), _ptr(dy, dt, "dy"), _ptr(dx, dt, "dx"),
            _ptr(dw, dt, "dw"), B, T, C, H, W, int(bool(residual)), _dtype_code(x),
            _stream(stream))


def _m_dsc_lowrank_fwd(x, z, U, y, H, W, residual=True, stream=None):
    B, T, C = _bt_c(x)
    R = z.shape[-1]
    dt = x.dtype
    return (_ptr(x, dt, "x"), _ptr(z, dt, "z"), _ptr(U, dt, "U"), _ptr(y, dt, "y"),
            B, T, C, H, W, R, int(bool(residual)), _dtype_code(x), _stream(stream))


def _m_dsc_lowrank_bwd(x, z, U, dy, dx, dz, dU, workspace, H, W, residual=True, stream=None):
    B, T, C = _bt_c(x)
    R = z.shape[-1]
    dt = x.dtype
    ws_ptr = _ptr(workspace, torch.uint8, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() if workspace is not None else 0
    return (_ptr(x, dt, "x"), _ptr(z, dt, "z"), _ptr(U, dt, "U"), _ptr(dy, dt, "dy"),
            _ptr(dx, dt, "dx"), _ptr(dz, dt, "dz"), _ptr(dU, dt, "dU"), ws_ptr, ws_bytes,
            B, T, C, H, W, R, int(bool(residual)), _dtype_code(x), _stream(stream))


def _m_dsc_lowrank_bwd_noalloc(x, z, U, dy, dx, dz, dU, H, W, residual=True, stream=None):
    B, T, C = _bt_c(x)
    R = z.shape[-1]
    dt = x.dtype
    return (_ptr(x, dt, "x"), _ptr(z, dt, "z"), _ptr(U, dt, "U"), _ptr(dy, dt, "dy"),
            _ptr(dx, dt, "dx"), _ptr(dz, dt, "dz"), _ptr(dU, dt, "dU"), B, T, C, H, W, R,
            int(bool(residual)), _dtype_code(x), _stream(stream))


def _m_dsc_headwise_decode(x, w, state, y, H, residual=True, stream=None):
    if x.dim() != 2:
        raise ValueError("x must be [B, C]")
    B, C = x.shape
    W = w.shape[-1]
    dt = x.dtype
    sp = _ptr(state, dt, "state") if W > 1 else None
    return (_ptr(x, dt, "x"), _ptr(w, dt, "w"), sp, _ptr(y, dt, "y"), B, C, H, W,
            int(bool(residual)), _dtype_code(x), _stream(stream))


def _m_dsc_lowrank_decode(x, z, U, state, y, H, W, residual=True, stream=None):
    if x.dim() != 2:
        raise ValueError("x must be [B, C]")
    B, C = x.shape
    R = z.shape[-1]
    dt = x.dtype
    sp = _ptr(state, dt, "state") if W > 1 else None
    return (_ptr(x, dt, "x"), _ptr(z, dt, "z"), _ptr(U, dt, "U"), sp, _ptr(y, dt, "y"),
            B, C, H, W, R, int(bool(residual)), _dtype_code(x), _stream(stream))


def _m_dsc_headwise_proj_decode(h, Wp, w, state, y, H, residual=True, stream=None):
    if h.dim() != 2 or Wp.dim() != 2:
        raise ValueError("h must be [B, D] and Wp [C, D]")
    B, D = h.shape
    C = Wp.shape[0]
    W = w.shape[-1]
    dt = h.dtype
    sp = _ptr(state, dt, "state") if W > 1 else None
    return (_ptr(h, dt, "h"), _ptr(Wp, dt, "Wp"), _ptr(w, dt, "w"), sp, _ptr(y, dt, "y"),
            B, D, C, H, W, int(bool(residual)), _dtype_code(h), _stream(stream))


def _m_dsc_lowrank_proj_decode(h, Wp, z, U, state, y, H, W, residual=True, stream=None):
    if h.dim() != 2 or Wp.dim() != 2:
        raise ValueError("h must be [B, D] and Wp [C, D]")
    B, D = h.shape
    C = Wp.shape[0]
    R = z.shape[-1]
    dt = h.dtype
    sp = _ptr(state, dt, "state") if W > 1 else None
    return (_ptr(h, dt, "h"), _ptr(Wp, dt, "Wp"), _ptr(z, dt, "z"), _ptr(U, dt, "U"), sp,
            _ptr(y, dt, "y"), B, D, C, H, W, R, int(bool(residual)), _dtype_code(h),
            _stream(stream))


def _m_dsc_static_fwd(x, w, y, residual=True, stream=None):
    B, T, C = _bt_c(x)
    W = w.shape[-1]
    dt = x.dtype
    return (_ptr(x, dt, "x"), _ptr(w, dt, "w"), _ptr(y, dt, "y"), B, T, C, W,
            int(bool(residual)), _dtype_code(x), _stream(stream))


def _m_dsc_static_bwd(x, w, dy, dx, dw, workspace, residual=True, stream=None):
    B, T, C = _bt_c(x)
    W = w.shape[-1]
    dt = x.dtype
    ws_ptr = _ptr(workspace, torch.uint8, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() if workspace is not None else 0
    return (_ptr(x, dt, "x"), _ptr(w, dt, "w"), _ptr(dy, dt, "dy"), _ptr(dx, dt, "dx"),
            _ptr(dw, dt, "dw"), ws_ptr, ws_bytes, B, T, C, W, int(bool(residual)),
            _dtype_code(x), _stream(stream))


def _call(name, args):
    _check(getattr(load(), name)(*args), name)


def dsc_headwise_fwd(x, w, y, H, residual=True, stream=None):
    """y[b,t,c] = residual*x + sum_k w[b,t,c//H,k] x[b,t-k,c]   (in place into y)."""
    _call("dsc_headwise_fwd", _m_dsc_headwise_fwd(x, w, y, H, residual, stream))


def dsc_headwise_bwd(x, w, dy, dx, dw, H, residual=True, stream=None):
    """dx, dw of the head-wise DSC (written in place)."""
    _call("dsc_headwise_bwd", _m_dsc_headwise_bwd(x, w, dy, dx, dw, H, residual, stream))


def dsc_lowrank_fwd(x, z, U, y, H, W, residual=True, stream=None):
    """y of the low-rank fused DSC (filters z_t U formed on-chip)."""
    _call("dsc_lowrank_fwd", _m_dsc_lowrank_fwd(x, z, U, y, H, W, residual, stream))


def dsc_lowrank_bwd_workspace_size(B, T, C, H, W, R, dtype) -> int:
    return int(load().dsc_lowrank_bwd_workspace_size(B, T, C, H, W, R, _DTYPES[dtype]))


def dsc_lowrank_bwd(x, z, U, dy, dx, dz, dU, workspace, H, W, residual=True, stream=None):
    """dx, dz, dU of the low-rank fused DSC; `workspace` is a uint8 CUDA tensor."""
    _call("dsc_lowrank_bwd",
          _m_dsc_lowrank_bwd(x, z, U, dy, dx, dz, dU, workspace, H, W, residual, stream))


def dsc_lowrank_bwd_noalloc(x, z, U, dy, dx, dz, dU, H, W, residual=True, stream=None):
    """dsc_lowrank_bwd with the library's own fixed scratch (no workspace)."""
    _call("dsc_lowrank_bwd_noalloc",
          _m_dsc_lowrank_bwd_noalloc(x, z, U, dy, dx, dz, dU, H, W, residual, stream))


def dsc_headwise_decode(x, w, state, y, H, residual=True, stream=None):
    """One decode step: y [B,C] from x [B,C], w [B,G,W] and state [B,W-1,C]
    (updated in place to hold the last W-1 inputs, newest first)."""
    _call("dsc_headwise_decode", _m_dsc_headwise_decode(x, w, state, y, H, residual, stream))


def dsc_lowrank_decode(x, z, U, state, y, H, W, residual=True, stream=None):
    """Low-rank decode step: taps z [B,R] U formed in fp32, then as above."""
    _call("dsc_lowrank_decode",
          _m_dsc_lowrank_decode(x, z, U, state, y, H, W, residual, stream))


def dsc_headwise_proj_decode(h, Wp, w, state, y, H, residual=True, stream=None):
    """Decode step merged with its projection: x = h [B,D] Wp[C,D]^T rounded
    once to the I/O type inside the kernel, then the head-wise decode step."""
    _call("dsc_headwise_proj_decode",
          _m_dsc_headwise_proj_decode(h, Wp, w, state, y, H, residual, stream))


def dsc_lowrank_proj_decode(h, Wp, z, U, state, y, H, W, residual=True, stream=None):
    """The same with the low-rank decode step (taps z [B,R] U in fp32)."""
    _call("dsc_lowrank_proj_decode",
          _m_dsc_lowrank_proj_decode(h, Wp, z, U, state, y, H, W, residual, stream))


def dsc_static_fwd(x, w, y, residual=True, stream=None):
    """Static short conv: y[b,t,c] = residual*x + sum_k w[c,k] x[b,t-k,c]; w is [C, W]."""
    _call("dsc_static_fwd", _m_dsc_static_fwd(x, w, y, residual, stream))


def dsc_static_bwd_workspace_size(B, T, C, W, dtype) -> int:
    return int(load().dsc_static_bwd_workspace_size(B, T, C, W, _DTYPES[dtype]))


def dsc_static_bwd(x, w, dy, dx, dw, workspace, residual=True, stream=None):
    """dx [B,T,C] and dw [C,W] of the static short conv; `workspace` is a uint8 CUDA tensor."""
    _call("dsc_static_bwd", _m_dsc_static_bwd(x, w, dy, dx, dw, workspace, residual, stream))


def dsc_headwise_proj_decode_selftest_timeout(h, Wp, w, state, y, H, wait_limit_ns,
                                              residual=True, stream=None):
    """Failure-path self-test of the tcgen05 merged decode kernel (bf16, 17 or
    more sequences): waits limited to wait_limit_ns and no loads issued; read
    the code with dsc_device_error() afterwards.  y and state are left
    unspecified."""
    a = _m_dsc_headwise_proj_decode(h, Wp, w, state, y, H, residual, stream)
    _call("dsc_headwise_proj_decode_selftest_timeout", a[:-1] + (int(wait_limit_ns), a[-1]))


def dsc_lowrank_fwd_selftest_timeout(x, z, U, y, H, W, wait_limit_ns, residual=True,
                                     stream=None):
    """Failure-path self-test of the tensor-core forward: every bounded wait
    limited to wait_limit_ns and no loads issued, so the waits run out; read
    the code with dsc_device_error() afterwards.  y is left unspecified."""
    a = _m_dsc_lowrank_fwd(x, z, U, y, H, W, residual, stream)
    _call("dsc_lowrank_fwd_selftest_timeout", a[:-1] + (int(wait_limit_ns), a[-1]))


def dsc_lowrank_bwd_selftest_timeout(x, z, U, dy, dx, dz, dU, workspace, H, W, wait_limit_ns,
                                     residual=True, stream=None):
    """Failure-path self-test of the tensor-core backward (as above)."""
    a = _m_dsc_lowrank_bwd(x, z, U, dy, dx, dz, dU, workspace, H, W, residual, stream)
    _call("dsc_lowrank_bwd_selftest_timeout", a[:-1] + (int(wait_limit_ns), a[-1]))


class BoundCall:
    """One C entry point with its argument tuple marshalled once.

    Calling it issues the same C call again (same pointers, sizes and
    stream) and raises DSCError on a status other than DSC_OK.  The tensors
    it was bound to must stay alive and unmoved while it is used."""

    __slots__ = ("name", "fn", "args", "keep")

    def __init__(self, name, args, keep):
        self.name = name
        self.fn = getattr(load(), name)
        self.args = args
        self.keep = keep          # the bound tensors, kept alive

    def __call__(self):
        rc = self.fn(*self.args)
        if rc != DSC_OK:
            raise DSCError(rc, self.name)


def bind(entry, *args, **kw):
    """Marshal the arguments of C entry point `entry` (e.g. "dsc_lowrank_bwd",
    same arguments as the Python function of that name) once; return a
    BoundCall that re-issues the call."""
    m = globals().get("_m_" + entry)
    if m is None:
        raise ValueError(f"no entry point {entry!r}")
    keep = [a for a in list(args) + list(kw.values()) if isinstance(a, torch.Tensor)]
    return BoundCall(entry, m(*args, **kw), keep)


# ------------------------------------------------------- conveniences --------

def headwise_fwd(x, w, H, residual=True):
    y = torch.empty_like(x)
    dsc_headwise_fwd(x, w, y, H, residual)
    return y


def headwise_bwd(x, w, dy, H, residual=True):
    dx = torch.empty_like(x)
    dw = torch.empty_like(w)
    dsc_headwise_bwd(x, w, dy, dx, dw, H, residual)
    return dx, dw


def lowrank_fwd(x, z, U, H, W, residual=True):
    y = torch.empty_like(x)
    dsc_lowrank_fwd(x, z, U, y, H, W, residual)
    return y


def lowrank_workspace(x, z, H, W):
    B, T, C = x.shape
    n = dsc_lowrank_bwd_workspace_size(B, T, C, H, W, z.shape[-1], x.dtype)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=x.device)


def lowrank_bwd(x, z, U, dy, H, W, residual=True, workspace=None):
    dx = torch.empty_like(x)
    dz = torch.empty_like(z)
    dU = torch.empty_like(U)
    if workspace is None:
        workspace = lowrank_workspace(x, z, H, W)
    dsc_lowrank_bwd(x, z, U, dy, dx, dz, dU, workspace, H, W, residual)
    return dx, dz, dU


def static_fwd(x, w, residual=True):
    y = torch.empty_like(x)
    dsc_static_fwd(x, w, y, residual)
    return y


def static_bwd(x, w, dy, residual=True, workspace=None):
    dx = torch.empty_like(x)
    dw = torch.empty_like(w)
    if workspace is None:
        B, T, C = x.shape
        n = dsc_static_bwd_workspace_size(B, T, C, w.shape[-1], x.dtype)
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=x.device)
    dsc_static_bwd(x, w, dy, dx, dw, workspace, residual)
    return dx, dw


def headwise_decode(x, w, state, H, residual=True):
    """One decode step (x [B,C], w [B,C/H,W]); the state [B,W-1,C] is updated
    in place.  Returns y [B,C]."""
    y = torch.empty_like(x)
    dsc_headwise_decode(x, w, state, y, H, residual)
    return y


def lowrank_decode(x, z, U, state, H, W, residual=True):
    y = torch.empty_like(x)
    dsc_lowrank_decode(x, z, U, state, y, H, W, residual)
    return y


def headwise_proj_decode(h, Wp, w, state, H, residual=True):
    """Decode step merged with its projection x = h [B,D] Wp[C,D]^T; the state
    is updated in place (its row 0 becomes x).  Returns y [B,C]."""
    y = torch.empty(h.shape[0], Wp.shape[0], dtype=h.dtype, device=h.device)
    dsc_headwise_proj_decode(h, Wp, w, state, y, H, residual)
    return y


def lowrank_proj_decode(h, Wp, z, U, state, H, W, residual=True):
    y = torch.empty(h.shape[0], Wp.shape[0], dtype=h.dtype, device=h.device)
    dsc_lowrank_proj_decode(h, Wp, z, U, state, y, H, W, residual)
    return y

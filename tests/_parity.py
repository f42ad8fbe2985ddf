"""Helpers for the GPU-vs-oracle parity tests.

Error measures (one reading of the stated bounds, applied to every output):
  forward    max |gpu - ref| / max |ref|        (max-norm relative)
  gradients  ||gpu - ref||_F / ||ref||_F         (Frobenius relative)
Bounds: bf16 I/O 2e-2 (forward) and 5e-2 (gradients); fp32 I/O 1e-5 (both).

Outputs are allocated inside guard bands filled with a NaN bit pattern; a
kernel that writes outside its tensor changes a guard and fails the test.
"""
import torch

TOL = {
    torch.bfloat16: {"fwd": 2e-2, "grad": 5e-2},
    torch.float32: {"fwd": 1e-5, "grad": 1e-5},
}
GUARD_BYTES = 256
_SENTINEL = {torch.bfloat16: 0x7FC3, torch.float32: 0x7FC00003}
_INT_VIEW = {torch.bfloat16: torch.int16, torch.float32: torch.int32}


def max_rel(gpu, ref):
    g = gpu.detach().double().cpu().reshape(-1)
    r = ref.double().reshape(-1)
    den = r.abs().max().item()
    return (g - r).abs().max().item() / (den if den > 0 else 1.0)


def fro_rel(gpu, ref):
    g = gpu.detach().double().cpu().reshape(-1)
    r = ref.double().reshape(-1)
    den = r.norm().item()
    return (g - r).norm().item() / (den if den > 0 else 1.0)


def assert_fwd(gpu, ref, dtype, what="y"):
    e = max_rel(gpu, ref)
    assert e <= TOL[dtype]["fwd"], f"{what}: max-rel error {e:.3e} > {TOL[dtype]['fwd']}"
    assert torch.isfinite(gpu).all(), f"{what}: non-finite output"
    return e


def assert_grad(gpu, ref, dtype, what):
    e = fro_rel(gpu, ref)
    assert e <= TOL[dtype]["grad"], f"{what}: Frobenius-rel error {e:.3e} > {TOL[dtype]['grad']}"
    assert torch.isfinite(gpu).all(), f"{what}: non-finite output"
    return e


class Guarded:
    """An output tensor living inside a larger buffer with sentinel guards."""

    def __init__(self, shape, dtype, device="cuda"):
        esz = torch.empty((), dtype=dtype).element_size()
        self.g = GUARD_BYTES // esz
        n = 1
        for s in shape:
            n *= s
        self.n = n
        self.dtype = dtype
        self.buf = torch.empty(n + 2 * self.g, dtype=dtype, device=device)
        self.buf.view(_INT_VIEW[dtype]).fill_(_SENTINEL[dtype])
        self.t = self.buf[self.g:self.g + n].view(shape)

    def guards_intact(self):
        iv = self.buf.view(_INT_VIEW[self.dtype])
        s = _SENTINEL[self.dtype]
        return bool((iv[:self.g] == s).all()) and bool((iv[self.g + self.n:] == s).all())


def assert_by_channel_set(gpu, ref, hot, dtype, what, grad):
    """The forward or gradient measure computed separately over the listed
    `hot` channels and over all the others (last axis = channels), so that a
    few large channels cannot hide errors in the ordinary ones."""
    g = gpu.detach().double().cpu()
    r = ref.double()
    C = g.shape[-1]
    mask = torch.zeros(C, dtype=torch.bool)
    mask[hot] = True
    out = {}
    for name, m in (("hot", mask), ("ordinary", ~mask)):
        e = (fro_rel if grad else max_rel)(g[..., m], r[..., m])
        bound = TOL[dtype]["grad" if grad else "fwd"]
        assert e <= bound, f"{what} ({name} channels): relative error {e:.3e} > {bound}"
        out[name] = e
    return out


def rows_of(t, rows):
    """Rows (flattened tokens) of a [B,T,...] tensor, on the CPU."""
    flat = t.reshape(t.shape[0] * t.shape[1], -1)
    return flat[rows.to(flat.device)].cpu()

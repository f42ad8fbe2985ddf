// dsc_abi.cu -- the extern "C" entry points declared in include/dsc.h:
// host-side validation, then dispatch to the kernel files.  Nothing here
// allocates, frees or synchronises.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dsc.h"
#include "dsc_internal.h"

namespace {

using dsc::Shape;

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Shape checks common to every entry point.  `R` is 0 for head-wise.
dsc_status_t check_shape(int64_t B, int64_t T, int64_t C, int64_t H, int64_t W,
                         int64_t R, dsc_dtype_t dt, bool lowrank) {
  if (dt != DSC_F32 && dt != DSC_BF16) return DSC_ERR_INVALID_ARG;
  if (B < 0 || T < 0 || C < 1 || H < 1 || W < 1) return DSC_ERR_INVALID_ARG;
  if (C % H != 0) return DSC_ERR_INVALID_ARG;
  if (lowrank && R < 1) return DSC_ERR_INVALID_ARG;
  // Index arithmetic is 64-bit; keep the element counts far from overflow.
  if (B > (int64_t(1) << 31) || T > (int64_t(1) << 31) || C > (int64_t(1) << 24))
    return DSC_ERR_INVALID_ARG;
  if (W > 4) return DSC_ERR_UNSUPPORTED;
  const int64_t vec = dt == DSC_BF16 ? 8 : 4;
  if (C % vec != 0) return DSC_ERR_ALIGNMENT;
  return DSC_OK;
}

dsc_status_t check_ptrs(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (p == nullptr) return DSC_ERR_INVALID_ARG;
  for (const void* p : ps)
    if (!aligned16(p)) return DSC_ERR_ALIGNMENT;
  return DSC_OK;
}

Shape make_shape(int64_t B, int64_t T, int64_t C, int64_t H, int64_t W, int64_t R,
                 int residual, dsc_dtype_t dt) {
  return Shape{B, T, C, H, W, R, residual ? 1 : 0, dt == DSC_BF16 ? 1 : 0};
}

dsc_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? DSC_OK : DSC_ERR_CUDA; }

// Checks of the projection-merged decode step beyond those of the decode step:
// D (the hidden size) positive, 16-byte rows, B small enough for the
// kernel's 32-bit sequence index.
dsc_status_t check_proj(int64_t B, int64_t D, dsc_dtype_t dtype) {
  if (D < 1 || D > (int64_t(1) << 24) || B > (int64_t(1) << 24)) return DSC_ERR_INVALID_ARG;
  if (D % (dtype == DSC_BF16 ? 8 : 4) != 0) return DSC_ERR_ALIGNMENT;
  return DSC_OK;
}

}  // namespace

extern "C" {

int dsc_abi_version(void) { return 1; }

const char* dsc_status_string(dsc_status_t s) {
  switch (s) {
    case DSC_OK: return "DSC_OK";
    case DSC_ERR_INVALID_ARG: return "DSC_ERR_INVALID_ARG";
    case DSC_ERR_ALIGNMENT: return "DSC_ERR_ALIGNMENT";
    case DSC_ERR_UNSUPPORTED: return "DSC_ERR_UNSUPPORTED";
    case DSC_ERR_WORKSPACE: return "DSC_ERR_WORKSPACE";
    case DSC_ERR_CUDA: return "DSC_ERR_CUDA";
  }
  return "DSC_ERR_UNKNOWN";
}

dsc_status_t dsc_headwise_fwd(const void* x, const void* w, void* y, int64_t B, int64_t T,
                              int64_t C, int64_t H, int64_t W, int residual,
                              dsc_dtype_t dtype, void* stream) {
  dsc_status_t st = check_shape(B, T, C, H, W, 0, dtype, false);
  if (st != DSC_OK) return st;
  if (B * T == 0) return DSC_OK;
  if ((st = check_ptrs({x, w, y})) != DSC_OK) return st;
  if (x == y) return DSC_ERR_INVALID_ARG;
  return from_cuda(dsc::headwise_fwd(x, w, y, make_shape(B, T, C, H, W, 0, residual, dtype),
                                     (cudaStream_t)stream));
}

dsc_status_t dsc_headwise_bwd(const void* x, const void* w, const void* dy, void* dx,
                              void* dw, int64_t B, int64_t T, int64_t C, int64_t H,
                              int64_t W, int residual, dsc_dtype_t dtype, void* stream) {
  dsc_status_t st = check_shape(B, T, C, H, W, 0, dtype, false);
  if (st != DSC_OK) return st;
  if (B * T == 0) return DSC_OK;
  if ((st = check_ptrs({x, w, dy, dx, dw})) != DSC_OK) return st;
  if (dx == x || dx == dy || dx == dw || dw == x || dw == w || dw == dy)
    return DSC_ERR_INVALID_ARG;
  return from_cuda(dsc::headwise_bwd(x, w, dy, dx, dw,
                                     make_shape(B, T, C, H, W, 0, residual, dtype),
                                     (cudaStream_t)stream));
}

dsc_status_t dsc_lowrank_fwd(const void* x, const void* z, const void* U, void* y,
                             int64_t B, int64_t T, int64_t C, int64_t H, int64_t W,
                             int64_t R, int residual, dsc_dtype_t dtype, void* stream) {
  dsc_status_t st = check_shape(B, T, C, H, W, R, dtype, true);
  if (st != DSC_OK) return st;
  const Shape s = make_shape(B, T, C, H, W, R, residual, dtype);
  if (!dsc::lowrank_supported(s)) return DSC_ERR_UNSUPPORTED;
  if (B * T == 0) return DSC_OK;
  if ((st = check_ptrs({x, z, U, y})) != DSC_OK) return st;
  if (x == y) return DSC_ERR_INVALID_ARG;
  if (dsc::lowrank_tc_supported(s)) {
    const cudaError_t e = dsc::lowrank_fwd_tc(x, z, U, y, s, (cudaStream_t)stream);
    if (e != cudaErrorNotSupported) return from_cuda(e);
  }
  return from_cuda(dsc::lowrank_fwd(x, z, U, y, s, (cudaStream_t)stream));
}

size_t dsc_lowrank_bwd_workspace_size(int64_t B, int64_t T, int64_t C, int64_t H,
                                      int64_t W, int64_t R, dsc_dtype_t dtype) {
  if (check_shape(B, T, C, H, W, R, dtype, true) != DSC_OK) return 0;
  const Shape s = make_shape(B, T, C, H, W, R, 0, dtype);
  if (!dsc::lowrank_supported(s) || B * T == 0) return 0;
  if (dsc::lowrank_bwd_tc_supported(s)) return dsc::lowrank_bwd_tc_workspace(s);
  return dsc::lowrank_bwd_workspace(s);
}

dsc_status_t dsc_lowrank_bwd(const void* x, const void* z, const void* U, const void* dy,
                             void* dx, void* dz, void* dU, void* workspace,
                             size_t workspace_bytes, int64_t B, int64_t T, int64_t C,
                             int64_t H, int64_t W, int64_t R, int residual,
                             dsc_dtype_t dtype, void* stream) {
  dsc_status_t st = check_shape(B, T, C, H, W, R, dtype, true);
  if (st != DSC_OK) return st;
  const Shape s = make_shape(B, T, C, H, W, R, residual, dtype);
  if (!dsc::lowrank_supported(s)) return DSC_ERR_UNSUPPORTED;
  if (B * T == 0) {
    // dU is a sum over zero tokens: all zeros.  Nothing else to write.
    if (dU == nullptr) return DSC_ERR_INVALID_ARG;
    const size_t bytes = (size_t)R * (C / H) * W * (dtype == DSC_BF16 ? 2 : 4);
    return from_cuda(cudaMemsetAsync(dU, 0, bytes, (cudaStream_t)stream));
  }
  if ((st = check_ptrs({x, z, U, dy, dx, dz, dU})) != DSC_OK) return st;
  if (dx == x || dx == dy || dz == z || dU == U) return DSC_ERR_INVALID_ARG;
  const bool tc = dsc::lowrank_bwd_tc_supported(s);
  const size_t need = tc ? dsc::lowrank_bwd_tc_workspace(s) : dsc::lowrank_bwd_workspace(s);
  if (need > 0) {
    if (workspace == nullptr || workspace_bytes < need) return DSC_ERR_WORKSPACE;
    if (!aligned16(workspace)) return DSC_ERR_ALIGNMENT;
  }
  if (tc)
    return from_cuda(dsc::lowrank_bwd_tc(x, z, U, dy, dx, dz, dU, workspace, s,
                                         (cudaStream_t)stream));
  return from_cuda(dsc::lowrank_bwd(x, z, U, dy, dx, dz, dU, workspace, s,
                                    (cudaStream_t)stream));
}

dsc_status_t dsc_headwise_decode(const void* x, const void* w, void* state, void* y, int64_t B,
                                 int64_t C, int64_t H, int64_t W, int residual,
                                 dsc_dtype_t dtype, void* stream) {
  dsc_status_t st = check_shape(B, 1, C, H, W, 0, dtype, false);
  if (st != DSC_OK) return st;
  if (B == 0) return DSC_OK;
  if ((st = check_ptrs({x, w, y})) != DSC_OK) return st;
  if (W > 1 && (st = check_ptrs({state})) != DSC_OK) return st;
  if (y == x || (W > 1 && (state == x || state == y))) return DSC_ERR_INVALID_ARG;
  return from_cuda(dsc::headwise_decode(x, w, state, y,
                                        make_shape(B, 1, C, H, W, 0, residual, dtype),
                                        (cudaStream_t)stream));
}

dsc_status_t dsc_lowrank_decode(const void* x, const void* z, const void* U, void* state,
                                void* y, int64_t B, int64_t C, int64_t H, int64_t W, int64_t R,
                                int residual, dsc_dtype_t dtype, void* stream) {
  dsc_status_t st = check_shape(B, 1, C, H, W, R, dtype, true);
  if (st != DSC_OK) return st;
  if (R > 32) return DSC_ERR_UNSUPPORTED;
  if (B == 0) return DSC_OK;
  if ((st = check_ptrs({x, z, U, y})) != DSC_OK) return st;
  if (W > 1 && (st = check_ptrs({state})) != DSC_OK) return st;
  if (y == x || (W > 1 && (state == x || state == y))) return DSC_ERR_INVALID_ARG;
  return from_cuda(dsc::lowrank_decode(x, z, U, state, y,
                                       make_shape(B, 1, C, H, W, R, residual, dtype),
                                       (cudaStream_t)stream));
}

dsc_status_t dsc_headwise_proj_decode(const void* h, const void* Wp, const void* w, void* state,
                                      void* y, int64_t B, int64_t D, int64_t C, int64_t H,
                                      int64_t W, int residual, dsc_dtype_t dtype, void* stream) {
  dsc_status_t st = check_shape(B, 1, C, H, W, 0, dtype, false);
  if (st != DSC_OK) return st;
  if ((st = check_proj(B, D, dtype)) != DSC_OK) return st;
  if (B == 0) return DSC_OK;
  if ((st = check_ptrs({h, Wp, w, y})) != DSC_OK) return st;
  if (W > 1 && (st = check_ptrs({state})) != DSC_OK) return st;
  if (y == h || y == Wp || (W > 1 && (state == h || state == y || state == Wp)))
    return DSC_ERR_INVALID_ARG;
  return from_cuda(dsc::headwise_proj_decode(h, Wp, w, state, y,
                                             make_shape(B, 1, C, H, W, 0, residual, dtype), D,
                                             (cudaStream_t)stream));
}

dsc_status_t dsc_headwise_proj_decode_selftest_timeout(const void* h, const void* Wp,
                                                      const void* w, void* state, void* y,
                                                      int64_t B, int64_t D, int64_t C, int64_t H,
                                                      int64_t W, int residual, dsc_dtype_t dtype,
                                                      uint64_t wait_limit_ns, void* stream) {
  dsc_status_t st = check_shape(B, 1, C, H, W, 0, dtype, false);
  if (st != DSC_OK) return st;
  if ((st = check_proj(B, D, dtype)) != DSC_OK) return st;
  if (B == 0 || wait_limit_ns < 1000 || wait_limit_ns > 1000000000ull) return DSC_ERR_INVALID_ARG;
  const Shape s = make_shape(B, 1, C, H, W, 0, residual, dtype);
  if (!dsc::headwise_proj_decode_uses_tc(s, D)) return DSC_ERR_UNSUPPORTED;
  if ((st = check_ptrs({h, Wp, w, y})) != DSC_OK) return st;
  if (W > 1 && (st = check_ptrs({state})) != DSC_OK) return st;
  if (y == h || y == Wp || (W > 1 && (state == h || state == y || state == Wp)))
    return DSC_ERR_INVALID_ARG;
  return from_cuda(dsc::proj_decode_tc_selftest(h, Wp, w, state, y, s, D, wait_limit_ns,
                                                (cudaStream_t)stream));
}

dsc_status_t dsc_lowrank_proj_decode(const void* h, const void* Wp, const void* z, const void* U,
                                     void* state, void* y, int64_t B, int64_t D, int64_t C,
                                     int64_t H, int64_t W, int64_t R, int residual,
                                     dsc_dtype_t dtype, void* stream) {
  dsc_status_t st = check_shape(B, 1, C, H, W, R, dtype, true);
  if (st != DSC_OK) return st;
  if ((st = check_proj(B, D, dtype)) != DSC_OK) return st;
  if (R > 32) return DSC_ERR_UNSUPPORTED;
  if (B == 0) return DSC_OK;
  if ((st = check_ptrs({h, Wp, z, U, y})) != DSC_OK) return st;
  if (W > 1 && (st = check_ptrs({state})) != DSC_OK) return st;
  if (y == h || y == Wp || (W > 1 && (state == h || state == y || state == Wp)))
    return DSC_ERR_INVALID_ARG;
  return from_cuda(dsc::lowrank_proj_decode(h, Wp, z, U, state, y,
                                            make_shape(B, 1, C, H, W, R, residual, dtype), D,
                                            (cudaStream_t)stream));
}

dsc_status_t dsc_static_fwd(const void* x, const void* w, void* y, int64_t B, int64_t T,
                            int64_t C, int64_t W, int residual, dsc_dtype_t dtype,
                            void* stream) {
  dsc_status_t st = check_shape(B, T, C, 1, W, 0, dtype, false);
  if (st != DSC_OK) return st;
  if (B * T == 0) return DSC_OK;
  if ((st = check_ptrs({x, w, y})) != DSC_OK) return st;
  if (x == y) return DSC_ERR_INVALID_ARG;
  return from_cuda(dsc::static_fwd(x, w, y, make_shape(B, T, C, 1, W, 0, residual, dtype),
                                   (cudaStream_t)stream));
}

size_t dsc_static_bwd_workspace_size(int64_t B, int64_t T, int64_t C, int64_t W,
                                     dsc_dtype_t dtype) {
  if (check_shape(B, T, C, 1, W, 0, dtype, false) != DSC_OK || B * T == 0) return 0;
  return dsc::static_bwd_workspace(make_shape(B, T, C, 1, W, 0, 0, dtype));
}

dsc_status_t dsc_static_bwd(const void* x, const void* w, const void* dy, void* dx, void* dw,
                            void* workspace, size_t workspace_bytes, int64_t B, int64_t T,
                            int64_t C, int64_t W, int residual, dsc_dtype_t dtype,
                            void* stream) {
  dsc_status_t st = check_shape(B, T, C, 1, W, 0, dtype, false);
  if (st != DSC_OK) return st;
  if (B * T == 0) {
    // dw is a sum over zero tokens: all zeros.  Nothing else to write.
    if (dw == nullptr) return DSC_ERR_INVALID_ARG;
    const size_t bytes = (size_t)C * W * (dtype == DSC_BF16 ? 2 : 4);
    return from_cuda(cudaMemsetAsync(dw, 0, bytes, (cudaStream_t)stream));
  }
  if ((st = check_ptrs({x, w, dy, dx, dw})) != DSC_OK) return st;
  if (dx == x || dx == dy || dx == dw || dw == x || dw == w || dw == dy)
    return DSC_ERR_INVALID_ARG;
  const Shape s = make_shape(B, T, C, 1, W, 0, residual, dtype);
  const size_t need = dsc::static_bwd_workspace(s);
  if (workspace == nullptr || workspace_bytes < need) return DSC_ERR_WORKSPACE;
  if (!aligned16(workspace)) return DSC_ERR_ALIGNMENT;
  return from_cuda(dsc::static_bwd(x, w, dy, dx, dw, workspace, s, (cudaStream_t)stream));
}

int dsc_lowrank_uses_tensor_cores(int64_t B, int64_t T, int64_t C, int64_t H, int64_t W,
                                  int64_t R, dsc_dtype_t dtype) {
  if (check_shape(B, T, C, H, W, R, dtype, true) != DSC_OK) return -1;
  const Shape s = make_shape(B, T, C, H, W, R, 0, dtype);
  if (!dsc::lowrank_supported(s)) return -1;
  return (dsc::lowrank_tc_supported(s) ? 1 : 0) | (dsc::lowrank_bwd_tc_supported(s) ? 2 : 0);
}

dsc_status_t dsc_device_error(unsigned int* code, int reset) {
  if (code == nullptr) return DSC_ERR_INVALID_ARG;
  unsigned int a = 0, b = 0, c = 0, d = 0;
  cudaError_t e = dsc::lowrank_tc_error(&a, reset != 0);
  if (e == cudaSuccess) e = dsc::headwise_tma_error(&b, reset != 0);
  if (e == cudaSuccess) e = dsc::proj_decode_tc_error(&c, reset != 0);
  if (e == cudaSuccess) e = dsc::static_tma_error(&d, reset != 0);
  *code = a != 0 ? a : b != 0 ? b : c != 0 ? c : d;
  return from_cuda(e);
}

dsc_status_t dsc_lowrank_fwd_selftest_timeout(const void* x, const void* z, const void* U,
                                              void* y, int64_t B, int64_t T, int64_t C,
                                              int64_t H, int64_t W, int64_t R, int residual,
                                              dsc_dtype_t dtype, uint64_t wait_limit_ns,
                                              void* stream) {
  dsc_status_t st = check_shape(B, T, C, H, W, R, dtype, true);
  if (st != DSC_OK) return st;
  if (B * T == 0 || wait_limit_ns < 1000 || wait_limit_ns > 1000000000ull)
    return DSC_ERR_INVALID_ARG;
  const Shape s = make_shape(B, T, C, H, W, R, residual, dtype);
  if (!dsc::lowrank_supported(s) || !dsc::lowrank_tc_supported(s)) return DSC_ERR_UNSUPPORTED;
  if ((st = check_ptrs({x, z, U, y})) != DSC_OK) return st;
  if (x == y) return DSC_ERR_INVALID_ARG;
  return from_cuda(
      dsc::lowrank_fwd_tc_selftest(x, z, U, y, s, wait_limit_ns, (cudaStream_t)stream));
}

dsc_status_t dsc_lowrank_bwd_selftest_timeout(const void* x, const void* z, const void* U,
                                              const void* dy, void* dx, void* dz, void* dU,
                                              void* workspace, size_t workspace_bytes,
                                              int64_t B, int64_t T, int64_t C, int64_t H,
                                              int64_t W, int64_t R, int residual,
                                              dsc_dtype_t dtype, uint64_t wait_limit_ns,
                                              void* stream) {
  dsc_status_t st = check_shape(B, T, C, H, W, R, dtype, true);
  if (st != DSC_OK) return st;
  if (B * T == 0 || wait_limit_ns < 1000 || wait_limit_ns > 1000000000ull)
    return DSC_ERR_INVALID_ARG;
  const Shape s = make_shape(B, T, C, H, W, R, residual, dtype);
  if (!dsc::lowrank_supported(s) || !dsc::lowrank_bwd_tc_supported(s)) return DSC_ERR_UNSUPPORTED;
  if ((st = check_ptrs({x, z, U, dy, dx, dz, dU})) != DSC_OK) return st;
  if (dx == x || dx == dy || dz == z || dU == U) return DSC_ERR_INVALID_ARG;
  const size_t need = dsc::lowrank_bwd_tc_workspace(s);
  if (workspace == nullptr || workspace_bytes < need) return DSC_ERR_WORKSPACE;
  if (!aligned16(workspace)) return DSC_ERR_ALIGNMENT;
  return from_cuda(dsc::lowrank_bwd_tc_selftest(x, z, U, dy, dx, dz, dU, workspace, s,
                                                wait_limit_ns, (cudaStream_t)stream));
}

int dsc_headwise_uses_tma(int64_t B, int64_t T, int64_t C, int64_t H, int64_t W,
                          dsc_dtype_t dtype) {
  if (check_shape(B, T, C, H, W, 0, dtype, false) != DSC_OK) return -1;
  const Shape s = make_shape(B, T, C, H, W, 0, 0, dtype);
  return (dsc::headwise_tma_supported(s, false) ? 1 : 0) |
         (dsc::headwise_tma_supported(s, true) ? 2 : 0);
}

}  // extern "C"

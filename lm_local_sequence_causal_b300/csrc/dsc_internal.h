// dsc_internal.h -- host-side interface between the C ABI layer (dsc_abi.cu)
// and the kernel files.  Arguments here are already validated.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace dsc {

struct Shape {
  int64_t B, T, C, H, W, R;  // R = 0 for the head-wise parameterisation
  int residual;
  int bf16;                  // 1 = bf16 I/O, 0 = fp32 I/O
  int64_t G() const { return C / H; }
  int64_t N() const { return B * T; }
};

// Head-wise kernels (headwise.cu).
cudaError_t headwise_fwd(const void* x, const void* w, void* y, const Shape& s,
                         cudaStream_t st);
cudaError_t headwise_bwd(const void* x, const void* w, const void* dy, void* dx,
                         void* dw, const Shape& s, cudaStream_t st);

// Low-rank kernels (lowrank_simt.cu).
bool lowrank_supported(const Shape& s);
cudaError_t lowrank_fwd(const void* x, const void* z, const void* U, void* y,
                        const Shape& s, cudaStream_t st);
size_t lowrank_bwd_workspace(const Shape& s);
cudaError_t lowrank_bwd(const void* x, const void* z, const void* U,
                        const void* dy, void* dx, void* dz, void* dU,
                        void* ws, const Shape& s, cudaStream_t st);

}  // namespace dsc

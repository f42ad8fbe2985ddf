// dsc_internal.h -- host-side interface between the C ABI layer (dsc_abi.cu)
// and the kernel files.  Arguments here are already validated.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

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

// Head-wise kernels with TMA-staged tiles (headwise_tma.cu): bf16 and the
// (H, W) pairs whose filter rows make a legal TMA box, C a multiple of the
// item width (64 or 128 channels).
bool headwise_tma_supported(const Shape& s, bool bwd);
cudaError_t headwise_fwd_tma(const void* x, const void* w, void* y, const Shape& s,
                             cudaStream_t st);
cudaError_t headwise_bwd_tma(const void* x, const void* w, const void* dy, void* dx, void* dw,
                             const Shape& s, cudaStream_t st);
cudaError_t headwise_tma_error(unsigned int* out, bool reset);

// Decode step with a carried state (decode.cu).
cudaError_t headwise_decode(const void* x, const void* w, void* state, void* y, const Shape& s,
                            cudaStream_t st);
cudaError_t lowrank_decode(const void* x, const void* z, const void* U, void* state, void* y,
                           const Shape& s, cudaStream_t st);

// Decode step merged with the projection of its input, x_t = h Wp^T with
// h [B, D] and Wp [C, D] (proj_decode.cu); s.T is 1, D a multiple of the
// 16-byte vector width.
cudaError_t headwise_proj_decode(const void* h, const void* Wp, const void* w, void* state,
                                 void* y, const Shape& s, int64_t D, cudaStream_t st);
cudaError_t lowrank_proj_decode(const void* h, const void* Wp, const void* z, const void* U,
                                void* state, void* y, const Shape& s, int64_t D,
                                cudaStream_t st);

// Static short convolution, filters w [C, W] constant over t (static_conv.cu).
// H = 1.  The backward needs a caller-owned fp32 workspace for the dw partials.
cudaError_t static_fwd(const void* x, const void* w, void* y, const Shape& s, cudaStream_t st);
size_t static_bwd_workspace(const Shape& s);
cudaError_t static_bwd(const void* x, const void* w, const void* dy, void* dx, void* dw,
                       void* ws, const Shape& s, cudaStream_t st);

// Low-rank kernels (lowrank_simt.cu).
bool lowrank_supported(const Shape& s);
cudaError_t lowrank_fwd(const void* x, const void* z, const void* U, void* y,
                        const Shape& s, cudaStream_t st);
size_t lowrank_bwd_workspace(const Shape& s);
cudaError_t lowrank_bwd(const void* x, const void* z, const void* U,
                        const void* dy, void* dx, void* dz, void* dU,
                        void* ws, const Shape& s, cudaStream_t st);

// Tensor-core (tcgen05) low-rank kernels (lowrank_tc.cu): bf16, R in
// {8, 16, 24, 32}, W <= 4, H = 1 or tied filters (the forward needs the
// chunk's U columns on 16-byte boundaries, see lowrank_tc_supported).  The
// *_tc functions return cudaErrorNotSupported when the shape is outside
// that set, so the caller can use the CUDA-core kernels.
bool lowrank_tc_supported(const Shape& s);
cudaError_t lowrank_fwd_tc(const void* x, const void* z, const void* U, void* y,
                           const Shape& s, cudaStream_t st);
// Backward on the tensor cores: bf16, R in {8, 16, 24, 32}, any H.
bool lowrank_bwd_tc_supported(const Shape& s);
size_t lowrank_bwd_tc_workspace(const Shape& s);
cudaError_t lowrank_bwd_tc(const void* x, const void* z, const void* U, const void* dy,
                           void* dx, void* dz, void* dU, void* ws, const Shape& s,
                           cudaStream_t st);
// Device error word of the tensor-core kernels (0 = no error; otherwise the
// code of the bounded wait that gave up).  Synchronous; diagnostic only.
cudaError_t lowrank_tc_error(unsigned int* out, bool reset);
// The decode step merged with its projection on the tensor core (bf16,
// W <= 4, R <= 32; any batch, in launches of up to 256 sequences).
bool proj_decode_tc_supported(const Shape& s, int64_t D);
cudaError_t proj_decode_tc(const void* h, const void* Wp, const void* w, const void* z,
                           const void* U, void* state, void* y, const Shape& s, int64_t D,
                           bool lowrank, cudaStream_t st);
cudaError_t proj_decode_tc_error(unsigned int* out, bool reset);
// Device error word of the TMA-staged static backward.
cudaError_t static_tma_error(unsigned int* out, bool reset);
// Failure-path self-test of the head-wise tcgen05 kernel: waits limited to
// wait_ns and a producer that issues no loads.
cudaError_t proj_decode_tc_selftest(const void* h, const void* Wp, const void* w, void* state,
                                    void* y, const Shape& s, int64_t D, uint64_t wait_ns,
                                    cudaStream_t st);
// Whether dsc_headwise_proj_decode takes the tcgen05 kernel for this shape.
bool headwise_proj_decode_uses_tc(const Shape& s, int64_t D);
// Self-test of the failure path: the same kernels with every bounded wait
// limited to wait_ns and a producer that issues no loads, so the waits of
// the other roles run out; the kernels record a code in the error word, free
// their TMEM and return.  Outputs are left unspecified.
cudaError_t lowrank_fwd_tc_selftest(const void* x, const void* z, const void* U, void* y,
                                    const Shape& s, uint64_t wait_ns, cudaStream_t st);
cudaError_t lowrank_bwd_tc_selftest(const void* x, const void* z, const void* U, const void* dy,
                                    void* dx, void* dz, void* dU, void* ws, const Shape& s,
                                    uint64_t wait_ns, cudaStream_t st);

// Host helpers (tmap.cu).
// 3-D tensor map over a dense row-major [d2][d1][d0] tensor of bf16 or fp32,
// box {b0, b1, 1}, swizzle 0/32/64/128 bytes, zero fill out of range.
bool make_tmap_3d(CUtensorMap* tm, const void* base, bool bf16, uint64_t d0, uint64_t d1,
                  uint64_t d2, uint32_t b0, uint32_t b1, int swizzle_bytes);
// 4-D bf16 tensor map with explicit strides (bytes) of dims 1..3, no swizzle.
bool make_tmap_4d_bf16(CUtensorMap* tm, const void* base, const uint64_t dims[4],
                       const uint64_t strides_bytes[3], const uint32_t box[4]);
int sm_count();
// Token ranges for a streaming grid of `ncb` channel blocks: as many CTAs as
// fit on the GPU at once (occupancy of `kernel` x SMs), at least 16 tokens
// each.
int64_t n_ranges(const void* kernel, int threads, int64_t ncb, int64_t N);

// Opt in to large dynamic shared memory, once per kernel and device.  The
// template parameter `Tag` keeps one record per kernel instance (all
// instances share a function type, so the type alone cannot tell them apart).
template <typename Tag, typename F>
cudaError_t set_smem(F* kernel, int bytes) {
  static std::mutex mu;
  static bool done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!done[dev]) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    done[dev] = true;
  }
  return cudaSuccess;
}


}  // namespace dsc

// decode.cu -- one-token (decode) step of Dynamic Short Convolutions with a
// carried state, head-wise and low-rank.
//
// The pages leave inference to future engineering ("Dynamic Short
// Convolutions: The 'Locality Bias' Transformers Were Missing", Limitations;
// "Technische Samenvatting: Dynamische Korte Convoluties Verbeteren
// Transformers", Beperkingen).  The step here is the forward definition
// (Methodologie: Mechanisme) evaluated at one new position t, with the last
// W-1 inputs of the sequence kept as state:
//   y[b,c]        = res*x_t[b,c] + w[b,g(c),0] x_t[b,c] + sum_{k>=1} w[b,g(c),k] state[b,k-1,c]
//   state'[b,0,c] = x_t[b,c],  state'[b,j,c] = state[b,j-1,c]   (j >= 1)
// with state[b,j] = x at time t-1-j (zero before the sequence start).  For
// the low-rank form the taps are w[b,g,k] = sum_r z_t[b,r] U[r,g*W+k] in
// fp32 (never rounded).  One thread owns one 16-byte vector of channels of
// one sequence: it reads the token and its W-1 state rows, writes y and the
// shifted state in place.  A decode step is a few kilobytes per sequence, so
// these kernels are latency-bound by nature; the taps come from L1/L2.
#include <algorithm>

#include "dsc_common.cuh"
#include "dsc_internal.h"

namespace dsc {
namespace {

constexpr int kThreads = 128;

template <typename T, int W>
__device__ __forceinline__ void step_and_shift(const float (&xv)[Vec<T>::N],
                                               const float (&taps)[Vec<T>::N][W],
                                               const uint4 (&sraw)[W > 1 ? W - 1 : 1],
                                               const uint4& xraw, int residual, T* yp, T* sp,
                                               int64_t C) {
  constexpr int V = Vec<T>::N;
  float sv[W > 1 ? W - 1 : 1][V];
#pragma unroll
  for (int j = 0; j < W - 1; ++j) unpack16<T>(sraw[j], sv[j]);
  float out[V];
#pragma unroll
  for (int v = 0; v < V; ++v) {
    float a = residual ? xv[v] : 0.f;
    a = fmaf(taps[v][0], xv[v], a);
#pragma unroll
    for (int k = 1; k < W; ++k) a = fmaf(taps[v][k], sv[k - 1][v], a);
    out[v] = a;
  }
  *reinterpret_cast<uint4*>(yp) = pack16<T>(out);
  // The state moves down one row; the token becomes row 0 (exact copies).
#pragma unroll
  for (int j = W - 2; j >= 1; --j) *reinterpret_cast<uint4*>(sp + j * C) = sraw[j - 1];
  if constexpr (W > 1) *reinterpret_cast<uint4*>(sp) = xraw;
}

template <typename T, int W>
__global__ void __launch_bounds__(kThreads)
hw_decode_kernel(const T* __restrict__ x, const T* __restrict__ w, T* __restrict__ state,
                 T* __restrict__ y, int64_t B, int64_t C, int64_t H, int residual) {
  constexpr int V = Vec<T>::N;
  const int64_t nvec = C / V;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= B * nvec) return;
  const int64_t b = i / nvec, c0 = (i - b * nvec) * V;
  const int64_t G = C / H;
  const uint4 xraw = ldg16(x + b * C + c0);
  float xv[V];
  unpack16<T>(xraw, xv);
  T* sp = state + b * (W - 1) * C + c0;
  uint4 sraw[W > 1 ? W - 1 : 1];
#pragma unroll
  for (int j = 0; j < W - 1; ++j) sraw[j] = *reinterpret_cast<const uint4*>(sp + j * C);
  float taps[V][W];
  const T* wb = w + b * G * W;
#pragma unroll
  for (int v = 0; v < V; ++v) {
    const int64_t g = (c0 + v) / H;
#pragma unroll
    for (int k = 0; k < W; ++k) taps[v][k] = to_f32(__ldg(wb + g * W + k));
  }
  step_and_shift<T, W>(xv, taps, sraw, xraw, residual, y + b * C + c0, sp, C);
}

template <typename T, int W>
__global__ void __launch_bounds__(kThreads)
lr_decode_kernel(const T* __restrict__ x, const T* __restrict__ z, const T* __restrict__ U,
                 T* __restrict__ state, T* __restrict__ y, int64_t B, int64_t C, int64_t H,
                 int R, int residual) {
  constexpr int V = Vec<T>::N;
  const int64_t nvec = C / V;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= B * nvec) return;
  const int64_t b = i / nvec, c0 = (i - b * nvec) * V;
  const int64_t GW = (C / H) * W;
  const uint4 xraw = ldg16(x + b * C + c0);
  float xv[V];
  unpack16<T>(xraw, xv);
  T* sp = state + b * (W - 1) * C + c0;
  uint4 sraw[W > 1 ? W - 1 : 1];
#pragma unroll
  for (int j = 0; j < W - 1; ++j) sraw[j] = *reinterpret_cast<const uint4*>(sp + j * C);
  float taps[V][W];
#pragma unroll
  for (int v = 0; v < V; ++v)
#pragma unroll
    for (int k = 0; k < W; ++k) taps[v][k] = 0.f;
  const T* zb = z + b * R;
  for (int r = 0; r < R; ++r) {
    const float zr = to_f32(__ldg(zb + r));
    const T* ur = U + static_cast<int64_t>(r) * GW;
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int64_t g = (c0 + v) / H;
#pragma unroll
      for (int k = 0; k < W; ++k) taps[v][k] = fmaf(zr, to_f32(__ldg(ur + g * W + k)), taps[v][k]);
    }
  }
  step_and_shift<T, W>(xv, taps, sraw, xraw, residual, y + b * C + c0, sp, C);
}

#define DSC_DEC_W_SWITCH(Wv, ...)                                     \
  switch (Wv) {                                                       \
    case 1: { constexpr int W_ = 1; __VA_ARGS__; } break;             \
    case 2: { constexpr int W_ = 2; __VA_ARGS__; } break;             \
    case 3: { constexpr int W_ = 3; __VA_ARGS__; } break;             \
    default: { constexpr int W_ = 4; __VA_ARGS__; } break;            \
  }

template <typename T>
cudaError_t hw_t(const void* x, const void* w, void* state, void* y, const Shape& s,
                 cudaStream_t st) {
  const int64_t n = s.B * (s.C / Vec<T>::N);
  const unsigned grid = static_cast<unsigned>((n + kThreads - 1) / kThreads);
  DSC_DEC_W_SWITCH(s.W, {
    hw_decode_kernel<T, W_><<<grid, kThreads, 0, st>>>(
        static_cast<const T*>(x), static_cast<const T*>(w), static_cast<T*>(state),
        static_cast<T*>(y), s.B, s.C, s.H, s.residual);
  })
  return cudaGetLastError();
}

template <typename T>
cudaError_t lr_t(const void* x, const void* z, const void* U, void* state, void* y,
                 const Shape& s, cudaStream_t st) {
  const int64_t n = s.B * (s.C / Vec<T>::N);
  const unsigned grid = static_cast<unsigned>((n + kThreads - 1) / kThreads);
  DSC_DEC_W_SWITCH(s.W, {
    lr_decode_kernel<T, W_><<<grid, kThreads, 0, st>>>(
        static_cast<const T*>(x), static_cast<const T*>(z), static_cast<const T*>(U),
        static_cast<T*>(state), static_cast<T*>(y), s.B, s.C, s.H, static_cast<int>(s.R),
        s.residual);
  })
  return cudaGetLastError();
}

}  // namespace

cudaError_t headwise_decode(const void* x, const void* w, void* state, void* y, const Shape& s,
                            cudaStream_t st) {
  return s.bf16 ? hw_t<__nv_bfloat16>(x, w, state, y, s, st)
                : hw_t<float>(x, w, state, y, s, st);
}

cudaError_t lowrank_decode(const void* x, const void* z, const void* U, void* state, void* y,
                           const Shape& s, cudaStream_t st) {
  return s.bf16 ? lr_t<__nv_bfloat16>(x, z, U, state, y, s, st)
                : lr_t<float>(x, z, U, state, y, s, st);
}

}  // namespace dsc

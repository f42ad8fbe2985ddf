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
// these kernels are latency-bound by nature: what matters is how many
// dependent memory round trips a thread makes.  The head-wise taps are W
// loads per channel, all issued together; the low-rank ones need R columns
// of U, which a block stages once in shared memory (below).
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

// Low-rank step.  The taps of a channel need a column of U for every rank r,
// and every sequence of the batch reads the same columns, so one block owns
// a slice of kLrCB channels for all sequences: it copies U[:, slice] once
// into shared memory (asynchronous 16-byte copies, all in flight together,
// so the copy costs one memory round trip whatever R is), then each thread
// forms the taps of its V channels for one sequence from z[b, :] and the
// staged slice.  Threads map to (sequence, channel vector) with the vector
// fastest; sequences beyond the block's kThreads / (kLrCB / V) are handled
// in further passes over the same staged slice.
constexpr int kLrCB = 32;      // channels per block
constexpr int kLrMaxR = 32;    // largest rank the entry point accepts

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned sa = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(sa), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
}

template <typename T, int W>
__global__ void __launch_bounds__(kThreads)
lr_decode_kernel(const T* __restrict__ x, const T* __restrict__ z, const T* __restrict__ U,
                 T* __restrict__ state, T* __restrict__ y, int64_t B, int64_t C, int64_t H,
                 int R, int residual) {
  constexpr int V = Vec<T>::N;
  constexpr int NVB = kLrCB / V;        // channel vectors per block
  constexpr int SP = kThreads / NVB;    // sequences per pass
  __shared__ __align__(16) T us[kLrMaxR * kLrCB * W];
  __shared__ float zs[SP * kLrMaxR];

  // The slice's groups g_lo..g_hi, i.e. U columns [col_lo, col_lo + ncol).
  const int64_t c_lo = static_cast<int64_t>(blockIdx.x) * kLrCB;
  const int64_t c_hi = c_lo + kLrCB < C ? c_lo + kLrCB : C;
  const int64_t GW = (C / H) * W;
  const int64_t g_lo = c_lo / H;
  const int64_t col_lo = g_lo * W;
  const int ncol = static_cast<int>(((c_hi - 1) / H + 1) * W - col_lo);
  const int tid = threadIdx.x;

  // Stage U[0:R, col_lo : col_lo + ncol] as rows of ncol elements.  The
  // 16-byte copies need 16-byte rows and a 16-byte start; other shapes take
  // element copies.
  if ((((GW | col_lo | static_cast<int64_t>(ncol)) * static_cast<int64_t>(sizeof(T))) & 15) == 0) {
    constexpr int E16 = 16 / static_cast<int>(sizeof(T));
    const int cpr = ncol / E16;
    for (int i = tid; i < R * cpr; i += kThreads) {
      const int r = i / cpr, j = i - r * cpr;
      cp_async16(us + r * ncol + j * E16, U + r * GW + col_lo + j * E16);
    }
  } else {
    for (int i = tid; i < R * ncol; i += kThreads) {
      const int r = i / ncol, j = i - r * ncol;
      us[i] = U[r * GW + col_lo + j];
    }
  }

  const int vl = tid % NVB, bl = tid / NVB;
  const int64_t c0 = c_lo + static_cast<int64_t>(vl) * V;
  const bool chan_ok = c0 < c_hi;
  // Offsets of this thread's channels' groups within a staged row.
  int off[V];
#pragma unroll
  for (int v = 0; v < V; ++v) off[v] = static_cast<int>(((c0 + v) / H - g_lo) * W);

  for (int64_t b0 = 0; b0 < B; b0 += SP) {
    const int64_t b = b0 + bl;
    const bool act = chan_ok && b < B;
    uint4 xraw = make_uint4(0, 0, 0, 0);
    uint4 sraw[W > 1 ? W - 1 : 1];
    T* sp = state + b * (W - 1) * C + c0;
    if (act) {
      xraw = ldg16(x + b * C + c0);
#pragma unroll
      for (int j = 0; j < W - 1; ++j) sraw[j] = *reinterpret_cast<const uint4*>(sp + j * C);
    }
    if (b0 > 0) __syncthreads();                 // the last pass has read zs
    const int nb = B - b0 < SP ? static_cast<int>(B - b0) : SP;
    for (int i = tid; i < nb * R; i += kThreads) zs[i] = to_f32(z[b0 * R + i]);
    if (b0 == 0) cp_async_wait_all();
    __syncthreads();
    if (!act) continue;

    float taps[V][W];
#pragma unroll
    for (int v = 0; v < V; ++v)
#pragma unroll
      for (int k = 0; k < W; ++k) taps[v][k] = 0.f;
    const float* zb = zs + bl * R;
    if (H == 1) {
      // The V channels' W taps are V*W consecutive elements: W 16-byte reads.
      const T* ub = us + vl * V * W;
      for (int r = 0; r < R; ++r) {
        const float zr = zb[r];
        float u[W][V];
#pragma unroll
        for (int j = 0; j < W; ++j)
          unpack16<T>(*reinterpret_cast<const uint4*>(ub + r * ncol + j * V), u[j]);
#pragma unroll
        for (int v = 0; v < V; ++v)
#pragma unroll
          for (int k = 0; k < W; ++k)
            taps[v][k] = fmaf(zr, u[(v * W + k) / V][(v * W + k) % V], taps[v][k]);
      }
    } else {
      for (int r = 0; r < R; ++r) {
        const float zr = zb[r];
        const T* ur = us + r * ncol;
#pragma unroll
        for (int v = 0; v < V; ++v)
#pragma unroll
          for (int k = 0; k < W; ++k) taps[v][k] = fmaf(zr, to_f32(ur[off[v] + k]), taps[v][k]);
      }
    }
    float xv[V];
    unpack16<T>(xraw, xv);
    step_and_shift<T, W>(xv, taps, sraw, xraw, residual, y + b * C + c0, sp, C);
  }
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
  if (s.R > kLrMaxR) return cudaErrorInvalidValue;
  const unsigned grid = static_cast<unsigned>((s.C + kLrCB - 1) / kLrCB);
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

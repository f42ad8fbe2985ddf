// static_conv.cu -- the static short convolution: the special case of DSC
// whose filters do not depend on the token (one per channel, w [C, W]).
//
// "Dynamic Short Convolutions: The 'Locality Bias' Transformers Were
// Missing", Methodology: Adaptive Filtering at Scale, 1. Mathematical
// Intuition (the standard convolution): the static causal depthwise
// convolution that DSC generalises, and the kernel family its Figure 1
// compares against,
//   y[b,t,c]  = res*x[b,t,c] + sum_{k<W} w[c,k] x[b,t-k,c]      (x = 0 before t = 0)
// and its chain rule:
//   dx[b,s,c] = res*dy[b,s,c] + sum_{k: s+k<T} w[c,k] dy[b,s+k,c]
//   dw[c,k]   = sum_{b,t} dy[b,t,c] x[b,t-k,c]                  (over all tokens)
// Same streaming scheme as the head-wise register kernels: a thread owns a
// vector of channels (16 bytes forward, 8 bytes backward) and walks a
// contiguous range of the flat token axis n = b*T + t (balanced ranges,
// sequence starts reset the causal window), with the loads of the next
// tokens in flight.  The taps are loaded once.  The backward accumulates dw
// over its range in registers and writes one fp32 partial per (range,
// channel, tap); a second kernel adds the partials in range order (bitwise
// reproducible).
#include <algorithm>

#include "dsc_common.cuh"
#include "dsc_internal.h"

namespace dsc {
namespace {

constexpr int kThreads = 128;
constexpr int kPF = 4;

struct Range {
  int64_t cb, r, n0, n1;
};
__device__ __forceinline__ Range range_of(int64_t ncb, int64_t nranges, int64_t N) {
  Range g;
  g.cb = blockIdx.x % ncb;
  g.r = blockIdx.x / ncb;
  g.n0 = N * g.r / nranges;
  g.n1 = N * (g.r + 1) / nranges;
  return g;
}

template <typename T, int W>
__device__ __forceinline__ void load_taps(const T* __restrict__ w, int64_t c0,
                                          float (&taps)[Vec<T>::N][W]) {
  constexpr int V = Vec<T>::N;
  float flat[V * W];
  load_chunk<T, V * W>(w + c0 * W, flat);
#pragma unroll
  for (int v = 0; v < V; ++v)
#pragma unroll
    for (int k = 0; k < W; ++k) taps[v][k] = flat[v * W + k];
}

template <typename T, int W>
__global__ void __launch_bounds__(kThreads)
static_fwd_kernel(const T* __restrict__ x, const T* __restrict__ w, T* __restrict__ y,
                  int64_t Tlen, int64_t C, int residual, int64_t N, int64_t ncb,
                  int64_t nranges) {
  constexpr int V = Vec<T>::N;
  const Range rg = range_of(ncb, nranges, N);
  const int64_t c0 = (rg.cb * blockDim.x + threadIdx.x) * V;
  if (c0 >= C) return;
  float taps[V][W];
  load_taps<T, W>(w, c0, taps);
  const T* xb = x + c0;
  T* yb = y + c0;
  int64_t t = rg.n0 % Tlen;
  float win[W > 1 ? W - 1 : 1][V];
#pragma unroll
  for (int j = 0; j < W - 1; ++j) {
    if (t - 1 - j >= 0) {
      unpack16<T>(ldg16(xb + (rg.n0 - 1 - j) * C), win[j]);
    } else {
#pragma unroll
      for (int v = 0; v < V; ++v) win[j][v] = 0.f;
    }
  }
  uint4 xr[kPF];
#pragma unroll
  for (int j = 0; j < kPF; ++j)
    if (rg.n0 + j < rg.n1) xr[j] = ldg16(xb + (rg.n0 + j) * C);
  for (int64_t nb = rg.n0; nb < rg.n1; nb += kPF) {
#pragma unroll
    for (int j = 0; j < kPF; ++j) {
      const int64_t n = nb + j;
      if (n < rg.n1) {
        if (t == 0) {
#pragma unroll
          for (int q = 0; q < W - 1; ++q)
#pragma unroll
            for (int v = 0; v < V; ++v) win[q][v] = 0.f;
        }
        float xv[V];
        unpack16<T>(xr[j], xv);
        if (n + kPF < rg.n1) xr[j] = ldg16(xb + (n + kPF) * C);
        float out[V];
#pragma unroll
        for (int v = 0; v < V; ++v) {
          float a = residual ? xv[v] : 0.f;
          a = fmaf(taps[v][0], xv[v], a);
#pragma unroll
          for (int k = 1; k < W; ++k) a = fmaf(taps[v][k], win[k - 1][v], a);
          out[v] = a;
        }
        stcs16(yb + n * C, pack16<T>(out));
#pragma unroll
        for (int q = W - 2; q > 0; --q)
#pragma unroll
          for (int v = 0; v < V; ++v) win[q][v] = win[q - 1][v];
        if constexpr (W > 1) {
#pragma unroll
          for (int v = 0; v < V; ++v) win[0][v] = xv[v];
        }
        if (++t == Tlen) t = 0;
      }
    }
  }
}

// Narrow channel vectors for the backward (kVB bytes a thread): a small
// per-thread state (taps, dw accumulators, load rings), so many threads fit
// on an SM.  A warp still reads 32*kVB contiguous bytes of a token row.
constexpr int kVB = 8;
constexpr int kRing = 4;   // dy ring: the W-row window plus kRing-W+1 rows of lead
constexpr int kRingX = 2;  // x ring: kRingX rows of lead

template <typename T> struct VecB { static constexpr int N = kVB / (int)sizeof(T); };

template <int B> struct RawOf;
template <> struct RawOf<4> { using type = uint32_t; };
template <> struct RawOf<8> { using type = uint2; };
template <> struct RawOf<16> { using type = uint4; };
using Raw = RawOf<kVB>::type;

__device__ __forceinline__ Raw ldgv(const void* p) { return __ldg(reinterpret_cast<const Raw*>(p)); }
__device__ __forceinline__ void stcsv(void* p, const Raw& v) { __stcs(reinterpret_cast<Raw*>(p), v); }

// The 32-bit words of a raw vector and back.
template <typename R>
__device__ __forceinline__ void raw_words(const R& u, uint32_t (&w)[sizeof(R) / 4]) {
  if constexpr (sizeof(R) == 4) {
    w[0] = u;
  } else if constexpr (sizeof(R) == 8) {
    w[0] = u.x;
    w[1] = u.y;
  } else {
    w[0] = u.x;
    w[1] = u.y;
    w[2] = u.z;
    w[3] = u.w;
  }
}
template <typename R>
__device__ __forceinline__ void words_raw(const uint32_t (&w)[sizeof(R) / 4], R& u) {
  if constexpr (sizeof(R) == 4) {
    u = w[0];
  } else if constexpr (sizeof(R) == 8) {
    u = make_uint2(w[0], w[1]);
  } else {
    u = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

template <typename T>
__device__ __forceinline__ void unpackv(const Raw& u, float (&f)[VecB<T>::N]) {
  uint32_t w[kVB / 4];
  raw_words<Raw>(u, w);
#pragma unroll
  for (int i = 0; i < kVB / 4; ++i) {
    if constexpr (sizeof(T) == 4) {
      f[i] = __uint_as_float(w[i]);
    } else {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
}

template <typename T>
__device__ __forceinline__ Raw packv(const float (&f)[VecB<T>::N]) {
  uint32_t w[kVB / 4];
#pragma unroll
  for (int i = 0; i < kVB / 4; ++i) {
    if constexpr (sizeof(T) == 4) {
      w[i] = __float_as_uint(f[i]);
    } else {
      __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
  }
  Raw u;
  words_raw<Raw>(w, u);
  return u;
}

// Backward in gather form.  The thread walks its tokens n in [n0, n1) with a
// ring of dy rows n .. n+kRing-1 in registers; at token n (time t)
//   dx[n]  = res*dy[n] + sum_{k: t+k<T} w[k] dy[n+k]
//   dw[k] += x[n] dy[n+k]                       (t+k < T)
// so every (x, dy) pair of the filter gradient is counted by the range that
// owns its x token, the dy rows up to W-1 past the range end are a halo, and
// no window of x or of partial dx sums is kept.  All threads of a CTA walk
// the same tokens, so the branches on t are uniform.
template <typename T, int W>
__global__ void __launch_bounds__(kThreads)
static_bwd_kernel(const T* __restrict__ x, const T* __restrict__ w, const T* __restrict__ dy,
                  T* __restrict__ dx, float* __restrict__ dw_part, int64_t Tlen, int64_t C,
                  int residual, int64_t N, int64_t ncb, int64_t nranges) {
  constexpr int V = VecB<T>::N;
  static_assert(W <= kRing && kRing % kRingX == 0, "ring sizes");
  const Range rg = range_of(ncb, nranges, N);
  const int64_t c0 = (rg.cb * blockDim.x + threadIdx.x) * V;
  if (c0 >= C) return;
  float taps[V][W];
#pragma unroll
  for (int v = 0; v < V; ++v)
#pragma unroll
    for (int k = 0; k < W; ++k) taps[v][k] = to_f32(__ldg(w + (c0 + v) * W + k));
  float dwa[V][W];
#pragma unroll
  for (int v = 0; v < V; ++v)
#pragma unroll
    for (int k = 0; k < W; ++k) dwa[v][k] = 0.f;
  const T* xb = x + c0;
  const T* gb = dy + c0;
  T* dxb = dx + c0;
  const int64_t n0 = rg.n0, n1 = rg.n1;
  const int64_t nend = n1 + W - 1 < N ? n1 + W - 1 : N;  // dy rows read: [n0, nend)
  Raw gr[kRing], xr[kRingX];
#pragma unroll
  for (int j = 0; j < kRing; ++j)
    if (n0 + j < nend) gr[j] = ldgv(gb + (n0 + j) * C);
#pragma unroll
  for (int j = 0; j < kRingX; ++j)
    if (n0 + j < n1) xr[j] = ldgv(xb + (n0 + j) * C);
  int64_t t = n0 % Tlen;
  for (int64_t nb = n0; nb < n1; nb += kRing) {
#pragma unroll
    for (int jj = 0; jj < kRing; ++jj) {
      const int64_t n = nb + jj;
      if (n < n1) {
        float xv[V];
        unpackv<T>(xr[jj % kRingX], xv);
        if (n + kRingX < n1) xr[jj % kRingX] = ldgv(xb + (n + kRingX) * C);
        float out[V];
        {
          float g[V];
          unpackv<T>(gr[jj], g);
#pragma unroll
          for (int v = 0; v < V; ++v) {
            out[v] = fmaf(taps[v][0], g[v], residual ? g[v] : 0.f);
            dwa[v][0] = fmaf(xv[v], g[v], dwa[v][0]);
          }
        }
#pragma unroll
        for (int k = 1; k < W; ++k) {
          if (t + k < Tlen) {
            float g[V];
            unpackv<T>(gr[(jj + k) % kRing], g);
#pragma unroll
            for (int v = 0; v < V; ++v) {
              out[v] = fmaf(taps[v][k], g[v], out[v]);
              dwa[v][k] = fmaf(xv[v], g[v], dwa[v][k]);
            }
          }
        }
        stcsv(dxb + n * C, packv<T>(out));
        if (n + kRing < nend) gr[jj] = ldgv(gb + (n + kRing) * C);
        if (++t == Tlen) t = 0;
      }
    }
  }
  float* dst = dw_part + rg.r * C * W + c0 * W;
#pragma unroll
  for (int v = 0; v < V; ++v)
#pragma unroll
    for (int k = 0; k < W; ++k) dst[v * W + k] = dwa[v][k];
}

// dw[i] = sum over ranges r of part[r][i], four outputs a thread.  A block
// of kRedSlices x 32 threads covers 128 outputs; slice s adds the ranges
// r = s, s + kRedSlices, ... in order, then the slices are added in order
// through shared memory: a fixed order, so dw is bitwise reproducible.
constexpr int kRedSlices = 8;

template <typename T>
__global__ void __launch_bounds__(kRedSlices * 32)
static_dw_reduce(const float* __restrict__ part, T* __restrict__ dw, int64_t n, int64_t nranges) {
  __shared__ float4 acc[kRedSlices][32];
  const int lane = threadIdx.x & 31, slice = threadIdx.x >> 5;
  const int64_t n4 = n / 4;
  const int64_t i4 = static_cast<int64_t>(blockIdx.x) * 32 + lane;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  if (i4 < n4) {
    const float4* src = reinterpret_cast<const float4*>(part) + i4;
    for (int64_t r = slice; r < nranges; r += kRedSlices) {
      const float4 v = __ldg(src + r * n4);
      a.x += v.x;
      a.y += v.y;
      a.z += v.z;
      a.w += v.w;
    }
  }
  acc[slice][lane] = a;
  __syncthreads();
  if (slice == 0 && i4 < n4) {
    float4 t = acc[0][lane];
#pragma unroll
    for (int q = 1; q < kRedSlices; ++q) {
      t.x += acc[q][lane].x;
      t.y += acc[q][lane].y;
      t.z += acc[q][lane].z;
      t.w += acc[q][lane].w;
    }
    T* o = dw + 4 * i4;
    o[0] = from_f32<T>(t.x);
    o[1] = from_f32<T>(t.y);
    o[2] = from_f32<T>(t.z);
    o[3] = from_f32<T>(t.w);
  }
}

// Token ranges: one wave of resident CTAs (occupancy x SMs over the channel
// blocks), at most kMaxRanges so the dw workspace has a bound that is a
// function of the shape only.
constexpr int64_t kMaxRanges = 512;

int64_t max_ranges(const Shape& s) {
  return std::max<int64_t>(1, std::min<int64_t>(kMaxRanges, s.N() / 16));
}

int64_t ranges_for(const void* kernel, int64_t ncb, const Shape& s) {
  return std::min<int64_t>(n_ranges(kernel, kThreads, ncb, s.N()), max_ranges(s));
}

#define DSC_ST_W_SWITCH(Wv, ...)                                      \
  switch (Wv) {                                                       \
    case 1: { constexpr int W_ = 1; __VA_ARGS__; } break;             \
    case 2: { constexpr int W_ = 2; __VA_ARGS__; } break;             \
    case 3: { constexpr int W_ = 3; __VA_ARGS__; } break;             \
    default: { constexpr int W_ = 4; __VA_ARGS__; } break;            \
  }

template <typename T>
cudaError_t fwd_t(const void* x, const void* w, void* y, const Shape& s, cudaStream_t st) {
  const int64_t ncb = (s.C / Vec<T>::N + kThreads - 1) / kThreads;
  DSC_ST_W_SWITCH(s.W, {
    const int64_t nr = ranges_for((const void*)static_fwd_kernel<T, W_>, ncb, s);
    static_fwd_kernel<T, W_><<<static_cast<unsigned>(ncb * nr), kThreads, 0, st>>>(
        static_cast<const T*>(x), static_cast<const T*>(w), static_cast<T*>(y), s.T, s.C,
        s.residual, s.N(), ncb, nr);
  })
  return cudaGetLastError();
}

template <typename T>
cudaError_t bwd_t(const void* x, const void* w, const void* dy, void* dx, void* dw, void* ws,
                  const Shape& s, cudaStream_t st) {
  const int64_t ncb = (s.C / VecB<T>::N + kThreads - 1) / kThreads;
  float* part = static_cast<float*>(ws);
  int64_t nr = 1;
  DSC_ST_W_SWITCH(s.W, {
    nr = ranges_for((const void*)static_bwd_kernel<T, W_>, ncb, s);
    static_bwd_kernel<T, W_><<<static_cast<unsigned>(ncb * nr), kThreads, 0, st>>>(
        static_cast<const T*>(x), static_cast<const T*>(w), static_cast<const T*>(dy),
        static_cast<T*>(dx), part, s.T, s.C, s.residual, s.N(), ncb, nr);
  })
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t n = s.C * s.W;  // a multiple of 4: C is a multiple of the vector width
  const unsigned blocks = static_cast<unsigned>((n / 4 + 31) / 32);
  static_dw_reduce<T><<<blocks, kRedSlices * 32, 0, st>>>(part, static_cast<T*>(dw), n, nr);
  return cudaGetLastError();
}

}  // namespace

size_t static_bwd_workspace(const Shape& s) {
  return static_cast<size_t>(max_ranges(s)) * s.C * s.W * sizeof(float);
}

cudaError_t static_fwd(const void* x, const void* w, void* y, const Shape& s, cudaStream_t st) {
  return s.bf16 ? fwd_t<__nv_bfloat16>(x, w, y, s, st) : fwd_t<float>(x, w, y, s, st);
}

cudaError_t static_bwd(const void* x, const void* w, const void* dy, void* dx, void* dw,
                       void* ws, const Shape& s, cudaStream_t st) {
  return s.bf16 ? bwd_t<__nv_bfloat16>(x, w, dy, dx, dw, ws, s, st)
                : bwd_t<float>(x, w, dy, dx, dw, ws, s, st);
}

}  // namespace dsc

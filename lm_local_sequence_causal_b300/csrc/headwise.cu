// headwise.cu -- head-wise Dynamic Short Convolution, forward and backward.
//
// y[b,t,c] = res*x[b,t,c] + sum_{k<W} w[b,t,c/H,k] * x[b,t-k,c]   (x = 0 before t = 0)
// ("Technische Samenvatting: Dynamische Korte Convoluties Verbeteren
// Transformers", Methodologie: Mechanisme, Parametrisatie item 2, Plaatsing.)
// The backward is the chain rule of that definition:
//   dx[b,s,c]   = res*dy[b,s,c] + sum_{k: s+k<T} w[b,s+k,c/H,k] dy[b,s+k,c]
//   dw[b,t,g,k] = sum_{c in group g} dy[b,t,c] x[b,t-k,c]
//
// Both passes are pure streams over HBM (about 2 flops per byte), so the
// design is about moving bytes: each thread owns one 16-byte vector of
// channels (8 bf16 or 4 fp32) and walks a tile of L tokens of one sequence,
// keeping the W-1 previous x rows (forward, dw) and the W pending dx rows
// (backward) in registers as a sliding window.  A warp therefore reads and
// writes 512 contiguous bytes per token row; the only re-read is the W-1 row
// halo at the start of each tile, which the neighbouring tile has just
// pulled into L2.  Filters are loaded as the contiguous chunk of the
// thread's groups (NG groups x W taps) with the widest aligned access.
//
// Fast paths: H divides the vector (NG = V/H groups per thread) or the vector
// divides H with H/V a power of two <= 32 (the H/V threads of one group are
// adjacent lanes and reduce dw by butterfly shuffles).  Every other H runs a
// plain per-channel path that is correct but not tuned.
#include <algorithm>

#include "dsc_common.cuh"
#include "dsc_internal.h"

namespace dsc {
namespace {

constexpr int kThreads = 128;

// The grid is one-dimensional over (sequence b, token tile, channel block),
// channel block fastest, so any B and T fit the launch limits.
struct Tile {
  int64_t cb, tt, b;
};
__device__ __forceinline__ Tile decode_tile(int64_t ncb, int64_t ntt) {
  int64_t i = blockIdx.x;
  Tile t;
  t.cb = i % ncb;
  i /= ncb;
  t.tt = i % ntt;
  t.b = i / ntt;
  return t;
}

// ------------------------------------------------------------ forward ----

template <typename T, int W, int NG>
__global__ void __launch_bounds__(kThreads)
hw_fwd_kernel(const T* __restrict__ x, const T* __restrict__ w, T* __restrict__ y,
              int64_t Tlen, int64_t C, int64_t H, int residual, int L, int64_t ncb,
              int64_t ntt) {
  constexpr int V = Vec<T>::N;
  const Tile tl = decode_tile(ncb, ntt);
  const int64_t cv = tl.cb * blockDim.x + threadIdx.x;
  const int64_t c0 = cv * V;
  if (c0 >= C) return;
  const int64_t G = C / H;
  const int64_t b = tl.b;
  const int64_t t0 = tl.tt * L;
  const int64_t t1 = t0 + L < Tlen ? t0 + L : Tlen;
  const T* xb = x + b * Tlen * C + c0;
  const T* wb = w + b * Tlen * G * W + (c0 / H) * W;
  T* yb = y + b * Tlen * C + c0;

  float win[W > 1 ? W - 1 : 1][V];  // win[j] = x[t-1-j]
#pragma unroll
  for (int j = 0; j < W - 1; ++j) {
    const int64_t t = t0 - 1 - j;
    if (t >= 0) {
      unpack16<T>(ldg16(xb + t * C), win[j]);
    } else {
#pragma unroll
      for (int v = 0; v < V; ++v) win[j][v] = 0.f;
    }
  }

#pragma unroll 2
  for (int64_t t = t0; t < t1; ++t) {
    float xv[V];
    unpack16<T>(ldg16(xb + t * C), xv);
    float taps[NG * W];
    load_chunk<T, NG * W>(wb + t * G * W, taps);
    float out[V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int gi = NG == 1 ? 0 : v / (V / NG);
      float a = residual ? xv[v] : 0.f;
      a = fmaf(taps[gi * W], xv[v], a);
#pragma unroll
      for (int k = 1; k < W; ++k) a = fmaf(taps[gi * W + k], win[k - 1][v], a);
      out[v] = a;
    }
    stcs16(yb + t * C, pack16<T>(out));
#pragma unroll
    for (int j = W - 2; j > 0; --j)
#pragma unroll
      for (int v = 0; v < V; ++v) win[j][v] = win[j - 1][v];
    if constexpr (W > 1) {
#pragma unroll
      for (int v = 0; v < V; ++v) win[0][v] = xv[v];
    }
  }
}

// ----------------------------------------------------------- backward ----

// One token step of the backward sweep is described in the file comment; the
// loop runs t over [t0, t1 + W - 1): step t adds the contributions of dy[t]
// to dx rows t-W+1..t (scatter form, so no filter row is kept), forms dw[t]
// when t is inside the tile, and retires dx row t-W+1.
template <typename T, int W, int NG>
__global__ void __launch_bounds__(kThreads)
hw_bwd_kernel(const T* __restrict__ x, const T* __restrict__ w,
              const T* __restrict__ dy, T* __restrict__ dx, T* __restrict__ dw,
              int64_t Tlen, int64_t C, int64_t H, int residual, int L, int tpg, int64_t ncb,
              int64_t ntt) {
  constexpr int V = Vec<T>::N;
  const Tile tl = decode_tile(ncb, ntt);
  const int64_t cv = tl.cb * blockDim.x + threadIdx.x;
  const int64_t nvec = C / V;
  // Lanes past the channel range leave together with their whole group
  // (C % H == 0), so the shuffle mask is the prefix of active lanes.
  const int64_t warp_base = cv - (threadIdx.x & 31);
  const int64_t nact = nvec - warp_base;
  const unsigned mask = nact >= 32 ? 0xffffffffu : nact > 0 ? ((1u << nact) - 1u) : 0u;
  if (cv >= nvec) return;
  const int64_t c0 = cv * V;
  const int64_t G = C / H;
  const int64_t b = tl.b;
  const int64_t t0 = tl.tt * L;
  const int64_t t1 = t0 + L < Tlen ? t0 + L : Tlen;
  const int64_t base = b * Tlen * C + c0;
  const int64_t wbase = b * Tlen * G * W + (c0 / H) * W;
  const bool leader = (NG > 1) || ((cv & (tpg - 1)) == 0);

  float xwin[W > 1 ? W - 1 : 1][V];  // x[t-1-j]
  float acc[W][V];                   // acc[j] = dx row t-(W-1)+j
#pragma unroll
  for (int j = 0; j < W - 1; ++j) {
    const int64_t t = t0 - 1 - j;
    if (t >= 0) {
      unpack16<T>(ldg16(x + base + t * C), xwin[j]);
    } else {
#pragma unroll
      for (int v = 0; v < V; ++v) xwin[j][v] = 0.f;
    }
  }
#pragma unroll
  for (int j = 0; j < W; ++j)
#pragma unroll
    for (int v = 0; v < V; ++v) acc[j][v] = 0.f;

  const int64_t tend = t1 + W - 1;
#pragma unroll 2
  for (int64_t t = t0; t < tend; ++t) {
    float g[V];
    float taps[NG * W];
    if (t < Tlen) {
      unpack16<T>(ldg16(dy + base + t * C), g);
      load_chunk<T, NG * W>(w + wbase + t * G * W, taps);
    } else {
#pragma unroll
      for (int v = 0; v < V; ++v) g[v] = 0.f;
#pragma unroll
      for (int i = 0; i < NG * W; ++i) taps[i] = 0.f;
    }
    // dx: row t enters the window; dy[t] feeds rows t-k through tap k.
#pragma unroll
    for (int v = 0; v < V; ++v) acc[W - 1][v] = (residual && t < t1) ? g[v] : 0.f;
#pragma unroll
    for (int k = 0; k < W; ++k) {
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int gi = NG == 1 ? 0 : v / (V / NG);
        acc[W - 1 - k][v] = fmaf(taps[gi * W + k], g[v], acc[W - 1 - k][v]);
      }
    }
    if (t < t1) {
      // dw[t, g, k] = sum over the group's channels of dy[t,c] x[t-k,c].
      float xv[V];
      unpack16<T>(ldg16(x + base + t * C), xv);
      float p[NG * W];
#pragma unroll
      for (int i = 0; i < NG * W; ++i) p[i] = 0.f;
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int gi = NG == 1 ? 0 : v / (V / NG);
        p[gi * W] = fmaf(g[v], xv[v], p[gi * W]);
#pragma unroll
        for (int k = 1; k < W; ++k) p[gi * W + k] = fmaf(g[v], xwin[k - 1][v], p[gi * W + k]);
      }
      if constexpr (NG == 1) {
        for (int off = 1; off < tpg; off <<= 1)
#pragma unroll
          for (int k = 0; k < W; ++k) p[k] += __shfl_xor_sync(mask, p[k], off);
      }
      if (leader) store_chunk<T, NG * W>(dw + wbase + t * G * W, p);
#pragma unroll
      for (int j = W - 2; j > 0; --j)
#pragma unroll
        for (int v = 0; v < V; ++v) xwin[j][v] = xwin[j - 1][v];
      if constexpr (W > 1) {
#pragma unroll
        for (int v = 0; v < V; ++v) xwin[0][v] = xv[v];
      }
    }
    // dx row t-W+1 has received every contribution.
    const int64_t s = t - (W - 1);
    if (s >= t0) stcs16(dx + base + s * C, pack16<T>(acc[0]));
#pragma unroll
    for (int j = 0; j < W - 1; ++j)
#pragma unroll
      for (int v = 0; v < V; ++v) acc[j][v] = acc[j + 1][v];
  }
}

// ------------------------------------------- generic (any H) fallbacks ----

// One thread per (token, channel): plain gather form, any H with C % H == 0.
template <typename T>
__global__ void hw_fwd_generic(const T* __restrict__ x, const T* __restrict__ w,
                               T* __restrict__ y, int64_t N, int64_t Tlen,
                               int64_t C, int64_t H, int64_t W, int residual) {
  const int64_t G = C / H;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < N * C;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / C, c = i % C, t = row % Tlen, g = c / H;
    float a = residual ? to_f32(x[i]) : 0.f;
    for (int64_t k = 0; k < W && t - k >= 0; ++k)
      a = fmaf(to_f32(w[(row * G + g) * W + k]), to_f32(x[i - k * C]), a);
    y[i] = from_f32<T>(a);
  }
}

template <typename T>
__global__ void hw_dx_generic(const T* __restrict__ w, const T* __restrict__ dy,
                              T* __restrict__ dx, int64_t N, int64_t Tlen,
                              int64_t C, int64_t H, int64_t W, int residual) {
  const int64_t G = C / H;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < N * C;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / C, c = i % C, t = row % Tlen, g = c / H;
    float a = residual ? to_f32(dy[i]) : 0.f;
    for (int64_t k = 0; k < W && t + k < Tlen; ++k)
      a = fmaf(to_f32(w[((row + k) * G + g) * W + k]), to_f32(dy[i + k * C]), a);
    dx[i] = from_f32<T>(a);
  }
}

// One thread per (token, group, tap).
template <typename T>
__global__ void hw_dw_generic(const T* __restrict__ x, const T* __restrict__ dy,
                              T* __restrict__ dw, int64_t N, int64_t Tlen,
                              int64_t C, int64_t H, int64_t W) {
  const int64_t G = C / H;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < N * G * W;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t k = i % W, g = (i / W) % G, row = i / (G * W), t = row % Tlen;
    float a = 0.f;
    if (t - k >= 0)
      for (int64_t c = g * H; c < (g + 1) * H; ++c)
        a = fmaf(to_f32(dy[row * C + c]), to_f32(x[(row - k) * C + c]), a);
    dw[i] = from_f32<T>(a);
  }
}

// ------------------------------------------------------------ dispatch ----

// Tokens per tile: long enough to amortise the W-1 row halo, short enough
// to give every SM several CTAs.
int tile_len(const Shape& s, int64_t ctas_x) {
  int64_t L = 64;
  while (L > 16 && ctas_x * s.B * ((s.T + L - 1) / L) < 4 * 148) L /= 2;
  while (ctas_x * s.B * ((s.T + L - 1) / L) > (int64_t(1) << 30)) L *= 2;
  return (int)L;
}

template <typename T>
int ng_of(int64_t H) {
  constexpr int V = Vec<T>::N;
  if (H < V && V % H == 0) return (int)(V / H);
  if (H % V == 0) {
    const int64_t tpg = H / V;
    if (tpg <= 32 && (tpg & (tpg - 1)) == 0) return 1;
  }
  return 0;  // generic path
}

#define DSC_W_SWITCH(Wv, ...)                                         \
  switch (Wv) {                                                       \
    case 1: { constexpr int W_ = 1; __VA_ARGS__; } break;             \
    case 2: { constexpr int W_ = 2; __VA_ARGS__; } break;             \
    case 3: { constexpr int W_ = 3; __VA_ARGS__; } break;             \
    default: { constexpr int W_ = 4; __VA_ARGS__; } break;            \
  }

#define DSC_NG_SWITCH(ng, ...)                                        \
  switch (ng) {                                                       \
    case 1: { constexpr int NG_ = 1; __VA_ARGS__; } break;            \
    case 2: { constexpr int NG_ = 2; __VA_ARGS__; } break;            \
    case 4: { constexpr int NG_ = 4; __VA_ARGS__; } break;            \
    default: { constexpr int NG_ = 8; __VA_ARGS__; } break;           \
  }

template <typename T>
cudaError_t fwd_t(const void* x, const void* w, void* y, const Shape& s, cudaStream_t st) {
  constexpr int V = Vec<T>::N;
  const int ng = ng_of<T>(s.H);
  if (ng == 0) {
    const int64_t n = s.N() * s.C;
    const int blocks = (int)std::min<int64_t>((n + 255) / 256, 148 * 16);
    hw_fwd_generic<T><<<blocks, 256, 0, st>>>((const T*)x, (const T*)w, (T*)y, s.N(),
                                              s.T, s.C, s.H, s.W, s.residual);
    return cudaGetLastError();
  }
  const int64_t nvec = s.C / V;
  const int threads = (int)std::min<int64_t>(kThreads, (nvec + 31) / 32 * 32);
  const int64_t gx = (nvec + threads - 1) / threads;
  const int L = tile_len(s, gx);
  const int64_t ntt = (s.T + L - 1) / L;
  const unsigned grid = (unsigned)(gx * ntt * s.B);
  DSC_W_SWITCH(s.W, DSC_NG_SWITCH(ng, {
    if constexpr (NG_ <= V)
      hw_fwd_kernel<T, W_, NG_><<<grid, threads, 0, st>>>(
          (const T*)x, (const T*)w, (T*)y, s.T, s.C, s.H, s.residual, L, gx, ntt);
  }))
  return cudaGetLastError();
}

template <typename T>
cudaError_t bwd_t(const void* x, const void* w, const void* dy, void* dx, void* dw,
                  const Shape& s, cudaStream_t st) {
  constexpr int V = Vec<T>::N;
  const int ng = ng_of<T>(s.H);
  if (ng == 0) {
    const int64_t n = s.N() * s.C;
    const int blocks = (int)std::min<int64_t>((n + 255) / 256, 148 * 16);
    hw_dx_generic<T><<<blocks, 256, 0, st>>>((const T*)w, (const T*)dy, (T*)dx, s.N(),
                                             s.T, s.C, s.H, s.W, s.residual);
    const int64_t nw = s.N() * s.G() * s.W;
    const int blocks_w = (int)std::min<int64_t>((nw + 255) / 256, 148 * 16);
    hw_dw_generic<T><<<blocks_w, 256, 0, st>>>((const T*)x, (const T*)dy, (T*)dw, s.N(),
                                               s.T, s.C, s.H, s.W);
    return cudaGetLastError();
  }
  const int64_t nvec = s.C / V;
  const int threads = (int)std::min<int64_t>(kThreads, (nvec + 31) / 32 * 32);
  const int64_t gx = (nvec + threads - 1) / threads;
  const int L = tile_len(s, gx);
  const int tpg = ng == 1 ? (int)(s.H / V) : 1;
  const int64_t ntt = (s.T + L - 1) / L;
  const unsigned grid = (unsigned)(gx * ntt * s.B);
  DSC_W_SWITCH(s.W, DSC_NG_SWITCH(ng, {
    if constexpr (NG_ <= V)
      hw_bwd_kernel<T, W_, NG_><<<grid, threads, 0, st>>>(
          (const T*)x, (const T*)w, (const T*)dy, (T*)dx, (T*)dw, s.T, s.C, s.H,
          s.residual, L, tpg, gx, ntt);
  }))
  return cudaGetLastError();
}

}  // namespace

cudaError_t headwise_fwd(const void* x, const void* w, void* y, const Shape& s,
                         cudaStream_t st) {
  return s.bf16 ? fwd_t<__nv_bfloat16>(x, w, y, s, st) : fwd_t<float>(x, w, y, s, st);
}

cudaError_t headwise_bwd(const void* x, const void* w, const void* dy, void* dx,
                         void* dw, const Shape& s, cudaStream_t st) {
  return s.bf16 ? bwd_t<__nv_bfloat16>(x, w, dy, dx, dw, s, st)
                : bwd_t<float>(x, w, dy, dx, dw, s, st);
}

}  // namespace dsc

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
#include <mutex>

#include "dsc_common.cuh"
#include "dsc_internal.h"

namespace dsc {
namespace {

constexpr int kThreads = 128;

// Work split: the B*T tokens are one flat axis n = b*T + t.  The grid is
// (channel block of 128 threads) x (token range); ranges are contiguous and
// balanced to +-1 token, and the grid is sized to the CTAs that fit on the
// GPU at once, so every CTA streams the same number of rows and there is no
// partial last wave.  A range may cross sequence boundaries: at t = 0 the
// causal window restarts from zero, and a tap only links rows of the same
// sequence.

// Tokens of look-ahead: each thread keeps the loads of the next kPF tokens
// in flight (a register ring), so a CTA has about kPF x 24-40 bytes per
// thread outstanding -- enough, at a few CTAs per SM, to cover HBM latency.
constexpr int kPF = 4;    // forward (x and the taps: 24 bytes a token)
constexpr int kPFB = 4;   // backward (dy, taps and x: 40 bytes a token)

struct Range {
  int64_t cb, n0, n1;
};
__device__ __forceinline__ Range decode_range(int64_t ncb, int64_t nranges, int64_t N) {
  Range r;
  r.cb = blockIdx.x % ncb;
  const int64_t i = blockIdx.x / ncb;
  r.n0 = N * i / nranges;
  r.n1 = N * (i + 1) / nranges;
  return r;
}

// ------------------------------------------------------------ forward ----

template <typename T, int W, int NG>
__global__ void __launch_bounds__(kThreads)
hw_fwd_kernel(const T* __restrict__ x, const T* __restrict__ w, T* __restrict__ y,
              int64_t Tlen, int64_t C, int64_t H, int residual, int64_t N, int64_t ncb,
              int64_t nranges) {
  constexpr int V = Vec<T>::N;
  const Range rg = decode_range(ncb, nranges, N);
  const int64_t cv = rg.cb * blockDim.x + threadIdx.x;
  const int64_t c0 = cv * V;
  if (c0 >= C) return;
  const int64_t G = C / H;
  const int64_t n0 = rg.n0, n1 = rg.n1;
  const T* xb = x + c0;
  const T* wb = w + (c0 / H) * W;
  T* yb = y + c0;

  int64_t t = n0 % Tlen;             // position of token n in its sequence
  float win[W > 1 ? W - 1 : 1][V];   // win[j] = x[n-1-j] (zero before the sequence start)
#pragma unroll
  for (int j = 0; j < W - 1; ++j) {
    if (t - 1 - j >= 0) {
      unpack16<T>(ldg16(xb + (n0 - 1 - j) * C), win[j]);
    } else {
#pragma unroll
      for (int v = 0; v < V; ++v) win[j][v] = 0.f;
    }
  }

  uint4 xr[kPF];
  RawChunk<T, NG * W> wr[kPF];
#pragma unroll
  for (int j = 0; j < kPF; ++j) {
    if (n0 + j < n1) {
      xr[j] = ldg16(xb + (n0 + j) * C);
      wr[j].load(wb + (n0 + j) * G * W);
    }
  }
  for (int64_t nb = n0; nb < n1; nb += kPF) {
#pragma unroll
    for (int j = 0; j < kPF; ++j) {
      const int64_t n = nb + j;
      if (n < n1) {
        if (t == 0) {
#pragma unroll
          for (int q = 0; q < W - 1; ++q)
#pragma unroll
            for (int v = 0; v < V; ++v) win[q][v] = 0.f;
        }
        float xv[V];
        unpack16<T>(xr[j], xv);
        float taps[NG * W];
        wr[j].unpack(taps);
        if (n + kPF < n1) {
          xr[j] = ldg16(xb + (n + kPF) * C);
          wr[j].load(wb + (n + kPF) * G * W);
        }
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

// ----------------------------------------------------------- backward ----

// One step n of the backward sweep (scatter form, so no filter row is kept):
// dy[n] feeds the dx rows n-k of the same sequence through tap k, dw[n] is
// formed when n is inside the range, and dx row n-W+1 is retired.  The steps
// run over [n0, n1 + W - 1) (cut at N), so the last rows of the range get
// the contributions of the next W-1 tokens.  The dy, w and x rows of the
// next kPF steps are in flight while a step computes.
template <typename T, int W, int NG>
__global__ void __launch_bounds__(kThreads)
hw_bwd_kernel(const T* __restrict__ x, const T* __restrict__ w,
              const T* __restrict__ dy, T* __restrict__ dx, T* __restrict__ dw,
              int64_t Tlen, int64_t C, int64_t H, int residual, int tpg, int64_t N,
              int64_t ncb, int64_t nranges) {
  constexpr int V = Vec<T>::N;
  const Range rg = decode_range(ncb, nranges, N);
  const int64_t cv = rg.cb * blockDim.x + threadIdx.x;
  const int64_t nvec = C / V;
  // Lanes past the channel range leave together with their whole group
  // (C % H == 0), so the shuffle mask is the prefix of active lanes.
  const int64_t warp_base = cv - (threadIdx.x & 31);
  const int64_t nact = nvec - warp_base;
  const unsigned mask = nact >= 32 ? 0xffffffffu : nact > 0 ? ((1u << nact) - 1u) : 0u;
  if (cv >= nvec) return;
  const int64_t c0 = cv * V;
  const int64_t G = C / H;
  const int64_t n0 = rg.n0, n1 = rg.n1;
  const int64_t wrow = G * W;
  const T* xb = x + c0;
  const T* gb = dy + c0;
  const T* wb = w + (c0 / H) * W;
  T* dxb = dx + c0;
  T* dwb = dw + (c0 / H) * W;
  const bool leader = (NG > 1) || ((cv & (tpg - 1)) == 0);

  int64_t t = n0 % Tlen;
  float xwin[W > 1 ? W - 1 : 1][V];  // x[n-1-j], zero before the sequence start
  float acc[W][V];                   // acc[j] = dx row n-(W-1)+j
#pragma unroll
  for (int j = 0; j < W - 1; ++j) {
    if (t - 1 - j >= 0) {
      unpack16<T>(ldg16(xb + (n0 - 1 - j) * C), xwin[j]);
    } else {
#pragma unroll
      for (int v = 0; v < V; ++v) xwin[j][v] = 0.f;
    }
  }
#pragma unroll
  for (int j = 0; j < W; ++j)
#pragma unroll
    for (int v = 0; v < V; ++v) acc[j][v] = 0.f;

  const int64_t nend = n1 + W - 1 < N ? n1 + W - 1 : N;
  uint4 gr[kPFB], xr[kPFB];
  RawChunk<T, NG * W> wr[kPFB];
#pragma unroll
  for (int j = 0; j < kPFB; ++j) {
    const int64_t n = n0 + j;
    if (n < nend) {
      gr[j] = ldg16(gb + n * C);
      wr[j].load(wb + n * wrow);
    }
    if (n < n1) xr[j] = ldg16(xb + n * C);
  }
  for (int64_t nb = n0; nb < nend; nb += kPFB) {
#pragma unroll
    for (int jj = 0; jj < kPFB; ++jj) {
      const int64_t n = nb + jj;
      if (n < nend) {
        const bool inside = n < n1;
        float g[V];
        unpack16<T>(gr[jj], g);
        float taps[NG * W];
        wr[jj].unpack(taps);
        float xv[V];
        if (inside) unpack16<T>(xr[jj], xv);
        const int64_t nn = n + kPFB;
        if (nn < nend) {
          gr[jj] = ldg16(gb + nn * C);
          wr[jj].load(wb + nn * wrow);
        }
        if (nn < n1) xr[jj] = ldg16(xb + nn * C);
        // dx: row n enters the window; dy[n] feeds rows n-k (same sequence).
#pragma unroll
        for (int v = 0; v < V; ++v) acc[W - 1][v] = (residual && inside) ? g[v] : 0.f;
#pragma unroll
        for (int k = 0; k < W; ++k) {
          if (t >= k) {
#pragma unroll
            for (int v = 0; v < V; ++v) {
              const int gi = NG == 1 ? 0 : v / (V / NG);
              acc[W - 1 - k][v] = fmaf(taps[gi * W + k], g[v], acc[W - 1 - k][v]);
            }
          }
        }
        if (inside) {
          if (t == 0) {
#pragma unroll
            for (int q = 0; q < W - 1; ++q)
#pragma unroll
              for (int v = 0; v < V; ++v) xwin[q][v] = 0.f;
          }
          // dw[n, g, k] = sum over the group's channels of dy[n,c] x[n-k,c].
          float p[NG * W];
#pragma unroll
          for (int i = 0; i < NG * W; ++i) p[i] = 0.f;
#pragma unroll
          for (int v = 0; v < V; ++v) {
            const int gi = NG == 1 ? 0 : v / (V / NG);
            p[gi * W] = fmaf(g[v], xv[v], p[gi * W]);
#pragma unroll
            for (int k = 1; k < W; ++k)
              p[gi * W + k] = fmaf(g[v], xwin[k - 1][v], p[gi * W + k]);
          }
          if constexpr (NG == 1) {
            for (int off = 1; off < tpg; off <<= 1)
#pragma unroll
              for (int k = 0; k < W; ++k) p[k] += __shfl_xor_sync(mask, p[k], off);
          }
          if (leader) store_chunk<T, NG * W>(dwb + n * wrow, p);
#pragma unroll
          for (int q = W - 2; q > 0; --q)
#pragma unroll
            for (int v = 0; v < V; ++v) xwin[q][v] = xwin[q - 1][v];
          if constexpr (W > 1) {
#pragma unroll
            for (int v = 0; v < V; ++v) xwin[0][v] = xv[v];
          }
        }
        // dx row n-W+1 has received every contribution.
        const int64_t sr = n - (W - 1);
        if (sr >= n0) stcs16(dxb + sr * C, pack16<T>(acc[0]));
#pragma unroll
        for (int q = 0; q < W - 1; ++q)
#pragma unroll
          for (int v = 0; v < V; ++v) acc[q][v] = acc[q + 1][v];
        if (++t == Tlen) t = 0;
      }
    }
  }
  // If the sweep stopped at the end of the data, the last W-1 rows are still
  // in the window; they are complete, so retire them here.
  if (nend < n1 + W - 1) {
#pragma unroll
    for (int j = 0; j < W - 1; ++j) {
      const int64_t sr = nend - (W - 1) + j;
      if (sr >= n0 && sr < n1) stcs16(dxb + sr * C, pack16<T>(acc[j]));
    }
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
  const int64_t N = s.N();
  DSC_W_SWITCH(s.W, DSC_NG_SWITCH(ng, {
    if constexpr (NG_ <= V) {
      auto kern = hw_fwd_kernel<T, W_, NG_>;
      const int64_t nr = n_ranges((const void*)kern, threads, gx, N);
      kern<<<(unsigned)(gx * nr), threads, 0, st>>>((const T*)x, (const T*)w, (T*)y, s.T, s.C,
                                                    s.H, s.residual, N, gx, nr);
    }
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
  const int tpg = ng == 1 ? (int)(s.H / V) : 1;
  const int64_t N = s.N();
  DSC_W_SWITCH(s.W, DSC_NG_SWITCH(ng, {
    if constexpr (NG_ <= V) {
      auto kern = hw_bwd_kernel<T, W_, NG_>;
      const int64_t nr = n_ranges((const void*)kern, threads, gx, N);
      kern<<<(unsigned)(gx * nr), threads, 0, st>>>((const T*)x, (const T*)w, (const T*)dy,
                                                    (T*)dx, (T*)dw, s.T, s.C, s.H, s.residual,
                                                    tpg, N, gx, nr);
    }
  }))
  return cudaGetLastError();
}

}  // namespace

cudaError_t headwise_fwd(const void* x, const void* w, void* y, const Shape& s,
                         cudaStream_t st) {
  if (headwise_tma_supported(s, false)) return headwise_fwd_tma(x, w, y, s, st);
  return s.bf16 ? fwd_t<__nv_bfloat16>(x, w, y, s, st) : fwd_t<float>(x, w, y, s, st);
}

cudaError_t headwise_bwd(const void* x, const void* w, const void* dy, void* dx,
                         void* dw, const Shape& s, cudaStream_t st) {
  if (headwise_tma_supported(s, true)) return headwise_bwd_tma(x, w, dy, dx, dw, s, st);
  return s.bf16 ? bwd_t<__nv_bfloat16>(x, w, dy, dx, dw, s, st)
                : bwd_t<float>(x, w, dy, dx, dw, s, st);
}

}  // namespace dsc

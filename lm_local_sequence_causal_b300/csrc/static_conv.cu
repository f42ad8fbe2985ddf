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
// bf16 with C a multiple of 64 (W <= 4) takes the TMA-staged kernels below
// (one CTA per 64-channel chunk and part of its token tiles, taps and dw
// accumulators in registers); the rest takes the register-streaming kernels:
// the same streaming scheme as the head-wise register kernels: a thread owns a
// vector of channels (16 bytes forward, 8 bytes backward) and walks a
// contiguous range of the flat token axis n = b*T + t (balanced ranges,
// sequence starts reset the causal window), with the loads of the next
// tokens in flight.  The taps are loaded once.  The backward accumulates dw
// over its range in registers and writes one fp32 partial per (range,
// channel, tap); a second kernel adds the partials in range order (bitwise
// reproducible).
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "dsc_common.cuh"
#include "dsc_internal.h"
#include "sm100.cuh"

namespace dsc {
namespace {

using namespace sm100;

// Set when a bounded wait of the TMA backward gives up: 1 = producer,
// 3 = epilogue, 4 = store.
__device__ unsigned int g_st_error = 0;

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

// ------------------------------------------- TMA-staged forward, backward ----
//
// bf16, W <= 4, C a multiple of 64.  The same streams as the register
// kernels above, staged by TMA: one CTA per (64-channel chunk c, part p of
// the chunk's 128-token tiles), so the chunk's taps stay in registers and,
// in the backward, dw accumulates in registers over every tile the CTA takes.
//   warp 0      TMA producer, a ring of 6 (forward) or 4 (backward) stages:
//               x rows [t0-W+1, t0+128) and, in the backward, dy rows
//               [t0, t0+127+W) of the chunk (rows before t = 0 and past T
//               read as zero: the causal padding and the dropped terms
//               s+k >= T).
//   warps 1-16  two groups of 8 warps taking alternate tiles; in a group,
//               warp w owns tokens 16w .. 16w+15 of the tile and lane l the
//               channel pair 2l, 2l+1, so a warp reads one 128-byte row of x
//               (and of dy) per token (4 bytes a lane) and keeps the W-row
//               windows in registers:
//                 y[t]   = res*x[t] + sum_k w[k] x[t-k]            (forward)
//                 dx[t]  = res*dy[t] + sum_k w[k] dy[t+k]          (backward)
//                 dw[k] += dy[t] x[t-k]
//               y or dx goes to a staged tile that one thread stores with TMA.
// At the end of the backward each group adds its 8 warps' dw (in warp order,
// through shared memory) and writes one fp32 partial per (part, group);
// static_dw_reduce adds the 2P partials of each (channel, tap) in a fixed
// order.
constexpr int kStBM = 128;
constexpr int kStNGRP = 8;
constexpr int kStThreads = (1 + 2 * kStNGRP) * 32;

__host__ __device__ constexpr int st_round1k(int b) { return (b + 1023) / 1024 * 1024; }

template <int W, bool BWD>
struct StLayout {
  // Stages: an even number (the two groups take alternate tiles; see the
  // head-wise TMA kernels), 6 for the forward's x-only stages, 4 for the
  // backward's x and dy.
  static constexpr int NST = BWD ? 4 : 6;
  static constexpr int XROWS = kStBM + W - 1;
  static constexpr int XBOX = XROWS * 128;            // one 64-channel box
  static constexpr int XBYTES = st_round1k(XBOX);
  static constexpr int STAGE = (BWD ? 2 : 1) * XBYTES;  // x (, dy)
  static constexpr int OBOX = kStBM * 128;            // staged y / dx tile of one group
  static constexpr int O_OFF = NST * STAGE;
  static constexpr int BAR_OFF = O_OFF + 2 * OBOX;
  // full[NST] empty[NST] ofull[2] ofree[2]
  static constexpr int NBAR = 2 * NST + 4;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int TOTAL = MISC_OFF + 16 + 1024;
  static constexpr uint32_t TX = (BWD ? 2 : 1) * XBOX;
  static_assert(NST % 2 == 0, "stages must be even");
  static_assert(TOTAL <= 227 * 1024, "static kernel shared memory");
  static_assert(kStNGRP * 32 * 2 * W * 4 <= OBOX, "dw scratch fits a staged tile");
};

// Byte address of the channel pair `cp` (4 bytes) of row `r` in a staged
// 64-channel tile with 128-byte rows and the TMA 128-byte swizzle.
__device__ __forceinline__ uint32_t pair_addr(uint32_t tile, uint32_t r, uint32_t cp) {
  return tile + sw128_offset(r, cp >> 2) + ((cp & 3u) << 2);
}

__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

__device__ __forceinline__ void sts32(uint32_t a, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

template <int W, bool BWD, bool RES>
__global__ void __launch_bounds__(kStThreads, 1)
st_tma(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dy,
       const __grid_constant__ CUtensorMap tm_out, const __nv_bfloat16* __restrict__ w,
       float* __restrict__ part, int ntl, int ntiles, int P, int64_t CW) {
  using L = StLayout<W, BWD>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = align1k(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = static_cast<int>(blockIdx.x) / P, pp = static_cast<int>(blockIdx.x) % P;
  // this CTA's tiles (b, tile) of the chunk: [tl0, tl1)
  const int tl0 = static_cast<int>(static_cast<long long>(ntl) * pp / P);
  const int tl1 = static_cast<int>(static_cast<long long>(ntl) * (pp + 1) / P);
  const int nmine = tl1 - tl0;
  const uint32_t bar_full = sb + L::BAR_OFF;
  const uint32_t bar_empty = bar_full + L::NST * 8;
  const uint32_t bar_ofull = bar_empty + L::NST * 8;
  const uint32_t bar_ofree = bar_ofull + 16;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFF);

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::NST; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kStNGRP);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(bar_ofull + 8 * g, kStNGRP);
      mbar_init(bar_ofree + 8 * g, 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_x);
    if constexpr (BWD) tma_prefetch_desc(&tm_dy);
    tma_prefetch_desc(&tm_out);
  }
  __syncthreads();

  if (warp == 0) {
    // ---------------------------------------------------------- producer --
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int it = 0;
      for (; it < nmine; ++it) {
        const int s = it % L::NST;
        if (!mbar_wait(bar_empty + 8 * s, ((it / L::NST) & 1) ^ 1, abort_flag, &g_st_error, 1))
          break;
        const int gt = tl0 + it, b = gt / ntiles, t0 = (gt - b * ntiles) * kStBM;
        const uint32_t full = bar_full + 8 * s;
        const uint32_t st = sb + s * L::STAGE;
        mbar_expect_tx(full, L::TX);
        tma_load_3d(st, &tm_x, full, chunk * 64, t0 - (W - 1), b, pol);
        if constexpr (BWD) tma_load_3d(st + L::XBYTES, &tm_dy, full, chunk * 64, t0, b, pol);
      }
      for (int j = std::max(0, it - L::NST); j < it; ++j)
        drain_wait(bar_full + 8 * (j % L::NST), (j / L::NST) & 1);
    }
  } else {
    // --------------------------------------------------------- epilogue --
    const int g = (warp - 1) >> 3;              // group: tiles it with it % 2 == g
    const int wg = (warp - 1) & 7;              // warp within the group: tokens 16wg ..
    const uint32_t cp = static_cast<uint32_t>(lane);   // channel pair of the chunk
    const bool storer = wg == 0 && lane == 0;
    const uint64_t pol = policy_evict_first();
    const uint32_t obuf = sb + L::O_OFF + g * L::OBOX;
    // the chunk's taps of this thread's two channels (fp32 pairs: channel
    // 2cp in .x, 2cp+1 in .y)
    float2 wt[W];
    {
      const __nv_bfloat16* wp = w + (static_cast<int64_t>(chunk) * 64 + 2 * cp) * W;
#pragma unroll
      for (int k = 0; k < W; ++k)
        wt[k] = make_float2(__bfloat162float(wp[k]), __bfloat162float(wp[W + k]));
    }
    float2 dwa[W];
#pragma unroll
    for (int k = 0; k < W; ++k) dwa[k] = make_float2(0.f, 0.f);
    auto pair = [](uint32_t v) {       // two bf16 -> fp32 pair (exact)
      return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
    };
    bool ok = true;
    for (int it = g; it < nmine; it += 2) {
      const int s = it % L::NST;
      const uint32_t aph = (it >> 1) & 1;
      if (storer) {
        bulk_wait_read<0>();                    // this group's previous store has read obuf
        mbar_arrive(bar_ofree + 8 * g);
      }
      ok = mbar_wait(bar_ofree + 8 * g, aph, abort_flag, &g_st_error, 3) &&
           mbar_wait(bar_full + 8 * s, (it / L::NST) & 1, abort_flag, &g_st_error, 3);
      if (!__all_sync(0xffffffffu, ok)) break;
      const uint32_t xt = sb + s * L::STAGE, dyt = xt + L::XBYTES;
      // Token r of the tile: dy row r + k holds dy[t+k]; x box row r + W-1-k
      // holds x[t-k].  Windows: gw[k] = dy row r+k, xw[k] = x box row r+W-1-k.
      const int r0 = 16 * wg;
      float2 gw[W], xw[W];
#pragma unroll
      for (int k = 0; k < W - 1; ++k) {
        if constexpr (BWD) gw[k + 1] = pair(lds32(pair_addr(dyt, r0 + k, cp)));
        xw[W - 2 - k] = pair(lds32(pair_addr(xt, r0 + k, cp)));
      }
#pragma unroll 4
      for (int r = r0; r < r0 + 16; ++r) {
#pragma unroll
        for (int k = 0; k < W - 1; ++k) {
          if constexpr (BWD) gw[k] = gw[k + 1];
          xw[W - 1 - k] = xw[W - 2 - k];
        }
        xw[0] = pair(lds32(pair_addr(xt, r + W - 1, cp)));
        float2 o;
        if constexpr (BWD) {
          gw[W - 1] = pair(lds32(pair_addr(dyt, r + W - 1, cp)));
          o = RES ? gw[0] : make_float2(0.f, 0.f);
#pragma unroll
          for (int k = 0; k < W; ++k) {
            o = __ffma2_rn(wt[k], gw[k], o);
            dwa[k] = __ffma2_rn(gw[0], xw[k], dwa[k]);
          }
        } else {
          // y[t] = res*x[t] + sum_k w[k] x[t-k]
          o = RES ? xw[0] : make_float2(0.f, 0.f);
#pragma unroll
          for (int k = 0; k < W; ++k) o = __ffma2_rn(wt[k], xw[k], o);
        }
        __nv_bfloat162 ob = __floats2bfloat162_rn(o.x, o.y);
        sts32(pair_addr(obuf, r, cp), *reinterpret_cast<uint32_t*>(&ob));
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar_empty + 8 * s);
        mbar_arrive(bar_ofull + 8 * g);
      }
      if (storer && mbar_wait(bar_ofull + 8 * g, aph, abort_flag, &g_st_error, 4)) {
        const int gt = tl0 + it, b = gt / ntiles, t0 = (gt - b * ntiles) * kStBM;
        tma_store_3d(&tm_out, obuf, chunk * 64, t0, b, pol);
        bulk_commit();
      }
    }
    if (storer) bulk_wait<0>();
    if constexpr (BWD) {
    // The group's dw: its 8 warps' sums added in warp order through the
    // group's staged tile (free once its last store has read it).
    named_bar_sync(1 + g, kStNGRP * 32);
    float* scratch = reinterpret_cast<float*>(smem + L::O_OFF + g * L::OBOX);
    // element e of thread (wg, lane) at scratch[e][wg][lane]: conflict-free
    const int me = wg * 32 + lane;
#pragma unroll
    for (int k = 0; k < W; ++k) {
      scratch[(2 * k) * kStNGRP * 32 + me] = dwa[k].x;
      scratch[(2 * k + 1) * kStNGRP * 32 + me] = dwa[k].y;
    }
    named_bar_sync(1 + g, kStNGRP * 32);
    if (wg == 0) {
      float sum[2 * W];
#pragma unroll
      for (int e = 0; e < 2 * W; ++e) sum[e] = 0.f;
      for (int q = 0; q < kStNGRP; ++q)
#pragma unroll
        for (int e = 0; e < 2 * W; ++e) sum[e] += scratch[e * kStNGRP * 32 + q * 32 + lane];
      // part[2 pp + g][c][k], channel c = 64 chunk + 2cp + (0 or 1)
      float* dst = part + static_cast<int64_t>(2 * pp + g) * CW +
                   (static_cast<int64_t>(chunk) * 64 + 2 * cp) * W;
#pragma unroll
      for (int k = 0; k < W; ++k) {
        dst[k] = sum[2 * k];
        dst[W + k] = sum[2 * k + 1];
      }
    }
    }
  }
  __syncthreads();
}

template <int W, bool BWD, bool RES>
struct StKernelTag {};

// Parts per chunk: the fewest waves times (tiles per CTA + a CTA's fixed
// cost, about kStCtaCost tiles: start-up, pipeline fill and drain, the dw
// sums), CTAs beyond one per SM running as further waves; at least one
// tile per part.  (Without the fixed cost the model chose 32 parts at
// C = 6144, 3072 CTAs of 4 tiles: 142 us under the profiler.)
constexpr double kStCtaCost = 4.0;

int st_parts(int64_t nchunks, int64_t ntl, int sms) {
  int best = 1;
  double bcost = -1;
  for (int64_t p = 1; p <= std::min<int64_t>(ntl, 64); ++p) {
    const double waves = std::ceil(static_cast<double>(nchunks * p) / sms);
    const double cost = waves * (std::ceil(static_cast<double>(ntl) / p) + kStCtaCost);
    if (bcost < 0 || cost < bcost - 1e-9) {
      bcost = cost;
      best = static_cast<int>(p);
    }
  }
  return best;
}

// out = y (forward) or dx (backward); dy and part only in the backward.
template <int W, bool BWD, bool RES>
cudaError_t st_tma_launch(const void* x, const void* w, const void* dy, void* out, float* part,
                          const Shape& s, int P, cudaStream_t st) {
  using L = StLayout<W, BWD>;
  CUtensorMap tx, tdy, tout;
  if (!make_tmap_3d(&tx, x, true, s.C, s.T, s.B, 64, L::XROWS, 128) ||
      !make_tmap_3d(&tout, out, true, s.C, s.T, s.B, 64, kStBM, 128))
    return cudaErrorInvalidValue;
  if constexpr (BWD) {
    if (!make_tmap_3d(&tdy, dy, true, s.C, s.T, s.B, 64, L::XROWS, 128))
      return cudaErrorInvalidValue;
  } else {
    tdy = tx;
  }
  const int ntiles = static_cast<int>((s.T + kStBM - 1) / kStBM);
  const int ntl = static_cast<int>(s.B * ntiles);
  const int64_t nchunks = s.C / 64;
  auto kern = st_tma<W, BWD, RES>;
  cudaError_t e = set_smem<StKernelTag<W, BWD, RES>>(kern, L::TOTAL);
  if (e != cudaSuccess) return e;
  kern<<<static_cast<unsigned>(nchunks * P), kStThreads, L::TOTAL, st>>>(
      tx, tdy, tout, static_cast<const __nv_bfloat16*>(w), part, ntl, ntiles, P, s.C * s.W);
  return cudaGetLastError();
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

// The TMA-staged kernels' parts per chunk for this shape, 0 if they do not
// apply (fp32, C not a multiple of 64, T or the tile count beyond their
// 32-bit indices, or, in the backward, more partial sums than the
// workspace holds).
int st_tma_parts(const Shape& s, bool bwd) {
  if (!s.bf16 || s.C % 64 != 0 || s.W > 4 || s.T >= (int64_t(1) << 30)) return 0;
  const int64_t ntl = s.B * ((s.T + kStBM - 1) / kStBM);
  if (ntl >= (int64_t(1) << 30)) return 0;
  const int sms = sm_count();
  if (sms <= 0) return 0;
  const int P = st_parts(s.C / 64, ntl, sms);
  if (s.C / 64 * P >= (int64_t(1) << 31)) return 0;
  return !bwd || 2 * P <= max_ranges(s) ? P : 0;
}

template <typename T>
cudaError_t fwd_t(const void* x, const void* w, void* y, const Shape& s, cudaStream_t st) {
  if (const int P = st_tma_parts(s, false); P > 0) {
    cudaError_t e = cudaSuccess;
    DSC_ST_W_SWITCH(s.W, {
      e = s.residual ? st_tma_launch<W_, false, true>(x, w, nullptr, y, nullptr, s, P, st)
                     : st_tma_launch<W_, false, false>(x, w, nullptr, y, nullptr, s, P, st);
    })
    return e;
  }
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
  if (const int P = st_tma_parts(s, true); P > 0) {
    cudaError_t e = cudaSuccess;
    DSC_ST_W_SWITCH(s.W, {
      e = s.residual ? st_tma_launch<W_, true, true>(x, w, dy, dx, part, s, P, st)
                     : st_tma_launch<W_, true, false>(x, w, dy, dx, part, s, P, st);
    })
    if (e != cudaSuccess) return e;
    const int64_t n = s.C * s.W;
    const unsigned blocks = static_cast<unsigned>((n / 4 + 31) / 32);
    static_dw_reduce<T><<<blocks, kRedSlices * 32, 0, st>>>(part, static_cast<T*>(dw), n, 2 * P);
    return cudaGetLastError();
  }
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

cudaError_t static_tma_error(unsigned int* out, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_st_error, sizeof(unsigned int));
  if (e != cudaSuccess || !reset) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_st_error, &zero, sizeof(unsigned int));
}

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

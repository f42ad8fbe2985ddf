// lowrank_simt.cu -- low-rank fused Dynamic Short Convolution on the CUDA
// cores (fp32 FMA), forward and backward.
//
// The filter of token t is w(t) = z_t U, z [B,T,R], U [R, G*W] with column
// j = g*W + k ("Technische Samenvatting: Dynamische Korte Convoluties
// Verbeteren Transformers", Parametrisatie item 1; Efficiente
// Trainingsimplementatie: Fused Low-Rank Kernel).  The kernels form the W
// taps of each (token, channel) in fp32 registers from z_t and the
// register-resident column block of U and apply them at once; w never
// touches memory.
//
// Backward (chain rule of the forward):
//   dx as in the head-wise backward, with the regenerated taps;
//   dw[t,g,k] = sum_{c in g} dy[t,c] x[t-k,c]   (on-chip only)
//   dz[t,r]   = sum_j dw[t,j] U[r,j]            (reduction over channels)
//   dU[r,j]   = sum_t z[t,r] dw[t,j]            (reduction over all tokens)
// The grid is (channel slices of 128) x (token splits).  Each CTA reduces
// its dz contribution over its 128 channels with a warp reduce-scatter and
// shared memory and writes one fp32 partial per (slice, token); each thread
// keeps its dU column block in registers over the whole split and writes
// one fp32 partial per (split, r, j).  A second kernel adds the partials in
// a fixed order, so results are reproducible bit for bit.
//
// One thread owns one channel: the R x W block of U it needs stays in
// registers, z rows are broadcast from shared memory.  Work per (token,
// channel) is R*W FMAs forward and 3*R*W backward.
#include <algorithm>

#include "dsc_common.cuh"
#include "dsc_internal.h"

namespace dsc {
namespace {

constexpr int kThreads = 128;   // channels per CTA
constexpr int kFwdTile = 64;    // tokens per forward CTA
constexpr int kChunk = 32;      // tokens per backward staging chunk

// Warp reduce-scatter of RT values: returns the sum over the 32 lanes of
// v[r] with r = lane >> (5 - log2 RT).  RT shuffles instead of 5 RT.
template <int RT>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[RT], int lane) {
  constexpr int LOG2RT = RT == 32 ? 5 : RT == 16 ? 4 : RT == 8 ? 3 : -1;
  static_assert(LOG2RT > 0, "RT must be 8, 16 or 32");
#pragma unroll
  for (int lvl = 0; lvl < LOG2RT; ++lvl) {
    const int off = 16 >> lvl;
    const int half = RT >> (lvl + 1);
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < RT / 2; ++i) {
      if (i < half) {
        const float keep = upper ? v[half + i] : v[i];
        const float send = upper ? v[i] : v[half + i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
      }
    }
  }
#pragma unroll
  for (int off = (1 << (5 - LOG2RT)) >> 1; off >= 1; off >>= 1)
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
  return v[0];
}

// ------------------------------------------------------------ forward ----

template <typename T, int W, int RT>
__global__ void __launch_bounds__(kThreads)
lr_fwd_simt(const T* __restrict__ x, const T* __restrict__ z, const T* __restrict__ U,
            T* __restrict__ y, int64_t Tlen, int64_t C, int64_t H, int R, int residual,
            int64_t ncb, int64_t ntt) {
  __shared__ float zs[kFwdTile][RT];
  const int tid = threadIdx.x;
  // one-dimensional grid over (b, token tile, channel block), channel block fastest
  const int64_t cb = blockIdx.x % ncb;
  const int64_t tt_ = (blockIdx.x / ncb) % ntt;
  const int64_t b = blockIdx.x / (ncb * ntt);
  const int64_t c = cb * kThreads + tid;
  const int64_t t0 = tt_ * kFwdTile;
  const int64_t t1 = std::min<int64_t>(t0 + kFwdTile, Tlen);
  const int64_t G = C / H;
  for (int i = tid; i < kFwdTile * RT; i += kThreads) {
    const int tt = i / RT, r = i % RT;
    zs[tt][r] = (r < R && t0 + tt < t1) ? to_f32(z[(b * Tlen + t0 + tt) * R + r]) : 0.f;
  }
  __syncthreads();
  if (c >= C) return;
  const int64_t g = c / H;
  float u[RT][W];
#pragma unroll
  for (int r = 0; r < RT; ++r)
#pragma unroll
    for (int k = 0; k < W; ++k) u[r][k] = r < R ? to_f32(U[(int64_t)r * G * W + g * W + k]) : 0.f;

  const T* xc = x + b * Tlen * C + c;
  T* yc = y + b * Tlen * C + c;
  float win[W > 1 ? W - 1 : 1];
#pragma unroll
  for (int j = 0; j < W - 1; ++j) win[j] = (t0 - 1 - j >= 0) ? to_f32(xc[(t0 - 1 - j) * C]) : 0.f;

  for (int64_t t = t0; t < t1; ++t) {
    const float xv = to_f32(xc[t * C]);
    const float* zr = zs[t - t0];
    float wk[W];
#pragma unroll
    for (int k = 0; k < W; ++k) wk[k] = 0.f;
#pragma unroll
    for (int r = 0; r < RT; ++r) {
      const float zz = zr[r];
#pragma unroll
      for (int k = 0; k < W; ++k) wk[k] = fmaf(zz, u[r][k], wk[k]);
    }
    float a = residual ? xv : 0.f;
    a = fmaf(wk[0], xv, a);
#pragma unroll
    for (int k = 1; k < W; ++k) a = fmaf(wk[k], win[k - 1], a);
    yc[t * C] = from_f32<T>(a);
#pragma unroll
    for (int j = W - 2; j > 0; --j) win[j] = win[j - 1];
    if constexpr (W > 1) win[0] = xv;
  }
}

// ----------------------------------------------------------- backward ----

template <typename T, int W, int RT>
__global__ void __launch_bounds__(kThreads)
lr_bwd_simt(const T* __restrict__ x, const T* __restrict__ z, const T* __restrict__ U,
            const T* __restrict__ dy, T* __restrict__ dx, float* __restrict__ dz_part,
            float* __restrict__ dU_part, int64_t N, int64_t Tlen, int64_t C, int64_t H,
            int R, int residual, int64_t split_len) {
  __shared__ float zs[kChunk][RT];
  __shared__ float red[kChunk][kThreads / 32][RT];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t c = (int64_t)blockIdx.x * kThreads + tid;
  const bool active = c < C;
  const int64_t slice = blockIdx.x, split = blockIdx.y;
  const int64_t n0 = split * split_len;
  const int64_t n1 = std::min<int64_t>(n0 + split_len, N);
  const int64_t G = C / H;
  const int64_t g = active ? c / H : 0;
  const int hl = (int)H;                          // lanes per group (power of two <= 32)
  const bool leader = active && ((c % H) == 0);

  float u[RT][W], dUa[RT][W];
#pragma unroll
  for (int r = 0; r < RT; ++r)
#pragma unroll
    for (int k = 0; k < W; ++k) {
      u[r][k] = (active && r < R) ? to_f32(U[(int64_t)r * G * W + g * W + k]) : 0.f;
      dUa[r][k] = 0.f;
    }

  float xwin[W > 1 ? W - 1 : 1];                  // x[n-1-j] of this channel
#pragma unroll
  for (int j = 0; j < W - 1; ++j) {
    const int64_t n = n0 - 1 - j;
    xwin[j] = (active && n >= 0) ? to_f32(x[n * C + c]) : 0.f;
  }
  float acc[W];                                   // acc[j] = dx row n-(W-1)+j
#pragma unroll
  for (int j = 0; j < W; ++j) acc[j] = 0.f;

  const int64_t nend = std::min<int64_t>(n1 + W - 1, N);
  for (int64_t cs = n0; cs < nend; cs += kChunk) {
    const int clen = (int)std::min<int64_t>(kChunk, nend - cs);
    for (int i = tid; i < kChunk * RT; i += kThreads) {
      const int tt = i / RT, r = i % RT;
      zs[tt][r] = (r < R && tt < clen) ? to_f32(z[(cs + tt) * R + r]) : 0.f;
    }
    __syncthreads();
    for (int tt = 0; tt < clen; ++tt) {
      const int64_t n = cs + tt;
      const int64_t t = n % Tlen;
      const float g_ = active ? to_f32(dy[n * C + c]) : 0.f;
      // regenerate the taps of token n
      float wk[W];
#pragma unroll
      for (int k = 0; k < W; ++k) wk[k] = 0.f;
#pragma unroll
      for (int r = 0; r < RT; ++r) {
        const float zz = zs[tt][r];
#pragma unroll
        for (int k = 0; k < W; ++k) wk[k] = fmaf(zz, u[r][k], wk[k]);
      }
      // dx scatter: dy[n] reaches rows n-k of the same sequence through tap k
      acc[W - 1] = (residual && n < n1) ? g_ : 0.f;
#pragma unroll
      for (int k = 0; k < W; ++k)
        if (t - k >= 0) acc[W - 1 - k] = fmaf(wk[k], g_, acc[W - 1 - k]);
      if (n < n1) {
        const float xv = active ? to_f32(x[n * C + c]) : 0.f;
        float dw[W];
        dw[0] = g_ * xv;
#pragma unroll
        for (int k = 1; k < W; ++k) dw[k] = (t - k >= 0) ? g_ * xwin[k - 1] : 0.f;
        for (int off = 1; off < hl; off <<= 1)
#pragma unroll
          for (int k = 0; k < W; ++k) dw[k] += __shfl_xor_sync(0xffffffffu, dw[k], off);
        if (!leader) {
#pragma unroll
          for (int k = 0; k < W; ++k) dw[k] = 0.f;
        }
        float q[RT];
#pragma unroll
        for (int r = 0; r < RT; ++r) {
          float s = 0.f;
#pragma unroll
          for (int k = 0; k < W; ++k) s = fmaf(dw[k], u[r][k], s);
          q[r] = s;
          const float zz = zs[tt][r];
#pragma unroll
          for (int k = 0; k < W; ++k) dUa[r][k] = fmaf(zz, dw[k], dUa[r][k]);
        }
        const float sum = warp_reduce_scatter<RT>(q, lane);
        constexpr int rep = 32 / RT;               // lanes holding the same r
        if ((lane % rep) == 0) red[tt][warp][lane / rep] = sum;
#pragma unroll
        for (int j = W - 2; j > 0; --j) xwin[j] = xwin[j - 1];
        if constexpr (W > 1) xwin[0] = xv;
      }
      const int64_t s_row = n - (W - 1);
      if (active && s_row >= n0) dx[s_row * C + c] = from_f32<T>(acc[0]);
#pragma unroll
      for (int j = 0; j < W - 1; ++j) acc[j] = acc[j + 1];
    }
    __syncthreads();
    // dz partial of this slice for the chunk's tokens inside the split
    const int nd = (int)std::max<int64_t>(0, std::min<int64_t>(clen, n1 - cs));
    for (int i = tid; i < nd * R; i += kThreads) {
      const int tt = i / R, r = i % R;
      float s = 0.f;
#pragma unroll
      for (int wp = 0; wp < kThreads / 32; ++wp) s += red[tt][wp][r];
      dz_part[(slice * N + cs + tt) * R + r] = s;
    }
    __syncthreads();
  }
  // When the split ends the data, the loop stops at N and the last W-1 rows
  // are still in the window; they are complete, so retire them here.
  if (nend == N) {
#pragma unroll
    for (int j = 0; j < W - 1; ++j) {
      const int64_t s_row = N - (W - 1) + j;
      if (active && s_row >= n0 && s_row < n1) dx[s_row * C + c] = from_f32<T>(acc[j]);
    }
  }
  if (leader) {
#pragma unroll
    for (int r = 0; r < RT; ++r)
      if (r < R)
#pragma unroll
        for (int k = 0; k < W; ++k)
          dU_part[(split * R + r) * G * W + g * W + k] = dUa[r][k];
  }
}

// dz = sum over slices of dz_part, dU = sum over splits of dU_part, in that
// fixed order; rounded once to the I/O type.
template <typename T>
__global__ void lr_reduce(const float* __restrict__ dz_part, const float* __restrict__ dU_part,
                          T* __restrict__ dz, T* __restrict__ dU, int64_t nz, int64_t S,
                          int64_t nU, int64_t P) {
  const int64_t total = nz + nU;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    float s = 0.f;
    if (i < nz) {
      for (int64_t k = 0; k < S; ++k) s += dz_part[k * nz + i];
      dz[i] = from_f32<T>(s);
    } else {
      const int64_t j = i - nz;
      for (int64_t k = 0; k < P; ++k) s += dU_part[k * nU + j];
      dU[j] = from_f32<T>(s);
    }
  }
}

// ------------------------------------------------------------ planning ----

struct BwdPlan {
  int64_t S, P, split_len;
  size_t dz_bytes, dU_bytes;
};

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

BwdPlan plan_bwd(const Shape& s) {
  BwdPlan p{};
  p.S = (s.C + kThreads - 1) / kThreads;
  const int64_t N = s.N();
  int64_t P = std::max<int64_t>(1, (4 * 148 + p.S - 1) / p.S);
  P = std::min<int64_t>(P, std::max<int64_t>(1, N / 64));
  p.split_len = (N + P - 1) / P;
  p.P = (N + p.split_len - 1) / p.split_len;
  p.dz_bytes = align256((size_t)p.S * N * s.R * sizeof(float));
  p.dU_bytes = align256((size_t)p.P * s.R * s.G() * s.W * sizeof(float));
  return p;
}

#define DSC_W_SWITCH(Wv, ...)                                         \
  switch (Wv) {                                                       \
    case 1: { constexpr int W_ = 1; __VA_ARGS__; } break;             \
    case 2: { constexpr int W_ = 2; __VA_ARGS__; } break;             \
    case 3: { constexpr int W_ = 3; __VA_ARGS__; } break;             \
    default: { constexpr int W_ = 4; __VA_ARGS__; } break;            \
  }

#define DSC_RT_SWITCH(R, ...)                                         \
  if ((R) <= 16) { constexpr int RT_ = 16; __VA_ARGS__; }             \
  else { constexpr int RT_ = 32; __VA_ARGS__; }

template <typename T>
cudaError_t fwd_t(const void* x, const void* z, const void* U, void* y, const Shape& s,
                  cudaStream_t st) {
  const int64_t ncb = (s.C + kThreads - 1) / kThreads;
  const int64_t ntt = (s.T + kFwdTile - 1) / kFwdTile;
  if (ncb * ntt * s.B > (int64_t(1) << 31) - 1) return cudaErrorInvalidConfiguration;
  const unsigned grid = (unsigned)(ncb * ntt * s.B);
  DSC_W_SWITCH(s.W, DSC_RT_SWITCH(s.R, {
    lr_fwd_simt<T, W_, RT_><<<grid, kThreads, 0, st>>>(
        (const T*)x, (const T*)z, (const T*)U, (T*)y, s.T, s.C, s.H, (int)s.R, s.residual,
        ncb, ntt);
  }))
  return cudaGetLastError();
}

template <typename T>
cudaError_t bwd_t(const void* x, const void* z, const void* U, const void* dy, void* dx,
                  void* dz, void* dU, void* ws, const Shape& s, cudaStream_t st) {
  const BwdPlan p = plan_bwd(s);
  float* dz_part = (float*)ws;
  float* dU_part = (float*)((char*)ws + p.dz_bytes);
  dim3 grid((unsigned)p.S, (unsigned)p.P);
  DSC_W_SWITCH(s.W, DSC_RT_SWITCH(s.R, {
    lr_bwd_simt<T, W_, RT_><<<grid, kThreads, 0, st>>>(
        (const T*)x, (const T*)z, (const T*)U, (const T*)dy, (T*)dx, dz_part, dU_part,
        s.N(), s.T, s.C, s.H, (int)s.R, s.residual, p.split_len);
  }))
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t nz = s.N() * s.R, nU = s.R * s.G() * s.W;
  const int blocks = (int)std::min<int64_t>((nz + nU + 255) / 256, 148 * 8);
  lr_reduce<T><<<blocks, 256, 0, st>>>(dz_part, dU_part, (T*)dz, (T*)dU, nz, p.S, nU, p.P);
  return cudaGetLastError();
}

}  // namespace

bool lowrank_supported(const Shape& s) {
  return s.R >= 1 && s.R <= 32 && s.H >= 1 && s.H <= 32 && (s.H & (s.H - 1)) == 0;
}

cudaError_t lowrank_fwd(const void* x, const void* z, const void* U, void* y,
                        const Shape& s, cudaStream_t st) {
  return s.bf16 ? fwd_t<__nv_bfloat16>(x, z, U, y, s, st) : fwd_t<float>(x, z, U, y, s, st);
}

size_t lowrank_bwd_workspace(const Shape& s) {
  const BwdPlan p = plan_bwd(s);
  return p.dz_bytes + p.dU_bytes;
}

cudaError_t lowrank_bwd(const void* x, const void* z, const void* U, const void* dy,
                        void* dx, void* dz, void* dU, void* ws, const Shape& s,
                        cudaStream_t st) {
  return s.bf16 ? bwd_t<__nv_bfloat16>(x, z, U, dy, dx, dz, dU, ws, s, st)
                : bwd_t<float>(x, z, U, dy, dx, dz, dU, ws, s, st);
}

}  // namespace dsc

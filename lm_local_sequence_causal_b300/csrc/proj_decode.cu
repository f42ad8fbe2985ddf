// proj_decode.cu -- decode step of Dynamic Short Convolutions merged with the
// projection that produces its input (inference, one new token per sequence).
//
// "Dynamic Short Convolutions: The 'Locality Bias' Transformers Were
// Missing", Limitations: for inference the convolution is to be merged into
// the matmul that precedes it.  In a decode step that matmul projects the
// new token's hidden state, x_t = h_t Wp^T (h [B, D]; Wp [C, D] as a linear
// layer stores its weight), and the step after it is the decode step of
// decode.cu:
//   y[b,c] = res*x[b,c] + w[b,g(c),0] x[b,c] + sum_{k>=1} w[b,g(c),k] state[b,k-1,c]
//   state[b,0,c] <- x[b,c],  state[b,j,c] <- state[b,j-1,c]
// Merged, x_t never goes to memory: the kernel rounds it once to the I/O type
// (the value the separate projection would store) and applies the step.
//
// At decode sizes the projection is a weight stream: Wp (C*D elements) is
// read once and everything else is small.  A warp owns RG = 4 output
// channels (rows of Wp).  Its lanes walk D in 16-byte pieces (lane l takes
// pieces l, l+32, ...), so each row is read in contiguous 512-byte runs, and
// every lane keeps fp32 partial sums (pairs, for the packed FMA) of its 4
// rows x NB sequences (NB = 1, 2, 4 or 8 by the batch), multiplying each Wp
// piece into the NB rows of h (which come from L1: every warp reads the same
// h).  A butterfly over the lane bits above 4*NB and a reduce-scatter over
// those below leave lane l < 4*NB with the finished x of row l / NB,
// sequence l % NB, and that lane runs the decode step for its (b, c).
// Batches above 8 go in blocks of 8; a warp re-reads its Wp rows (from L2)
// for each block.  This CUDA-core kernel serves fp32 and bf16 batches of up
// to 4 sequences; bf16 batches of 5 to 16 take the warp-level tensor-core
// kernel below, and larger ones the tcgen05 kernel of proj_decode_tc.cu
// (D split over a cluster, partial sums through distributed shared memory).
#include <cuda_bf16.h>

#include <algorithm>

#include "dsc_common.cuh"
#include "dsc_internal.h"

namespace dsc {
namespace {

constexpr int kPdThreads = 128;
constexpr int RG = 4;        // output channels per warp item

// A 16-byte piece as fp32 pairs: bf16 -> 4 pairs (elements 2i, 2i+1), fp32 -> 2 pairs.
template <typename T>
struct Pairs {
  static constexpr int N = Vec<T>::N / 2;
};

template <typename T>
__device__ __forceinline__ void to_pairs(const uint4& u, float2 (&p)[Pairs<T>::N]) {
  if constexpr (sizeof(T) == 2) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      p[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
  } else {
    p[0] = make_float2(__uint_as_float(u.x), __uint_as_float(u.y));
    p[1] = make_float2(__uint_as_float(u.z), __uint_as_float(u.w));
  }
}

// 16-byte load of streamed data (Wp, read once) that does not allocate in
// L1, so the Wp stream does not evict h, which every warp re-reads from L1.
__device__ __forceinline__ uint4 ldg16_stream(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

// One step of the warp reduce-scatter: lanes with bit HALF set keep the
// upper half of their 2*HALF values and send the lower half to the partner
// lane (lane ^ HALF), which does the opposite; each adds what it receives.
template <int NV, int HALF>
__device__ __forceinline__ void reduce_scatter_step(float (&v)[NV], int lane) {
  const bool hi = (lane & HALF) != 0;
#pragma unroll
  for (int j = 0; j < HALF; ++j) {
    const float send = hi ? v[j] : v[j + HALF];
    const float keep = hi ? v[j + HALF] : v[j];
    v[j] = keep + __shfl_xor_sync(0xffffffffu, send, HALF);
  }
}

// Warp-wide sums of NV values (a power of two <= 32) per lane: afterwards
// v[0] of lane l is the sum over all lanes of value l % NV.
template <int NV>
__device__ __forceinline__ void warp_sum_scatter(float (&v)[NV], int lane) {
#pragma unroll
  for (int m = 16; m >= NV; m >>= 1)
#pragma unroll
    for (int j = 0; j < NV; ++j) v[j] += __shfl_xor_sync(0xffffffffu, v[j], m);
  if constexpr (NV >= 32) reduce_scatter_step<NV, 16>(v, lane);
  if constexpr (NV >= 16) reduce_scatter_step<NV, 8>(v, lane);
  if constexpr (NV >= 8) reduce_scatter_step<NV, 4>(v, lane);
  if constexpr (NV >= 4) reduce_scatter_step<NV, 2>(v, lane);
  if constexpr (NV >= 2) reduce_scatter_step<NV, 1>(v, lane);
}

template <typename T, int W, bool LOWRANK, int NB>
__global__ void __launch_bounds__(kPdThreads)
proj_decode_kernel(const T* __restrict__ h, const T* __restrict__ Wp, const T* __restrict__ w,
                   const T* __restrict__ z, const T* __restrict__ U, T* __restrict__ state,
                   T* __restrict__ y, int B, int D, int C, int H, int R, int residual) {
  constexpr int V = Vec<T>::N;             // elements per 16-byte piece
  constexpr int NP = Pairs<T>::N;
  constexpr int NV = RG * NB;              // finished values per warp item and block
  // Pieces of each row a lane has in flight at once (more when the
  // accumulators are few).
  constexpr int UF = NB <= 2 ? 4 : 2;
  const int lane = threadIdx.x & 31;
  const long long warp0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const int nitems = (C + RG - 1) / RG;
  const int npieces = D / V;
  for (long long item = warp0; item < nitems; item += nwarps) {
    const int c0 = static_cast<int>(item) * RG;
    const int nr = min(RG, C - c0);
    for (int b0 = 0; b0 < B; b0 += NB) {
      const int nb = min(NB, B - b0);
      // This lane's (b, c) after the reduction, and its step operands,
      // fetched now so their latency hides behind the Wp stream.
      const int r = lane / NB, b = lane % NB;
      const bool mine = lane < NV && r < nr && b < nb;
      const int c = c0 + r;
      const int64_t bg = b0 + b;
      const int64_t g = mine ? c / H : 0;
      T tap_raw[LOWRANK ? 1 : W];
      T sr[W > 1 ? W - 1 : 1];
      if (mine) {
        if constexpr (!LOWRANK) {
          const T* wb = w + (bg * (C / H) + g) * W;
#pragma unroll
          for (int k = 0; k < W; ++k) tap_raw[k] = wb[k];
        }
        if constexpr (W > 1) {
          const T* sp = state + bg * (W - 1) * C + c;
#pragma unroll
          for (int j = 0; j < W - 1; ++j) sr[j] = sp[static_cast<int64_t>(j) * C];
        }
      }
      float2 acc[RG][NB];
#pragma unroll
      for (int rr = 0; rr < RG; ++rr)
#pragma unroll
        for (int bb = 0; bb < NB; ++bb) acc[rr][bb] = make_float2(0.f, 0.f);
      const T* hb = h + static_cast<int64_t>(b0) * D;
      for (int p0 = lane; p0 < npieces; p0 += 32 * UF) {
        uint4 raw[UF][RG];
#pragma unroll
        for (int u = 0; u < UF; ++u)
#pragma unroll
          for (int rr = 0; rr < RG; ++rr) {
            const int p = p0 + 32 * u;
            raw[u][rr] = (p < npieces && rr < nr)
                             ? ldg16_stream(Wp + static_cast<int64_t>(c0 + rr) * D + p * V)
                             : make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
        for (int u = 0; u < UF; ++u) {
          const int p = p0 + 32 * u;
          if (p >= npieces) break;
          uint4 hraw[NB];
#pragma unroll
          for (int bb = 0; bb < NB; ++bb)
            hraw[bb] = bb < nb ? ldg16(hb + static_cast<int64_t>(bb) * D + p * V)
                               : make_uint4(0u, 0u, 0u, 0u);
          float2 wv[RG][NP];
#pragma unroll
          for (int rr = 0; rr < RG; ++rr) to_pairs<T>(raw[u][rr], wv[rr]);
#pragma unroll
          for (int bb = 0; bb < NB; ++bb) {
            float2 hv[NP];
            to_pairs<T>(hraw[bb], hv);
#pragma unroll
            for (int rr = 0; rr < RG; ++rr)
#pragma unroll
              for (int i = 0; i < NP; ++i) acc[rr][bb] = __ffma2_rn(wv[rr][i], hv[i], acc[rr][bb]);
          }
        }
      }
      float v[NV];
#pragma unroll
      for (int rr = 0; rr < RG; ++rr)
#pragma unroll
        for (int bb = 0; bb < NB; ++bb) v[rr * NB + bb] = acc[rr][bb].x + acc[rr][bb].y;
      warp_sum_scatter<NV>(v, lane);
      // ---- the decode step of (b, c) = (b0 + lane % NB, c0 + lane / NB)
      if (!mine) continue;
      const T xs = from_f32<T>(v[0]);      // x_t as the projection would store it
      const float xf = to_f32(xs);
      float taps[W];
      if constexpr (!LOWRANK) {
#pragma unroll
        for (int k = 0; k < W; ++k) taps[k] = to_f32(tap_raw[k]);
      } else {
        const int64_t GW = static_cast<int64_t>(C / H) * W;
#pragma unroll
        for (int k = 0; k < W; ++k) taps[k] = 0.f;
#pragma unroll 8
        for (int q = 0; q < R; ++q) {
          const float zq = to_f32(z[bg * R + q]);
          const T* uq = U + q * GW + g * W;
#pragma unroll
          for (int k = 0; k < W; ++k) taps[k] = fmaf(zq, to_f32(uq[k]), taps[k]);
        }
      }
      float a = residual ? xf : 0.f;
      a = fmaf(taps[0], xf, a);
      if constexpr (W > 1) {
        T* sp = state + bg * (W - 1) * C + c;
#pragma unroll
        for (int k = 1; k < W; ++k) a = fmaf(taps[k], to_f32(sr[k - 1]), a);
        // the state moves down one row; x_t becomes row 0 (exact copies)
#pragma unroll
        for (int j = W - 2; j >= 1; --j) sp[static_cast<int64_t>(j) * C] = sr[j - 1];
        sp[0] = xs;
      }
      y[bg * C + c] = from_f32<T>(a);
    }
  }
}

// ---------------------------------------------------------------------------
// bf16: the projection on the warp-level tensor-core MMA (mma.sync m16n8k16,
// bf16 in, fp32 accumulate).  A CTA owns 8 output channels (the MMA's N) and
// its 4 warps split D: warp w takes the 32-element chunks w, w+4, w+8, ...
// Lane (g, q) = (lane / 4, lane % 4) loads 16 bytes of Wp row c0 + g at
// offset 8q of a chunk and 16 bytes of h rows g and g+8 of a 16-sequence
// block (the MMA's M) at the same offset.  The contraction index may be
// ordered freely as long as both operands agree; here K slots 2q, 2q+1,
// 2q+8, 2q+9 of MMA s (s = 0, 1) hold elements 8q + 4s + 0..3 of the chunk,
// so each lane's 16-byte loads are its A and B fragments as they are.  The
// four warps' partial sums meet in shared memory (added in warp order), and
// thread t runs the decode step of sequence t / 8, channel c0 + t % 8.
// Wp is read once per pass of up to 16*MB sequences (later passes from L2).
// The tcgen05 MMA needs M >= 64 rows per CTA, i.e. 128 rows of Wp on M and
// 48 CTAs at C = 6144, too few SMs to stream Wp at HBM speed without a
// cross-CTA split of D; proj_decode_tc.cu makes that split for batches of
// more than 16 sequences, and up to 16 this kernel, whose CTAs own 8 rows
// and need no cross-CTA reduction, is as fast.

constexpr int kMmaThreads = 128;   // 4 warps split D
constexpr int kMmaN = 8;           // output channels per CTA
constexpr int kSeg = 8;            // chunks of a warp's Wp loads in flight

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int W, bool LOWRANK, int MB>
__global__ void __launch_bounds__(kMmaThreads)
proj_decode_mma(const __nv_bfloat16* __restrict__ h, const __nv_bfloat16* __restrict__ Wp,
                const __nv_bfloat16* __restrict__ w, const __nv_bfloat16* __restrict__ z,
                const __nv_bfloat16* __restrict__ U, __nv_bfloat16* __restrict__ state,
                __nv_bfloat16* __restrict__ y, int B, int D, int C, int H, int R,
                int residual) {
  using T = __nv_bfloat16;
  __shared__ float part[4][MB][16][kMmaN];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  const int nchunks = (D + 31) / 32;
  const int nblk = (C + kMmaN - 1) / kMmaN;
  // the (sequence, channel) of this thread's decode steps
  const int m = threadIdx.x / kMmaN, n = threadIdx.x % kMmaN;
  for (int cb = blockIdx.x; cb < nblk; cb += gridDim.x) {
    const int c0 = cb * kMmaN;
    const bool row_ok = c0 + g < C;
    const T* wrow = Wp + static_cast<int64_t>(c0 + g) * D;
    const int c = c0 + n;
    for (int b0 = 0; b0 < B; b0 += 16 * MB) {
      // Step operands of this thread, fetched before the projection.
      T tap_raw[MB][LOWRANK ? 1 : W];
      T sr[MB][W > 1 ? W - 1 : 1];
#pragma unroll
      for (int mb = 0; mb < MB; ++mb) {
        const int64_t bg = b0 + 16 * mb + m;
        if (bg < B && c < C) {
          if constexpr (!LOWRANK) {
            const T* wb = w + (bg * (C / H) + c / H) * W;
#pragma unroll
            for (int k = 0; k < W; ++k) tap_raw[mb][k] = wb[k];
          }
          if constexpr (W > 1) {
            const T* sp = state + bg * (W - 1) * C + c;
#pragma unroll
            for (int j = 0; j < W - 1; ++j) sr[mb][j] = sp[static_cast<int64_t>(j) * C];
          }
        }
      }
      float acc[MB][4];
#pragma unroll
      for (int mb = 0; mb < MB; ++mb)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[mb][i] = 0.f;
      for (int j0 = warp; j0 < nchunks; j0 += 4 * kSeg) {
        uint4 wq[kSeg];
#pragma unroll
        for (int sg = 0; sg < kSeg; ++sg) {
          const int d = 32 * (j0 + 4 * sg) + 8 * q;
          wq[sg] = (row_ok && d < D) ? ldg16_stream(wrow + d) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int mb = 0; mb < MB; ++mb) {
          const int r0 = b0 + 16 * mb + g, r1 = r0 + 8;
          const T* h0p = h + static_cast<int64_t>(r0) * D;
          const T* h1p = h + static_cast<int64_t>(r1) * D;
#pragma unroll
          for (int sg = 0; sg < kSeg; ++sg) {
            if (j0 + 4 * sg >= nchunks) break;              // the same for the whole warp
            const int d = 32 * (j0 + 4 * sg) + 8 * q;
            const uint4 h0 = (r0 < B && d < D) ? ldg16(h0p + d) : make_uint4(0u, 0u, 0u, 0u);
            const uint4 h1 = (r1 < B && d < D) ? ldg16(h1p + d) : make_uint4(0u, 0u, 0u, 0u);
            mma_bf16_16816(acc[mb], h0.x, h1.x, h0.y, h1.y, wq[sg].x, wq[sg].y);
            mma_bf16_16816(acc[mb], h0.z, h1.z, h0.w, h1.w, wq[sg].z, wq[sg].w);
          }
        }
      }
      // D fragment: (row g, cols 2q, 2q+1) and (row g+8, cols 2q, 2q+1)
#pragma unroll
      for (int mb = 0; mb < MB; ++mb) {
        part[warp][mb][g][2 * q] = acc[mb][0];
        part[warp][mb][g][2 * q + 1] = acc[mb][1];
        part[warp][mb][g + 8][2 * q] = acc[mb][2];
        part[warp][mb][g + 8][2 * q + 1] = acc[mb][3];
      }
      __syncthreads();
#pragma unroll
      for (int mb = 0; mb < MB; ++mb) {
        const int64_t bg = b0 + 16 * mb + m;
        if (bg >= B || c >= C) continue;
        const float xsum = ((part[0][mb][m][n] + part[1][mb][m][n]) + part[2][mb][m][n]) +
                           part[3][mb][m][n];
        const T xs = from_f32<T>(xsum);    // x_t as the projection would store it
        const float xf = to_f32(xs);
        float taps[W];
        if constexpr (!LOWRANK) {
#pragma unroll
          for (int k = 0; k < W; ++k) taps[k] = to_f32(tap_raw[mb][k]);
        } else {
          const int64_t GW = static_cast<int64_t>(C / H) * W;
          const int64_t gg = c / H;
#pragma unroll
          for (int k = 0; k < W; ++k) taps[k] = 0.f;
#pragma unroll 8
          for (int rr = 0; rr < R; ++rr) {
            const float zr = to_f32(z[bg * R + rr]);
            const T* ur = U + rr * GW + gg * W;
#pragma unroll
            for (int k = 0; k < W; ++k) taps[k] = fmaf(zr, to_f32(ur[k]), taps[k]);
          }
        }
        float a = residual ? xf : 0.f;
        a = fmaf(taps[0], xf, a);
        if constexpr (W > 1) {
          T* sp = state + bg * (W - 1) * C + c;
#pragma unroll
          for (int k = 1; k < W; ++k) a = fmaf(taps[k], to_f32(sr[mb][k - 1]), a);
#pragma unroll
          for (int j = W - 2; j >= 1; --j) sp[static_cast<int64_t>(j) * C] = sr[mb][j - 1];
          sp[0] = xs;
        }
        y[bg * C + c] = from_f32<T>(a);
      }
      __syncthreads();                       // part is rewritten by the next pass
    }
  }
}

template <bool LOWRANK>
cudaError_t launch_mma(const void* h, const void* Wp, const void* w, const void* z,
                       const void* U, void* state, void* y, const Shape& s, int64_t D,
                       cudaStream_t st) {
  using T = __nv_bfloat16;
  const int64_t nblk = (s.C + kMmaN - 1) / kMmaN;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorNoDevice;
  const unsigned g =
      static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>(nblk, int64_t(sms) * 16)));
  const int B = static_cast<int>(s.B), Di = static_cast<int>(D), C = static_cast<int>(s.C),
            H = static_cast<int>(s.H), R = static_cast<int>(s.R);
  const T* ph = static_cast<const T*>(h);
  const T* pW = static_cast<const T*>(Wp);
  const T* pw = static_cast<const T*>(w);
  const T* pz = static_cast<const T*>(z);
  const T* pU = static_cast<const T*>(U);
  T* ps = static_cast<T*>(state);
  T* py = static_cast<T*>(y);
  // One 16-sequence block per pass: batches of more than 16 sequences take
  // the tcgen05 kernel (proj_decode_tc.cu), so a call here has one pass.
#define DSC_PDM_LAUNCH(Wv, MBv)                                                                 \
  proj_decode_mma<Wv, LOWRANK, MBv><<<g, kMmaThreads, 0, st>>>(ph, pW, pw, pz, pU, ps, py, B, \
                                                              Di, C, H, R, s.residual)
#define DSC_PDM_MB(Wv) DSC_PDM_LAUNCH(Wv, 1)
  switch (s.W) {
    case 1: DSC_PDM_MB(1); break;
    case 2: DSC_PDM_MB(2); break;
    case 3: DSC_PDM_MB(3); break;
    default: DSC_PDM_MB(4); break;
  }
#undef DSC_PDM_MB
#undef DSC_PDM_LAUNCH
  return cudaGetLastError();
}

template <typename T, bool LOWRANK>
cudaError_t launch_t(const void* h, const void* Wp, const void* w, const void* z, const void* U,
                     void* state, void* y, const Shape& s, int64_t D, cudaStream_t st) {
  const int64_t nitems = (s.C + RG - 1) / RG;
  const int64_t warps_per_cta = kPdThreads / 32;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorNoDevice;
  const int64_t grid =
      std::max<int64_t>(1, std::min<int64_t>((nitems + warps_per_cta - 1) / warps_per_cta,
                                             static_cast<int64_t>(sms) * 16));
  const int B = static_cast<int>(s.B), Di = static_cast<int>(D), C = static_cast<int>(s.C),
            H = static_cast<int>(s.H), R = static_cast<int>(s.R);
  const T* ph = static_cast<const T*>(h);
  const T* pW = static_cast<const T*>(Wp);
  const T* pw = static_cast<const T*>(w);
  const T* pz = static_cast<const T*>(z);
  const T* pU = static_cast<const T*>(U);
  T* ps = static_cast<T*>(state);
  T* py = static_cast<T*>(y);
  const unsigned g = static_cast<unsigned>(grid);
  // Sequences per block: the batch rounded up to 1, 2, 4 or 8.
  const int nbt = s.B <= 1 ? 1 : s.B <= 2 ? 2 : s.B <= 4 ? 4 : 8;
#define DSC_PD_LAUNCH(Wv, NBv)                                                              \
  proj_decode_kernel<T, Wv, LOWRANK, NBv><<<g, kPdThreads, 0, st>>>(ph, pW, pw, pz, pU, ps, \
                                                                    py, B, Di, C, H, R,     \
                                                                    s.residual)
#define DSC_PD_NB(Wv)                       \
  switch (nbt) {                            \
    case 1: DSC_PD_LAUNCH(Wv, 1); break;    \
    case 2: DSC_PD_LAUNCH(Wv, 2); break;    \
    case 4: DSC_PD_LAUNCH(Wv, 4); break;    \
    default: DSC_PD_LAUNCH(Wv, 8); break;   \
  }
  switch (s.W) {
    case 1: DSC_PD_NB(1); break;
    case 2: DSC_PD_NB(2); break;
    case 3: DSC_PD_NB(3); break;
    default: DSC_PD_NB(4); break;
  }
#undef DSC_PD_NB
#undef DSC_PD_LAUNCH
  return cudaGetLastError();
}

// bf16 batches up to this size take the CUDA-core kernel: with few
// sequences its packed FMAs are cheap, and its 4 x 4 Wp pieces in flight
// per lane stream Wp faster than the MMA kernel's 8 (measured at D = 2048,
// C = 6144: 8.2 against 10.1 us per step at B = 1, 10.0 against 10.3 at
// B = 4, 16.0 against 10.3 at B = 8).  fp32 always takes it.
constexpr int64_t kSimtMaxB = 4;
// bf16 batches from this size take the tcgen05 kernel of proj_decode_tc.cu
// (measured at D = 2048, C = 6144: 12.7 against 15.0 us per step at B = 17,
// 14.9 against 26.9 at B = 64; at B = 16 the two are even, and the warp-MMA
// kernel's 16-sequence blocks fit that batch exactly).
constexpr int64_t kTcMinB = 17;

}  // namespace

bool headwise_proj_decode_uses_tc(const Shape& s, int64_t D) {
  return s.bf16 && s.B >= kTcMinB && proj_decode_tc_supported(s, D);
}

cudaError_t headwise_proj_decode(const void* h, const void* Wp, const void* w, void* state,
                                 void* y, const Shape& s, int64_t D, cudaStream_t st) {
  if (s.bf16 && s.B >= kTcMinB && proj_decode_tc_supported(s, D))
    return proj_decode_tc(h, Wp, w, nullptr, nullptr, state, y, s, D, false, st);
  if (s.bf16 && s.B > kSimtMaxB)
    return launch_mma<false>(h, Wp, w, nullptr, nullptr, state, y, s, D, st);
  if (s.bf16)
    return launch_t<__nv_bfloat16, false>(h, Wp, w, nullptr, nullptr, state, y, s, D, st);
  return launch_t<float, false>(h, Wp, w, nullptr, nullptr, state, y, s, D, st);
}

cudaError_t lowrank_proj_decode(const void* h, const void* Wp, const void* z, const void* U,
                                void* state, void* y, const Shape& s, int64_t D,
                                cudaStream_t st) {
  if (s.bf16 && s.B >= kTcMinB && proj_decode_tc_supported(s, D))
    return proj_decode_tc(h, Wp, nullptr, z, U, state, y, s, D, true, st);
  if (s.bf16 && s.B > kSimtMaxB)
    return launch_mma<true>(h, Wp, nullptr, z, U, state, y, s, D, st);
  if (s.bf16) return launch_t<__nv_bfloat16, true>(h, Wp, nullptr, z, U, state, y, s, D, st);
  return launch_t<float, true>(h, Wp, nullptr, z, U, state, y, s, D, st);
}

}  // namespace dsc

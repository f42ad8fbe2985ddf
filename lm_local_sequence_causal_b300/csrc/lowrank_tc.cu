// lowrank_tc.cu -- low-rank fused Dynamic Short Convolution on the
// 5th-generation tensor cores (tcgen05) with TMA-staged tiles.
//
// The filters of token t are w(t) = z_t U, z [B,T,R], U [R, C*W] with
// column j = c*W + k ("Technische Samenvatting: Dynamische Korte
// Convoluties Verbeteren Transformers", Parametrisatie item 1; Efficiente
// Trainingsimplementatie: Fused Low-Rank Kernel).  For a tile of 128 tokens
// and a chunk of 64 channels the filters are one small GEMM,
//     Wt[128 tokens x 64*W columns] = Z[128 x R] * U[R x 64*W],
// which the tensor core computes into TMEM (fp32, never rounded, never
// written to memory); the CUDA cores then read each token's row of Wt and
// apply the W taps to x.  The contraction has K = R = 16, so the tensor core
// is busy for a few percent of the time; the kernel is built to stream x and
// y at HBM speed around it.
//
// Forward kernel, one persistent CTA per SM, warp-specialised:
//   warp 0      TMA producer: per work item (b, 128-token tile, 64-channel
//               chunk) one box of x rows [t0-W+1, t0+128) x 64 channels
//               (128-byte swizzled rows; rows before t = 0 and past T read
//               as zero, which is the causal zero padding) and the z rows of
//               the tile, into a 4-stage ring.
//   warp 1      allocates 512 TMEM columns; one lane issues the MMAs
//               (M = 128, N = 64*W, K = 16 per instruction) into one of two
//               TMEM accumulators and commits them to mbarriers.
//   warps 2-9   epilogue: warp (w % 4) owns TMEM lanes 32*(w % 4) .. +31 =
//               those tokens; warps 2-5 take channels 0-31 of the chunk,
//               warps 6-9 channels 32-63.  Each thread loads its token's
//               W taps for 8 channels at a time (tcgen05.ld), reads
//               x[t-k] for the same 8 channels from the staged tile (16-byte
//               swizzled reads, no bank conflicts), forms
//               y = res*x + sum_k w_k x[t-k] in fp32, rounds once to bf16 and
//               writes a staged y tile that one thread stores with TMA.
// The U columns of the CTA's chunks are placed in shared memory once, in the
// K-major 32-byte-swizzled layout the MMA reads.  Work items are handed out
// as contiguous ranges, chunk-major, and the grid is at least the number of
// chunks, so a CTA meets at most two chunks.
//
// Every mbarrier wait is bounded (sm100.cuh); on a timeout the kernel
// records a code in the device error word, lets its in-flight copies land,
// frees its TMEM and returns.
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "dsc_common.cuh"
#include "dsc_internal.h"
#include "sm100.cuh"

namespace dsc {
namespace {

using namespace sm100;

// Set when a bounded wait gives up: 1 = producer, 2 = MMA issuer,
// 3 = epilogue, 4 = y store.  Cleared only by lowrank_tc_error(reset).
__device__ unsigned int g_tc_error = 0;

constexpr int BM = 128;     // tokens per tile = TMEM lanes
constexpr int CC = 64;      // channels per chunk = one 128-byte swizzled row
constexpr int NST = 4;      // input pipeline stages
constexpr int NEPI = 8;     // epilogue warps
constexpr int kFwdThreads = (2 + NEPI) * 32;
constexpr uint32_t kTmemCols = 512;

__host__ __device__ constexpr int round1k(int b) { return (b + 1023) / 1024 * 1024; }

template <int W, int KS>
struct FwdLayout {
  static constexpr int XROWS = BM + W - 1;
  static constexpr int XBOX = XROWS * 128;            // bytes of one x box
  static constexpr int XBYTES = round1k(XBOX);
  static constexpr int ZBYTES = BM * 32;              // one K-step of z (4 KB)
  static constexpr int NCOL = CC * W;                 // MMA N
  static constexpr int BBYTES = round1k(NCOL * 32);   // one K-step of U
  static constexpr int YBYTES = BM * 128;
  static constexpr int X_OFF = 0;
  static constexpr int Z_OFF = X_OFF + NST * XBYTES;
  static constexpr int B_OFF = Z_OFF + NST * KS * ZBYTES;
  static constexpr int Y_OFF = B_OFF + 2 * KS * BBYTES;
  static constexpr int BAR_OFF = Y_OFF + 2 * YBYTES;
  // full[NST] empty[NST] accf[2] acce[2] yfull[2] yfree[2]
  static constexpr int NBAR = 2 * NST + 8;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int TOTAL = MISC_OFF + 16 + 1024;  // + slack to align the base
  static constexpr uint32_t TX = XBOX + KS * ZBYTES;  // bytes landing per stage
};

__device__ __forceinline__ unsigned char* align1k(unsigned char* p) {
  return reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
}

struct Item {
  int chunk, b, t0;
};
__device__ __forceinline__ Item decode(long long i, int nbt, int ntiles) {
  Item it;
  it.chunk = static_cast<int>(i / nbt);
  const int rem = static_cast<int>(i - static_cast<long long>(it.chunk) * nbt);
  it.b = rem / ntiles;
  it.t0 = (rem - it.b * ntiles) * BM;
  return it;
}

// Fill the K-major 32-byte-swizzled B operand of chunk `chunk`: row n (the
// chunk's column c*W + k), K-element r = U[r, chunk*64*W + n] (zero past R
// or past the channel count).
template <int W, int KS>
__device__ void fill_u_tile(unsigned char* dst, const __nv_bfloat16* __restrict__ U, int chunk,
                            int C, int R) {
  using L = FwdLayout<W, KS>;
  const int64_t GW = static_cast<int64_t>(C) * W;
  for (int idx = threadIdx.x; idx < KS * L::NCOL * 16; idx += blockDim.x) {
    const int ks = idx / (L::NCOL * 16);
    const int rem = idx - ks * L::NCOL * 16;
    const int n = rem >> 4, k = rem & 15;
    const int r = ks * 16 + k;
    const int64_t col = static_cast<int64_t>(chunk) * L::NCOL + n;
    __nv_bfloat16 v = __float2bfloat16_rn(0.f);
    if (r < R && col < GW) v = U[static_cast<int64_t>(r) * GW + col];
    *reinterpret_cast<__nv_bfloat16*>(dst + ks * L::BBYTES + sw32_offset(n, k)) = v;
  }
}

// Wait for a phase during teardown: ignores the abort flag, bounded in time.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer() - t0 > kWaitLimitNs) return;
}

template <int W, int KS>
__global__ void __launch_bounds__(kFwdThreads, 1)
lr_fwd_tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_z,
          const __grid_constant__ CUtensorMap tm_y, const __nv_bfloat16* __restrict__ U, int C,
          int R, int ntiles, int nbt, int nchunks, int residual) {
  using L = FwdLayout<W, KS>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = align1k(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const long long items = static_cast<long long>(nchunks) * nbt;
  const long long i0 = items * blockIdx.x / gridDim.x;
  const long long i1 = items * (blockIdx.x + 1) / gridDim.x;

  const uint32_t bar_full = sb + L::BAR_OFF;
  const uint32_t bar_empty = bar_full + NST * 8;
  const uint32_t bar_accf = bar_empty + NST * 8;
  const uint32_t bar_acce = bar_accf + 16;
  const uint32_t bar_yfull = bar_acce + 16;
  const uint32_t bar_yfree = bar_yfull + 16;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1 + NEPI);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_accf + 8 * a, 1);
      mbar_init(bar_acce + 8 * a, NEPI);
      mbar_init(bar_yfull + 8 * a, NEPI);
      mbar_init(bar_yfree + 8 * a, 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_z);
    tma_prefetch_desc(&tm_y);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);

  const int chunk_first = i1 > i0 ? static_cast<int>(i0 / nbt) : 0;
  const int chunk_last = i1 > i0 ? static_cast<int>((i1 - 1) / nbt) : -1;
  for (int bsel = 0; bsel < 2; ++bsel)
    if (chunk_first + bsel <= chunk_last)
      fill_u_tile<W, KS>(smem + L::B_OFF + bsel * KS * L::BBYTES, U, chunk_first + bsel, C, R);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------- producer --
    if (lane == 0) {
      const uint64_t pol_stream = policy_evict_first();
      const uint64_t pol_keep = policy_evict_last();   // z is re-read for every chunk
      int it = 0;
      for (long long i = i0; i < i1; ++i, ++it) {
        const int s = it % NST;
        const uint32_t ph = (it / NST) & 1;
        if (!mbar_wait(bar_empty + 8 * s, ph ^ 1, abort_flag, &g_tc_error, 1)) break;
        const Item itm = decode(i, nbt, ntiles);
        const uint32_t full = bar_full + 8 * s;
        mbar_expect_tx(full, L::TX);
        tma_load_3d(sb + L::X_OFF + s * L::XBYTES, &tm_x, full, itm.chunk * CC,
                    itm.t0 - (W - 1), itm.b, pol_stream);
        for (int ks = 0; ks < KS; ++ks)
          tma_load_3d(sb + L::Z_OFF + (s * KS + ks) * L::ZBYTES, &tm_z, full, ks * 16, itm.t0,
                      itm.b, pol_keep);
      }
      // Let every load this thread issued land before the CTA can exit.
      for (int j = std::max(0, it - NST); j < it; ++j)
        drain_wait(bar_full + 8 * (j % NST), (j / NST) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, L::NCOL);
      int it = 0;
      for (long long i = i0; i < i1; ++i, ++it) {
        const int s = it % NST;
        const uint32_t ph = (it / NST) & 1;
        const int a = it & 1;
        const uint32_t aph = (it >> 1) & 1;
        if (!mbar_wait(bar_acce + 8 * a, aph ^ 1, abort_flag, &g_tc_error, 2)) break;
        if (!mbar_wait(bar_full + 8 * s, ph, abort_flag, &g_tc_error, 2)) break;
        tc_fence_after();
        const int bsel = static_cast<int>(i / nbt) - chunk_first;
        const uint32_t d = tmem + a * 256;
        for (int ks = 0; ks < KS; ++ks) {
          const uint64_t ad = desc_kmajor_sw32(sb + L::Z_OFF + (s * KS + ks) * L::ZBYTES);
          const uint64_t bd = desc_kmajor_sw32(sb + L::B_OFF + (bsel * KS + ks) * L::BBYTES);
          mma_bf16(d, ad, bd, idesc, ks > 0 ? 1u : 0u);
        }
        mma_commit(bar_accf + 8 * a);
        mma_commit(bar_empty + 8 * s);
      }
      if (it > 0) drain_wait(bar_accf + 8 * ((it - 1) & 1), ((it - 1) >> 1) & 1);
    }
  } else {
    // --------------------------------------------------------- epilogue --
    const int lg = warp & 3;                 // TMEM lane group of this warp
    const int h = (warp - 2) >> 2;           // channel half of the chunk
    const int tl = lg * 32 + lane;           // token within the tile
    const bool storer = (warp == 2 && lane == 0);
    const uint64_t pol_y = policy_evict_first();
    const uint32_t tbase = tmem + (static_cast<uint32_t>(lg * 32) << 16);
    int it = 0;
    for (long long i = i0; i < i1; ++i, ++it) {
      const int s = it % NST;
      const uint32_t ph = (it / NST) & 1;
      const int a = it & 1;
      const uint32_t aph = (it >> 1) & 1;
      const uint32_t ybuf = sb + L::Y_OFF + a * L::YBYTES;
      if (storer) {
        bulk_wait_read<1>();                 // the store that used this buffer has read it
        mbar_arrive(bar_yfree + 8 * a);
      }
      // Every lane waits; the warp leaves together if any wait gave up, so
      // the .sync.aligned TMEM loads below always run converged.
      bool ok = mbar_wait(bar_yfree + 8 * a, aph, abort_flag, &g_tc_error, 3) &&
                mbar_wait(bar_accf + 8 * a, aph, abort_flag, &g_tc_error, 3) &&
                mbar_wait(bar_full + 8 * s, ph, abort_flag, &g_tc_error, 3);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t xt = sb + L::X_OFF + s * L::XBYTES;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int cch = 4 * h + q;           // 16-byte chunk of the 128-byte row
        uint32_t acc[8 * W];
        tmem_ld_cols<8 * W>(tbase + a * 256 + (h * 32 + q * 8) * W, acc);
        float xv[W][8];
#pragma unroll
        for (int k = 0; k < W; ++k) {
          const uint32_t row = tl + (W - 1) - k;
          unpack16<__nv_bfloat16>(lds128(xt + sw128_offset(row, cch)), xv[k]);
        }
        tmem_wait_ld();
        tmem_regs_ready<8 * W>(acc);
        float out[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          float v = residual ? xv[0][c] : 0.f;
#pragma unroll
          for (int k = 0; k < W; ++k) v = fmaf(__uint_as_float(acc[c * W + k]), xv[k][c], v);
          out[c] = v;
        }
        sts128(ybuf + sw128_offset(tl, cch), pack16<__nv_bfloat16>(out));
      }
      tc_fence_before();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar_acce + 8 * a);
        mbar_arrive(bar_empty + 8 * s);
        mbar_arrive(bar_yfull + 8 * a);
      }
      // On a failed wait the store is skipped; the abort flag is up, so the
      // whole warp leaves at the next item's waits.
      if (storer && mbar_wait(bar_yfull + 8 * a, aph, abort_flag, &g_tc_error, 4)) {
        const Item itm = decode(i, nbt, ntiles);
        tma_store_3d(&tm_y, ybuf, itm.chunk * CC, itm.t0, itm.b, pol_y);
        bulk_commit();
      }
    }
    if (storer) bulk_wait<0>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ host ----

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

template <int W, int KS>
cudaError_t launch_fwd(const void* x, const void* z, const void* U, void* y, const Shape& s,
                       cudaStream_t st) {
  using L = FwdLayout<W, KS>;
  CUtensorMap tx, tz, ty;
  if (!make_tmap_3d(&tx, x, true, s.C, s.T, s.B, CC, BM + W - 1, 128) ||
      !make_tmap_3d(&tz, z, true, s.R, s.T, s.B, 16, BM, 32) ||
      !make_tmap_3d(&ty, y, true, s.C, s.T, s.B, CC, BM, 128))
    return cudaErrorNotSupported;
  const int ntiles = static_cast<int>((s.T + BM - 1) / BM);
  const int nchunks = static_cast<int>((s.C + CC - 1) / CC);
  const long long nbt = static_cast<long long>(s.B) * ntiles;
  const long long items = nbt * nchunks;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorNoDevice;
  long long grid = std::min<long long>(sms, items);
  grid = std::max<long long>(grid, nchunks);
  auto kern = lr_fwd_tc<W, KS>;
  cudaError_t e = set_smem<L>(kern, L::TOTAL);
  if (e != cudaSuccess) return e;
  kern<<<static_cast<unsigned>(grid), kFwdThreads, L::TOTAL, st>>>(
      tx, tz, ty, static_cast<const __nv_bfloat16*>(U), static_cast<int>(s.C),
      static_cast<int>(s.R), ntiles, static_cast<int>(nbt), nchunks, s.residual);
  return cudaGetLastError();
}

}  // namespace

bool lowrank_tc_supported(const Shape& s) {
  return s.bf16 && s.H == 1 && (s.R == 16 || s.R == 32) && s.W >= 1 && s.W <= 4 &&
         s.B * ((s.T + BM - 1) / BM) < (int64_t(1) << 30) && s.T < (int64_t(1) << 30) &&
         s.C < (int64_t(1) << 24);
}

cudaError_t lowrank_fwd_tc(const void* x, const void* z, const void* U, void* y,
                           const Shape& s, cudaStream_t st) {
  if (!lowrank_tc_supported(s)) return cudaErrorNotSupported;
  const bool k2 = s.R > 16;
  switch (s.W) {
    case 1: return k2 ? launch_fwd<1, 2>(x, z, U, y, s, st) : launch_fwd<1, 1>(x, z, U, y, s, st);
    case 2: return k2 ? launch_fwd<2, 2>(x, z, U, y, s, st) : launch_fwd<2, 1>(x, z, U, y, s, st);
    case 3: return k2 ? launch_fwd<3, 2>(x, z, U, y, s, st) : launch_fwd<3, 1>(x, z, U, y, s, st);
    default: return k2 ? launch_fwd<4, 2>(x, z, U, y, s, st) : launch_fwd<4, 1>(x, z, U, y, s, st);
  }
}

cudaError_t lowrank_tc_error(unsigned int* out, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_tc_error, sizeof(unsigned int));
  if (e != cudaSuccess || !reset) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(unsigned int));
}

}  // namespace dsc

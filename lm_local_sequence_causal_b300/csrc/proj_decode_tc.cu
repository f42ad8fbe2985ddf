// proj_decode_tc.cu -- the decode step merged with its projection on the
// 5th-generation tensor core, for batches of more than a few sequences.
//
// What it computes is the merged step of proj_decode.cu ("Dynamic Short
// Convolutions: The 'Locality Bias' Transformers Were Missing",
// Limitations: the convolution merged into the matmul before it):
//   x[b,c] = sum_d h[b,d] Wp[c,d]      rounded once to bf16
//   y[b,c] = res*x[b,c] + w[b,g(c),0] x[b,c] + sum_{k>=1} w[b,g(c),k] state[b,k-1,c]
//   state[b,0,c] <- x[b,c],  state[b,j,c] <- state[b,j-1,c]
// with w = z U for the low-rank form.
//
// The projection is a weight stream (Wp, C x D, read once) against a few
// rows of h.  Transposed, x^T = Wp h^T is an MMA with M = 128 channels (rows
// of Wp: the A operand), N = the batch rounded up to 16 (rows of h: the B
// operand) and K = D, both operands K-major as they lie in memory, so TMA
// brings 128-byte-swizzled boxes of 64 D-elements of Wp (128 rows) and h (N
// rows) straight into the tensor core's layout, and the fp32 accumulator
// lives in TMEM (128 lanes = channels, N columns = sequences).  C / 128
// channel tiles alone would leave most SMs idle (48 at C = 6144), so D is
// split over a cluster of KS CTAs (the largest KS <= 8 whose clusters all
// fit on the device at once): rank q takes a contiguous range of D's
// 64-element blocks.  The KS partial tiles
// meet through distributed shared memory: rank q finishes the sequences
// b = q, q + KS, ... of the tile, so every rank stores its partial sums of
// those sequences into rank q's shared memory (stores, which do not stall
// the way remote loads do); q then adds the KS partials in rank order (a
// fixed order: the result does not depend on scheduling), rounds x and runs
// the decode step, one thread per channel, so the loads and stores of w,
// state and y are contiguous along the channels.
//
// Roles (8 warps): warp 0 lane 0 issues the TMA loads of a ring of stages,
// warp 1 owns TMEM and lane 0 issues the MMAs, warps 2-7 prefetch the
// decode step's operands into L2; after the K loop all eight warps run the
// epilogue (warps w and w + 4 read TMEM lanes 32 (w mod 4) .. + 31 and take
// alternate chunks of columns).  Every mbarrier wait is bounded in time (a
// broken pipeline sets an error code and the kernel returns); both cluster
// barriers are reached by every thread of every CTA whatever happened before
// them, so no CTA waits on one that left.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "dsc_common.cuh"
#include "dsc_internal.h"
#include "sm100.cuh"

namespace dsc {
namespace {

using namespace sm100;

__device__ unsigned int g_pd_error = 0;

constexpr int kPdtThreads = 256;            // 8 warps
constexpr int kPdtM = 128;                  // channels per CTA (the MMA's M)
constexpr int kPdtMaxN = 256;               // sequences per launch (the MMA's N)
constexpr int kPdtMaxStages = 8;
constexpr int kPdtMaxCluster = 8;
constexpr int kPdtABytes = kPdtM * 128;     // one stage of Wp: 128 rows x 64 bf16
constexpr int kPdtSmem = 227 * 1024;        // opt-in; a launch uses what its N needs
constexpr int kPdtMisc = 2 * kPdtMaxStages * 8 + 8 + 16;   // full, empty, done; flag, TMEM slot

struct PdtArgs {
  const __nv_bfloat16* w;      // head-wise taps [B][C/H][W]
  const __nv_bfloat16* z;      // low-rank factors [B][R]
  const __nv_bfloat16* U;      // [R][(C/H) W]
  __nv_bfloat16* state;        // [B][W-1][C]
  __nv_bfloat16* y;            // [B][C]
  int B, C, H, R, residual;
  int N;                       // MMA N: B rounded up to 16
  int nkb;                     // 64-element blocks of D
  int nst;                     // pipeline stages
  unsigned long long wns;      // wait limit
  int withhold;                // self-test: the producer issues no loads, so waits run out
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

// Every thread of every CTA of the cluster; writes before it (shared memory
// included) are visible to reads after it anywhere in the cluster.
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_map(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

__device__ __forceinline__ void dsmem_st(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Remote 16-byte store into another CTA's shared memory (address from mapa).
__device__ __forceinline__ void dsmem_st4u(uint32_t addr, uint4 v) {
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// The push of a cluster of KSC = 1, 2, 4 or 8 CTAs: chunks of 4 KSC
// accumulator columns (the two column halves alternate chunks, j a
// multiple of 4 KSC); rank q gets columns j + q + KSC e (e < 4) at its slots
// j / KSC + e, one 16-byte store (a local one for this CTA's own rank).
// `mine` is the shared-memory address of this thread's slot row.
template <int KSC>
__device__ __forceinline__ void push_tile(uint32_t tl, uint32_t mine, uint32_t rank, int half,
                                          int N, int B) {
  constexpr int CH = 4 * KSC;
  for (int j = half * CH; j < N && j < B; j += 2 * CH) {
    uint32_t v[CH];
    tmem_ld_cols<CH>(tl + j, v);
    tmem_wait_ld();
    tmem_regs_ready<CH>(v);
    const uint32_t at = mine + 4u * static_cast<uint32_t>(j / KSC);
#pragma unroll
    for (int q = 0; q < KSC; ++q) {
      const uint4 f = make_uint4(v[q], v[q + KSC], v[q + 2 * KSC], v[q + 3 * KSC]);
      if (q == static_cast<int>(rank)) sts128(at, f);
      else dsmem_st4u(dsmem_map(at, static_cast<uint32_t>(q)), f);
    }
  }
}

// Row length (floats) of a channel's slots: room for every column of the
// MMA's N rounded up to a multiple of 8 (the epilogue reads batches of 4
// slots), and an odd number of 16-byte units, so 8 lanes reading or writing
// 16 bytes of 8 rows hit 8 different bank groups.
__host__ __device__ __forceinline__ int slot_ld(int N, int KS) {
  return ((N + KS - 1) / KS + 7) / 8 * 8 + 4;
}

// K-major operand with 128-byte rows and the 128-byte swizzle (8-row atoms
// 1024 bytes apart), as TMA writes a box of 64 bf16 per row.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

template <int W, bool LOWRANK>
__global__ void __launch_bounds__(kPdtThreads, 1)
proj_decode_tc_kernel(const __grid_constant__ CUtensorMap tm_wp,
                      const __grid_constant__ CUtensorMap tm_h, const PdtArgs a) {
  using T = __nv_bfloat16;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = align1k(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.N;
  const uint32_t stage_bytes = kPdtABytes + static_cast<uint32_t>(N) * 128u;
  const uint32_t misc = sb + a.nst * stage_bytes;
  const uint32_t bar_full = misc, bar_empty = misc + kPdtMaxStages * 8;
  const uint32_t bar_done = misc + 2 * kPdtMaxStages * 8;
  volatile int* abort_flag =
      reinterpret_cast<volatile int*>(smem + a.nst * stage_bytes + 2 * kPdtMaxStages * 8 + 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + a.nst * stage_bytes +
                                                    2 * kPdtMaxStages * 8 + 12);
  const uint32_t KS = cluster_size(), rank = cluster_rank();
  const int tile = static_cast<int>(blockIdx.x / KS);
  const int c_tile = tile * kPdtM;
  // This rank's blocks of D: [kb0, kb1), never empty (the host keeps KS <= nkb).
  const int kb0 = static_cast<int>((static_cast<long long>(a.nkb) * rank) / KS);
  const int kb1 = static_cast<int>((static_cast<long long>(a.nkb) * (rank + 1)) / KS);
  const int nk = kb1 - kb0;
  uint32_t tcols = 32;
  while (tcols < static_cast<uint32_t>(N)) tcols <<= 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.nst; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_wp);
    tma_prefetch_desc(&tm_h);
  }
  // Launched as a programmatic dependent: the barrier set-up above may
  // overlap the previous kernel in the stream; TMEM is taken, and every
  // input read (after the block barrier below), only once that kernel ended.
  if (warp == 1) {
    griddep_wait();
    tmem_alloc(smem_u32(tmem_slot), tcols);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // -------------------------------------------------------- producer --
    if (lane == 0) {
      const uint64_t pol_wp = policy_evict_first();   // read once
      const uint64_t pol_h = policy_evict_last();     // read by every tile
      int i = 0;
      for (; i < nk && !a.withhold; ++i) {
        const int s = i % a.nst;
        const uint32_t ph = (i / a.nst) & 1;
        if (!mbar_wait(bar_empty + 8 * s, ph ^ 1, abort_flag, &g_pd_error, 1, a.wns)) break;
        const uint32_t st = sb + s * stage_bytes;
        mbar_expect_tx(bar_full + 8 * s, stage_bytes);
        const int d0 = (kb0 + i) * 64;
        tma_load_3d(st, &tm_wp, bar_full + 8 * s, d0, c_tile, 0, pol_wp);
        tma_load_3d(st + kPdtABytes, &tm_h, bar_full + 8 * s, d0, 0, 0, pol_h);
      }
      // Let every load this thread issued land before the CTA can exit.
      for (int j = std::max(0, i - a.nst); j < i; ++j)
        drain_wait(bar_full + 8 * (j % a.nst), (j / a.nst) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer --
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kPdtM, static_cast<uint32_t>(N));
      for (int i = 0; i < nk; ++i) {
        const int s = i % a.nst;
        if (!mbar_wait(bar_full + 8 * s, (i / a.nst) & 1, abort_flag, &g_pd_error, 2, a.wns))
          break;
        tc_fence_after();
        const uint32_t st = sb + s * stage_bytes;
        const uint64_t ad = desc_sw128(st), bd = desc_sw128(st + kPdtABytes);
        // Four K-steps of 16 elements: 32 bytes further along each row.
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16(tmem, ad + static_cast<uint64_t>(2 * kk), bd + static_cast<uint64_t>(2 * kk),
                   idesc, (i > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar_empty + 8 * s);
      }
      // Signals once every MMA issued above has completed (also after an
      // early exit, so the epilogue never reads TMEM under a running MMA).
      mma_commit(bar_done);
    }
  } else {
    // ------------------------------------------------------ prefetcher --
    // Warps 2-7 have nothing to do during the K loop: they bring the decode
    // step's operands of this rank's sequences (state rows, taps or z) into
    // L2, so the epilogue's loads are L2 hits.  Lines are 128 bytes; a run
    // of n bytes at p is covered by the lines of p, p + 128, ..., p + n - 1.
    const int pt = threadIdx.x - 64, npt = kPdtThreads - 64;
    const int64_t C = a.C, G = C / a.H;
    const int cn = static_cast<int>(std::min<int64_t>(kPdtM, C - c_tile));   // channels here
    const int64_t g_lo = c_tile / a.H, g_hi = (c_tile + cn - 1) / a.H;
    const int srow = cn * 2;                                   // bytes of a state row here
    const int trow = LOWRANK ? a.R * 2 : static_cast<int>(g_hi - g_lo + 1) * W * 2;
    const int sl = W > 1 ? (W - 1) * ((srow + 127) / 128 + 1) : 0;      // lines per sequence
    const int tlines = (trow + 127) / 128 + 1;
    const int per_b = sl + tlines;
    const int nmine = (a.B - static_cast<int>(rank) + static_cast<int>(KS) - 1) /
                      static_cast<int>(KS);
    for (int i = pt; i < nmine * per_b; i += npt) {
      const int bi = i / per_b, li = i - bi * per_b;
      const int64_t b = rank + static_cast<int64_t>(KS) * bi;
      const char* base;
      int off, len;
      if (li < sl) {
        const int j = li / ((srow + 127) / 128 + 1), l = li - j * ((srow + 127) / 128 + 1);
        base = reinterpret_cast<const char*>(a.state + (b * (W - 1) + j) * C + c_tile);
        off = l * 128;
        len = srow;
      } else {
        const int l = li - sl;
        base = LOWRANK ? reinterpret_cast<const char*>(a.z + b * a.R)
                       : reinterpret_cast<const char*>(a.w + (b * G + g_lo) * W);
        off = l * 128;
        len = trow;
      }
      prefetch_l2(base + std::min(off, len - 1));
    }
  }

  // ---------------------------------------------------------- epilogue --
  // Every CTA of the cluster first finishes its K loop (so no stage of any
  // CTA is still read by an MMA or written by TMA); then each CTA pushes its
  // partial sums to the rank that finishes each sequence: rank p writes
  // x_p[b, c] into rank q = b % KS, slot [p][c][b / KS] (a row of ld floats
  // per channel).  With KS = 1, 2, 4 or 8, a TMEM load of 4 KS columns
  // gives each rank 4 consecutive slots, one 16-byte store.  After a second
  // cluster barrier every rank adds its slots locally.
  __syncwarp();
  bool ok = mbar_wait(bar_done, 0, abort_flag, &g_pd_error, 3, a.wns);
  ok = __all_sync(0xffffffffu, ok) && !*abort_flag;
  griddep_launch_dependents();     // the next kernel may start its prologue
  tc_fence_after();
  tc_fence_before();
  cluster_sync();
  const int nbq = (a.B + static_cast<int>(KS) - 1) / static_cast<int>(KS);   // slots per rank
  const int ld = slot_ld(N, static_cast<int>(KS));
  float* slots = reinterpret_cast<float*>(smem);  // [KS][128][ld] fp32, in the stage ring
  const int lg = warp & 3, half = warp >> 2;     // TMEM lane group; which chunks
  const int row = lg * 32 + lane;                // channel within the tile
  if (ok) {
    tc_fence_after();
    const uint32_t tl = tmem + (static_cast<uint32_t>(lg * 32) << 16);
    const uint32_t mine = smem_u32(slots + (rank * kPdtM + row) * ld);
    switch (KS) {
      case 1: push_tile<1>(tl, mine, rank, half, N, a.B); break;
      case 2: push_tile<2>(tl, mine, rank, half, N, a.B); break;
      case 4: push_tile<4>(tl, mine, rank, half, N, a.B); break;
      case 8: push_tile<8>(tl, mine, rank, half, N, a.B); break;
      default: break;
    }
    if (KS != 1 && KS != 2 && KS != 4 && KS != 8) {
      for (int j = half * 8; j < N && j < a.B; j += 16) {
        uint32_t v[8];
        tmem_ld8(tl + j, v);
        tmem_wait_ld();
        tmem_regs_ready<8>(v);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t b = static_cast<uint32_t>(j + e);
          const uint32_t q = b % KS, bl = b / KS;
          const uint32_t at = mine + 4u * bl;
          if (q == rank) slots[(rank * kPdtM + row) * ld + bl] = __uint_as_float(v[e]);
          else dsmem_st(dsmem_map(at, q), __uint_as_float(v[e]));
        }
      }
    }
  }
  tc_fence_before();
  cluster_sync();

  // Decode steps of this rank's sequences b = rank + KS * bl: thread t takes
  // channel t % 128 and half of the slots (t / 128 picks the half), NBX
  // consecutive slots at a time, with every load of a batch issued before
  // its stores.
  const int c = c_tile + (threadIdx.x & (kPdtM - 1));
  const int sub = threadIdx.x >> 7;              // 0 or 1
  if (ok && !*abort_flag && c < a.C) {
    const int64_t C = a.C;
    const int64_t G = C / a.H, g = c / a.H;
    const int cl = c - c_tile;
    constexpr int NBX = 4;     // 8 was slower (more registers, fewer loads in flight)
    const int units = (nbq + NBX - 1) / NBX, u_half = (units + 1) / 2;
    const int u0 = sub ? u_half : 0, u1 = sub ? units : u_half;
    for (int u = u0; u < u1; ++u) {
      const int bl0 = u * NBX;
      int bb[NBX];
      bool on[NBX];
#pragma unroll
      for (int j = 0; j < NBX; ++j) {
        bb[j] = static_cast<int>(rank) + static_cast<int>(KS) * (bl0 + j);
        on[j] = bl0 + j < nbq && bb[j] < a.B;
      }
      float taps[NBX][W];
      if constexpr (!LOWRANK) {
#pragma unroll
        for (int j = 0; j < NBX; ++j) {
          const T* wb = a.w + (static_cast<int64_t>(on[j] ? bb[j] : 0) * G + g) * W;
#pragma unroll
          for (int k = 0; k < W; ++k) taps[j][k] = on[j] ? __bfloat162float(wb[k]) : 0.f;
        }
      } else {
        // z[b] U[:, g W + k] in fp32; each U column is loaded once per batch.
        const int64_t GW = G * W;
#pragma unroll
        for (int j = 0; j < NBX; ++j)
#pragma unroll
          for (int k = 0; k < W; ++k) taps[j][k] = 0.f;
        for (int r = 0; r < a.R; ++r) {
          float u[W];
#pragma unroll
          for (int k = 0; k < W; ++k) u[k] = __bfloat162float(a.U[r * GW + g * W + k]);
#pragma unroll
          for (int j = 0; j < NBX; ++j) {
            const float zr =
                on[j] ? __bfloat162float(a.z[static_cast<int64_t>(bb[j]) * a.R + r]) : 0.f;
#pragma unroll
            for (int k = 0; k < W; ++k) taps[j][k] = fmaf(zr, u[k], taps[j][k]);
          }
        }
      }
      T sv[NBX][W > 1 ? W - 1 : 1];
      if constexpr (W > 1) {
#pragma unroll
        for (int j = 0; j < NBX; ++j) {
          const T* sp = a.state + static_cast<int64_t>(on[j] ? bb[j] : 0) * (W - 1) * C + c;
#pragma unroll
          for (int i = 0; i < W - 1; ++i) sv[j][i] = on[j] ? sp[i * C] : __float2bfloat16_rn(0.f);
        }
      }
      // The KS partials in rank order, four slots per 16-byte load.
      float xsum[NBX];
#pragma unroll
      for (int j = 0; j < NBX; ++j) xsum[j] = 0.f;
      for (int p = 0; p < static_cast<int>(KS); ++p) {
#pragma unroll
        for (int h4 = 0; h4 < NBX / 4; ++h4) {
          const uint4 v = lds128(smem_u32(slots + (p * kPdtM + cl) * ld + bl0 + 4 * h4));
          xsum[4 * h4 + 0] += __uint_as_float(v.x);
          xsum[4 * h4 + 1] += __uint_as_float(v.y);
          xsum[4 * h4 + 2] += __uint_as_float(v.z);
          xsum[4 * h4 + 3] += __uint_as_float(v.w);
        }
      }
#pragma unroll
      for (int j = 0; j < NBX; ++j) {
        if (!on[j]) continue;
        const int b = bb[j];
        const T xs = __float2bfloat16_rn(xsum[j]);   // x as the projection would store it
        const float xf = __bfloat162float(xs);
        float acc = a.residual ? xf : 0.f;
        acc = fmaf(taps[j][0], xf, acc);
        if constexpr (W > 1) {
          T* sp = a.state + static_cast<int64_t>(b) * (W - 1) * C + c;
#pragma unroll
          for (int k = 1; k < W; ++k) acc = fmaf(taps[j][k], __bfloat162float(sv[j][k - 1]), acc);
#pragma unroll
          for (int i = W - 2; i >= 1; --i) sp[i * C] = sv[j][i - 1];
          sp[0] = xs;
        }
        a.y[static_cast<int64_t>(b) * C + c] = __float2bfloat16_rn(acc);
      }
    }
  }
  tc_fence_after();
  if (warp == 1) {
    drain_wait(bar_done, 0);
    tc_fence_after();
    tmem_dealloc(tmem, tcols);
  }
}

template <int W, bool LOWRANK>
struct PdtKernelTag {};

// Launch configuration of a cluster of `ks` CTAs with the full shared-memory
// opt-in (every launch keeps one CTA per SM: its stages take > 113 KB).
void cluster_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute (&attr)[2], unsigned grid,
                    unsigned ks, size_t smem, cudaStream_t st) {
  cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kPdtThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // A programmatic dependent of the previous kernel in the stream (the
  // kernel waits for it before its first load).
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
}

// How many clusters of `ks` CTAs fit on the device at once (cached per
// device).  The SMs of a cluster come from one GPC, so this is below
// SMs / ks where a GPC's SM count is not a multiple of ks (45 clusters of 3
// on 148 SMs).
template <int W, bool LOWRANK>
int max_clusters(int ks) {
  static std::mutex mu;
  static int cache[64][kPdtMaxCluster + 1] = {};     // value + 1; 0 = not asked yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev][ks] == 0) {
    auto kern = proj_decode_tc_kernel<W, LOWRANK>;
    int n = 0;
    if (set_smem<PdtKernelTag<W, LOWRANK>>(kern, kPdtSmem) == cudaSuccess) {
      cudaLaunchConfig_t cfg;
      cudaLaunchAttribute attr[2];
      cluster_config(cfg, attr, static_cast<unsigned>(ks), static_cast<unsigned>(ks), kPdtSmem,
                     nullptr);
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
    }
    cache[dev][ks] = n + 1;
  }
  return cache[dev][ks] - 1;
}

template <int W, bool LOWRANK>
cudaError_t run_w(const void* h, const void* Wp, const void* w, const void* z, const void* U,
                  void* state, void* y, const Shape& s, int64_t D, cudaStream_t st,
                  uint64_t wait_ns, int withhold) {
  using T = __nv_bfloat16;
  auto kern = proj_decode_tc_kernel<W, LOWRANK>;
  cudaError_t e = set_smem<PdtKernelTag<W, LOWRANK>>(kern, kPdtSmem);
  if (e != cudaSuccess) return e;
  const int ntile = static_cast<int>((s.C + kPdtM - 1) / kPdtM);
  const int nkb = static_cast<int>((D + 63) / 64);
  // The widest split of D whose clusters all fit at once (one wave): a
  // second wave of a few clusters costs as much as the first.
  int ks = 1;
  for (int k = std::min(kPdtMaxCluster, nkb); k >= 2; --k)
    if (max_clusters<W, LOWRANK>(k) >= ntile) {
      ks = k;
      break;
    }
  CUtensorMap twp;
  if (!make_tmap_3d(&twp, Wp, true, D, s.C, 1, 64, kPdtM, 128)) return cudaErrorInvalidValue;
  const int64_t G = s.G();
  for (int64_t b0 = 0; b0 < s.B; b0 += kPdtMaxN) {
    const int nb = static_cast<int>(std::min<int64_t>(kPdtMaxN, s.B - b0));
    PdtArgs a;
    a.N = (nb + 15) / 16 * 16;
    const size_t stage = kPdtABytes + static_cast<size_t>(a.N) * 128;
    // The partial sums pushed to a rank: KS x 128 rows of slot_ld floats.
    const size_t slots = static_cast<size_t>(ks) * kPdtM * slot_ld(a.N, ks) * sizeof(float);
    const size_t room = kPdtSmem - 1024 - kPdtMisc;
    a.nst = static_cast<int>(std::min<size_t>(kPdtMaxStages, room / stage));
    if (a.nst < 2 || a.nst * stage < slots) return cudaErrorInvalidValue;
    const size_t smem = a.nst * stage + kPdtMisc + 1024;
    CUtensorMap th;
    if (!make_tmap_3d(&th, static_cast<const T*>(h) + b0 * D, true, D, nb, 1, 64, a.N, 128))
      return cudaErrorInvalidValue;
    a.w = LOWRANK ? nullptr : static_cast<const T*>(w) + b0 * G * s.W;
    a.z = LOWRANK ? static_cast<const T*>(z) + b0 * s.R : nullptr;
    a.U = static_cast<const T*>(U);
    a.state = s.W > 1 ? static_cast<T*>(state) + b0 * (s.W - 1) * s.C : nullptr;
    a.y = static_cast<T*>(y) + b0 * s.C;
    a.B = nb;
    a.C = static_cast<int>(s.C);
    a.H = static_cast<int>(s.H);
    a.R = static_cast<int>(s.R);
    a.residual = s.residual;
    a.nkb = nkb;
    a.wns = wait_ns;
    a.withhold = withhold;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    cluster_config(cfg, attr, static_cast<unsigned>(ntile * ks), static_cast<unsigned>(ks), smem,
                   st);
    e = cudaLaunchKernelEx(&cfg, kern, twp, th, a);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

bool proj_decode_tc_supported(const Shape& s, int64_t D) {
  return s.bf16 && s.W >= 1 && s.W <= 4 && s.R <= 32 && D >= 8 && D % 8 == 0 &&
         s.C <= (int64_t(1) << 24) && s.B >= 1;
}

namespace {

cudaError_t run(const void* h, const void* Wp, const void* w, const void* z, const void* U,
                void* state, void* y, const Shape& s, int64_t D, bool lowrank, cudaStream_t st,
                uint64_t wait_ns, int withhold) {
  if (!proj_decode_tc_supported(s, D)) return cudaErrorNotSupported;
#define DSC_PDT_W(Wv)                                                                         \
  return lowrank ? run_w<Wv, true>(h, Wp, w, z, U, state, y, s, D, st, wait_ns, withhold)    \
                 : run_w<Wv, false>(h, Wp, w, z, U, state, y, s, D, st, wait_ns, withhold)
  switch (s.W) {
    case 1: DSC_PDT_W(1);
    case 2: DSC_PDT_W(2);
    case 3: DSC_PDT_W(3);
    default: DSC_PDT_W(4);
  }
#undef DSC_PDT_W
}

}  // namespace

cudaError_t proj_decode_tc(const void* h, const void* Wp, const void* w, const void* z,
                           const void* U, void* state, void* y, const Shape& s, int64_t D,
                           bool lowrank, cudaStream_t st) {
  return run(h, Wp, w, z, U, state, y, s, D, lowrank, st, kWaitLimitNs, 0);
}

cudaError_t proj_decode_tc_selftest(const void* h, const void* Wp, const void* w, void* state,
                                    void* y, const Shape& s, int64_t D, uint64_t wait_ns,
                                    cudaStream_t st) {
  return run(h, Wp, w, nullptr, nullptr, state, y, s, D, false, st, wait_ns, 1);
}

cudaError_t proj_decode_tc_error(unsigned int* out, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_pd_error, sizeof(unsigned int));
  if (e != cudaSuccess || !reset) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_pd_error, &zero, sizeof(unsigned int));
}

}  // namespace dsc

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
// apply the W taps to x.  The contraction has K = R (16 at the QKV size;
// ranks up to 32, padded to 16 or 32 with zeros), so the tensor core is busy
// for a few percent of the time; the kernel is built to stream x and y at
// HBM speed around it.
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
//   warps 2-17  epilogue, two groups of 8 warps taking alternate items (each
//               with its own TMEM accumulator, so the groups overlap); in a
//               group, warp (w % 4) owns TMEM lanes 32*(w % 4) .. +31 = those
//               tokens and the two warps of each lane group split the
//               chunk's channels.  Each thread loads its token's W taps for
//               8 channels at a time (tcgen05.ld), reads x[t-k] for the same
//               8 channels from the staged tile (16-byte swizzled reads, no
//               bank conflicts), forms y = res*x + sum_k w_k x[t-k] in fp32,
//               rounds once to bf16 and writes the warp's own staging box
//               (32 tokens x 32 channels), which the warp stores with TMA.
// Each stage also carries the chunk's U columns, loaded by TMA straight from
// U's natural [R, C*W] layout (MN-major operand, 128-byte swizzle).  Work
// items are handed out round-robin (item i to CTA i mod grid) in tile-major
// order, so the CTAs working side by side read neighbouring 128-byte pieces
// of the same rows of x.
//
// Every mbarrier wait is bounded (sm100.cuh); on a timeout the kernel
// records a code in the device error word, lets its in-flight copies land,
// frees its TMEM and returns.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "dsc_common.cuh"
#include "dsc_internal.h"
#include "sm100.cuh"

namespace dsc {
namespace {

using namespace sm100;

// Set when a bounded wait gives up: 1 = producer, 2 = MMA issuer,
// 3 = epilogue, 4 = y store, 5 = second MMA issuer (backward dz/dU).
// Cleared only by lowrank_tc_error(reset).
__device__ unsigned int g_tc_error = 0;

constexpr int BM = 128;     // tokens per tile = TMEM lanes
constexpr int CC = 64;      // channels per chunk = one 128-byte swizzled row
constexpr int NST = 4;      // input pipeline stages
// The forward's two epilogue groups take alternate items; an even stage
// count keeps every stage with one group, so a group's parity wait on a
// stage is never two phases ahead of the barrier.
static_assert(NST % 2 == 0, "forward stages must be even");
constexpr int NEPI_F = 16;  // forward epilogue warps: two groups of 8 that take alternate items
constexpr int NGRP = 8;     // warps per forward epilogue group (4 lane groups x 2 channel halves)
constexpr int kFwdThreads = (2 + NEPI_F) * 32;
constexpr int NEPI = 8;     // warps per backward epilogue group (4 lane groups x 2 channel halves)
// producer, D-MMA issuer, dx group, dw group, dz/dU-MMA issuer
constexpr int kBwdThreads = (3 + 2 * NEPI) * 32;
constexpr int kDzduWarp = 2 + 2 * NEPI;
// The dx warps read the backward's D accumulator and hand it back in
// kDParts channel parts of 64 / kDParts channels each.
constexpr int kDParts = 2;
constexpr uint32_t kTmemCols = 512;

__host__ __device__ constexpr int round1k(int b) { return (b + 1023) / 1024 * 1024; }

// HP = min(H, 8): channels of an 8-channel piece that share one filter.  A
// 64-channel chunk uses (64/H)*W consecutive columns of U; they are loaded
// as NA atoms of 64 columns (the tail of the last atom is not read back).
template <int W, int KS, int HP>
struct FwdLayout {
  static constexpr int XROWS = BM + W - 1;
  static constexpr int XBOX = XROWS * 128;            // bytes of one x box
  static constexpr int XBYTES = round1k(XBOX);
  static constexpr int ZBYTES = BM * 32;              // one K-step of z (4 KB)
  static constexpr int NA = (W + HP - 1) / HP;        // 64-column U atoms per chunk
  static constexpr int NCOL = 64 * NA;                // MMA N
  static constexpr int UATOM = KS * 16 * 128;         // 64 U columns x R rows (2 or 4 KB)
  static constexpr int UBYTES = NA * UATOM;
  static constexpr int STAGE = XBYTES + KS * ZBYTES + round1k(UBYTES);
  // Staged y: every epilogue warp has its own box(es) of 32 tokens x 32
  // channels (64-byte rows, 64-byte swizzle) that it stores with TMA; two
  // per warp where shared memory allows, so a warp never waits for its
  // previous store to be read.
  static constexpr int YBOX = 32 * 64;
  static constexpr int Z_IN = XBYTES;                 // offsets inside a stage
  static constexpr int U_IN = XBYTES + KS * ZBYTES;
  static constexpr int Y_OFF = NST * STAGE;
  // full[NST] empty[NST] accf[2] acce[2]
  static constexpr int NBAR = 2 * NST + 4;
  static constexpr int total(int nyb) {
    return Y_OFF + NEPI_F * nyb * YBOX + NBAR * 8 + 16 + 1024;   // + slack to align the base
  }
  static constexpr int NYB = total(2) <= 227 * 1024 ? 2 : 1;
  static constexpr int BAR_OFF = Y_OFF + NEPI_F * NYB * YBOX;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int TOTAL = MISC_OFF + 16 + 1024;
  static constexpr uint32_t TX = XBOX + KS * ZBYTES + UBYTES;  // bytes landing per stage
};


// Work item i of the forward -> (b, token tile, chunk): tile-major, so the
// CTAs working side by side (items i, i+1, ... handed out round-robin) read
// neighbouring 128-byte pieces of the same rows of x.  32-bit arithmetic:
// the host admits fewer than 2^31 items (lowrank_tc_supported).
struct Item {
  int chunk, b, t0;
};
__device__ __forceinline__ Item decode_tm(long long i, int nchunks, int ntiles) {
  Item it;
  const unsigned ii = static_cast<unsigned>(i);
  const unsigned tile = ii / static_cast<unsigned>(nchunks);
  it.chunk = static_cast<int>(ii - tile * static_cast<unsigned>(nchunks));
  it.b = static_cast<int>(tile / static_cast<unsigned>(ntiles));
  it.t0 = static_cast<int>(tile - static_cast<unsigned>(it.b) * static_cast<unsigned>(ntiles)) * BM;
  return it;
}

// fp32 pairs for the packed FMA (fma.rn.f32x2).
__device__ __forceinline__ float2 f2(uint32_t lo, uint32_t hi) {
  return make_float2(__uint_as_float(lo), __uint_as_float(hi));
}
// The two bf16 of a 32-bit word as an fp32 pair (exact).
__device__ __forceinline__ float2 bf2f(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
// Byte offset of the 16-byte chunk `chunk` (0..3) of row `row` in a tile
// with 64-byte rows stored by TMA with SWIZZLE_64B (address bits 4-5 XORed
// with bits 7-8; the tile 512-byte aligned).
__device__ __forceinline__ uint32_t sw64_offset(uint32_t row, uint32_t chunk) {
  const uint32_t o = row * 64u + chunk * 16u;
  return o ^ ((o >> 3) & 0x30u);
}

__device__ __forceinline__ uint32_t f2bf(float2 v) {
  __nv_bfloat162 h = __floats2bfloat162_rn(v.x, v.y);
  return *reinterpret_cast<uint32_t*>(&h);
}


// Shared-memory descriptor (fields as in sm100.cuh); layout 0 = no swizzle
// (8-row x 16-byte core matrices), 2 = 128-byte swizzle, 6 = 32-byte swizzle.
__device__ __forceinline__ uint64_t make_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t layout) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(layout) << 61);
}

// kind::f16 instruction descriptor with operand majors (0 = K-major, 1 = MN-major).
__host__ __device__ constexpr uint32_t idesc_major(uint32_t M, uint32_t N, uint32_t amaj,
                                                   uint32_t bmaj) {
  return idesc_bf16_f32(M, N) | (amaj << 15) | (bmaj << 16);
}

// RES: y includes the residual x (a template parameter: as a runtime flag
// its select sat in every piece of the epilogue, measured 2% slower).
template <int W, int KS, int HP, bool RES>
__global__ void __launch_bounds__(kFwdThreads, 1)
lr_fwd_tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_z,
          const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_y,
          int ntiles, int nbt, int nchunks, int hshift, uint64_t wns, int withhold, int C,
          int T) {
  using L = FwdLayout<W, KS, HP>;
  const int ucols = (CC >> hshift) * W;      // U columns of one chunk (H = 2^hshift)
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = align1k(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const long long items = static_cast<long long>(nchunks) * nbt;
  // this CTA's items: blockIdx.x, blockIdx.x + gridDim.x, ...
  const int nmine = items > blockIdx.x
                        ? static_cast<int>((items - 1 - blockIdx.x) / gridDim.x) + 1
                        : 0;

  const uint32_t bar_full = sb + L::BAR_OFF;
  const uint32_t bar_empty = bar_full + NST * 8;
  const uint32_t bar_accf = bar_empty + NST * 8;
  const uint32_t bar_acce = bar_accf + 16;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1 + NGRP);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_accf + 8 * a, 1);
      mbar_init(bar_acce + 8 * a, NGRP);
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_z);
    tma_prefetch_desc(&tm_u);
    tma_prefetch_desc(&tm_y);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------- producer --
    if (lane == 0) {
      const uint64_t pol_stream = policy_evict_first();
      const uint64_t pol_keep = policy_evict_last();   // z and U are re-read by many items
      int it = 0;
      for (; it < nmine && !withhold; ++it) {
        const int s = it % NST;
        const uint32_t ph = (it / NST) & 1;
        if (!mbar_wait(bar_empty + 8 * s, ph ^ 1, abort_flag, &g_tc_error, 1, wns)) break;
        const Item itm = decode_tm(blockIdx.x + static_cast<long long>(it) * gridDim.x,
                                   nchunks, ntiles);
        const uint32_t full = bar_full + 8 * s;
        const uint32_t st = sb + s * L::STAGE;
        mbar_expect_tx(full, L::TX);
        tma_load_3d(st, &tm_x, full, itm.chunk * CC, itm.t0 - (W - 1), itm.b, pol_stream);
        for (int ks = 0; ks < KS; ++ks)
          tma_load_3d(st + L::Z_IN + ks * L::ZBYTES, &tm_z, full, ks * 16, itm.t0, itm.b,
                      pol_keep);
        for (int a = 0; a < L::NA; ++a)
          tma_load_3d(st + L::U_IN + a * L::UATOM, &tm_u, full, itm.chunk * ucols + a * 64, 0, 0,
                      pol_keep);
      }
      // Let every load this thread issued land before the CTA can exit.
      for (int j = std::max(0, it - NST); j < it; ++j)
        drain_wait(bar_full + 8 * (j % NST), (j / NST) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      // A = z tile (K-major, 32-byte swizzle); B = the chunk's U columns in
      // natural order (MN-major, 128-byte swizzle, 64-column atoms).
      constexpr uint32_t idesc = idesc_major(BM, L::NCOL, 0, 1);
      int it = 0;
      for (; it < nmine; ++it) {
        const int s = it % NST;
        const uint32_t ph = (it / NST) & 1;
        const int a = it & 1;
        const uint32_t aph = (it >> 1) & 1;
        if (!mbar_wait(bar_acce + 8 * a, aph ^ 1, abort_flag, &g_tc_error, 2, wns)) break;
        if (!mbar_wait(bar_full + 8 * s, ph, abort_flag, &g_tc_error, 2, wns)) break;
        tc_fence_after();
        const uint32_t st = sb + s * L::STAGE;
        const uint32_t d = tmem + a * 256;
        for (int ks = 0; ks < KS; ++ks) {
          const uint64_t ad = desc_kmajor_sw32(st + L::Z_IN + ks * L::ZBYTES);
          const uint64_t bd = make_desc(st + L::U_IN + ks * 2048, L::UATOM, 1024, 2);
          mma_bf16(d, ad, bd, idesc, ks > 0 ? 1u : 0u);
        }
        mma_commit(bar_accf + 8 * a);
        mma_commit(bar_empty + 8 * s);
      }
      if (it > 0) drain_wait(bar_accf + 8 * ((it - 1) & 1), ((it - 1) >> 1) & 1);
    }
  } else {
    // --------------------------------------------------------- epilogue --
    // Two independent groups of 8 warps: group g takes the items it with
    // it % 2 == g, using TMEM accumulator g, so one group's loads, math and
    // stores overlap the other group's.  A warp owns 32 tokens (its TMEM
    // lanes) and 32 channels (four 8-channel pieces) of the item and stores
    // them itself from its staging box, so no group-wide barrier sits on
    // the output path; the accumulator is handed back right after the
    // warp's last TMEM load.
    const int g = (warp - 2) >> 3;
    const int lg = warp & 3;                 // TMEM lane group of this warp
    const int h = ((warp - 2) >> 2) & 1;     // channel half of the chunk
    const int tl = lg * 32 + lane;           // token within the tile
    const uint64_t pol_y = policy_evict_first();
    const uint32_t tbase = tmem + (static_cast<uint32_t>(lg * 32) << 16) + g * 256;
    const uint32_t ybase = sb + L::Y_OFF + (warp - 2) * L::NYB * L::YBOX;
    for (int it = g; it < nmine; it += 2) {
      const int s = it % NST;
      const uint32_t ph = (it / NST) & 1;
      const uint32_t aph = (it >> 1) & 1;
      // Every lane waits; the warp leaves together if any wait gave up, so
      // the .sync.aligned TMEM loads below always run converged.
      bool ok = mbar_wait(bar_accf + 8 * g, aph, abort_flag, &g_tc_error, 3, wns) &&
                mbar_wait(bar_full + 8 * s, ph, abort_flag, &g_tc_error, 3, wns);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t xt = sb + s * L::STAGE;
      const uint32_t ybuf = ybase + ((it >> 1) % L::NYB) * L::YBOX;
      if (lane == 0) bulk_wait_read<L::NYB - 1>();   // this box's previous store has read it
      __syncwarp();
      // Four 8-channel pieces per warp; tap k of the chunk's filter group gl
      // is column gl*W + k, and channel c of the chunk uses group c / H.
      constexpr int NCP = 8 / HP * W;        // TMEM columns of one piece
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int cch = 4 * h + q;           // 16-byte chunk of the 128-byte row
        uint32_t acc[NCP];
        // first filter group of the piece: cch*8/H (H = HP below 8)
        const int g0 = HP < 8 ? cch * 8 / HP : (cch * 8) >> hshift;
        tmem_ld_cols<NCP>(tbase + g0 * W, acc);
        uint4 xr[W];
#pragma unroll
        for (int k = 0; k < W; ++k) xr[k] = lds128(xt + sw128_offset(tl + (W - 1) - k, cch));
        tmem_wait_ld();
        tmem_regs_ready<NCP>(acc);
        if (q == 3) {                         // the accumulator is in registers
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_acce + 8 * g);
        }
        float2 o[4];
        const uint32_t x0[4] = {xr[0].x, xr[0].y, xr[0].z, xr[0].w};
#pragma unroll
        for (int p = 0; p < 4; ++p) o[p] = RES ? bf2f(x0[p]) : make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < W; ++k) {
          const uint32_t xw[4] = {xr[k].x, xr[k].y, xr[k].z, xr[k].w};
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            // channels 2p, 2p+1 of the piece use filter groups (2p)/HP, (2p+1)/HP
            const float2 wk = f2(acc[((2 * p) / HP) * W + k], acc[((2 * p + 1) / HP) * W + k]);
            o[p] = __ffma2_rn(wk, bf2f(xw[p]), o[p]);
          }
        }
        sts128(ybuf + sw64_offset(lane, q),
               make_uint4(f2bf(o[0]), f2bf(o[1]), f2bf(o[2]), f2bf(o[3])));
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar_empty + 8 * s);
        const Item itm = decode_tm(blockIdx.x + static_cast<long long>(it) * gridDim.x,
                                   nchunks, ntiles);
        const int cbox = itm.chunk * CC + 32 * h, tbox = itm.t0 + 32 * lg;
        // Boxes wholly past C or T are skipped; partly outside ones are
        // clipped by the tensor map.
        if (cbox < C && tbox < T) tma_store_3d(&tm_y, ybuf, cbox, tbox, itm.b, pol_y);
        bulk_commit();
      }
    }
    if (lane == 0) bulk_wait<0>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------ backward ----
//
// Chain rule of the forward (the pages state no backward; this is derived):
//   dx[s,c]   = res*dy[s,c] + sum_{k: s+k<T} w[s+k,c,k] dy[s+k,c]
//   dw[t,c,k] = dy[t,c] x[t-k,c]                          (kept on-chip, bf16)
//   dz[t,r]   = sum_{c,k} dw[t,c,k] U[r,c*W+k]            (over all channels)
//   dU[r,c*W+k] = sum_{b,t} z[t,r] dw[t,c,k]              (over all tokens)
// One pass over x, dy, z per (128-token tile, 64-channel chunk) item, four
// kinds of tensor-core MMA (all M = 128, fp32 accumulators in TMEM):
//   D_k[s,c]  = sum_r z[s+k,r] U[r,c*W+k]   (N = 64, K = R; the z operand is a
//               row-interleaved tile whose start moves 16 bytes per row, so
//               the shift by k tokens is a descriptor offset)  -> dx
//   dz[t,r]  += dw[t,:] U[r,:]^T            (N = R, K = 64*W; dw K-major)
//   dU^T[j,r]+= dw[:,j]^T z[:,r]            (N = R, K = 128 tokens; dw read
//               MN-major from the same tile, z MN-major from the same tile
//               as the D_k operand)
// dw lives in four 16 KB tiles (one per tap, 128 tokens x 64 channels,
// 128-byte swizzle), written once by the epilogue and read by both
// contractions.  The grid is S channel slices x P token splits; a CTA walks
// its slice chunk by chunk and, inside a chunk, its split tile by tile.  It
// keeps the dz accumulators of all its tiles and the dU accumulator of its
// current chunk in TMEM, and writes one fp32 partial per (slice, token) and
// per (split, column); a second kernel adds them in a fixed order.
//
// Roles: warp 0 producer (TMA boxes of x [t0-W+1, t0+128), dy [t0, t0+127+W)
// and z [t0, t0+127+W), plus one 1-D bulk copy of the chunk's U tiles per
// chunk), warp 1 TMEM owner and issuer of the D_k MMAs, warp 18 issuer of
// the dz and dU MMAs (two issuers, so the dx path never waits behind the dw
// path), warps 2-9 the dx group (reads
// D_k and dy, writes dx from registers, and frees each 32-channel half of D
// so the MMAs of the next item can start on it), warps 10-17 the dw group (forms dw into the
// dw tiles one tap pair at a time; at chunk ends it reads out the dU
// accumulator, at the end the dz ones).  The two groups run independently.

// RK = K-steps of 16 ranks (R padded to 16 * RK with zeros).
template <int W, int RK>
struct BwdLayout {
  static constexpr int RP = 16 * RK;                      // padded rank
  static constexpr int NT = W <= 2 ? 2 : 4;               // dw taps incl. zero padding
  static constexpr int XROWS = BM + W - 1;
  static constexpr int XBOX = XROWS * 128;
  static constexpr int XBYTES = round1k(XBOX);
  static constexpr int ZBOX = XROWS * 2 * RP;             // [RP/8 groups][XROWS][16 B]
  static constexpr int ZBYTES = round1k(ZBOX);
  static constexpr int NSTB = RK == 1 ? 3 : 2;
  static constexpr int STAGE = 2 * XBYTES + ZBYTES;       // x, dy, z
  static constexpr int UTAP = 2048 * RK;                  // U tile of one tap: [RP r][64 c]
  static constexpr int UBYTES = W * UTAP;                 // U tiles of one chunk
  static constexpr int UALLOC = round1k(UBYTES);
  static constexpr int DWTAP = BM * 128;                  // one tap of dw (16 KB)
  // Staged dx: for each warp of the dx group and each D part, one box of
  // 32 tokens x 16 channels (32-byte rows, 32-byte swizzle) that the warp
  // stores with TMA itself.
  static constexpr int DXBOX = 32 * 32;
  static constexpr int STG_OFF = 0;
  static constexpr int U_OFF = NSTB * STAGE;
  static constexpr int DW_OFF = U_OFF + 2 * UALLOC;
  static constexpr int DX_OFF = DW_OFF + NT * DWTAP;
  static constexpr int BAR_OFF = DX_OFF + NEPI * kDParts * DXBOX;
  // full[3] empty[3] dfull[P] dempty[P] dwfull[2] dwfree[2] ufull[2] ufree[2]
  // uafull[2] uaempty[2] dzfull  (P = kDParts)
  static constexpr int NBAR = 2 * NSTB + 2 * kDParts + 4 + 8 + 1;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int TOTAL = MISC_OFF + 16 + 1024;
  static constexpr uint32_t TX = 2 * XBOX + ZBOX;
  static constexpr int TM_D = 0;                          // W x 64 columns
  static constexpr int TM_DU = W * 64;                    // 2 buffers x NT/2 x RP
  static constexpr int TM_DZ = TM_DU + NT * RP;           // RP per tile of the split
  static constexpr int TPS_MAX = (512 - TM_DZ) / RP;
};

struct BwdArgs {
  float* dz_part;          // [S][B*T][RP]
  float* dU_part;          // [P][RP][C*W]
  const unsigned char* uimg;  // [nchunks][W][RP rows][128 B] swizzled U tiles
  int T, C, ntiles, nchunks, S, P, ntl;
  // Bounded waits give up after wait_ns; withhold != 0 makes the producer
  // issue no loads at all, so every wait of the other roles runs out (the
  // self-test of the failure path; 0 in normal use).
  unsigned long long wait_ns;
  int withhold;
};

// RES: dx includes the residual dy (a template parameter: as the runtime
// flag it was a select per 8-channel piece on the dx warps' path, measured
// 2% slower).
template <int W, int RK, bool RES>
__global__ void __launch_bounds__(kBwdThreads, 1)
lr_bwd_tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dy,
          const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_dx,
          const BwdArgs args) {
  using L = BwdLayout<W, RK>;
  constexpr int NST_ = L::NSTB;
  constexpr int RP = L::RP;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = align1k(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t wns = args.wait_ns;

  // This CTA's channel slice [ch0, ch1) and token-tile split [tl0, tl1).
  const int slice = blockIdx.x % args.S, split = blockIdx.x / args.S;
  const int ch0 = static_cast<int>(static_cast<long long>(args.nchunks) * slice / args.S);
  const int ch1 = static_cast<int>(static_cast<long long>(args.nchunks) * (slice + 1) / args.S);
  const int tl0 = static_cast<int>(static_cast<long long>(args.ntl) * split / args.P);
  const int tl1 = static_cast<int>(static_cast<long long>(args.ntl) * (split + 1) / args.P);
  const int ntile = tl1 - tl0, nchunk = ch1 - ch0;
  const int nitems = ntile * nchunk;
  const int64_t CW = static_cast<int64_t>(args.C) * W;
  const int64_t Ntok = static_cast<int64_t>(args.ntl / args.ntiles) * args.T;

  const uint32_t bar_full = sb + L::BAR_OFF;
  const uint32_t bar_empty = bar_full + NST_ * 8;
  const uint32_t bar_dfull = bar_empty + NST_ * 8;     // [kDParts]: one per channel part of D
  const uint32_t bar_dempty = bar_dfull + 8 * kDParts;  // [kDParts]
  const uint32_t bar_dwfull = bar_dempty + 8 * kDParts;  // [2]: one per tap pair of the dw tiles
  const uint32_t bar_dwfree = bar_dwfull + 16;   // [2]
  const uint32_t bar_ufull = bar_dwfree + 16;
  const uint32_t bar_ufree = bar_ufull + 16;
  const uint32_t bar_uafull = bar_ufree + 16;
  const uint32_t bar_uaempty = bar_uafull + 16;
  const uint32_t bar_dzfull = bar_uaempty + 16;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST_; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 2 + 2 * NEPI);   // both MMA issuers, both groups
    }
    for (int hh = 0; hh < kDParts; ++hh) {
      mbar_init(bar_dfull + 8 * hh, 1);
      mbar_init(bar_dempty + 8 * hh, NEPI);
    }
    for (int pr = 0; pr < 2; ++pr) {
      mbar_init(bar_dwfull + 8 * pr, NEPI);
      mbar_init(bar_dwfree + 8 * pr, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_ufull + 8 * a, 1);
      mbar_init(bar_ufree + 8 * a, 2);                // both MMA issuers read U
      mbar_init(bar_uafull + 8 * a, 1);
      mbar_init(bar_uaempty + 8 * a, NEPI);
    }
    mbar_init(bar_dzfull, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_dy);
    tma_prefetch_desc(&tm_z);
    tma_prefetch_desc(&tm_dx);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  // Taps past W of the padded dw tiles stay zero for the whole kernel.
  for (int i = threadIdx.x; i < (L::NT - W) * L::DWTAP / 16; i += blockDim.x)
    sts128(sb + L::DW_OFF + W * L::DWTAP + 16 * i, make_uint4(0, 0, 0, 0));
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The setup above touches no global memory.  From here on the kernel reads
  // its inputs and writes its outputs, so it waits for the kernels it depends
  // on (a no-op unless launched as a programmatic dependent), and lets the
  // reduction kernel that follows it be scheduled.
  griddep_wait();
  griddep_launch_dependents();

  // item n -> (local chunk lc = n / ntile, local tile lt = n % ntile), tracked
  // item by item in every role
  if (warp == 0) {
    // ---------------------------------------------------------- producer --
    if (lane == 0) {
      const uint64_t pol_stream = policy_evict_first();
      const uint64_t pol_keep = policy_evict_last();
      // item n = chunk lc, tile lt of the split = tile tt of sequence b
      const int b_first = tl0 / args.ntiles, tt_first = tl0 - b_first * args.ntiles;
      int lc = 0, lt = 0, b = b_first, tt = tt_first;
      auto next_item = [&]() {
        if (++lt == ntile) {
          lt = 0;
          ++lc;
          b = b_first;
          tt = tt_first;
        } else if (++tt == args.ntiles) {
          tt = 0;
          ++b;
        }
      };
      int n = 0;
      for (; n < nitems && !args.withhold; ++n, next_item()) {
        if (lt == 0) {
          const int ub = lc & 1;
          if (!mbar_wait(bar_ufree + 8 * ub, ((lc >> 1) & 1) ^ 1, abort_flag, &g_tc_error, 1,
                         wns))
            break;
          const uint32_t uf = bar_ufull + 8 * ub;
          mbar_expect_tx(uf, L::UBYTES);
          asm volatile(
              "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
              "[%0], [%1], %2, [%3], %4;" ::"r"(sb + L::U_OFF + ub * L::UALLOC),
              "l"(args.uimg + static_cast<size_t>(ch0 + lc) * L::UBYTES), "r"(L::UBYTES),
              "r"(uf), "l"(pol_keep)
              : "memory");
        }
        const int s = n % NST_;
        const uint32_t ph = (n / NST_) & 1;
        if (!mbar_wait(bar_empty + 8 * s, ph ^ 1, abort_flag, &g_tc_error, 1, wns)) break;
        const int t0 = tt * BM;
        const int c0 = (ch0 + lc) * CC;
        const uint32_t full = bar_full + 8 * s;
        const uint32_t st = sb + L::STG_OFF + s * L::STAGE;
        mbar_expect_tx(full, L::TX);
        tma_load_3d(st, &tm_x, full, c0, t0 - (W - 1), b, pol_stream);
        tma_load_3d(st + L::XBYTES, &tm_dy, full, c0, t0, b, pol_stream);
        asm volatile(
            "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::"
            "cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(st + 2 * L::XBYTES),
            "l"(reinterpret_cast<uint64_t>(&tm_z)), "r"(0), "r"(t0), "r"(0), "r"(b), "r"(full),
            "l"(pol_keep)
            : "memory");
      }
      for (int j = std::max(0, n - NST_); j < n; ++j)
        drain_wait(bar_full + 8 * (j % NST_), (j / NST_) & 1);
      const int nl = n > 0 ? (n - 1) / ntile + 1 : 0;      // chunks whose U load was issued
      for (int lc = std::max(0, nl - 2); lc < nl; ++lc)
        drain_wait(bar_ufull + 8 * (lc & 1), (lc >> 1) & 1);
    }
  } else if (warp == 1) {
    // --------------------------------------------------- D-MMA issuer --
    // D_k for every item: one MMA of N = 64 (the chunk's channels) per tap
    // and K-step, A = z K-major (shifted k rows), B = U MN-major.  The dx
    // group hands D back in kDParts channel parts, each right after loading
    // it into registers, so the next item's D is formed while the dx group
    // still computes on the current one.
    if (lane == 0) {
      const uint32_t zsbo = L::XROWS * 16;                    // stride of the two z halves
      int issued[kDParts] = {};
      bool ok = true;
      int lc = 0, lt = 0;                          // chunk and tile of item n
      auto next_item = [&]() {
        if (++lt == ntile) {
          lt = 0;
          ++lc;
        }
      };
      for (int n = 0; n < nitems && ok; ++n, next_item()) {
        const int s = n % NST_;
        if (lt == 0)
          ok = mbar_wait(bar_ufull + 8 * (lc & 1), (lc >> 1) & 1, abort_flag, &g_tc_error, 2,
                         wns);
        ok = ok && mbar_wait(bar_full + 8 * s, (n / NST_) & 1, abort_flag, &g_tc_error, 2, wns);
        if (!ok) break;
        const uint32_t zt = sb + L::STG_OFF + s * L::STAGE + 2 * L::XBYTES;
        const uint32_t ut = sb + L::U_OFF + (lc & 1) * L::UALLOC;
        // Descriptor bases; every operand below starts a multiple of 16
        // bytes further, which is that many units added to the start field
        // (shared-memory addresses stay below 256 KB, so it cannot carry).
        const uint64_t zd0 = make_desc(zt, zsbo, 128, 0);
        const uint64_t ud0 = make_desc(ut, 16, 1024, 2);
        // Once every part is free; every part is signalled on completion.
#pragma unroll
        for (int hh = 0; hh < kDParts; ++hh)
          ok = ok && mbar_wait(bar_dempty + 8 * hh, (n & 1) ^ 1, abort_flag, &g_tc_error, 2, wns);
        if (!ok) break;
        tc_fence_after();
        {
          constexpr uint32_t id_d64 = idesc_major(BM, CC, 0, 1);
#pragma unroll
          for (int k = 0; k < W; ++k)
#pragma unroll
            for (int ks = 0; ks < RK; ++ks)
              mma_bf16(tmem + L::TM_D + k * 64,
                       zd0 + static_cast<uint64_t>((16 * k + 2 * ks * zsbo) >> 4),
                       ud0 + static_cast<uint64_t>((k * L::UTAP + ks * 2048) >> 4),
                       id_d64, ks > 0 ? 1u : 0u);
#pragma unroll
          for (int hh = 0; hh < kDParts; ++hh) {
            mma_commit(bar_dfull + 8 * hh);
            ++issued[hh];
          }
        }
        if (!ok) break;
        mma_commit(bar_empty + 8 * s);
        if (lt == ntile - 1) mma_commit(bar_ufree + 8 * (lc & 1));
      }
      // Let every MMA this thread issued finish before TMEM is freed.
      for (int hh = 0; hh < kDParts; ++hh)
        if (issued[hh] > 0) drain_wait(bar_dfull + 8 * hh, (issued[hh] - 1) & 1);
    }
  } else if (warp == kDzduWarp) {
    // ------------------------------------------------- dz/dU-MMA issuer --
    // dz and dU for every item, one tap pair at a time as the dw group
    // finishes writing it.
    if (lane == 0) {
      constexpr uint32_t id_dz = idesc_major(BM, RP, 0, 0);   // A dw K-major, B U K-major
      constexpr uint32_t id_du = idesc_major(BM, RP, 1, 1);   // A dw^T MN-major, B z MN-major
      const uint32_t zsbo = L::XROWS * 16;
      bool ok = true;
      int issued_pair[2] = {0, 0};
      int lc = 0, lt = 0;                          // chunk and tile of item m
      auto next_item = [&]() {
        if (++lt == ntile) {
          lt = 0;
          ++lc;
        }
      };
      for (int m = 0; m < nitems && ok; ++m, next_item()) {
        const int s = m % NST_;
        const int ub = lc & 1;
        if (lt == 0) {
          ok = mbar_wait(bar_ufull + 8 * ub, (lc >> 1) & 1, abort_flag, &g_tc_error, 5, wns);
          if (lc >= 2)
            ok = ok && mbar_wait(bar_uaempty + 8 * ub, ((lc >> 1) & 1) ^ 1, abort_flag,
                                 &g_tc_error, 5, wns);
        }
        ok = ok && mbar_wait(bar_full + 8 * s, (m / NST_) & 1, abort_flag, &g_tc_error, 5, wns);
        if (!ok) break;
        const uint32_t dw = sb + L::DW_OFF;
        const uint32_t ut = sb + L::U_OFF + ub * L::UALLOC;
        const uint32_t zt = sb + L::STG_OFF + s * L::STAGE + 2 * L::XBYTES;
        // Descriptor bases (offsets below are multiples of 16 bytes, added to
        // the start field as for the D MMAs).
        const uint64_t dza = make_desc(dw, 16, 1024, 2), dzb = make_desc(ut, 16, 1024, 2);
        const uint64_t dua = make_desc(dw, L::DWTAP, 1024, 2), dub = make_desc(zt, 128, zsbo, 0);
        const uint32_t tdz = tmem + L::TM_DZ + lt * RP;
        const uint32_t tdu = tmem + L::TM_DU + ub * (L::NT / 2) * RP;
        const uint32_t first_dz = lc > 0 ? 1u : 0u, first_du = lt > 0 ? 1u : 0u;
#pragma unroll
        for (int pr = 0; pr < L::NT / 2; ++pr) {
          ok = mbar_wait(bar_dwfull + 8 * pr, m & 1, abort_flag, &g_tc_error, 5, wns);
          if (!ok) break;
          tc_fence_after();
          // Two accumulation chains, interleaved so that consecutive MMAs
          // never feed each other:
          //   dz[t, :]   (+)= the pair's 128 columns (tap-major, 16 per K-step)
          //   dU^T[j', :](+)= the tile's 128 tokens; M block pr = taps 2pr, 2pr+1
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int q = 8 * pr + i;
            const int k = q >> 2, cb = q & 3;
            if (k < W)
              mma_bf16(tdz, dza + static_cast<uint64_t>((k * L::DWTAP + cb * 32) >> 4),
                       dzb + static_cast<uint64_t>((k * L::UTAP + cb * 32) >> 4), id_dz,
                       q > 0 ? 1u : first_dz);
            mma_bf16(tdu + pr * RP,
                     dua + static_cast<uint64_t>((2 * pr * L::DWTAP + i * 2048) >> 4),
                     dub + static_cast<uint64_t>((i * 256) >> 4), id_du, i > 0 ? 1u : first_du);
          }
          mma_commit(bar_dwfree + 8 * pr);
          ++issued_pair[pr];
        }
        if (!ok) break;
        mma_commit(bar_empty + 8 * s);
        if (lt == ntile - 1) {
          mma_commit(bar_uafull + 8 * ub);
          mma_commit(bar_ufree + 8 * ub);
        }
      }
      if (ok && nitems > 0) mma_commit(bar_dzfull);
      // Let every MMA this thread issued finish before TMEM is freed.
      for (int pr = 0; pr < 2; ++pr)
        if (issued_pair[pr] > 0) drain_wait(bar_dwfree + 8 * pr, (issued_pair[pr] - 1) & 1);
    }
  } else {
    // ---------------------------------------------------------- epilogues --
    // Two groups of 8 warps that run independently, item by item:
    //   warps 2-9   (dx group): dx = res*dy + sum_k D_k dy[t+k], stored from
    //               registers; frees each half of D for the next item's MMAs.
    //   warps 10-17 (dw group): dw tiles, one tap pair at a time; the dU
    //               readout at chunk ends and the dz readout at the end.
    // In each group warp (w % 4) owns TMEM lanes 32*(w % 4) .. +31 (tokens)
    // and the two warps of a lane group split the chunk's channels.
    const bool dx_group = warp < 2 + NEPI;
    const int lg = warp & 3;
    const int h = ((warp - 2) >> 2) & 1;
    const int tl = lg * 32 + lane;
    const uint32_t tlane = static_cast<uint32_t>(lg * 32) << 16;
    bool ok = true;
    if (dx_group) {
      // dx[t] = res*dy[t] + sum_k D_k[t] dy[t+k]: each thread reads dy rows
      // t .. t+W-1 from the staged tile (the 128-byte swizzle keeps the 32
      // rows of a warp's read conflict-free).  Per D part a warp owns 32
      // tokens x 16 channels: it loads their W taps from TMEM in one go and
      // hands the part back to the MMA issuer at once, then writes dx into
      // its own 1 KB staging box, which it stores with TMA.
      const int wd = warp - 2;                              // 0..7 within the group
      const uint32_t dxst = sb + L::DX_OFF + wd * kDParts * L::DXBOX;
      const uint64_t pol_dx = policy_evict_first();
      // Item n = chunk lc, tile lt of the split = tile tt of sequence b,
      // advanced item by item (no division on this path).
      const int b_first = tl0 / args.ntiles, tt_first = tl0 - b_first * args.ntiles;
      int lc = 0, lt = 0, b = b_first, tt = tt_first;
      auto next_item = [&]() {
        if (++lt == ntile) {
          lt = 0;
          ++lc;
          b = b_first;
          tt = tt_first;
        } else if (++tt == args.ntiles) {
          tt = 0;
          ++b;
        }
      };
      for (int n = 0; n < nitems; ++n, next_item()) {
        const int s = n % NST_;
        const int t0 = tt * BM;
        const int c0 = (ch0 + lc) * CC;
        const uint32_t dyt = sb + L::STG_OFF + s * L::STAGE + L::XBYTES;
        ok = mbar_wait(bar_full + 8 * s, (n / NST_) & 1, abort_flag, &g_tc_error, 3, wns);
        if (!__all_sync(0xffffffffu, ok)) break;
        // The warp's box of a part: tokens t0 + 32*lg .. +31, channels
        // c0 + 32*hh + 16*h .. +15 (two 8-channel pieces).
        constexpr int PPC = CC / kDParts / 16;
        const bool box_in = t0 + 32 * lg < args.T;
#pragma unroll 1
        for (int hh = 0; hh < kDParts; ++hh) {
          ok = __all_sync(0xffffffffu, mbar_wait(bar_dfull + 8 * hh, n & 1, abort_flag,
                                                 &g_tc_error, 3, wns));
          if (!ok) break;
          tc_fence_after();
          uint32_t dk[PPC][W][8];
#pragma unroll
          for (int q = 0; q < PPC; ++q)
#pragma unroll
            for (int k = 0; k < W; ++k)
              tmem_ld8(tmem + tlane + L::TM_D + k * 64 + 8 * (2 * PPC * hh + PPC * h + q),
                       dk[q][k]);
          tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < PPC; ++q)
#pragma unroll
            for (int k = 0; k < W; ++k) tmem_regs_ready<8>(dk[q][k]);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(bar_dempty + 8 * hh);
            bulk_wait_read<1>();          // this box's previous store has read it
          }
          __syncwarp();
          const uint32_t box = dxst + hh * L::DXBOX;
#pragma unroll
          for (int q = 0; q < PPC; ++q) {
            const int cch = 2 * PPC * hh + PPC * h + q;
            float2 o[4];
#pragma unroll
            for (int k = 0; k < W; ++k) {
              const uint4 g = lds128(dyt + sw128_offset(tl + k, cch));
              const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
              if (k == 0) {
#pragma unroll
                for (int p = 0; p < 4; ++p)
                  o[p] = RES ? bf2f(gw[p]) : make_float2(0.f, 0.f);
              }
#pragma unroll
              for (int p = 0; p < 4; ++p)
                o[p] = __ffma2_rn(f2(dk[q][k][2 * p], dk[q][k][2 * p + 1]), bf2f(gw[p]), o[p]);
            }
            sts128(box + sw32_offset(lane, 8 * q),
                   make_uint4(f2bf(o[0]), f2bf(o[1]), f2bf(o[2]), f2bf(o[3])));
          }
          fence_proxy_async_smem();
          __syncwarp();
          const int cbox = c0 + 32 * hh + 16 * h;
          if (lane == 0) {
            // Boxes wholly past C or T are skipped; partly outside ones are
            // clipped by the tensor map.
            if (box_in && cbox < args.C)
              tma_store_3d(&tm_dx, box, cbox, t0 + 32 * lg, b, pol_dx);
            bulk_commit();
          }
        }
        if (!ok) break;
        if (lane == 0) mbar_arrive(bar_empty + 8 * s);
      }
      if (lane == 0) bulk_wait<0>();
    } else {
      // dw[t,c,k] = dy[t,c] x[t-k,c].  Thread (chunk wc of 8 channels, run of
      // 4 tokens) keeps a window of x rows in registers, so each x and dy row
      // is read once.  The product of two bf16 is exact in fp32, so one
      // bf16x2 multiply (round to nearest) gives the same bf16 as the fp32
      // product rounded once.
      const int wt = threadIdx.x - (2 + NEPI) * 32;     // 0..255 in the dw group
      const int wc = wt & 7;                            // 16-byte chunk of the row
      const int r0 = (wt >> 3) * 4;                     // first token of the run
      int lc = 0, lt = 0;                               // chunk and tile of item n
      auto next_item = [&]() {
        if (++lt == ntile) {
          lt = 0;
          ++lc;
        }
      };
      for (int n = 0; n < nitems; ++n, next_item()) {
        const int s = n % NST_;
        const int c0 = (ch0 + lc) * CC;
        const uint32_t xt = sb + L::STG_OFF + s * L::STAGE, dyt = xt + L::XBYTES;
        ok = mbar_wait(bar_full + 8 * s, (n / NST_) & 1, abort_flag, &g_tc_error, 3, wns);
        if (!__all_sync(0xffffffffu, ok)) break;
        // x box row r holds token t0 - (W-1) + r; token r0 + i needs rows
        // r0 + i + (W-1) - k.
        uint4 xw[4 + W - 1];
#pragma unroll
        for (int j = 0; j < 4 + W - 1; ++j) xw[j] = lds128(xt + sw128_offset(r0 + j, wc));
        uint4 gw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) gw[i] = lds128(dyt + sw128_offset(r0 + i, wc));
#pragma unroll
        for (int pr = 0; pr < L::NT / 2; ++pr) {
          ok = mbar_wait(bar_dwfree + 8 * pr, (n & 1) ^ 1, abort_flag, &g_tc_error, 3, wns);
          if (!__all_sync(0xffffffffu, ok)) break;
#pragma unroll
          for (int k = 2 * pr; k < 2 * pr + 2; ++k) {
            if (k < W) {
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gw[i]);
                const __nv_bfloat162* x2 =
                    reinterpret_cast<const __nv_bfloat162*>(&xw[i + (W - 1) - k]);
                __nv_bfloat162 p2[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) p2[e] = __hmul2(g2[e], x2[e]);
                sts128(sb + L::DW_OFF + k * L::DWTAP + sw128_offset(r0 + i, wc),
                       *reinterpret_cast<const uint4*>(p2));
              }
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_dwfull + 8 * pr);
        }
        if (!ok) break;
        if (lane == 0) mbar_arrive(bar_empty + 8 * s);
        // End of a chunk: read out its dU^T accumulator (TMEM lanes = columns).
        if (lt == ntile - 1) {
          const int ub = lc & 1;
          ok = mbar_wait(bar_uafull + 8 * ub, (lc >> 1) & 1, abort_flag, &g_tc_error, 3, wns);
          if (!__all_sync(0xffffffffu, ok)) break;
          tc_fence_after();
          if (h < L::NT / 2) {
            uint32_t v[RP];
#pragma unroll
            for (int ks = 0; ks < RK; ++ks)
              tmem_ld16(tmem + tlane + L::TM_DU + ub * (L::NT / 2) * RP + h * RP + 16 * ks,
                        v + 16 * ks);
            tmem_wait_ld();
            tmem_regs_ready<RP>(v);
            const int jp = h * 128 + tl;                  // tap-major column of the chunk
            const int k = jp >> 6, c = c0 + (jp & 63);
            if (k < W && c < args.C) {
              float* dst = args.dU_part + static_cast<size_t>(split) * RP * CW +
                           static_cast<int64_t>(c) * W + k;
#pragma unroll
              for (int r = 0; r < RP; ++r)
                dst[static_cast<int64_t>(r) * CW] = __uint_as_float(v[r]);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_uaempty + 8 * ub);
        }
      }
      // The dz accumulators of every tile of the split.
      if (ok && nitems > 0) {
        ok = mbar_wait(bar_dzfull, 0, abort_flag, &g_tc_error, 3, wns);
        if (__all_sync(0xffffffffu, ok)) {
          tc_fence_after();
          for (int lt = h; lt < ntile; lt += 2) {
            uint32_t v[RP];
#pragma unroll
            for (int ks = 0; ks < RK; ++ks)
              tmem_ld16(tmem + tlane + L::TM_DZ + lt * RP + 16 * ks, v + 16 * ks);
            tmem_wait_ld();
            tmem_regs_ready<RP>(v);
            const int gt = tl0 + lt;
            const int b = gt / args.ntiles, t = (gt - b * args.ntiles) * BM + tl;
            if (t < args.T) {
              float4* dst = reinterpret_cast<float4*>(
                  args.dz_part + (static_cast<size_t>(slice) * Ntok +
                                  static_cast<int64_t>(b) * args.T + t) * RP);
#pragma unroll
              for (int i = 0; i < RP / 4; ++i)
                dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                     __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// U rearranged into the shared-memory image of the backward's U tiles: for
// chunk ch and tap k, a [RP r][64 c] tile with 128-byte rows and the TMA
// 128-byte swizzle, element (r, c) = U[r, ((64*ch + c)/H)*W + k] (zero past
// C and for the padding ranks r >= R).  With tied filters (H > 1) every
// channel gets its group's column, so the kernel sees per-channel filters
// that are equal within a group; dU of a group is then the sum of the
// per-channel dU over its H channels (the tied reduction below).
template <int W, int RK>
__global__ void lr_u_image(const __nv_bfloat16* __restrict__ U, unsigned char* __restrict__ img,
                           int C, int H, int R, int nchunks) {
  constexpr int RP = 16 * RK;
  // The backward kernel launched after this one waits for it to complete
  // before it reads the image; it may be scheduled at once.
  griddep_launch_dependents();
  const int64_t GW = static_cast<int64_t>(C / H) * W;
  const int total = nchunks * W * RP * 8;              // 16-byte pieces
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const int piece = i & 7, r = (i >> 3) % RP, tile = (i >> 3) / RP;
    const int k = tile % W, ch = tile / W;
    uint32_t w4[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      uint32_t pair = 0;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int c = ch * CC + piece * 8 + 2 * e + hh;
        uint32_t bits = 0;
        if (c < C && r < R)
          bits = __bfloat16_as_ushort(
              U[static_cast<int64_t>(r) * GW + static_cast<int64_t>(c / H) * W + k]);
        pair |= bits << (16 * hh);
      }
      w4[e] = pair;
    }
    const uint32_t off = static_cast<uint32_t>(r) * 128u + ((static_cast<uint32_t>(piece) ^ (r & 7u)) << 4);
    *reinterpret_cast<uint4*>(img + static_cast<size_t>(tile) * (2048 * RK) + off) =
        make_uint4(w4[0], w4[1], w4[2], w4[3]);
  }
}

// dz[n, r] = sum_s dz_part[s][n][r]; dU[r, j] = sum_p dU_part[p][r][j]; fixed
// order, fp32, rounded once to bf16.  Four outputs per thread.  The partials
// hold RP >= R ranks (R a multiple of 8); the padding ranks are skipped.
__global__ void lr_reduce_tc(const float* __restrict__ dz_part, const float* __restrict__ dU_part,
                             __nv_bfloat16* __restrict__ dz, __nv_bfloat16* __restrict__ dU,
                             int64_t nz4, int S, int64_t nU4, int P, int R, int RP, int64_t CW) {
  griddep_wait();        // the partial sums of the backward kernel launched before this one
  const int64_t total = nz4 + nU4;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4* src;
    int64_t stride;
    int cnt;
    __nv_bfloat16* out;
    int64_t j;
    if (i < nz4) {
      // i = n * RP/4 + r/4 in the partials; written at n * R + r
      const int64_t n = i / (RP / 4);
      const int r = static_cast<int>(i - n * (RP / 4)) * 4;
      if (r >= R) continue;
      src = reinterpret_cast<const float4*>(dz_part) + i;
      stride = nz4;
      cnt = S;
      out = dz;
      j = (n * R + r) / 4;
    } else {
      // the first R rows of each split's [RP][C*W] partial
      j = i - nz4;
      src = reinterpret_cast<const float4*>(dU_part) + j;
      stride = static_cast<int64_t>(RP) * CW / 4;
      cnt = P;
      out = dU;
    }
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p = 0; p < cnt; ++p) {
      const float4 v = __ldcs(src + p * stride);
      a.x += v.x;
      a.y += v.y;
      a.z += v.z;
      a.w += v.w;
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y), hi = __floats2bfloat162_rn(a.z, a.w);
    uint2 pk = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
    *reinterpret_cast<uint2*>(out + 4 * j) = pk;
  }
}

// Tied filters: dU[r, g*W + k] = sum_p sum_{h<H} dU_part[p][r][(g*H + h)*W + k],
// p outer and h inner (a fixed order), one output a thread.
__global__ void lr_reduce_du_tied(const float* __restrict__ dU_part,
                                  __nv_bfloat16* __restrict__ dU, int R, int RP, int H, int W,
                                  int64_t GW, int P) {
  const int64_t CW = GW * H;
  const int64_t total = static_cast<int64_t>(R) * GW;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / GW, j = i - r * GW;
    const int64_t g = j / W, k = j - g * W;
    const float* src = dU_part + r * CW + g * H * W + k;
    float a = 0.f;
    for (int p = 0; p < P; ++p) {
      const float* sp = src + static_cast<int64_t>(p) * RP * CW;
      for (int h = 0; h < H; ++h) a += __ldcs(sp + h * W);
    }
    dU[i] = __float2bfloat16_rn(a);
  }
}

// ------------------------------------------------------------------ host ----


// Wait limit of the bounded waits and the self-test switch (withhold: the
// producer issues no loads, so every other role's wait runs out).
struct Diag {
  uint64_t wait_ns = kWaitLimitNs;
  int withhold = 0;
};

// Launch as a programmatic dependent of the previous kernel in the stream:
// it may be scheduled before that kernel ends and waits for it in
// griddep_wait().
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem,
                       cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// The shared-memory opt-in is recorded per kernel instance; the two RES
// instances of a layout are two kernels.
template <int W, int KS, int HP, bool RES>
struct FwdKernelTag {};

template <int W, int KS, int HP, bool RES>
cudaError_t launch_fwd(const void* x, const void* z, const void* U, void* y, const Shape& s,
                       cudaStream_t st, const Diag& dg) {
  using L = FwdLayout<W, KS, HP>;
  CUtensorMap tx, tz, tu, ty;
  if (!make_tmap_3d(&tx, x, true, s.C, s.T, s.B, CC, BM + W - 1, 128) ||
      !make_tmap_3d(&tz, z, true, s.R, s.T, s.B, 16, BM, 32) ||
      !make_tmap_3d(&tu, U, true, s.G() * s.W, s.R, 1, 64, 16 * KS, 128) ||
      !make_tmap_3d(&ty, y, true, s.C, s.T, s.B, 32, 32, 64))
    return cudaErrorInvalidValue;
  const int ntiles = static_cast<int>((s.T + BM - 1) / BM);
  const int nchunks = static_cast<int>((s.C + CC - 1) / CC);
  const long long nbt = static_cast<long long>(s.B) * ntiles;
  const long long items = nbt * nchunks;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorNoDevice;
  const long long grid = std::min<long long>(sms, items);
  auto kern = lr_fwd_tc<W, KS, HP, RES>;
  cudaError_t e = set_smem<FwdKernelTag<W, KS, HP, RES>>(kern, L::TOTAL);
  if (e != cudaSuccess) return e;
  kern<<<static_cast<unsigned>(grid), kFwdThreads, L::TOTAL, st>>>(
      tx, tz, tu, ty, ntiles, static_cast<int>(nbt), nchunks,
      __builtin_ctzll(static_cast<unsigned long long>(s.H)), dg.wait_ns, dg.withhold,
      static_cast<int>(s.C), static_cast<int>(s.T));
  return cudaGetLastError();
}

// ---- backward host side

struct TcBwdPlan {
  int S = 0, P = 0, ntiles = 0, nchunks = 0, ntl = 0;
  size_t dz_off = 0, dU_off = 0, img_off = 0, total = 0;
};

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int rk_of(int64_t R) { return R > 16 ? 2 : 1; }

int tps_max(int64_t W, int RK) {
  if (RK == 2) {
    switch (W) {
      case 1: return BwdLayout<1, 2>::TPS_MAX;
      case 2: return BwdLayout<2, 2>::TPS_MAX;
      case 3: return BwdLayout<3, 2>::TPS_MAX;
      default: return BwdLayout<4, 2>::TPS_MAX;
    }
  }
  switch (W) {
    case 1: return BwdLayout<1, 1>::TPS_MAX;
    case 2: return BwdLayout<2, 1>::TPS_MAX;
    case 3: return BwdLayout<3, 1>::TPS_MAX;
    default: return BwdLayout<4, 1>::TPS_MAX;
  }
}

// Choose S channel slices x P token splits (S * P CTAs, one per SM when
// possible): each CTA's dz accumulators must fit TMEM (tiles per split <=
// tps_max), and the estimate balances the largest CTA's streamed bytes
// against the fp32 partial sums written and re-read by the reduction.
TcBwdPlan plan_bwd_tc(const Shape& s, int nsm) {
  TcBwdPlan p;
  p.ntiles = static_cast<int>((s.T + BM - 1) / BM);
  p.nchunks = static_cast<int>((s.C + CC - 1) / CC);
  p.ntl = static_cast<int>(s.B * p.ntiles);
  const int RK = rk_of(s.R);
  const size_t RP = 16 * static_cast<size_t>(RK);
  const int tmax = tps_max(s.W, RK);
  const double item = 3.0 * BM * CC * 2;
  const double N = static_cast<double>(s.B) * s.T, CW = static_cast<double>(s.C) * s.W;
  double best = -1;
  const int pmin = (p.ntl + tmax - 1) / tmax;
  for (int P = pmin; P <= std::max(pmin, std::min(p.ntl, nsm)); ++P) {
    const int tps = (p.ntl + P - 1) / P;
    if (tps > tmax) continue;
    const int S = std::max(1, std::min(p.nchunks, nsm / P));
    const int cps = (p.nchunks + S - 1) / S;
    const double waves = std::ceil(static_cast<double>(S) * P / nsm);
    const double cost = waves * cps * tps * item + 2.0 * 64.0 * (S * N + P * CW) / (S * P);
    if (best < 0 || cost < best) {
      best = cost;
      p.S = S;
      p.P = P;
    }
  }
  p.dz_off = 0;
  p.dU_off = align_up(static_cast<size_t>(p.S) * s.B * s.T * RP * sizeof(float), 256);
  p.img_off = p.dU_off + align_up(static_cast<size_t>(p.P) * RP * s.C * s.W * sizeof(float), 256);
  p.total = p.img_off + align_up(static_cast<size_t>(p.nchunks) * s.W * 2048 * RK, 256);
  return p;
}

// One shared-memory opt-in record per backward kernel instance (the RES
// instances of a layout are two kernels).
template <int W, int RK, bool RES>
struct BwdKernelTag {};

template <int W, int RK, bool RES>
cudaError_t launch_bwd(const void* x, const void* z, const void* U, const void* dy, void* dx,
                       void* dz, void* dU, void* ws, const Shape& s, const TcBwdPlan& p,
                       cudaStream_t st, const Diag& dg) {
  using L = BwdLayout<W, RK>;
  CUtensorMap tx, tdy, tz, tdx;
  // z [B][T][R] seen as [B][R/8 groups][T][8]: group g of token t at byte
  // offset t*2R + 16g.  The box covers RP/8 groups; groups past R/8 read as
  // zero (the padding ranks).
  const uint64_t R = static_cast<uint64_t>(s.R);
  const uint64_t zd[4] = {8, static_cast<uint64_t>(s.T), R / 8, static_cast<uint64_t>(s.B)};
  const uint64_t zs[3] = {R * 2, 16, static_cast<uint64_t>(s.T) * R * 2};
  const uint32_t zb[4] = {8, static_cast<uint32_t>(L::XROWS), static_cast<uint32_t>(L::RP / 8), 1};
  if (!make_tmap_3d(&tx, x, true, s.C, s.T, s.B, CC, L::XROWS, 128) ||
      !make_tmap_3d(&tdy, dy, true, s.C, s.T, s.B, CC, L::XROWS, 128) ||
      !make_tmap_3d(&tdx, dx, true, s.C, s.T, s.B, 16, 32, 32) ||
      !make_tmap_4d_bf16(&tz, z, zd, zs, zb))
    return cudaErrorInvalidValue;
  unsigned char* base = static_cast<unsigned char*>(ws);
  BwdArgs a;
  a.dz_part = reinterpret_cast<float*>(base + p.dz_off);
  a.dU_part = reinterpret_cast<float*>(base + p.dU_off);
  a.uimg = base + p.img_off;
  a.T = static_cast<int>(s.T);
  a.C = static_cast<int>(s.C);
  a.ntiles = p.ntiles;
  a.nchunks = p.nchunks;
  a.S = p.S;
  a.P = p.P;
  a.ntl = p.ntl;
  a.wait_ns = dg.wait_ns;
  a.withhold = dg.withhold;
  {
    const int pieces = p.nchunks * W * L::RP * 8;
    lr_u_image<W, RK><<<std::min(1184, (pieces + 255) / 256), 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(U), base + p.img_off, static_cast<int>(s.C),
        static_cast<int>(s.H), static_cast<int>(s.R), p.nchunks);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  static_assert(L::TOTAL <= 227 * 1024, "backward shared memory");
  auto kern = lr_bwd_tc<W, RK, RES>;
  cudaError_t e = set_smem<BwdKernelTag<W, RK, RES>>(kern, L::TOTAL);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, static_cast<unsigned>(p.S * p.P), kBwdThreads, L::TOTAL, st, tx, tdy, tz,
                 tdx, a);
  if (e != cudaSuccess) return e;
  // Per-channel dU partials reduce straight to dU when H = 1; tied filters
  // add their H channels in a second small kernel.
  const int64_t nz4 = s.B * s.T * L::RP / 4, nU4 = s.H == 1 ? s.R * s.C * s.W / 4 : 0;
  const int blocks = static_cast<int>(std::min<int64_t>((nz4 + nU4 + 255) / 256, 148 * 8));
  e = launch_pdl(lr_reduce_tc, static_cast<unsigned>(blocks), 256u, 0, st,
                 static_cast<const float*>(a.dz_part), static_cast<const float*>(a.dU_part),
                 static_cast<__nv_bfloat16*>(dz), static_cast<__nv_bfloat16*>(dU), nz4, p.S, nU4,
                 p.P, static_cast<int>(s.R), static_cast<int>(L::RP), s.C * s.W);
  if (e != cudaSuccess || s.H == 1) return e;
  const int64_t GW = s.G() * s.W;
  const int tb = static_cast<int>(std::min<int64_t>((s.R * GW + 255) / 256, 148 * 8));
  lr_reduce_du_tied<<<tb, 256, 0, st>>>(a.dU_part, static_cast<__nv_bfloat16*>(dU),
                                        static_cast<int>(s.R), L::RP, static_cast<int>(s.H),
                                        W, GW, p.P);
  return cudaGetLastError();
}

template <int KS, int HP, bool RES>
cudaError_t fwd_res(const void* x, const void* z, const void* U, void* y, const Shape& s,
                    cudaStream_t st, const Diag& dg) {
  switch (s.W) {
    case 1: return launch_fwd<1, KS, HP, RES>(x, z, U, y, s, st, dg);
    case 2: return launch_fwd<2, KS, HP, RES>(x, z, U, y, s, st, dg);
    case 3: return launch_fwd<3, KS, HP, RES>(x, z, U, y, s, st, dg);
    default: return launch_fwd<4, KS, HP, RES>(x, z, U, y, s, st, dg);
  }
}

template <int KS, int HP>
cudaError_t fwd_hp(const void* x, const void* z, const void* U, void* y, const Shape& s,
                   cudaStream_t st, const Diag& dg) {
  return s.residual ? fwd_res<KS, HP, true>(x, z, U, y, s, st, dg)
                    : fwd_res<KS, HP, false>(x, z, U, y, s, st, dg);
}

template <int KS>
cudaError_t fwd_w(const void* x, const void* z, const void* U, void* y, const Shape& s, int hp,
                  cudaStream_t st, const Diag& dg) {
  switch (hp) {
    case 1: return fwd_hp<KS, 1>(x, z, U, y, s, st, dg);
    case 2: return fwd_hp<KS, 2>(x, z, U, y, s, st, dg);
    case 4: return fwd_hp<KS, 4>(x, z, U, y, s, st, dg);
    default: return fwd_hp<KS, 8>(x, z, U, y, s, st, dg);
  }
}

template <int W, int RK>
cudaError_t bwd_res(const void* x, const void* z, const void* U, const void* dy, void* dx,
                    void* dz, void* dU, void* ws, const Shape& s, const TcBwdPlan& p,
                    cudaStream_t st, const Diag& dg) {
  return s.residual ? launch_bwd<W, RK, true>(x, z, U, dy, dx, dz, dU, ws, s, p, st, dg)
                    : launch_bwd<W, RK, false>(x, z, U, dy, dx, dz, dU, ws, s, p, st, dg);
}

cudaError_t bwd_dispatch(const void* x, const void* z, const void* U, const void* dy, void* dx,
                         void* dz, void* dU, void* ws, const Shape& s, cudaStream_t st,
                         const Diag& dg) {
  const int nsm = sm_count();
  if (nsm <= 0) return cudaErrorNoDevice;
  const TcBwdPlan p = plan_bwd_tc(s, nsm);
  if (rk_of(s.R) == 2) {
    switch (s.W) {
      case 1: return bwd_res<1, 2>(x, z, U, dy, dx, dz, dU, ws, s, p, st, dg);
      case 2: return bwd_res<2, 2>(x, z, U, dy, dx, dz, dU, ws, s, p, st, dg);
      case 3: return bwd_res<3, 2>(x, z, U, dy, dx, dz, dU, ws, s, p, st, dg);
      default: return bwd_res<4, 2>(x, z, U, dy, dx, dz, dU, ws, s, p, st, dg);
    }
  }
  switch (s.W) {
    case 1: return bwd_res<1, 1>(x, z, U, dy, dx, dz, dU, ws, s, p, st, dg);
    case 2: return bwd_res<2, 1>(x, z, U, dy, dx, dz, dU, ws, s, p, st, dg);
    case 3: return bwd_res<3, 1>(x, z, U, dy, dx, dz, dU, ws, s, p, st, dg);
    default: return bwd_res<4, 1>(x, z, U, dy, dx, dz, dU, ws, s, p, st, dg);
  }
}

}  // namespace

bool lowrank_bwd_tc_supported(const Shape& s) {
  return s.bf16 && s.H >= 1 && s.R >= 8 && s.R <= 32 && s.R % 8 == 0 && s.W >= 1 && s.W <= 4 &&
         s.B * ((s.T + BM - 1) / BM) < (int64_t(1) << 30) && s.T < (int64_t(1) << 30) &&
         s.C < (int64_t(1) << 24);
}

size_t lowrank_bwd_tc_workspace(const Shape& s) {
  if (!lowrank_bwd_tc_supported(s)) return 0;
  const int nsm = sm_count();
  return plan_bwd_tc(s, nsm > 0 ? nsm : 148).total;
}

cudaError_t lowrank_bwd_tc(const void* x, const void* z, const void* U, const void* dy,
                           void* dx, void* dz, void* dU, void* ws, const Shape& s,
                           cudaStream_t st) {
  if (!lowrank_bwd_tc_supported(s)) return cudaErrorNotSupported;
  return bwd_dispatch(x, z, U, dy, dx, dz, dU, ws, s, st, Diag{});
}

cudaError_t lowrank_bwd_tc_selftest(const void* x, const void* z, const void* U, const void* dy,
                                    void* dx, void* dz, void* dU, void* ws, const Shape& s,
                                    uint64_t wait_ns, cudaStream_t st) {
  if (!lowrank_bwd_tc_supported(s)) return cudaErrorNotSupported;
  Diag dg;
  dg.wait_ns = wait_ns;
  dg.withhold = 1;
  return bwd_dispatch(x, z, U, dy, dx, dz, dU, ws, s, st, dg);
}

// Forward: tied filters need whole groups in a 64-channel chunk and a U
// column offset per chunk ((64/H)*W columns) on a 16-byte boundary, which
// TMA requires; the U rows ((C/H)*W columns) must be a multiple of 16 bytes.
bool lowrank_tc_supported(const Shape& s) {
  const bool pow2 = (s.H & (s.H - 1)) == 0;
  const bool tie_ok = s.H == 1 || (pow2 && s.H <= 64 && (64 / s.H * s.W) % 8 == 0 &&
                                   (s.G() * s.W) % 8 == 0);
  return s.bf16 && tie_ok && s.R >= 8 && s.R <= 32 && s.R % 8 == 0 && s.W >= 1 && s.W <= 4 &&
         s.B * ((s.T + BM - 1) / BM) < (int64_t(1) << 30) && s.T < (int64_t(1) << 30) &&
         s.C < (int64_t(1) << 24) &&
         s.B * ((s.T + BM - 1) / BM) * ((s.C + CC - 1) / CC) < (int64_t(1) << 31);
}

namespace {
cudaError_t fwd_dispatch(const void* x, const void* z, const void* U, void* y, const Shape& s,
                         cudaStream_t st, const Diag& dg) {
  const int hp = s.H >= 8 ? 8 : static_cast<int>(s.H);
  switch (s.R > 16 ? 2 : 1) {
    case 1: return fwd_w<1>(x, z, U, y, s, hp, st, dg);
    default: return fwd_w<2>(x, z, U, y, s, hp, st, dg);
  }
}
}  // namespace

cudaError_t lowrank_fwd_tc(const void* x, const void* z, const void* U, void* y,
                           const Shape& s, cudaStream_t st) {
  if (!lowrank_tc_supported(s)) return cudaErrorNotSupported;
  return fwd_dispatch(x, z, U, y, s, st, Diag{});
}

cudaError_t lowrank_fwd_tc_selftest(const void* x, const void* z, const void* U, void* y,
                                    const Shape& s, uint64_t wait_ns, cudaStream_t st) {
  if (!lowrank_tc_supported(s)) return cudaErrorNotSupported;
  Diag dg;
  dg.wait_ns = wait_ns;
  dg.withhold = 1;
  return fwd_dispatch(x, z, U, y, s, st, dg);
}

cudaError_t lowrank_tc_error(unsigned int* out, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_tc_error, sizeof(unsigned int));
  if (e != cudaSuccess || !reset) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(unsigned int));
}

}  // namespace dsc

// headwise_tma.cu -- head-wise Dynamic Short Convolution, forward and backward,
// with TMA-staged tiles (bf16; the (H, W) pairs listed at `item_width`).
//
// y[b,t,c] = res*x[b,t,c] + sum_{k<W} w[b,t,c/H,k] * x[b,t-k,c]   (x = 0 before t = 0)
// ("Technische Samenvatting: Dynamische Korte Convoluties Verbeteren
// Transformers", Methodologie: Mechanisme, Parametrisatie item 2, Plaatsing.)
// Backward (chain rule of that definition):
//   dx[b,s,c]   = res*dy[b,s,c] + sum_{k: s+k<T} w[b,s+k,c/H,k] dy[b,s+k,c]
//   dw[b,t,g,k] = sum_{c in group g} dy[b,t,c] x[b,t-k,c]
//
// Pure streams over HBM.  A work item is (b, 128-token tile, chunk of 64 or
// 128 channels); one persistent CTA per SM takes items round-robin in
// tile-major order, so neighbouring CTAs read neighbouring pieces of the
// same rows.
//   warp 0      TMA producer, 4-stage ring: x rows [t0-W+1, t0+128) (the
//               rows before t = 0 read as zero: the causal padding), in the
//               backward also dy rows and w rows [t0, t0+127+W) (rows past T
//               read as zero, which drops the terms with s+k >= T), and the
//               w rows of the tile: the chunk's groups x W taps.
//   warps 1-16  two independent groups of 8 warps that take alternate items,
//               each with its own staged output tiles; in a group the warp
//               (lane group lg = w % 4, half h) owns tokens 32*lg .. +31 and
//               half of the chunk's channels (8-channel pieces, which make
//               whole groups since H >= 8; in the H = 64 backward a warp
//               owns 16 tokens, two adjacent lanes each, see TOK2).  Outputs
//               go to staged tiles that one thread of the group stores with
//               TMA (dw of the padded-box layouts from registers).
// Every mbarrier wait is bounded (sm100.cuh); a timeout records a code in
// this file's device error word and the CTA returns.
#include <cuda_bf16.h>

#include <algorithm>

#include "dsc_common.cuh"
#include "dsc_internal.h"
#include "sm100.cuh"

namespace dsc {
namespace {

using namespace sm100;

// Set when a bounded wait gives up: 1 = producer, 3 = epilogue, 4 = store.
__device__ unsigned int g_hw_error = 0;

constexpr int BM = 128;      // tokens per tile
constexpr int NGRP = 8;      // warps per epilogue group
constexpr int kThreads = (1 + 2 * NGRP) * 32;

__host__ __device__ constexpr int round1k(int b) { return (b + 1023) / 1024 * 1024; }

// Shared-memory layout of one configuration: items of 128 tokens x CW
// channels (CW = 64 or 128; x, dy and outputs move as CW/64 boxes of 64
// channels with 128-byte swizzle).  BWD adds the dy boxes, a longer w box
// (the dx terms need w[s+k]) and the staged dw tile.
template <int W, int H, bool BWD, int CW>
struct HwLayout {
  static constexpr int NB = CW / 64;                  // 64-channel boxes per item
  static constexpr int GI = CW / H;                   // groups per item
  // PADW: the item's taps (GI*W elements) are not a whole number of 16-byte
  // units (e.g. 4 groups x 3 taps = 24 bytes), so no TMA box can start at
  // them.  The box is then 16 elements wide and starts at the 8-element
  // boundary at or below them: the taps sit 0 or 4 elements into it (GI*W
  // is a multiple of 4 and at most 12), and dw goes straight from
  // registers to global memory instead of through a staged TMA store.
  static constexpr bool PADW = (GI * W * 2) % 16 != 0;
  static_assert(!PADW || ((GI * W) % 4 == 0 && GI * W <= 12), "padded filter box");
  static constexpr int WROW = PADW ? 32 : GI * W * 2;  // bytes of one row of the w box
  // TOK2 (backward with a group wider than half the item, H = 64 on 64-channel
  // items): two adjacent lanes share a token, each taking half the item's
  // channels, so the group's dw is one shuffle away instead of in another warp.
  static constexpr bool TOK2 = BWD && H > CW / 2;
  static_assert(!TOK2 || (H == CW && PADW), "two-lane tokens: one group per item");
  static constexpr int WSW = (WROW == 32 || WROW == 64) ? WROW : 0;  // swizzle of the w box
  static constexpr int XROWS = BM + W - 1;
  static constexpr int XBOX = XROWS * 128;            // one 64-channel box
  static constexpr int XBYTES = round1k(XBOX);
  static constexpr int WROWS = BWD ? XROWS : BM;
  static constexpr int WBOX = WROWS * WROW;
  static constexpr int WBYTES = round1k(WBOX);
  static constexpr int DY_IN = NB * XBYTES;           // offsets inside a stage
  static constexpr int W_IN = (BWD ? 2 : 1) * NB * XBYTES;
  static constexpr int STAGE = W_IN + WBYTES;
  static constexpr int OBOX = BM * 128;               // one staged 64-channel output box
  static constexpr int OBYTES = NB * OBOX;            // staged y / dx tile of one group
  static constexpr int DWBYTES = (BWD && !PADW) ? round1k(BM * WROW) : 0;  // staged dw tile
  // Shared memory of the layout with `nst` stages.
  static constexpr int total(int nst) {
    return nst * STAGE + 2 * OBYTES + 2 * DWBYTES + (2 * nst + 4) * 8 + 16 + 1024;
  }
  // Stages: 6 in the forward when they fit (measured 87 instead of 94 us
  // with 4 at the QKV size), else 4 when they fit, else 2.  Always even:
  // the two epilogue groups take alternate items, so with an even count
  // each stage serves one group only and a group waits on a stage's barrier
  // at most one phase ahead of its last use.  With an odd count a stage
  // alternates between the groups, a group can wait two phases ahead, and
  // the parity wait then returns on the phase before (the data of the other
  // group's item, still loading).
  static constexpr int NST = (!BWD && total(6) <= 227 * 1024) ? 6
                             : total(4) <= 227 * 1024            ? 4
                                                                 : 2;
  static_assert(NST % 2 == 0, "stages must be even");
  static constexpr int O_OFF = NST * STAGE;
  static constexpr int DW_OFF = O_OFF + 2 * OBYTES;
  static constexpr int BAR_OFF = DW_OFF + 2 * DWBYTES;
  // full[NST] empty[NST] ofull[2] ofree[2]
  static constexpr int NBAR = 2 * NST + 4;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int TOTAL = MISC_OFF + 16 + 1024;
  static constexpr uint32_t TX = (BWD ? 2 : 1) * NB * XBOX + WBOX;
};

// Byte offset of byte `o` of row `r` in a w tile of `row` bytes per row
// stored by TMA with a `sw`-byte swizzle (0, 32 or 64).
template <int row, int sw>
__device__ __forceinline__ uint32_t wtile_offset(uint32_t r, uint32_t o) {
  const uint32_t a = r * row + o;
  if constexpr (sw == 32) return a ^ ((a >> 3) & 0x10u);
  if constexpr (sw == 64) return a ^ ((a >> 3) & 0x30u);
  return a;
}

__device__ __forceinline__ float lds_bf16(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return __uint_as_float(static_cast<uint32_t>(v) << 16);
}

// Two fp32 rounded to nearest-even bf16, packed (first in the low half).
__device__ __forceinline__ uint32_t f2bf2(float a, float b) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(a))) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(b))) << 16);
}

__device__ __forceinline__ void sts_bf16(uint32_t addr, float f) {
  const unsigned short v = __bfloat16_as_ushort(__float2bfloat16_rn(f));
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// The W taps of filter group gl in row r of the staged w tile, as fp32.
// W = 2 or 4 taps are one 4- or 8-byte load (their offset is a multiple of
// the access size, so it stays inside one 16-byte swizzle unit): threads on
// consecutive rows then meet at most two to a bank, where W separate 2-byte
// loads meet eight to a bank on 32-byte rows.
template <int W, int row, int sw>
__device__ __forceinline__ void load_taps(uint32_t wt, uint32_t r, int e0, float (&t)[W]) {
  const uint32_t a = wt + wtile_offset<row, sw>(r, static_cast<uint32_t>(e0) * 2);
  if constexpr (W == 4) {
    uint32_t lo, hi;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(lo), "=r"(hi) : "r"(a));
    t[0] = __uint_as_float(lo << 16);
    t[1] = __uint_as_float(lo & 0xffff0000u);
    t[2] = __uint_as_float(hi << 16);
    t[3] = __uint_as_float(hi & 0xffff0000u);
  } else if constexpr (W == 2) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    t[0] = __uint_as_float(v << 16);
    t[1] = __uint_as_float(v & 0xffff0000u);
  } else {
#pragma unroll
    for (int k = 0; k < W; ++k)
      t[k] = lds_bf16(wt + wtile_offset<row, sw>(r, static_cast<uint32_t>(e0 + k) * 2));
  }
}

struct HwItem {
  int chunk, b, t0;
};
// Work item i -> (chunk, b, t0), tile-major.  (The same in 32-bit
// arithmetic measured 5% slower in the forward at the QKV size: 82.0 against
// 77.9 us; the compiler scheduled the epilogue differently.)
__device__ __forceinline__ HwItem hw_decode(long long i, int nchunks, int ntiles) {
  HwItem it;
  const long long tile = i / nchunks;
  it.chunk = static_cast<int>(i - tile * nchunks);
  it.b = static_cast<int>(tile / ntiles);
  it.t0 = static_cast<int>(tile - static_cast<long long>(it.b) * ntiles) * BM;
  return it;
}

// The residual term: in the backward a template parameter RES (no
// per-channel select in its epilogue: 125.0 -> 121.5 us at the QKV size);
// the forward keeps the runtime flag `residual` (RES is false there), which
// measured faster (77.4 against 80.2 us: the compiler gave the template
// version 72 registers instead of 80 and a tighter schedule).
template <int W, int H, bool BWD, int CW, bool RES>
__global__ void __launch_bounds__(kThreads, 1)
hw_tma_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dy,
              const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_out,
              const __grid_constant__ CUtensorMap tm_dw, int ntiles, int nbt, int nchunks,
              int residual, __nv_bfloat16* __restrict__ dw_out, int T, int64_t GW) {
  static_assert(!RES || BWD, "RES is the backward's compile-time residual flag");
  using L = HwLayout<W, H, BWD, CW>;
  constexpr int NST = L::NST;
  constexpr int NB = L::NB;
  constexpr int PPW = CW / 16;                         // 8-channel pieces per warp
  // A thread's pieces start on a group boundary, so a group's taps can be
  // loaded at its first piece (with TOK2 the item is one group).
  static_assert((PPW * 8) % H == 0 || L::TOK2, "pieces start on a group boundary");
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = align1k(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long items = static_cast<long long>(nchunks) * nbt;
  const int nmine = items > blockIdx.x
                        ? static_cast<int>((items - 1 - blockIdx.x) / gridDim.x) + 1
                        : 0;
  const uint32_t bar_full = sb + L::BAR_OFF;
  const uint32_t bar_empty = bar_full + NST * 8;
  const uint32_t bar_ofull = bar_empty + NST * 8;
  const uint32_t bar_ofree = bar_ofull + 16;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFF);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, NGRP);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(bar_ofull + 8 * g, NGRP);
      mbar_init(bar_ofree + 8 * g, 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_out);
    if constexpr (BWD) {
      tma_prefetch_desc(&tm_dy);
      if constexpr (!L::PADW) tma_prefetch_desc(&tm_dw);
    }
  }
  __syncthreads();

  if (warp == 0) {
    // ---------------------------------------------------------- producer --
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int it = 0;
      for (; it < nmine; ++it) {
        const int s = it % NST;
        if (!mbar_wait(bar_empty + 8 * s, ((it / NST) & 1) ^ 1, abort_flag, &g_hw_error, 1))
          break;
        const HwItem itm =
            hw_decode(blockIdx.x + static_cast<long long>(it) * gridDim.x, nchunks, ntiles);
        const uint32_t full = bar_full + 8 * s;
        const uint32_t st = sb + s * L::STAGE;
        mbar_expect_tx(full, L::TX);
#pragma unroll
        for (int j = 0; j < NB; ++j) {
          tma_load_3d(st + j * L::XBYTES, &tm_x, full, itm.chunk * CW + 64 * j, itm.t0 - (W - 1),
                      itm.b, pol);
          if constexpr (BWD)
            tma_load_3d(st + L::DY_IN + j * L::XBYTES, &tm_dy, full, itm.chunk * CW + 64 * j,
                        itm.t0, itm.b, pol);
        }
        const int wx = itm.chunk * L::GI * W;
        tma_load_3d(st + L::W_IN, &tm_w, full, L::PADW ? (wx & ~7) : wx, itm.t0, itm.b, pol);
      }
      for (int j = std::max(0, it - NST); j < it; ++j)
        drain_wait(bar_full + 8 * (j % NST), (j / NST) & 1);
    }
  } else {
    // --------------------------------------------------------- epilogue --
    const int g = (warp - 1) >> 3;             // group: items it with it % 2 == g
    // The thread's token of the tile (tl) and channel half of the item (h):
    // a warp owns 32 tokens and one half, or with TOK2 16 tokens, two
    // adjacent lanes per token.
    const int lg = warp & 3;
    const int h = L::TOK2 ? (lane & 1) : ((warp - 1) >> 2) & 1;
    const int tl = L::TOK2 ? ((warp - 1) & 7) * 16 + (lane >> 1) : lg * 32 + lane;
    const bool storer = ((warp - 1) & 7) == 0 && lane == 0;
    const uint64_t pol = policy_evict_first();
    const uint32_t obuf = sb + L::O_OFF + g * L::OBYTES;
    const uint32_t dwbuf = sb + L::DW_OFF + g * L::DWBYTES;
    // TRACK: the group's items (g, g+2, ... of this CTA) are followed step by
    // step: the global item moves by 2 * gridDim.x, i.e. dch chunks and dtl
    // (b, tile) steps with carries.  Used by the backward with H >= 16, where
    // it measured faster than decoding each item with divisions (QKV pair
    // 119.6 -> 117.6 us, H = 64 147.5 -> 144.3 us); the forward and H = 8
    // measured slower with it (78 -> 82 us, 130 -> 137 us: the compiler
    // scheduled their epilogues differently) and decode each item.
    constexpr bool TRACK = BWD && H >= 16;
    HwItem trk{};
    int ctl = 0, dtl = 0, dch = 0;
    if constexpr (TRACK) {
      trk = hw_decode(blockIdx.x + static_cast<long long>(g) * gridDim.x, nchunks, ntiles);
      const int istep = 2 * static_cast<int>(gridDim.x);
      dtl = istep / nchunks;
      dch = istep - dtl * nchunks;
      ctl = trk.t0 / BM;
    }
    auto next_item = [&]() {
      if constexpr (TRACK) {
        trk.chunk += dch;
        int adv = dtl;
        if (trk.chunk >= nchunks) {
          trk.chunk -= nchunks;
          ++adv;
        }
        ctl += adv;
        while (ctl >= ntiles) {
          ctl -= ntiles;
          ++trk.b;
        }
        trk.t0 = ctl * BM;
      }
    };
    for (int it = g; it < nmine; it += 2, next_item()) {
      const int s = it % NST;
      const uint32_t aph = (it >> 1) & 1;
      if (storer) {
        bulk_wait_read<0>();                   // this group's previous stores have read
        mbar_arrive(bar_ofree + 8 * g);
      }
      bool ok = mbar_wait(bar_ofree + 8 * g, aph, abort_flag, &g_hw_error, 3) &&
                mbar_wait(bar_full + 8 * s, (it / NST) & 1, abort_flag, &g_hw_error, 3);
      if (!__all_sync(0xffffffffu, ok)) break;
      const uint32_t st = sb + s * L::STAGE;
      const uint32_t wt = st + L::W_IN;
      // PADW: the item's taps start woff elements into the w box.
      const HwItem itm0 =
          TRACK ? trk
                : hw_decode(blockIdx.x + static_cast<long long>(it) * gridDim.x, nchunks, ntiles);
      const int woff = L::PADW ? (itm0.chunk * L::GI * W) & 7 : 0;
      if constexpr (!BWD) {
        // y = res*x + sum_k w[t,g,k] x[t-k].  A group's taps are loaded at
        // its first piece: a new group starts where 8q is a multiple of H
        // (the thread's first piece starts one, as 8*PPW is a multiple of H
        // or the item holds one group).
        float taps[W];
#pragma unroll
        for (int q = 0; q < PPW; ++q) {
          const int cch = PPW * h + q;           // 8-channel piece of the item
          const int gl = cch * 8 / H;            // its filter group within the item
          const uint32_t xt = st + (cch >> 3) * L::XBYTES;
          if ((q * 8) % H == 0) load_taps<W, L::WROW, L::WSW>(wt, tl, woff + gl * W, taps);
          float xv[W][8];
#pragma unroll
          for (int k = 0; k < W; ++k)
            unpack16<__nv_bfloat16>(lds128(xt + sw128_offset(tl + (W - 1) - k, cch & 7)), xv[k]);
          float out[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            float v = residual ? xv[0][c] : 0.f;
#pragma unroll
            for (int k = 0; k < W; ++k) v = fmaf(taps[k], xv[k][c], v);
            out[c] = v;
          }
          sts128(obuf + (cch >> 3) * L::OBOX + sw128_offset(tl, cch & 7),
                 pack16<__nv_bfloat16>(out));
        }
      } else {
        // dx = res*dy + sum_k w[t+k,g,k] dy[t+k];  dw[t,g,k] = sum_{c in g} dy[t,c] x[t-k,c]
        [[maybe_unused]] uint32_t dwp[L::PADW ? (PPW * 8 / H) * W / 2 + 1 : 1];
        float p[W];
#pragma unroll
        for (int k = 0; k < W; ++k) p[k] = 0.f;
        float wk[W];                             // tap k of row tl + k (the filter of token t+k)
#pragma unroll
        for (int q = 0; q < PPW; ++q) {
          const int cch = PPW * h + q;
          const int gl = cch * 8 / H;
          const uint32_t xt = st + (cch >> 3) * L::XBYTES;
          const uint32_t dyt = st + L::DY_IN + (cch >> 3) * L::XBYTES;
          // loaded at the group's first piece, as in the forward
          if ((q * 8) % H == 0) {
#pragma unroll
            for (int k = 0; k < W; ++k) {
              float row_taps[W];
              load_taps<W, L::WROW, L::WSW>(wt, tl + k, woff + gl * W, row_taps);
              wk[k] = row_taps[k];
            }
          }
          float gv[W][8];
#pragma unroll
          for (int k = 0; k < W; ++k)
            unpack16<__nv_bfloat16>(lds128(dyt + sw128_offset(tl + k, cch & 7)), gv[k]);
          float out[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            float v = RES ? gv[0][c] : 0.f;
#pragma unroll
            for (int k = 0; k < W; ++k) v = fmaf(wk[k], gv[k][c], v);
            out[c] = v;
          }
          sts128(obuf + (cch >> 3) * L::OBOX + sw128_offset(tl, cch & 7),
                 pack16<__nv_bfloat16>(out));
#pragma unroll
          for (int k = 0; k < W; ++k) {
            float xv[8];
            unpack16<__nv_bfloat16>(lds128(xt + sw128_offset(tl + (W - 1) - k, cch & 7)), xv);
#pragma unroll
            for (int c = 0; c < 8; ++c) p[k] = fmaf(gv[0][c], xv[c], p[k]);
          }
          // The last 8-channel piece of a group: its W taps are complete.
          if (!L::TOK2 && ((cch + 1) * 8) % H == 0) {
            if constexpr (L::TOK2) {
            } else if constexpr (L::PADW) {
              // bf16 pairs in registers; written below in 4-byte stores.  The
              // warp's pieces hold whole groups (PPW*8 is a multiple of H),
              // so the piece's group within the warp is q*8/H.
              static_assert((PPW * 8) % H == 0, "whole groups per warp");
              const int gw = ((q * 8) / H) * W;     // first element of the group within the warp
#pragma unroll
              for (int k = 0; k < W; ++k) {
                const uint32_t v = __bfloat16_as_ushort(__float2bfloat16_rn(p[k]));
                const int e = gw + k;
                if (e & 1) dwp[e >> 1] |= v << 16;
                else dwp[e >> 1] = v;
                p[k] = 0.f;
              }
            } else if constexpr (W == 4 || W == 2) {
              // the group's taps in one 8- or 4-byte store
              uint32_t pk[2];
              pk[0] = f2bf2(p[0], p[1]);
              if constexpr (W == 4) pk[1] = f2bf2(p[2], p[3]);
              const uint32_t a = dwbuf + wtile_offset<L::WROW, L::WSW>(tl, (gl * W) * 2);
              if constexpr (W == 4)
                asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(a), "r"(pk[0]), "r"(pk[1])
                             : "memory");
              else
                asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(pk[0]) : "memory");
#pragma unroll
              for (int k = 0; k < W; ++k) p[k] = 0.f;
            } else {
#pragma unroll
              for (int k = 0; k < W; ++k) {
                sts_bf16(dwbuf + wtile_offset<L::WROW, L::WSW>(tl, (gl * W + k) * 2), p[k]);
                p[k] = 0.f;
              }
            }
          }
        }
        if constexpr (L::TOK2) {
          // The token's two lanes hold the sums over their halves of the
          // group; the even lane adds them and writes the W taps (8 bytes at
          // an 8-byte multiple: W = 4 and the group index times 4).
          static_assert(W == 4, "two-lane tokens are built for W = 4");
#pragma unroll
          for (int k = 0; k < W; ++k) p[k] += __shfl_xor_sync(0xffffffffu, p[k], 1);
          const int t = itm0.t0 + tl;
          if (h == 0 && t < T) {
            uint2* dst = reinterpret_cast<uint2*>(
                dw_out + (static_cast<int64_t>(itm0.b) * T + t) * GW +
                static_cast<int64_t>(itm0.chunk) * L::GI * W);
            *dst = make_uint2(f2bf2(p[0], p[1]), f2bf2(p[2], p[3]));
          }
        } else if constexpr (L::PADW) {
          // The warp's groups are contiguous in dw: (PPW*8/H)*W elements of
          // 2 bytes starting at a 4-byte multiple (GI*W and the groups
          // before this warp's are multiples of 4 and 2 elements).
          constexpr int NE = (PPW * 8 / H) * W;
          static_assert(NE % 2 == 0, "whole bf16 pairs");
          const int t = itm0.t0 + tl;
          if (t < T) {
            uint32_t* dst = reinterpret_cast<uint32_t*>(
                dw_out + (static_cast<int64_t>(itm0.b) * T + t) * GW +
                (static_cast<int64_t>(itm0.chunk) * L::GI + (PPW * h * 8) / H) * W);
#pragma unroll
            for (int e = 0; e < NE / 2; ++e) dst[e] = dwp[e];
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar_empty + 8 * s);
        mbar_arrive(bar_ofull + 8 * g);
      }
      if (storer && mbar_wait(bar_ofull + 8 * g, aph, abort_flag, &g_hw_error, 4)) {
        const HwItem itm =
            TRACK ? trk
                  : hw_decode(blockIdx.x + static_cast<long long>(it) * gridDim.x, nchunks, ntiles);
#pragma unroll
        for (int j = 0; j < NB; ++j)
          tma_store_3d(&tm_out, obuf + j * L::OBOX, itm.chunk * CW + 64 * j, itm.t0, itm.b, pol);
        if constexpr (BWD && !L::PADW)
          tma_store_3d(&tm_dw, dwbuf, itm.chunk * L::GI * W, itm.t0, itm.b, pol);
        bulk_commit();
      }
    }
    if (storer) bulk_wait<0>();
  }
  __syncthreads();
}

// One shared-memory opt-in record per kernel instance.
template <int W, int H, bool BWD, int CW, bool RES>
struct HwKernelTag {};

template <int W, int H, bool BWD, int CW, bool RES>
cudaError_t launch_res(const void* x, const void* dy, const void* w, void* out, void* dw,
                       const Shape& s, cudaStream_t st) {
  using L = HwLayout<W, H, BWD, CW>;
  const uint64_t GW = static_cast<uint64_t>(s.C / H) * W;
  CUtensorMap tx, tdy, tw, tout, tdw;
  if (!make_tmap_3d(&tx, x, true, s.C, s.T, s.B, 64, L::XROWS, 128) ||
      !make_tmap_3d(&tw, w, true, GW, s.T, s.B, L::WROW / 2, L::WROWS, L::WSW) ||
      !make_tmap_3d(&tout, out, true, s.C, s.T, s.B, 64, BM, 128))
    return cudaErrorInvalidValue;
  if constexpr (BWD) {
    if (!make_tmap_3d(&tdy, dy, true, s.C, s.T, s.B, 64, L::XROWS, 128))
      return cudaErrorInvalidValue;
    if constexpr (L::PADW) {
      tdw = tw;                                 // unused: dw is written from registers
    } else {
      if (!make_tmap_3d(&tdw, dw, true, GW, s.T, s.B, L::GI * W, BM, L::WSW))
        return cudaErrorInvalidValue;
    }
  } else {
    tdy = tx;
    tdw = tw;
  }
  const int ntiles = static_cast<int>((s.T + BM - 1) / BM);
  const int nchunks = static_cast<int>(s.C / CW);
  const long long nbt = static_cast<long long>(s.B) * ntiles;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorNoDevice;
  const long long grid = std::min<long long>(sms, nbt * nchunks);
  auto kern = hw_tma_kernel<W, H, BWD, CW, RES>;
  cudaError_t e = set_smem<HwKernelTag<W, H, BWD, CW, RES>>(kern, L::TOTAL);
  if (e != cudaSuccess) return e;
  kern<<<static_cast<unsigned>(grid), kThreads, L::TOTAL, st>>>(
      tx, tdy, tw, tout, tdw, ntiles, static_cast<int>(nbt), nchunks, s.residual,
      static_cast<__nv_bfloat16*>(dw), static_cast<int>(s.T), static_cast<int64_t>(GW));
  return cudaGetLastError();
}

template <int W, int H, bool BWD, int CW>
cudaError_t launch(const void* x, const void* dy, const void* w, void* out, void* dw,
                   const Shape& s, cudaStream_t st) {
  if constexpr (BWD) {
    if (s.residual) return launch_res<W, H, BWD, CW, true>(x, dy, w, out, dw, s, st);
  }
  return launch_res<W, H, BWD, CW, false>(x, dy, w, out, dw, s, st);
}

// Channel width of the item for (H, W) and C, 0 if there is no TMA path.
// The pairs are those whose filter rows make a TMA box of a multiple of 16
// bytes.  The narrowest legal item is 64 channels for H = 8, (16, 2),
// (16, 4) and (32, 4), 128 for (16, 1), (16, 3), (32, 2) and (64, 4).  The
// forward of (8, 1), (16, 2) and (32, 4) takes 128-channel items when C
// allows (measured 3 to 15% faster at C = 6144); for the others, (16, 4)
// included, the wider item leaves room for only two stages and is slower.
// The backward of (16, 3) takes 64-channel items with the padded filter box
// (24-byte filter rows; see PADW in the layout): 128-channel items with
// 48-byte rows do not fit shared memory with two stages.  The backward of
// (64, 4) takes 64-channel items too (one group per item, two lanes per
// token: TOK2), which leave room for four stages where 128-channel items
// leave two.  Its filter tensor
// rows (3C/16 elements) must still be a multiple of 16 bytes for the tensor
// map, so C is a multiple of 128.
int item_width(int64_t H, int64_t W, bool bwd, int64_t C) {
  const bool narrow = (H == 8 && W >= 1 && W <= 4) || (H == 16 && (W == 2 || W == 4)) ||
                      (H == 32 && W == 4);
  const bool wide_only = (H == 16 && (W == 1 || W == 3)) || (H == 32 && W == 2) ||
                         (H == 64 && W == 4);
  const bool wide_fwd = (H == 8 && W == 1) || (H == 16 && W == 2) || (H == 32 && W == 4);
  if (bwd && H == 16 && W == 3) return C % 128 == 0 ? 64 : 0;
  if (bwd && H == 64 && W == 4) return C % 128 == 0 ? 64 : 0;
  if (wide_only) return C % 128 == 0 ? 128 : 0;
  if (!narrow) return 0;
  if (!bwd && wide_fwd && C % 128 == 0) return 128;
  return C % 64 == 0 ? 64 : 0;
}

template <bool BWD, int CW>
cudaError_t dispatch_cw(const void* x, const void* dy, const void* w, void* out, void* dw,
                        const Shape& s, cudaStream_t st) {
  if constexpr (CW == 64) {
    switch (s.H * 8 + s.W) {
      case 8 * 8 + 1: return launch<1, 8, BWD, 64>(x, dy, w, out, dw, s, st);
      case 8 * 8 + 2: return launch<2, 8, BWD, 64>(x, dy, w, out, dw, s, st);
      case 8 * 8 + 3: return launch<3, 8, BWD, 64>(x, dy, w, out, dw, s, st);
      case 8 * 8 + 4: return launch<4, 8, BWD, 64>(x, dy, w, out, dw, s, st);
      case 16 * 8 + 2: return launch<2, 16, BWD, 64>(x, dy, w, out, dw, s, st);
      case 16 * 8 + 3:
        if constexpr (BWD) return launch<3, 16, true, 64>(x, dy, w, out, dw, s, st);
        break;
      case 64 * 8 + 4:
        if constexpr (BWD) return launch<4, 64, true, 64>(x, dy, w, out, dw, s, st);
        break;
      case 16 * 8 + 4: return launch<4, 16, BWD, 64>(x, dy, w, out, dw, s, st);
      case 32 * 8 + 4: return launch<4, 32, BWD, 64>(x, dy, w, out, dw, s, st);
      default: break;
    }
  } else {
    switch (s.H * 8 + s.W) {
      case 16 * 8 + 1: return launch<1, 16, BWD, 128>(x, dy, w, out, dw, s, st);
      case 16 * 8 + 3:
        if constexpr (!BWD) return launch<3, 16, false, 128>(x, dy, w, out, dw, s, st);
        break;
      case 32 * 8 + 2: return launch<2, 32, BWD, 128>(x, dy, w, out, dw, s, st);
      case 64 * 8 + 4: return launch<4, 64, BWD, 128>(x, dy, w, out, dw, s, st);
      default: break;
    }
    if constexpr (!BWD) {
      switch (s.H * 8 + s.W) {
        case 8 * 8 + 1: return launch<1, 8, false, 128>(x, dy, w, out, dw, s, st);
        case 16 * 8 + 2: return launch<2, 16, false, 128>(x, dy, w, out, dw, s, st);
        case 32 * 8 + 4: return launch<4, 32, false, 128>(x, dy, w, out, dw, s, st);
        default: break;
      }
    }
  }
  return cudaErrorNotSupported;
}

template <bool BWD>
cudaError_t dispatch(const void* x, const void* dy, const void* w, void* out, void* dw,
                     const Shape& s, cudaStream_t st) {
  if (item_width(s.H, s.W, BWD, s.C) == 128)
    return dispatch_cw<BWD, 128>(x, dy, w, out, dw, s, st);
  return dispatch_cw<BWD, 64>(x, dy, w, out, dw, s, st);
}

}  // namespace

bool headwise_tma_supported(const Shape& s, bool bwd) {
  if (!s.bf16) return false;
  const int cw = item_width(s.H, s.W, bwd, s.C);
  return cw > 0 && s.T < (int64_t(1) << 30) &&
         s.B * ((s.T + BM - 1) / BM) < (int64_t(1) << 30) && s.C < (int64_t(1) << 24);
}

cudaError_t headwise_fwd_tma(const void* x, const void* w, void* y, const Shape& s,
                             cudaStream_t st) {
  if (!headwise_tma_supported(s, false)) return cudaErrorNotSupported;
  return dispatch<false>(x, nullptr, w, y, nullptr, s, st);
}

cudaError_t headwise_bwd_tma(const void* x, const void* w, const void* dy, void* dx, void* dw,
                             const Shape& s, cudaStream_t st) {
  if (!headwise_tma_supported(s, true)) return cudaErrorNotSupported;
  return dispatch<true>(x, dy, w, dx, dw, s, st);
}

cudaError_t headwise_tma_error(unsigned int* out, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_hw_error, sizeof(unsigned int));
  if (e != cudaSuccess || !reset) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_hw_error, &zero, sizeof(unsigned int));
}

}  // namespace dsc

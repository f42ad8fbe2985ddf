// tmap.cu -- host-side helpers for the kernels: encoding of tensor maps
// (through the driver entry point, so the library needs no link-time
// libcuda), the SM count of the current device, and the token-range split of
// the streaming kernels.  Host code only.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "dsc_internal.h"

namespace dsc {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

bool make_tmap_3d(CUtensorMap* tm, const void* base, bool bf16, uint64_t d0, uint64_t d1,
                  uint64_t d2, uint32_t b0, uint32_t b1, int swizzle_bytes) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const uint64_t esz = bf16 ? 2 : 4;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * esz, d0 * d1 * esz};
  const cuuint32_t box[3] = {b0, b1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_NONE;
  if (swizzle_bytes == 32) sw = CU_TENSOR_MAP_SWIZZLE_32B;
  if (swizzle_bytes == 64) sw = CU_TENSOR_MAP_SWIZZLE_64B;
  if (swizzle_bytes == 128) sw = CU_TENSOR_MAP_SWIZZLE_128B;
  const CUresult r =
      fn(tm, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
         const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
         CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_4d_bf16(CUtensorMap* tm, const void* base, const uint64_t dims[4],
                       const uint64_t strides_bytes[3], const uint32_t box[4]) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t d[4] = {dims[0], dims[1], dims[2], dims[3]};
  const cuuint64_t st[3] = {strides_bytes[0], strides_bytes[1], strides_bytes[2]};
  const cuuint32_t bx[4] = {box[0], box[1], box[2], box[3]};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), d, st,
                        bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static int cache[64] = {};
  if (dev < 0 || dev >= 64) return 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

// Resident CTAs per SM of `kernel` at `threads` threads, cached per kernel
// (keyed by its address: every instance of one template shares a type).
static int blocks_per_sm(const void* kernel, int threads) {
  static std::mutex mu;
  static const void* keys[64] = {};
  static int vals[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < 64; ++i) {
    if (keys[i] == kernel) return vals[i];
    if (keys[i] == nullptr) {
      int nb = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, threads, 0) != cudaSuccess ||
          nb <= 0)
        nb = 2;
      keys[i] = kernel;
      vals[i] = nb;
      return nb;
    }
  }
  return 2;
}

// Token ranges for a grid of `ncb` channel blocks: as many CTAs as fit on
// the GPU at once (occupancy of this kernel x SMs), at least 16 tokens each.
int64_t n_ranges(const void* kernel, int threads, int64_t ncb, int64_t N) {
  const int per_sm = blocks_per_sm(kernel, threads);
  const int sms = sm_count() > 0 ? sm_count() : 148;
  int64_t r = std::max<int64_t>(1, static_cast<int64_t>(per_sm) * sms / ncb);
  r = std::min<int64_t>(r, std::max<int64_t>(1, N / 16));
  return std::min<int64_t>(r, (int64_t(1) << 31) / ncb - 1);
}

}  // namespace dsc

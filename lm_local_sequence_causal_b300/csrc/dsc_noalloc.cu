// dsc_noalloc.cu -- dsc_lowrank_bwd_noalloc: the low-rank backward for
// callers that cannot allocate device memory.
//
// Who needs it: code that runs where no allocator is available or allowed,
// for example a plugin loaded into a host program that owns all device
// memory and hands out none, a service with a fixed memory budget that
// forbids allocation once it is up, or a latency-critical path where the
// implicit device synchronisation of cudaMalloc/cudaFree cannot be
// tolerated.  Such callers can still pass their inputs and outputs, but not
// the fp32 partial-sum workspace that dsc_lowrank_bwd needs.
//
// This entry point takes that workspace from a fixed array compiled into
// the library (a file-scope __device__ array of kScratchBytes), so it calls
// no allocating routine at all.  Each GPU that loads the library holds the
// array until the process exits.  The kernels and their launch plan are the
// ones dsc_lowrank_bwd runs; only the workspace pointer differs.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/dsc.h"

namespace {

constexpr size_t kScratchBytes = DSC_LOWRANK_BWD_NOALLOC_MAX_BYTES;
constexpr int kMaxDevices = 64;

// The shared scratch.  In host code this name is only a host-side stand-in:
// its device address must be fetched with cudaGetSymbolAddress on each
// device before a kernel may use it.
static __device__ __align__(256) unsigned char g_dsc_scratch[kScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch on the current device; fetched once per
// device (the first call on a device does this set-up).
dsc_status_t scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return DSC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dsc_scratch) != cudaSuccess || p == nullptr)
      return DSC_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return DSC_OK;
}

}  // namespace

extern "C" dsc_status_t dsc_lowrank_bwd_noalloc(
    const void* x, const void* z, const void* U, const void* dy, void* dx, void* dz,
    void* dU, int64_t B, int64_t T, int64_t C, int64_t H, int64_t W, int64_t R,
    int residual, dsc_dtype_t dtype, void* stream) {
  // Size check first: a problem whose partial sums do not fit is refused
  // before anything is touched.  (An invalid shape reports 0 here and is
  // then rejected by dsc_lowrank_bwd's own checks.)
  const size_t need = dsc_lowrank_bwd_workspace_size(B, T, C, H, W, R, dtype);
  if (need > kScratchBytes) return DSC_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    const dsc_status_t st = scratch_on_current_device(&scratch);
    if (st != DSC_OK) return st;
  }
  // The backward writes every partial sum before it reads it, so whatever
  // the previous call left in the scratch needs no clearing.
  return dsc_lowrank_bwd(x, z, U, dy, dx, dz, dU, scratch, need > 0 ? kScratchBytes : 0, B, T,
                         C, H, W, R, residual, dtype, stream);
}

// flce_noalloc.cu -- flce_forward_noalloc: the forward pass for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the point where
// they need the loss: code running inside a custom allocator or memory-pool
// callback, runtimes that hand out a fixed device arena and forbid further
// allocation, or hosts where an allocation could trigger a synchronising
// garbage-collection or defragmentation pass. They can still pass their inputs and
// outputs. This entry point takes no workspace: its scratch (the forward's partial
// softmax statistics, target logits, loss partial sums and the device error word)
// lives in one file-scope device array of kNoAllocScratchBytes.
//
// Properties:
//  * The array takes 64 MiB of device memory on every GPU where it is used, from the
//    first call on that GPU (when CUDA loads this module) until the process exits.
//    That holds under CUDA's default lazy module loading; with
//    CUDA_MODULE_LOADING=EAGER the module, and so the array, is loaded on every device
//    the process uses, whether or not this entry point is ever called.
//  * The first call on a device, with that device current, looks the array's
//    device address up with cudaGetSymbolAddress (the host-side name of a
//    __device__ array is only a stand-in, never a device pointer) and keeps it for the
//    life of the process. Make that first call before any stream capture. A device
//    reset (cudaDeviceReset, or a primary context released and created again) makes
//    the kept address stale: do not use this entry point after one.
//  * Its error word is internal. A bad target gives that row's loss (and the reduced
//    loss) NaN, as in flce_forward; a pipeline wait that ran out gives NaN in every lse
//    and loss value of the call.
//  * Every call on a device shares the one array and it keeps the previous call's
//    contents. Each call clears what must start at zero (the error word) itself; all
//    other scratch is fully overwritten. Calls whose execution overlaps on the GPU
//    (other streams, other host threads, concurrent graph nodes) race on the array:
//    serialise them.
//  * Shapes whose forward scratch (flce_workspace_size(N, D, V, 0)) exceeds the
//    array are refused with FLCE_ERR_WORKSPACE_TOO_SMALL before anything runs.
//  * It calls no cudaMalloc, cudaFree or other allocating routine.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/flce.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_flce_noalloc_scratch[kNoAllocScratchBytes];

void* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (looked up once per device).
flce_status scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return FLCE_ERR_UNSUPPORTED_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_flce_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return FLCE_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return FLCE_OK;
}

}  // namespace

extern "C" flce_status flce_forward_noalloc(const void* X, const void* W, const int32_t* targets, int64_t N,
                                            int64_t D, int64_t V, int32_t ignore_index, float label_smoothing,
                                            float zloss_scale, flce_reduction red, float* loss, float* lse,
                                            struct CUstream_st* stream) {
  const size_t need = flce_workspace_size(N, D, V, 0);
  if (need > kNoAllocScratchBytes) return FLCE_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const flce_status st = scratch_on_current_device(&scratch);
  if (st != FLCE_OK) return st;
  return flce_forward(X, W, targets, N, D, V, ignore_index, label_smoothing, zloss_scale, red, loss, lse, scratch,
                      kNoAllocScratchBytes, stream);
}

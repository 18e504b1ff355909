// moe_noalloc.cu — routing (router, top-k, softmax weights, histogram, permutation) for callers
// that cannot allocate device memory.
//
// moe_route_topk needs a caller-provided workspace. Some callers have no way to provide one:
// runtimes that freeze their allocator after start-up, and embedders that own no device
// allocator at all (a plugin handed only input and output buffers). moe_route_topk_noalloc
// serves them: its workspace is a fixed device array owned by this library, so a call allocates
// nothing (no cudaMalloc, no cudaFree, no allocating library routine).
//
// The array is file-scope static device memory of kNoAllocScratchBytes (4 MiB). Every GPU that
// loads the library keeps it until the process exits. The first call on a device looks up the
// array's device address (cudaGetSymbolAddress) and caches it per device ordinal; the cache
// does not survive a cudaDeviceReset of that device in the same process. All calls share the
// array, so calls whose executions overlap on the GPU (for example on two streams) race and
// must be serialised by the caller. The array keeps the previous call's contents; each call
// first clears the control words that must start at zero. The status word is not cleared: a
// device-side timeout stays recorded until moe_read_device_status(NULL, ...) reads and clears
// it.
#include "../../include/moe_nvfp4.h"
#include "moe_internal.cuh"

#include <mutex>

namespace {

// 4 MiB: enough for the routing workspace of, e.g., 512 tokens x 512 experts x top-10 at
// hidden 4096, or 8 tokens x 1024 experts x top-32.
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;

static __device__ __align__(256) unsigned char g_route_scratch[kNoAllocScratchBytes];

// Device address of g_route_scratch per device (host code must not use the symbol itself: on the
// host it names a shadow variable, not device memory).
void* scratch_address(int device, cudaError_t* err) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  *err = cudaSuccess;
  if (device < 0 || device >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[device]) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_route_scratch);
    if (*err != cudaSuccess) return nullptr;
    addr[device] = p;
  }
  return addr[device];
}

}  // namespace

namespace moe {
// The fixed array of the current device (for reading its status word), or null.
void* noalloc_scratch_of_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  cudaError_t e;
  return scratch_address(dev, &e);
}
}  // namespace moe

extern "C" {

moe_status moe_route_topk_noalloc(const uint16_t* x, const uint16_t* router_w, int T, int H, int E,
                                  int k, int32_t* idx, float* w, int32_t* counts, int32_t* offsets,
                                  int32_t* perm, void* stream) {
  size_t need = 0;
  const moe_status st = moe_route_workspace_size(T, H, E, k, &need);  // validates the sizes
  if (st != MOE_OK) return st;
  if (need > kNoAllocScratchBytes) return MOE_ERR_WORKSPACE;   // beyond the fixed array
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  cudaError_t e;
  void* ws = scratch_address(dev, &e);
  if (!ws) return MOE_ERR_CUDA;
  // The control words before and after the status word (router ticket, counts of the call)
  // must start at zero; the status word keeps an earlier call's error until it is read.
  static_assert(moe::kCtlStatus == 1, "control word layout");
  unsigned char* ctl = static_cast<unsigned char*>(ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  e = cudaMemsetAsync(ctl, 0, moe::kCtlStatus * 4, s);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(ctl + (moe::kCtlStatus + 1) * 4, 0,
                        (moe::kCtlWords - moe::kCtlStatus - 1) * 4, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  return moe_route_topk(x, router_w, T, H, E, k, idx, w, counts, offsets, perm, ws,
                        kNoAllocScratchBytes, stream);
}

}  // extern "C"

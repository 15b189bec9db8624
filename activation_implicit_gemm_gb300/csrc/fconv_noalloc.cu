// fconv_run_noalloc: fconv_run for callers that cannot allocate device memory.
//
// The workspace that fconv_run takes from the caller (the weight copy, the repacked X and
// the split-K partial sums of the tensor-core route) comes here from one fixed, file-scope
// device array. Host code never uses the array's name as an address (on the host it is
// only a stand-in symbol): the device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, and handed to the unchanged fconv_run
// path as its workspace. Plans that need no workspace never look it up.
#include <cuda_runtime.h>

#include <mutex>

#include "fconv_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[FCONV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];  // device address of the array, per device
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (set-up on first use).
fconv_status scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return FCONV_E_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return FCONV_E_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return FCONV_E_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return FCONV_OK;
}

}  // namespace

extern "C" fconv_status fconv_run_noalloc(const fconv_plan* plan, const void* x, const void* w,
                                          const void* b, const void* z, void* y, void* stream) {
  if (!plan) return FCONV_E_NULL;
  size_t need = 0;
  fconv_status st = fconv_plan_workspace_size(plan, &need);
  if (st != FCONV_OK) return st;
  if (need > (size_t)FCONV_NOALLOC_SCRATCH_BYTES) return FCONV_E_WORKSPACE;
  if (need == 0) return fconv_run(plan, x, w, b, z, y, nullptr, 0, stream);
  void* scratch = nullptr;
  st = scratch_for_current_device(&scratch);
  if (st != FCONV_OK) return st;
  return fconv_run(plan, x, w, b, z, y, scratch, (size_t)FCONV_NOALLOC_SCRATCH_BYTES, stream);
}

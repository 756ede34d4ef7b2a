// i8lt_backward_input_noalloc: the backward to the input for callers that
// cannot allocate device memory.  Its scratch (status word, grad_bias partial
// sums, fp16 copy of grad_output) lives in one static device array that the
// CUDA runtime places on every GPU that loads this library; the call then
// runs the ordinary i8lt_backward_input on that array.
#include <cuda_runtime.h>

#include <mutex>

#include "i8lt.h"

namespace {

// Scratch held by every GPU that loads the library, until the process exits.
constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(I8LT_NOALLOC_SCRATCH_BYTES);
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The host-side
// symbol is only a stand-in: the address comes from the runtime, once per
// device, with that device current, and is kept for the life of the process
// (a cudaDeviceReset would invalidate it; the header says so).
int scratch_on_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return I8LT_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return I8LT_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return I8LT_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return I8LT_OK;
}

}  // namespace

extern "C" int i8lt_backward_input_noalloc(const void* G, int gt, int64_t M, int64_t N, const int8_t* CB,
                                           const float* SCB, int64_t K, const void* addend, void* grad_A,
                                           void* grad_bias, int bt, void* stream) {
  if (gt != I8LT_F16 && gt != I8LT_BF16 && gt != I8LT_F32) return I8LT_ERR_UNSUPPORTED_DTYPE;
  if (M < 0 || N <= 0 || K <= 0) return I8LT_ERR_INVALID_ARG;
  const size_t need = i8lt_backward_workspace_size(M, N, gt);
  if (need == 0) return I8LT_ERR_INVALID_ARG;
  if (need > kNoAllocScratchBytes) return I8LT_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  if (int st = scratch_on_current_device(&scratch)) return st;
  return i8lt_backward_input(G, gt, M, N, CB, SCB, K, addend, grad_A, grad_bias, bt, scratch,
                             kNoAllocScratchBytes, stream);
}

extern "C" int i8lt_noalloc_read_device_status(int32_t* status, void* stream) {
  void* scratch = nullptr;
  if (int st = scratch_on_current_device(&scratch)) return st;
  // the status word sits at the start of the scratch, as in every workspace
  return i8lt_read_device_status(scratch, status, nullptr, stream);
}

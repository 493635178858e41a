// The library's device error word.
//
// Kernels that wait on hardware (mbarrier phases of tensor-core commits)
// bound every wait; when one gives up, the kernel sets a bit of
// g_ss_error_flags (atomicOr) and finishes without further waiting.  The host
// reads and clears the word with ss_check_device_errors.
#include <cuda_runtime.h>

#include <mutex>

#include "launch.h"

__device__ unsigned int g_ss_error_flags = 0;

namespace selscan {

namespace {
constexpr int kMaxDev = 64;
std::mutex g_mu;
unsigned int* g_flag_ptr[kMaxDev] = {};

}  // namespace

cudaError_t error_flags_ptr(unsigned int** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_flag_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_ss_error_flags);
    if (e != cudaSuccess) return e;
    g_flag_ptr[dev] = static_cast<unsigned int*>(p);
  }
  *out = g_flag_ptr[dev];
  return cudaSuccess;
}

cudaError_t read_clear_error_flags(cudaStream_t s, unsigned int* out) {
  unsigned int* p = nullptr;
  cudaError_t e = error_flags_ptr(&p);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyAsync(out, p, sizeof(unsigned int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && *out) e = cudaMemsetAsync(p, 0, sizeof(unsigned int), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e;
}

}  // namespace selscan

// ss_scan_bwd_noalloc: the backward scan for callers that cannot allocate
// device memory themselves.
//
// Who needs it: code that runs where cudaMalloc is not available or not
// allowed, e.g. a plugin loaded into a host application that owns all device
// memory and hands out only the tensors it manages, or a latency-critical
// loop that must never call into the allocator (cudaMalloc/cudaFree can
// synchronise the device).  Such a caller can still pass its inputs and
// outputs, but has no way to provide ss_scan_bwd's workspace.
//
// This entry point uses a fixed scratch buffer that lives in the library
// itself: a file-scope __device__ array of kScratchBytes.  Every GPU that
// loads the library holds those bytes until the process exits.  Problems
// whose workspace (ss_scan_bwd_workspace_size) exceeds kScratchBytes are
// rejected with SS_ERR_SCRATCH_LIMIT before anything is launched.
//
// In host code the array's name does not denote a device address, so the
// first call on each device looks the address up with cudaGetSymbolAddress
// (with that device current) and caches it; later calls reuse the cached
// address.  With lazy module loading (the CUDA default) that first lookup is
// also what loads the library's device code, and with it the array, onto the
// device: the first call on a device does take device memory.  Make it at
// initialisation, outside allocation-sensitive code and before any stream
// capture begins.
//
// All calls share the one buffer and it keeps whatever the last call left
// in it.  The backward kernels write every scratch word before they read
// it, so nothing needs clearing between calls.  Two calls whose work
// overlaps on the GPU (e.g. on different streams without ordering) race on
// the buffer and corrupt each other's results: order them on one stream or
// with events.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/selscan.h"

// ss_scan_bwd's argument checks (api.cu), without the workspace pair.
extern "C" ss_status selscan_check_bwd_args(
    const void* u, const void* delta, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* delta_bias, const void* dy, int64_t Bsz,
    int64_t Dch, int64_t L, int64_t N, ss_dtype dtype, void* du, void* ddelta, float* dA,
    float* dB, float* dC, float* dD, void* dz, float* ddelta_bias);

constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB

// The scratch buffer (one per device, allocated when the module loads).
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up once per device).
ss_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return SS_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SS_OK;
}

}  // namespace

extern "C" {

size_t ss_scan_bwd_noalloc_max_scratch(void) { return kScratchBytes; }

ss_status ss_scan_bwd_noalloc(const void* u, const void* delta, const float* A, const void* B,
                              const void* C, const float* D, const void* z,
                              const float* delta_bias, int softplus, const void* dy,
                              int64_t Bsz, int64_t Dch, int64_t L, int64_t N, ss_dtype dtype,
                              void* du, void* ddelta, float* dA, float* dB, float* dC,
                              float* dD, void* dz, float* ddelta_bias, ss_stream_t stream) {
  // ss_scan_bwd's checks first (same status for the same bad arguments),
  // then the scratch limit
  ss_status st = selscan_check_bwd_args(u, delta, A, B, C, D, z, delta_bias, dy, Bsz, Dch, L, N,
                                         dtype, du, ddelta, dA, dB, dC, dD, dz, ddelta_bias);
  if (st != SS_OK) return st;
  size_t need = 0;
  st = ss_scan_bwd_workspace_size(Bsz, Dch, L, N, dtype, &need);
  if (st != SS_OK) return st;
  if (need > kScratchBytes) return SS_ERR_SCRATCH_LIMIT;
  void* ws = nullptr;
  if (need > 0) {
    st = scratch_address(&ws);
    if (st != SS_OK) return st;
  }
  // Same checks and the same three stages as ss_scan_bwd, on the static buffer.
  return ss_scan_bwd(u, delta, A, B, C, D, z, delta_bias, softplus, dy, Bsz, Dch, L, N, dtype,
                     du, ddelta, dA, dB, dC, dD, dz, ddelta_bias, ws, kScratchBytes, stream);
}

}  // extern "C"

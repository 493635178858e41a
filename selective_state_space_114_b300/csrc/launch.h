// Internal launcher interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace selscan {

enum class Dt { F32 = 0, BF16 = 1, F16 = 2 };

struct ScanArgs {
  const void* u;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* D;           // nullable
  const void* z;            // nullable
  const float* delta_bias;  // nullable
  int softplus;
  int64_t Bsz, Dch, L;
  Dt dt;
  const float* h0 = nullptr;  // forward only: state before step 0, [Bsz][Dch][N] (nullable = 0)
  int N = 16;                 // state size: 8, 16, 32 or 64
};

struct BwdOut {
  const void* dy;
  void* du;
  void* ddelta;
  float* dA;
  float* dB;
  float* dC;
  float* dD;           // nullable iff D null
  void* dz;            // nullable iff z null
  float* ddelta_bias;  // nullable iff delta_bias null
};

struct StepArgs {
  float* h;
  const void* u;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const void* z;
  const float* delta_bias;
  int softplus;
  int64_t Bsz, Dch;
  Dt dt;
  void* y;
  int N = 16;  // state size: 8, 16, 32 or 64
};

// Forward: writes y and (if non-null) h_last; with h_chunks non-null also the
// state entering every kScanChunk-step chunk, [Bsz][Dch][chunk][N], when the
// kernel the shape takes can (the row-sequential one); returns
// cudaErrorNotSupported before launching anything when it cannot.
// Requires Bsz*Dch*L > 0.
cudaError_t launch_scan_fwd(const ScanArgs& a, void* y, float* h_last, cudaStream_t s,
                            float* h_chunks = nullptr);

// Chunk of the backward (steps), and of the forward's chunk states.
constexpr int kScanChunk = 128;

// Forward with chunk states: also writes, into the backward's workspace, the
// state entering every kScanChunk-step chunk ([Bsz][Dch][chunk][N] fp32 at
// bwd_chunk_states_offset), so that the backward need not recompute them.
// Kernels that cannot write them run the backward's state summaries instead.
size_t bwd_chunk_states_offset(int64_t Bsz, int64_t Dch, int64_t L, int64_t N);

// Backward workspace size (bytes) and the launch of one of its stages.
// Requires Bsz*Dch*L > 0.
enum BwdPhase : int {
  kBwdStates = 0,         // chunk states and adjoint carries (summaries + carries)
  kBwdReverse = 1,        // the reverse pass
  kBwdReduce = 2,         // fixed-order reduction of the partials
  kBwdAdjointStates = 3,  // adjoint carries only: the chunk states are saved
  kBwdChunkStates = 4,    // chunk states only (for the forward)
};
size_t bwd_workspace_bytes(int64_t Bsz, int64_t Dch, int64_t L, int64_t N);
cudaError_t launch_scan_bwd(int phase, const ScanArgs& a, const BwdOut& o, void* ws,
                            cudaStream_t s);

// The library's device error word: bits set by kernels whose bounded waits
// gave up.  error_flags_ptr: its device address on the current device;
// read_clear_error_flags: copy it to the host and clear it (synchronises s).
constexpr unsigned int kErrXprojTimeout = 1u << 0;  // input projection: a tensor-core wait
cudaError_t error_flags_ptr(unsigned int** out);
cudaError_t read_clear_error_flags(cudaStream_t s, unsigned int* out);

// One decode step.  Requires Bsz*Dch > 0.
cudaError_t launch_step(const StepArgs& a, cudaStream_t s);

struct ConvArgs {
  const void* x;
  const float* w;     // [Dch][K]
  const float* bias;  // nullable
  int silu;
  int64_t Bsz, Dch, L;
  int K;              // 1 .. 4
  Dt dt;
  void* u;            // forward output
};

struct ConvGrads {
  const void* g;  // dL/du
  void* dx;
  float* dw;
  float* dbias;   // nullable iff bias null
};

// Causal depthwise conv1d + silu: phase 0 forward (writes a.u), phase 1
// backward (writes o.dx, o.dw, o.dbias).  Requires Bsz*Dch*L > 0.
cudaError_t launch_conv(int phase, const ConvArgs& a, const ConvGrads& o, cudaStream_t s);

struct XprojArgs {
  const void* u;    // [Bsz][Dch][L]
  const void* Wx;   // [R + 2N][Dch]
  const void* Wdt;  // [Dch][R]
  int64_t Bsz, Dch, L, R, N;
  Dt dt;            // BF16 or F16
  void* delta;      // [Bsz][Dch][L]
  void* B;          // [Bsz][N][L]
  void* C;          // [Bsz][N][L]
  unsigned int* err = nullptr;     // device error word (kErrXprojTimeout)
  int test_stuck_wait = 0;         // test hook: also wait on a barrier nothing arrives at
};

// Input projection (x_proj then dt_proj) on the tensor cores.  Requires
// Bsz*Dch*L > 0, L, Dch, R multiples of 8, R >= 8, N >= 1, R + 2N <= 256.
cudaError_t launch_xproj(const XprojArgs& a, cudaStream_t s);
size_t xproj_smem_bytes(int64_t R, int64_t N);
cudaError_t xproj_wait_failures(int* out);

}  // namespace selscan

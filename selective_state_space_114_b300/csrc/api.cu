// C ABI of libselscan: argument checks, then dispatch to the kernels on the
// caller's stream.  Declarations and contracts: include/selscan.h.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/selscan.h"
#include "launch.h"

using selscan::Dt;

namespace {

constexpr int64_t kMaxDim = int64_t(1) << 40;

bool misaligned(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u); }

bool bad_size(int64_t x) { return x < 0 || x > kMaxDim; }

bool product_too_big(int64_t a, int64_t b, int64_t c) {
  // a*b*c*16 (state-expanded element count) must fit comfortably in int64
  if (a == 0 || b == 0 || c == 0) return false;
  const double p = (double)a * (double)b * (double)c;
  return p > 1e17;
}

ss_status cuda_status(cudaError_t e) { return e == cudaSuccess ? SS_OK : SS_ERR_CUDA; }

bool known_dtype(ss_dtype d) { return d == SS_F32 || d == SS_BF16 || d == SS_F16; }

Dt to_dt(ss_dtype d) { return d == SS_BF16 ? Dt::BF16 : d == SS_F16 ? Dt::F16 : Dt::F32; }

// State sizes every entry point takes.
bool n_ok(int64_t N) { return N == 8 || N == 16 || N == 32 || N == 64; }

}  // namespace

extern "C" {

const char* ss_status_str(ss_status s) {
  switch (s) {
    case SS_OK: return "SS_OK";
    case SS_ERR_NULL: return "SS_ERR_NULL: a required pointer is NULL";
    case SS_ERR_SHAPE: return "SS_ERR_SHAPE: a size is negative or too large";
    case SS_ERR_DTYPE: return "SS_ERR_DTYPE: unknown dtype";
    case SS_ERR_N_UNSUPPORTED:
      return "SS_ERR_N_UNSUPPORTED: N must be 8, 16, 32 or 64";
    case SS_ERR_ALIGN: return "SS_ERR_ALIGN: a pointer is not 16-byte aligned";
    case SS_ERR_WORKSPACE: return "SS_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case SS_ERR_CUDA: return "SS_ERR_CUDA: the CUDA runtime reported an error";
    case SS_ERR_SCRATCH_LIMIT:
      return "SS_ERR_SCRATCH_LIMIT: the problem needs more scratch than the static buffer of "
             "ss_scan_bwd_noalloc holds";
    case SS_ERR_TIMEOUT:
      return "SS_ERR_TIMEOUT: a kernel's bounded wait on the hardware gave up (its outputs are "
             "incomplete)";
  }
  return "unknown ss_status";
}

int ss_version(void) { return 10000; }

namespace {

// ws non-null: also the chunk states, into the backward's workspace.
ss_status run_fwd(const void* u, const void* delta, const float* A, const void* B, const void* C,
                  const float* D, const void* z, const float* delta_bias, int softplus,
                  const float* h0, int64_t Bsz, int64_t Dch, int64_t L, int64_t N, ss_dtype dtype,
                  void* y, float* h_last, ss_stream_t stream, void* ws = nullptr,
                  size_t ws_bytes = 0, bool save = false) {
  if (!known_dtype(dtype)) return SS_ERR_DTYPE;
  if (bad_size(Bsz) || bad_size(Dch) || bad_size(L) || bad_size(N)) return SS_ERR_SHAPE;
  if (Bsz > 65535 || product_too_big(Bsz, Dch, L)) return SS_ERR_SHAPE;
  if (!n_ok(N)) return SS_ERR_N_UNSUPPORTED;
  const bool work = Bsz > 0 && Dch > 0 && L > 0;
  if (work && (!u || !delta || !A || !B || !C || !y)) return SS_ERR_NULL;
  if (misaligned(u) || misaligned(delta) || misaligned(A) || misaligned(B) || misaligned(C) ||
      misaligned(D) || misaligned(z) || misaligned(delta_bias) || misaligned(y) ||
      misaligned(h_last) || misaligned(h0))
    return SS_ERR_ALIGN;
  if (save && work) {
    const size_t need = selscan::bwd_workspace_bytes(Bsz, Dch, L, N);
    if (!ws || misaligned(ws) || ws_bytes < need) return SS_ERR_WORKSPACE;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!work) {
    if (h_last && Bsz > 0 && Dch > 0) {
      const size_t bytes = sizeof(float) * (size_t)(Bsz * Dch * N);
      if (!h0) return cuda_status(cudaMemsetAsync(h_last, 0, bytes, s));
      if (h0 != h_last)
        return cuda_status(cudaMemcpyAsync(h_last, h0, bytes, cudaMemcpyDeviceToDevice, s));
    }
    return SS_OK;
  }
  selscan::ScanArgs a{u, delta, A, B, C, D, z, delta_bias, softplus ? 1 : 0,
                      Bsz, Dch, L, to_dt(dtype), h0, (int)N};
  if (!save) return cuda_status(selscan::launch_scan_fwd(a, y, h_last, s));
  float* hc = reinterpret_cast<float*>(static_cast<char*>(ws) +
                                       selscan::bwd_chunk_states_offset(Bsz, Dch, L, N));
  cudaError_t e = selscan::launch_scan_fwd(a, y, h_last, s, hc);
  if (e == cudaErrorNotSupported) {
    // a chunked forward kernel: the backward's state summaries write them
    e = selscan::launch_scan_fwd(a, y, h_last, s);
    if (e == cudaSuccess) {
      selscan::BwdOut none{};
      e = selscan::launch_scan_bwd(selscan::kBwdChunkStates, a, none, ws, s);
    }
  }
  return cuda_status(e);
}

}  // namespace

ss_status ss_scan_fwd(const void* u, const void* delta, const float* A, const void* B,
                      const void* C, const float* D, const void* z, const float* delta_bias,
                      int softplus, int64_t Bsz, int64_t Dch, int64_t L, int64_t N,
                      ss_dtype dtype, void* y, float* h_last, ss_stream_t stream) {
  return run_fwd(u, delta, A, B, C, D, z, delta_bias, softplus, nullptr, Bsz, Dch, L, N, dtype,
                 y, h_last, stream);
}

ss_status ss_scan_fwd_save(const void* u, const void* delta, const float* A, const void* B,
                           const void* C, const float* D, const void* z,
                           const float* delta_bias, int softplus, int64_t Bsz, int64_t Dch,
                           int64_t L, int64_t N, ss_dtype dtype, void* y, float* h_last,
                           void* workspace, size_t workspace_bytes, ss_stream_t stream) {
  return run_fwd(u, delta, A, B, C, D, z, delta_bias, softplus, nullptr, Bsz, Dch, L, N, dtype,
                 y, h_last, stream, workspace, workspace_bytes, true);
}

ss_status ss_scan_fwd_from_state(const void* u, const void* delta, const float* A,
                                 const void* B, const void* C, const float* D, const void* z,
                                 const float* delta_bias, int softplus, const float* h0,
                                 int64_t Bsz, int64_t Dch, int64_t L, int64_t N, ss_dtype dtype,
                                 void* y, float* h_last, ss_stream_t stream) {
  return run_fwd(u, delta, A, B, C, D, z, delta_bias, softplus, h0, Bsz, Dch, L, N, dtype, y,
                 h_last, stream);
}

ss_status ss_scan_bwd_workspace_size(int64_t Bsz, int64_t Dch, int64_t L, int64_t N,
                                     ss_dtype dtype, size_t* bytes) {
  if (!bytes) return SS_ERR_NULL;
  if (!known_dtype(dtype)) return SS_ERR_DTYPE;
  if (bad_size(Bsz) || bad_size(Dch) || bad_size(L) || bad_size(N)) return SS_ERR_SHAPE;
  if (Bsz > 65535 || product_too_big(Bsz, Dch, L)) return SS_ERR_SHAPE;
  if (!n_ok(N)) return SS_ERR_N_UNSUPPORTED;
  *bytes = (Bsz > 0 && Dch > 0 && L > 0) ? selscan::bwd_workspace_bytes(Bsz, Dch, L, N) : 0;
  return SS_OK;
}

namespace {

// Checks shared by ss_scan_bwd and its three stages.  Returns SS_OK with
// *work = false when there is nothing to compute (the zero gradients have
// then been written by zero_grads when phase covers them).
ss_status check_bwd(const void* u, const void* delta, const float* A, const void* B,
                    const void* C, const float* D, const void* z, const float* delta_bias,
                    const void* dy, int64_t Bsz, int64_t Dch, int64_t L, int64_t N,
                    ss_dtype dtype, void* du, void* ddelta, float* dA, float* dB, float* dC,
                    float* dD, void* dz, float* ddelta_bias, void* workspace,
                    size_t workspace_bytes, bool* work, bool check_workspace = true) {
  if (!known_dtype(dtype)) return SS_ERR_DTYPE;
  if (bad_size(Bsz) || bad_size(Dch) || bad_size(L) || bad_size(N)) return SS_ERR_SHAPE;
  if (Bsz > 65535 || product_too_big(Bsz, Dch, L)) return SS_ERR_SHAPE;
  if (!n_ok(N)) return SS_ERR_N_UNSUPPORTED;
  *work = Bsz > 0 && Dch > 0 && L > 0;
  if (*work && (!u || !delta || !A || !B || !C || !dy || !du || !ddelta || !dA || !dB || !dC))
    return SS_ERR_NULL;
  if (*work && ((D != nullptr) != (dD != nullptr) || (z != nullptr) != (dz != nullptr) ||
                (delta_bias != nullptr) != (ddelta_bias != nullptr)))
    return SS_ERR_NULL;
  if (misaligned(u) || misaligned(delta) || misaligned(A) || misaligned(B) || misaligned(C) ||
      misaligned(D) || misaligned(z) || misaligned(delta_bias) || misaligned(dy) ||
      misaligned(du) || misaligned(ddelta) || misaligned(dA) || misaligned(dB) ||
      misaligned(dC) || misaligned(dD) || misaligned(dz) || misaligned(ddelta_bias))
    return SS_ERR_ALIGN;
  if (*work && check_workspace) {
    const size_t need = selscan::bwd_workspace_bytes(Bsz, Dch, L, N);
    if (!workspace || misaligned(workspace) || workspace_bytes < need) return SS_ERR_WORKSPACE;
  }
  return SS_OK;
}

// Empty sequence or batch: every gradient that has elements is zero.
ss_status zero_grads(int64_t Bsz, int64_t Dch, int64_t L, int64_t N, float* dA, float* dB,
                     float* dC, float* dD, float* ddelta_bias, cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  if (Dch > 0) {
    if (dA) e = cudaMemsetAsync(dA, 0, sizeof(float) * (size_t)(Dch * N), s);
    if (e == cudaSuccess && dD) e = cudaMemsetAsync(dD, 0, sizeof(float) * (size_t)Dch, s);
    if (e == cudaSuccess && ddelta_bias)
      e = cudaMemsetAsync(ddelta_bias, 0, sizeof(float) * (size_t)Dch, s);
  }
  if (e == cudaSuccess && Bsz > 0 && L > 0) {
    if (dB) e = cudaMemsetAsync(dB, 0, sizeof(float) * (size_t)(Bsz * N * L), s);
    if (e == cudaSuccess && dC) e = cudaMemsetAsync(dC, 0, sizeof(float) * (size_t)(Bsz * N * L), s);
  }
  return cuda_status(e);
}

// phase < 0: all three stages in order; kBwdStates (or kBwdAdjointStates),
// kBwdReverse, kBwdReduce: one stage.  saved: the chunk states are in the
// workspace already (ss_scan_fwd_save), so the first stage computes the
// adjoint carries only.
ss_status run_bwd(int phase, bool saved, const void* u, const void* delta, const float* A, const void* B,
                  const void* C, const float* D, const void* z, const float* delta_bias,
                  int softplus, const void* dy, int64_t Bsz, int64_t Dch, int64_t L, int64_t N,
                  ss_dtype dtype, void* du, void* ddelta, float* dA, float* dB, float* dC,
                  float* dD, void* dz, float* ddelta_bias, void* workspace,
                  size_t workspace_bytes, ss_stream_t stream) {
  bool work = false;
  ss_status st = check_bwd(u, delta, A, B, C, D, z, delta_bias, dy, Bsz, Dch, L, N, dtype, du,
                           ddelta, dA, dB, dC, dD, dz, ddelta_bias, workspace, workspace_bytes,
                           &work);
  if (st != SS_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!work) {
    if (phase < 0 || phase == selscan::kBwdReduce)
      return zero_grads(Bsz, Dch, L, N, dA, dB, dC, dD, ddelta_bias, s);
    return SS_OK;
  }
  selscan::ScanArgs a{u, delta, A, B, C, D, z, delta_bias, softplus ? 1 : 0,
                      Bsz, Dch, L, to_dt(dtype), nullptr, (int)N};
  selscan::BwdOut o{dy, du, ddelta, dA, dB, dC, dD, dz, ddelta_bias};
  for (int ph = 0; ph < 3; ++ph) {
    if (phase >= 0 && ph != phase) continue;
    const int launch = (ph == selscan::kBwdStates && saved) ? selscan::kBwdAdjointStates : ph;
    cudaError_t e = selscan::launch_scan_bwd(launch, a, o, workspace, s);
    if (e != cudaSuccess) return SS_ERR_CUDA;
  }
  return SS_OK;
}

}  // namespace

// ss_scan_bwd's argument checks without the workspace pair (for
// ss_scan_bwd_noalloc, which supplies its own); internal to the library.
__attribute__((visibility("hidden"))) ss_status selscan_check_bwd_args(
    const void* u, const void* delta, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* delta_bias, const void* dy, int64_t Bsz,
    int64_t Dch, int64_t L, int64_t N, ss_dtype dtype, void* du, void* ddelta, float* dA,
    float* dB, float* dC, float* dD, void* dz, float* ddelta_bias) {
  bool work = false;
  return check_bwd(u, delta, A, B, C, D, z, delta_bias, dy, Bsz, Dch, L, N, dtype, du, ddelta,
                   dA, dB, dC, dD, dz, ddelta_bias, nullptr, 0, &work, false);
}

#define SS_BWD_PARAMS                                                                        \
  const void *u, const void *delta, const float *A, const void *B, const void *C,             \
      const float *D, const void *z, const float *delta_bias, int softplus, const void *dy,    \
      int64_t Bsz, int64_t Dch, int64_t L, int64_t N, ss_dtype dtype, void *du, void *ddelta, \
      float *dA, float *dB, float *dC, float *dD, void *dz, float *ddelta_bias,               \
      void *workspace, size_t workspace_bytes, ss_stream_t stream
#define SS_BWD_ARGS                                                                          \
  u, delta, A, B, C, D, z, delta_bias, softplus, dy, Bsz, Dch, L, N, dtype, du, ddelta, dA, dB, \
      dC, dD, dz, ddelta_bias, workspace, workspace_bytes, stream

ss_status ss_scan_bwd(SS_BWD_PARAMS) { return run_bwd(-1, false, SS_BWD_ARGS); }
ss_status ss_scan_bwd_states(SS_BWD_PARAMS) {
  return run_bwd(selscan::kBwdStates, false, SS_BWD_ARGS);
}
ss_status ss_scan_bwd_reverse(SS_BWD_PARAMS) {
  return run_bwd(selscan::kBwdReverse, false, SS_BWD_ARGS);
}
ss_status ss_scan_bwd_reduce(SS_BWD_PARAMS) {
  return run_bwd(selscan::kBwdReduce, false, SS_BWD_ARGS);
}
ss_status ss_scan_bwd_saved(SS_BWD_PARAMS) { return run_bwd(-1, true, SS_BWD_ARGS); }
ss_status ss_scan_bwd_states_saved(SS_BWD_PARAMS) {
  return run_bwd(selscan::kBwdStates, true, SS_BWD_ARGS);
}

ss_status ss_step(float* h, const void* u_t, const void* delta_t, const float* A,
                  const void* B_t, const void* C_t, const float* D, const void* z_t,
                  const float* delta_bias, int softplus, int64_t Bsz, int64_t Dch, int64_t N,
                  ss_dtype dtype, void* y_t, ss_stream_t stream) {
  if (!known_dtype(dtype)) return SS_ERR_DTYPE;
  if (bad_size(Bsz) || bad_size(Dch) || bad_size(N)) return SS_ERR_SHAPE;
  if (Bsz > 65535 || product_too_big(Bsz, Dch, 4)) return SS_ERR_SHAPE;
  if (!n_ok(N)) return SS_ERR_N_UNSUPPORTED;
  if (Bsz == 0 || Dch == 0) return SS_OK;
  if (!h || !u_t || !delta_t || !A || !B_t || !C_t || !y_t) return SS_ERR_NULL;
  if (misaligned(h) || misaligned(u_t) || misaligned(delta_t) || misaligned(A) ||
      misaligned(B_t) || misaligned(C_t) || misaligned(D) || misaligned(z_t) ||
      misaligned(delta_bias) || misaligned(y_t))
    return SS_ERR_ALIGN;
  selscan::StepArgs a{h, u_t, delta_t, A, B_t, C_t, D, z_t, delta_bias, softplus ? 1 : 0,
                      Bsz, Dch, to_dt(dtype), y_t, (int)N};
  return cuda_status(selscan::launch_step(a, reinterpret_cast<cudaStream_t>(stream)));
}

ss_status ss_conv1d_silu_fwd(const void* x, const float* w, const float* bias, int silu,
                             int64_t Bsz, int64_t Dch, int64_t L, int64_t K, ss_dtype dtype,
                             void* u, ss_stream_t stream) {
  if (!known_dtype(dtype)) return SS_ERR_DTYPE;
  if (bad_size(Bsz) || bad_size(Dch) || bad_size(L) || K < 1 || K > 4) return SS_ERR_SHAPE;
  if (product_too_big(Bsz, Dch, L)) return SS_ERR_SHAPE;
  const bool work = Bsz > 0 && Dch > 0 && L > 0;
  if (work && (!x || !w || !u)) return SS_ERR_NULL;
  if (misaligned(x) || misaligned(w) || misaligned(bias) || misaligned(u)) return SS_ERR_ALIGN;
  if (!work) return SS_OK;
  selscan::ConvArgs a{x, w, bias, silu ? 1 : 0, Bsz, Dch, L, (int)K, to_dt(dtype), u};
  selscan::ConvGrads o{nullptr, nullptr, nullptr, nullptr};
  return cuda_status(selscan::launch_conv(0, a, o, reinterpret_cast<cudaStream_t>(stream)));
}

ss_status ss_conv1d_silu_bwd(const void* x, const float* w, const float* bias, int silu,
                             const void* du, int64_t Bsz, int64_t Dch, int64_t L, int64_t K,
                             ss_dtype dtype, void* dx, float* dw, float* dbias,
                             ss_stream_t stream) {
  if (!known_dtype(dtype)) return SS_ERR_DTYPE;
  if (bad_size(Bsz) || bad_size(Dch) || bad_size(L) || K < 1 || K > 4) return SS_ERR_SHAPE;
  if (product_too_big(Bsz, Dch, L) || Dch > 0x7fffffff) return SS_ERR_SHAPE;
  const bool work = Bsz > 0 && Dch > 0 && L > 0;
  if (Dch > 0 && !dw) return SS_ERR_NULL;
  if (Dch > 0 && (bias != nullptr) != (dbias != nullptr)) return SS_ERR_NULL;
  if (work && (!x || !w || !du || !dx)) return SS_ERR_NULL;
  if (misaligned(x) || misaligned(w) || misaligned(bias) || misaligned(du) || misaligned(dx) ||
      misaligned(dw) || misaligned(dbias))
    return SS_ERR_ALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!work) {
    if (Dch == 0) return SS_OK;
    cudaError_t e = cudaMemsetAsync(dw, 0, sizeof(float) * (size_t)(Dch * K), s);
    if (e == cudaSuccess && dbias) e = cudaMemsetAsync(dbias, 0, sizeof(float) * (size_t)Dch, s);
    return cuda_status(e);
  }
  selscan::ConvArgs a{x, w, bias, silu ? 1 : 0, Bsz, Dch, L, (int)K, to_dt(dtype), nullptr};
  selscan::ConvGrads o{du, dx, dw, dbias};
  return cuda_status(selscan::launch_conv(1, a, o, s));
}

namespace {
int g_xproj_stuck_wait = 0;  // test hook state (ss_debug_xproj_stuck_wait)
}  // namespace

ss_status ss_check_device_errors(ss_stream_t stream) {
  unsigned int flags = 0;
  if (selscan::read_clear_error_flags(reinterpret_cast<cudaStream_t>(stream), &flags) !=
      cudaSuccess)
    return SS_ERR_CUDA;
  return flags ? SS_ERR_TIMEOUT : SS_OK;
}

void ss_debug_xproj_stuck_wait(int on) { g_xproj_stuck_wait = on ? 1 : 0; }

ss_status ss_xproj(const void* u, const void* Wx, const void* Wdt, int64_t Bsz, int64_t Dch,
                   int64_t L, int64_t R, int64_t N, ss_dtype dtype, void* delta, void* B, void* C,
                   ss_stream_t stream) {
  if (dtype != SS_BF16 && dtype != SS_F16) return SS_ERR_DTYPE;
  if (bad_size(Bsz) || bad_size(Dch) || bad_size(L) || bad_size(R) || bad_size(N))
    return SS_ERR_SHAPE;
  if (product_too_big(Bsz, Dch, L) || R < 8 || R % 8 || N < 1 || R + 2 * N > 256 || Dch % 8 ||
      L % 8 || Bsz * ((L + 127) / 128) > 0x7fffffff)
    return SS_ERR_SHAPE;
  const bool work = Bsz > 0 && Dch > 0 && L > 0;
  if (work && (!u || !Wx || !Wdt || !delta || !B || !C)) return SS_ERR_NULL;
  if (misaligned(u) || misaligned(Wx) || misaligned(Wdt) || misaligned(delta) || misaligned(B) ||
      misaligned(C))
    return SS_ERR_ALIGN;
  if (!work) return SS_OK;
  unsigned int* err = nullptr;
  if (selscan::error_flags_ptr(&err) != cudaSuccess) return SS_ERR_CUDA;
  selscan::XprojArgs a{u, Wx, Wdt, Bsz, Dch, L, R, N, to_dt(dtype), delta, B, C, err,
                       g_xproj_stuck_wait};
  return cuda_status(selscan::launch_xproj(a, reinterpret_cast<cudaStream_t>(stream)));
}

int ss_xproj_wait_failures(void) {
  int n = 0;
  return selscan::xproj_wait_failures(&n) == cudaSuccess ? n : -1;
}

}  // extern "C"

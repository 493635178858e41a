// One-token recurrent step (the "RNN form" used for decoding: "mamba.py" page,
// gittoolsai.com, update of 2024-01-17 on the step function; "Mamba 7.9.1",
// lpnh.cn, section 6.2 on streaming with a carried state):
//   delta = softplus(delta_t + bias); h <- exp(delta A) h + delta B_t u_t;
//   y_t = (C_t . h + D u_t) silu(z_t)
// Bandwidth-bound on the float32 state (128 bytes read and written per row):
// one thread per (batch, channel) row keeps its 16 states in registers, with
// four 16-byte loads and stores of h in flight; A, B_t and C_t are small and
// come from the caches.
#include "common.cuh"
#include "launch.h"

namespace selscan {

namespace {

template <typename Io>
__device__ __forceinline__ void load16(const typename Io::T* p, float (&v)[kN]) {
  if constexpr (Io::kVec == 8) {
    unpack_bf16x8(*reinterpret_cast<const uint4*>(p), v);
    unpack_bf16x8(*reinterpret_cast<const uint4*>(p + 8), v + 8);
  } else {
#pragma unroll
    for (int k = 0; k < kN / 4; ++k) {
      const float4 w = *reinterpret_cast<const float4*>(p + 4 * k);
      v[4 * k] = w.x;
      v[4 * k + 1] = w.y;
      v[4 * k + 2] = w.z;
      v[4 * k + 3] = w.w;
    }
  }
}

template <typename Io>
__global__ void __launch_bounds__(256) step_kernel(StepArgs p) {
  using T = typename Io::T;
  const int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= p.Bsz * p.Dch) return;
  const int64_t b = row / p.Dch, d = row % p.Dch;
  float4* hp = reinterpret_cast<float4*>(p.h + row * kN);
  float4 h4[kN / 4];
#pragma unroll
  for (int k = 0; k < kN / 4; ++k) h4[k] = hp[k];
  const float uu = Io::to_f(static_cast<const T*>(p.u)[row]);
  const float x = Io::to_f(static_cast<const T*>(p.delta)[row]) +
                  (p.delta_bias ? p.delta_bias[d] : 0.f);
  const float dt = p.softplus ? softplus_fast(x) : x;
  const float zz = p.z ? Io::to_f(static_cast<const T*>(p.z)[row]) : 0.f;
  const float Dd = p.D ? p.D[d] : 0.f;
  float Bv[kN], Cv[kN];
  load16<Io>(static_cast<const T*>(p.B) + b * kN, Bv);
  load16<Io>(static_cast<const T*>(p.C) + b * kN, Cv);
  const float4* Ap = reinterpret_cast<const float4*>(p.A + d * kN);
  const float dtu = dt * uu;
  float y = Dd * uu;
#pragma unroll
  for (int k = 0; k < kN / 4; ++k) {
    const float4 a = Ap[k];
    float4 hv = h4[k];
    hv.x = fmaf(ex2f(dt * a.x * kLog2e), hv.x, dtu * Bv[4 * k]);
    hv.y = fmaf(ex2f(dt * a.y * kLog2e), hv.y, dtu * Bv[4 * k + 1]);
    hv.z = fmaf(ex2f(dt * a.z * kLog2e), hv.z, dtu * Bv[4 * k + 2]);
    hv.w = fmaf(ex2f(dt * a.w * kLog2e), hv.w, dtu * Bv[4 * k + 3]);
    hp[k] = hv;
    y = fmaf(Cv[4 * k], hv.x, y);
    y = fmaf(Cv[4 * k + 1], hv.y, y);
    y = fmaf(Cv[4 * k + 2], hv.z, y);
    y = fmaf(Cv[4 * k + 3], hv.w, y);
  }
  if (p.z) y *= zz * sigmoid_f(zz);
  static_cast<T*>(p.y)[row] = Io::from_f(y);
}

}  // namespace

cudaError_t launch_step(const StepArgs& a, cudaStream_t s) {
  const int64_t rows = a.Bsz * a.Dch;
  const unsigned blocks = (unsigned)((rows + 255) / 256);
  if (a.dt == Dt::BF16)
    step_kernel<IoBf16><<<blocks, 256, 0, s>>>(a);
  else
    step_kernel<IoF32><<<blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace selscan

// One-token recurrent step (the "RNN form" used for decoding: "mamba.py" page,
// gittoolsai.com, update of 2024-01-17 on the step function; "Mamba 7.9.1",
// lpnh.cn, section 6.2 on streaming with a carried state):
//   delta = softplus(delta_t + bias); h <- exp(delta A) h + delta B_t u_t;
//   y_t = (C_t . h + D u_t) silu(z_t)
// Bandwidth-bound on the float32 state: four threads per (batch, channel) row,
// each updating four states with one 16-byte load and store, so a warp moves
// 512 contiguous bytes of h per access; the C.h sum is finished with two
// shuffles inside the group of four.
#include "common.cuh"
#include "launch.h"

namespace selscan {

namespace {

template <typename Io>
__device__ __forceinline__ void load4(const typename Io::T* p, float (&v)[4]) {
  using T = typename Io::T;
  if constexpr (sizeof(T) == 2) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);  // four 16-bit elements
    const T* e = reinterpret_cast<const T*>(&w);
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = Io::to_f(e[i]);
  } else {
    const float4 w = *reinterpret_cast<const float4*>(p);
    v[0] = w.x;
    v[1] = w.y;
    v[2] = w.z;
    v[3] = w.w;
  }
}

// Grid: x = blocks of kStepRowsPerCta channels, y = batch.  Quad qi of a CTA
// owns channels d0 + qi + 64 m (m < kStepRowsPerThread): each of its loads and
// stores of h covers 64 consecutive channels (4 KB) per CTA, every thread
// keeps kStepRowsPerThread 16-byte state loads in flight, and the batch index
// comes from the grid (no division).
constexpr int kStepThreads = 256;
constexpr int kStepRowsPerThread = 1;
constexpr int kStepRowsPerCta = kStepThreads / 4 * kStepRowsPerThread;

template <typename Io>
__global__ void __launch_bounds__(kStepThreads) step_kernel(StepArgs p) {
  using T = typename Io::T;
  constexpr int M = kStepRowsPerThread;
  const int q = threadIdx.x & 3;  // states 4q .. 4q+3
  const int qi = threadIdx.x >> 2;
  const int64_t b = blockIdx.y;
  const int64_t d0 = (int64_t)blockIdx.x * kStepRowsPerCta + qi;

  float Bv[4], Cv[4];
  load4<Io>(static_cast<const T*>(p.B) + b * kN + 4 * q, Bv);
  load4<Io>(static_cast<const T*>(p.C) + b * kN + 4 * q, Cv);
  float4 hv[M], Av[M];
  float uu[M], xx[M], zz[M];
  bool valid[M];
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const int64_t d = d0 + 64 * m;
    valid[m] = d < p.Dch;
    const int64_t rr = b * p.Dch + (valid[m] ? d : 0);
    hv[m] = valid[m] ? *reinterpret_cast<const float4*>(p.h + rr * kN + 4 * q)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    Av[m] = valid[m] ? *reinterpret_cast<const float4*>(p.A + d * kN + 4 * q)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    uu[m] = valid[m] ? Io::to_f(static_cast<const T*>(p.u)[rr]) : 0.f;
    xx[m] = valid[m] ? Io::to_f(static_cast<const T*>(p.delta)[rr]) +
                           (p.delta_bias ? p.delta_bias[d] : 0.f)
                     : 0.f;
    zz[m] = (valid[m] && p.z) ? Io::to_f(static_cast<const T*>(p.z)[rr]) : 0.f;
  }
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const int64_t d = d0 + 64 * m;
    const int64_t rr = b * p.Dch + (valid[m] ? d : 0);
    const float dt = p.softplus ? softplus_fast(xx[m]) : xx[m];
    const float dtu = dt * uu[m];
    float4 h = hv[m];
    h.x = fmaf(ex2f(dt * Av[m].x * kLog2e), h.x, dtu * Bv[0]);
    h.y = fmaf(ex2f(dt * Av[m].y * kLog2e), h.y, dtu * Bv[1]);
    h.z = fmaf(ex2f(dt * Av[m].z * kLog2e), h.z, dtu * Bv[2]);
    h.w = fmaf(ex2f(dt * Av[m].w * kLog2e), h.w, dtu * Bv[3]);
    if (valid[m]) *reinterpret_cast<float4*>(p.h + rr * kN + 4 * q) = h;
    float yp = fmaf(Cv[0], h.x, fmaf(Cv[1], h.y, fmaf(Cv[2], h.z, Cv[3] * h.w)));
    yp += __shfl_xor_sync(0xffffffffu, yp, 1);
    yp += __shfl_xor_sync(0xffffffffu, yp, 2);
    if (valid[m] && q == 0) {
      float y = fmaf(p.D ? p.D[d] : 0.f, uu[m], yp);
      if (p.z) y *= zz[m] * sigmoid_f(zz[m]);
      static_cast<T*>(p.y)[rr] = Io::from_f(y);
    }
  }
}

}  // namespace

cudaError_t launch_step(const StepArgs& a, cudaStream_t s) {
  const dim3 grid((unsigned)((a.Dch + kStepRowsPerCta - 1) / kStepRowsPerCta), (unsigned)a.Bsz);
  if (a.dt == Dt::BF16)
    step_kernel<IoBf16><<<grid, kStepThreads, 0, s>>>(a);
  else if (a.dt == Dt::F16)
    step_kernel<IoF16><<<grid, kStepThreads, 0, s>>>(a);
  else
    step_kernel<IoF32><<<grid, kStepThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace selscan

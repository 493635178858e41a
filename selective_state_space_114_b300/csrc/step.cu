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

template <typename Io>
__global__ void __launch_bounds__(256) step_kernel(StepArgs p) {
  using T = typename Io::T;
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t rows = p.Bsz * p.Dch;
  const int64_t row = gid >> 2;
  const int q = threadIdx.x & 3;  // states 4q .. 4q+3
  const bool valid = row < rows;
  const int64_t rr = valid ? row : 0;
  const int64_t b = rr / p.Dch, d = rr % p.Dch;

  float yp = 0.f, uu = 0.f, zz = 0.f;
  float4 hv = make_float4(0.f, 0.f, 0.f, 0.f);
  if (valid) {
    uu = Io::to_f(static_cast<const T*>(p.u)[rr]);
    const float x = Io::to_f(static_cast<const T*>(p.delta)[rr]) +
                    (p.delta_bias ? p.delta_bias[d] : 0.f);
    const float dt = p.softplus ? softplus_fast(x) : x;
    const float4 Av = *reinterpret_cast<const float4*>(p.A + d * kN + 4 * q);
    float Bv[4], Cv[4];
    load4<Io>(static_cast<const T*>(p.B) + b * kN + 4 * q, Bv);
    load4<Io>(static_cast<const T*>(p.C) + b * kN + 4 * q, Cv);
    hv = *reinterpret_cast<const float4*>(p.h + rr * kN + 4 * q);
    const float dtu = dt * uu;
    hv.x = fmaf(ex2f(dt * Av.x * kLog2e), hv.x, dtu * Bv[0]);
    hv.y = fmaf(ex2f(dt * Av.y * kLog2e), hv.y, dtu * Bv[1]);
    hv.z = fmaf(ex2f(dt * Av.z * kLog2e), hv.z, dtu * Bv[2]);
    hv.w = fmaf(ex2f(dt * Av.w * kLog2e), hv.w, dtu * Bv[3]);
    *reinterpret_cast<float4*>(p.h + rr * kN + 4 * q) = hv;
    yp = fmaf(Cv[0], hv.x, fmaf(Cv[1], hv.y, fmaf(Cv[2], hv.z, Cv[3] * hv.w)));
    if (p.z) zz = Io::to_f(static_cast<const T*>(p.z)[rr]);
  }
  yp += __shfl_xor_sync(0xffffffffu, yp, 1);
  yp += __shfl_xor_sync(0xffffffffu, yp, 2);
  if (valid && q == 0) {
    float y = fmaf(p.D ? p.D[d] : 0.f, uu, yp);
    if (p.z) y *= zz * sigmoid_f(zz);
    static_cast<T*>(p.y)[rr] = Io::from_f(y);
  }
}

}  // namespace

cudaError_t launch_step(const StepArgs& a, cudaStream_t s) {
  const int64_t threads = a.Bsz * a.Dch * 4;
  const unsigned blocks = (unsigned)((threads + 255) / 256);
  if (a.dt == Dt::BF16)
    step_kernel<IoBf16><<<blocks, 256, 0, s>>>(a);
  else if (a.dt == Dt::F16)
    step_kernel<IoF16><<<blocks, 256, 0, s>>>(a);
  else
    step_kernel<IoF32><<<blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace selscan

// One-token recurrent step (the "RNN form" used for decoding: "mamba.py" page,
// gittoolsai.com, update of 2024-01-17 on the step function; "Mamba 7.9.1",
// lpnh.cn, section 6.2 on streaming with a carried state):
//   delta = softplus(delta_t + bias); h <- exp(delta A) h + delta B_t u_t;
//   y_t = (C_t . h + D u_t) silu(z_t)
// Bandwidth-bound on the float32 state: four threads per (batch, channel) row,
// each updating N / 4 states (with N = 16 one 16-byte load and store, so a
// warp moves 512 contiguous bytes of h per access); the C.h sum is finished
// with two shuffles inside the group of four.
// Successive steps overlap (programmatic dependent launch): a step lets the
// next one start at once; the next loads its token, A, D and delta_bias, then
// waits for the previous grid to complete before it reads or writes h and y.
#include "common.cuh"
#include "launch.h"

namespace selscan {

namespace {

// SPL consecutive elements as float (SPL = 2: one 4- or 8-byte load; SPL a
// multiple of 4: 8- or 16-byte loads).
template <typename Io, int SPL>
__device__ __forceinline__ void load_spl(const typename Io::T* p, float (&v)[SPL]) {
  using T = typename Io::T;
  if constexpr (sizeof(T) == 2) {
    if constexpr (SPL == 2) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
      const T* e = reinterpret_cast<const T*>(&w);
      v[0] = Io::to_f(e[0]);
      v[1] = Io::to_f(e[1]);
    } else {
#pragma unroll
      for (int c = 0; c < SPL / 4; ++c) {
        const uint2 w = reinterpret_cast<const uint2*>(p)[c];  // four 16-bit elements
        const T* e = reinterpret_cast<const T*>(&w);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[4 * c + i] = Io::to_f(e[i]);
      }
    }
  } else if constexpr (SPL % 4 == 0) {
#pragma unroll
    for (int c = 0; c < SPL / 4; ++c) {
      const float4 w = reinterpret_cast<const float4*>(p)[c];
      v[4 * c] = w.x;
      v[4 * c + 1] = w.y;
      v[4 * c + 2] = w.z;
      v[4 * c + 3] = w.w;
    }
  } else {
    const float2 w = *reinterpret_cast<const float2*>(p);
    v[0] = w.x;
    v[1] = w.y;
  }
}

// Grid: x = blocks of 64 channels, y = batch.  Quad qi of a CTA owns channel
// d0 + qi; each load and store of h covers 64 consecutive channels per CTA,
// and the batch index comes from the grid (no division).
constexpr int kStepThreads = 256;
constexpr int kStepRowsPerCta = kStepThreads / 4;

template <typename Io, int NS>
__global__ void __launch_bounds__(kStepThreads) step_kernel(StepArgs p) {
  using T = typename Io::T;
  constexpr int SPL = NS / 4;
  const int q = threadIdx.x & 3;  // states SPL q .. SPL q + SPL - 1
  const int64_t b = blockIdx.y;
  const int64_t d = (int64_t)blockIdx.x * kStepRowsPerCta + (threadIdx.x >> 2);
  const bool valid = d < p.Dch;
  const int64_t dd = valid ? d : 0;
  const int64_t rr = b * p.Dch + dd;

  // the next step may be scheduled now; it waits below for this grid to end
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // every load first (rows past Dch read row 0 of the batch and store nothing);
  // the token's inputs before the wait, the state after it
  float Bv[SPL], Cv[SPL], hv[SPL], Av[SPL];
  load_spl<Io, SPL>(static_cast<const T*>(p.B) + b * NS + SPL * q, Bv);
  load_spl<Io, SPL>(static_cast<const T*>(p.C) + b * NS + SPL * q, Cv);
  load_spl<IoF32, SPL>(p.A + dd * NS + SPL * q, Av);
  const float uu = Io::to_f(static_cast<const T*>(p.u)[rr]);
  const float x = Io::to_f(static_cast<const T*>(p.delta)[rr]) +
                  (p.delta_bias ? p.delta_bias[dd] : 0.f);
  const float zz = p.z ? Io::to_f(static_cast<const T*>(p.z)[rr]) : 0.f;
  const float Dd = (valid && p.D) ? p.D[d] : 0.f;
  // the previous kernel of the stream has completed and its writes are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  load_spl<IoF32, SPL>(p.h + rr * NS + SPL * q, hv);

  const float dt = p.softplus ? softplus_fast(x) : x;
  const float dtu = dt * uu;
  float yp = 0.f;
#pragma unroll
  for (int i = 0; i < SPL; ++i) {
    hv[i] = fmaf(ex2f(dt * Av[i] * kLog2e), hv[i], dtu * Bv[i]);
    yp = fmaf(Cv[i], hv[i], yp);
  }
  if (valid) {
    float* hp = p.h + rr * NS + SPL * q;
    if constexpr (SPL % 4 == 0) {
#pragma unroll
      for (int c = 0; c < SPL / 4; ++c)
        reinterpret_cast<float4*>(hp)[c] =
            make_float4(hv[4 * c], hv[4 * c + 1], hv[4 * c + 2], hv[4 * c + 3]);
    } else {
      *reinterpret_cast<float2*>(hp) = make_float2(hv[0], hv[1]);
    }
  }
  yp += __shfl_xor_sync(0xffffffffu, yp, 1);
  yp += __shfl_xor_sync(0xffffffffu, yp, 2);
  if (valid && q == 0) {
    float y = fmaf(Dd, uu, yp);
    if (p.z) y *= zz * sigmoid_f(zz);
    static_cast<T*>(p.y)[rr] = Io::from_f(y);
  }
}

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel of the stream runs, and waits for it (griddepcontrol)
// before it touches the state.
template <typename Io, int NS>
cudaError_t launch_step_ns(const StepArgs& a, const dim3& grid, cudaStream_t s) {
  return launch_pdl(step_kernel<Io, NS>, grid, dim3(kStepThreads), 0, s, a);
}

template <typename Io>
cudaError_t launch_step_t(const StepArgs& a, const dim3& grid, cudaStream_t s) {
  switch (a.N) {
    case 8: return launch_step_ns<Io, 8>(a, grid, s);
    case 16: return launch_step_ns<Io, 16>(a, grid, s);
    case 32: return launch_step_ns<Io, 32>(a, grid, s);
    case 64: return launch_step_ns<Io, 64>(a, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_step(const StepArgs& a, cudaStream_t s) {
  const dim3 grid((unsigned)((a.Dch + kStepRowsPerCta - 1) / kStepRowsPerCta), (unsigned)a.Bsz);
  if (a.dt == Dt::BF16) return launch_step_t<IoBf16>(a, grid, s);
  if (a.dt == Dt::F16) return launch_step_t<IoF16>(a, grid, s);
  return launch_step_t<IoF32>(a, grid, s);
}

}  // namespace selscan

// Causal depthwise conv1d + silu: the step of the Mamba block that produces
// the scan input u from the in-projection output x ("Mamba 7.9.1", lpnh.cn,
// section 4.1: d_conv = 4; the "mamba.py" page, resources section: the
// minimal implementation uses a plain Conv1d there):
//   c_t = bias_d + sum_{k<K} w[d][k] x_{t-(K-1)+k}   (x_s = 0 for s < 0)
//   u_t = c_t sigmoid(c_t)                          (c_t without silu)
// and its backward (g = dL/du, gc = g silu'(c)):
//   dx_s = sum_k w[d][k] gc_{s+(K-1)-k},  dw[d][k] = sum_{b,t} gc_t x_{t-(K-1)+k},
//   dbias_d = sum_{b,t} gc_t.
// Both are bandwidth-bound elementwise passes with a K-1 halo.
#include "common.cuh"
#include "launch.h"

namespace selscan {

namespace {

constexpr int kConvThreads = 256;
constexpr int kConvBwdRun = 2;  // consecutive vectors per backward item

// silu'(c) = s (1 + c (1 - s)), s = sigmoid(c)
__device__ __forceinline__ float silu_grad(float c) {
  const float s = sigmoid_f(c);
  return s * fmaf(c, 1.f - s, 1.f);
}

// ---------------------------------------------------------------------------
// forward: grid (vector blocks of a row, rows); each thread computes
// kConvVpt output vectors of kVec elements, all loads issued first.
// ---------------------------------------------------------------------------
constexpr int kConvVpt = 2;
constexpr int kConvFwdThreads = 128;  // 128 x 2 vectors = a 2048-step bf16 row per CTA

template <typename Io, int K, bool kVec>
__global__ void __launch_bounds__(kConvFwdThreads)
    conv_fwd_kernel(ConvArgs p, int64_t vecs_per_row) {
  pdl_wait();
  using T = typename Io::T;
  constexpr int V = Io::kVec;
  const int64_t row = (int64_t)blockIdx.y + (int64_t)blockIdx.z * gridDim.y;
  if (row >= p.Bsz * p.Dch) return;
  const int64_t d = row % p.Dch, L = p.L;
  const T* xr = static_cast<const T*>(p.x) + row * L;
  T* ur = static_cast<T*>(p.u) + row * L;
  float w[K];
#pragma unroll
  for (int k = 0; k < K; ++k) w[k] = p.w[d * K + k];
  const float bias = p.bias ? p.bias[d] : 0.f;
  const int64_t v0 = (int64_t)blockIdx.x * (kConvFwdThreads * kConvVpt) + threadIdx.x;
  float cur[kConvVpt][V], prev[kConvVpt][V];
#pragma unroll
  for (int m = 0; m < kConvVpt; ++m) {
    const int64_t t0 = (v0 + m * kConvFwdThreads) * V;
    const bool in = v0 + m * kConvFwdThreads < vecs_per_row;
    load_kt<Io, V, kVec>(xr, t0, L, in, cur[m]);
    if (K > 1) load_kt<Io, V, kVec>(xr, t0 - V, L, in && t0 > 0, prev[m]);
  }
#pragma unroll
  for (int m = 0; m < kConvVpt; ++m) {
    const int64_t v = v0 + m * kConvFwdThreads;
    if (v >= vecs_per_row) break;
    float xx[V + K - 1];  // x_{t0-(K-1)} .. x_{t0+V-1}
#pragma unroll
    for (int i = 0; i < K - 1; ++i) xx[i] = prev[m][V - (K - 1) + i];
#pragma unroll
    for (int i = 0; i < V; ++i) xx[K - 1 + i] = cur[m][i];
    float out[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
      float c = bias;
#pragma unroll
      for (int k = 0; k < K; ++k) c = fmaf(w[k], xx[i + k], c);
      out[i] = p.silu ? c * sigmoid_f(c) : c;
    }
    store_kt<Io, V, kVec>(ur, v * V, L, true, out);
  }
  pdl_trigger();  // the main work is done: the next kernel may be scheduled
}

// ---------------------------------------------------------------------------
// backward: one CTA per channel d, all batches (threads stride over the
// channel's (batch, vector) items; registers capped for four CTAs per SM); dx
// written elementwise, dw and dbias reduced in the CTA in a fixed order
// (bitwise reproducible).
// ---------------------------------------------------------------------------
template <typename Io, int K, bool kVec>
__global__ void __launch_bounds__(kConvThreads, 4) conv_bwd_kernel(ConvArgs p, ConvGrads o) {
  pdl_wait();
  using T = typename Io::T;
  constexpr int V = Io::kVec;
  __shared__ float red[K + 1][kConvThreads];
  const int tid = threadIdx.x;
  const int64_t d = blockIdx.x, L = p.L;
  float w[K];
#pragma unroll
  for (int k = 0; k < K; ++k) w[k] = p.w[d * K + k];
  const float bias = p.bias ? p.bias[d] : 0.f;
  float dw[K], db = 0.f;
#pragma unroll
  for (int k = 0; k < K; ++k) dw[k] = 0.f;
  // items: (batch, run of kConvBwdRun consecutive vectors) of this channel;
  // a run loads its K-1 halo steps on each side once
  constexpr int S = kConvBwdRun * V;  // steps per item
  const int64_t runs = (L + S - 1) / S;
  const int64_t items = p.Bsz * runs;
  // the item index it = b * runs + v advances by kConvThreads per pass: keep
  // (b, v) incrementally instead of dividing every pass
  int64_t b = tid / runs, v = tid - (tid / runs) * runs;
  const int64_t bstep = kConvThreads / runs, vstep = kConvThreads - bstep * runs;
  for (int64_t it = tid; it < items; it += kConvThreads) {
    const int64_t t0 = v * S;
    const int64_t row = b * p.Dch + d;
    const T* xr = static_cast<const T*>(p.x) + row * L;
    const T* gr = static_cast<const T*>(o.g) + row * L;
    v += vstep;
    b += bstep;
    if (v >= runs) {
      v -= runs;
      ++b;
    }
    // x_{t0-(K-1)} .. x_{t0+S-1+(K-1)} and g_{t0} .. g_{t0+S-1+(K-1)}; the
    // loads give 0 at and past L, so gc = 0 there and no step past L adds
    // to dw, dbias or dx
    float xx[S + 2 * (K - 1)], gg[S + K - 1];
    {
      float prev[V], cur[S], next[V], gcur[S], gnext[V];
#pragma unroll
      for (int r = 0; r < kConvBwdRun; ++r) {
        float* c = cur + r * V;
        float* gc_ = gcur + r * V;
        load_kt<Io, V, kVec>(xr, t0 + r * V, L, true, *reinterpret_cast<float(*)[V]>(c));
        load_kt<Io, V, kVec>(gr, t0 + r * V, L, true, *reinterpret_cast<float(*)[V]>(gc_));
      }
      if (K > 1) {
        load_kt<Io, V, kVec>(xr, t0 - V, L, t0 > 0, prev);
        load_kt<Io, V, kVec>(xr, t0 + S, L, true, next);
        load_kt<Io, V, kVec>(gr, t0 + S, L, true, gnext);
      }
#pragma unroll
      for (int q = 0; q < K - 1; ++q) {
        xx[q] = prev[V - (K - 1) + q];
        xx[K - 1 + S + q] = next[q];
        gg[S + q] = gnext[q];
      }
#pragma unroll
      for (int q = 0; q < S; ++q) {
        xx[K - 1 + q] = cur[q];
        gg[q] = gcur[q];
      }
    }
    // gc_t for t = t0 .. t0+S-1+(K-1)
    float gc[S + K - 1];
#pragma unroll
    for (int q = 0; q < S + K - 1; ++q) {
      float c = bias;
#pragma unroll
      for (int k = 0; k < K; ++k) c = fmaf(w[k], xx[q + k], c);
      gc[q] = p.silu ? gg[q] * silu_grad(c) : gg[q];
    }
    float dx[S];
#pragma unroll
    for (int q = 0; q < S; ++q) {
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < K; ++k) acc = fmaf(w[k], gc[q + (K - 1) - k], acc);
      dx[q] = acc;
      db += gc[q];
#pragma unroll
      for (int k = 0; k < K; ++k) dw[k] = fmaf(gc[q], xx[q + k], dw[k]);
    }
    store_kt<Io, S, kVec>(static_cast<T*>(o.dx) + row * L, t0, L, true, dx);
  }
#pragma unroll
  for (int k = 0; k < K; ++k) red[k][tid] = dw[k];
  red[K][tid] = db;
  __syncthreads();
  for (int s = kConvThreads / 2; s > 0; s >>= 1) {
    if (tid < s) {
#pragma unroll
      for (int k = 0; k <= K; ++k) red[k][tid] += red[k][tid + s];
    }
    __syncthreads();
  }
  if (tid <= K) {
    const float r = red[tid][0];
    if (tid < K)
      o.dw[d * K + tid] = r;
    else if (o.dbias)
      o.dbias[d] = r;
  }
  pdl_trigger();  // the main work is done: the next kernel may be scheduled
}

template <typename Io, int K>
cudaError_t launch_conv_k(int phase, const ConvArgs& a, const ConvGrads& o, cudaStream_t s) {
  const bool vec = a.L % Io::kVec == 0;
  if (phase == 0) {
    const int64_t vpr = (a.L + Io::kVec - 1) / Io::kVec;
    const int64_t rows = a.Bsz * a.Dch;
    const int64_t gy = rows < 65535 ? rows : 65535, gz = (rows + gy - 1) / gy;
    dim3 grid((unsigned)((vpr + kConvFwdThreads * kConvVpt - 1) / (kConvFwdThreads * kConvVpt)),
              (unsigned)gy, (unsigned)gz);
    if (vec)
      return launch_pdl(conv_fwd_kernel<Io, K, true>, grid, dim3(kConvFwdThreads), 0, s, a, vpr);
    else
      return launch_pdl(conv_fwd_kernel<Io, K, false>, grid, dim3(kConvFwdThreads), 0, s, a, vpr);
  } else {
    if (vec)
      return launch_pdl(conv_bwd_kernel<Io, K, true>, dim3((unsigned)a.Dch), dim3(kConvThreads), 0,
                        s, a, o);
    else
      return launch_pdl(conv_bwd_kernel<Io, K, false>, dim3((unsigned)a.Dch), dim3(kConvThreads), 0,
                        s, a, o);
  }
}

template <typename Io>
cudaError_t launch_conv_t(int phase, const ConvArgs& a, const ConvGrads& o, cudaStream_t s) {
  switch (a.K) {
    case 1: return launch_conv_k<Io, 1>(phase, a, o, s);
    case 2: return launch_conv_k<Io, 2>(phase, a, o, s);
    case 3: return launch_conv_k<Io, 3>(phase, a, o, s);
    default: return launch_conv_k<Io, 4>(phase, a, o, s);
  }
}

}  // namespace

cudaError_t launch_conv(int phase, const ConvArgs& a, const ConvGrads& o, cudaStream_t s) {
  if (a.dt == Dt::BF16) return launch_conv_t<IoBf16>(phase, a, o, s);
  if (a.dt == Dt::F16) return launch_conv_t<IoF16>(phase, a, o, s);
  return launch_conv_t<IoF32>(phase, a, o, s);
}

}  // namespace selscan

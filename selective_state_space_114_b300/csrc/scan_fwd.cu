// Forward selective scan: discretisation, state recurrence, contraction with
// C, D skip and silu gate fused in one pass; the state never leaves the SM.
//
// Fusion and on-chip state follow the "hardware-aware" scan described on the
// "mamba.py" page (gittoolsai.com, performance section: the state lives only
// in fast memory, cutting HBM traffic by O(N)); the recurrence is the
// sequential loop of the "PyTorch 한 파일에서의 Mamba 구현" thread
// (news.hada.io, topic 12448), evaluated here as a chunked parallel scan.
//
// Grid: x = channel groups of R = 2W rows, y = batch.  Each warp holds two
// rows; lanes of a half-warp split the current 256-step chunk into 16-step
// segments (see common.cuh).  The CTA stages B and C of its batch for the
// chunk once in shared memory (as float) and every row reuses them.  The
// state crossing chunk boundaries lives in shared memory (carry), so a CTA
// walks the whole sequence with no second pass.
#include "common.cuh"
#include "launch.h"

namespace selscan {

template <typename Io, int W, bool kVec>
__global__ void __launch_bounds__(W * 32)
    scan_fwd_kernel(ScanArgs p, typename Io::T* __restrict__ y_out, float* __restrict__ h_last) {
  using T = typename Io::T;
  constexpr int R = 2 * W;
  constexpr int NT = W * 32;
  extern __shared__ float4 smem4[];
  float* Bs = reinterpret_cast<float*>(smem4);  // [kN][kChunk] slot-permuted
  float* Cs = Bs + kN * kChunk;                 // [kN][kChunk]
  float* carry = Cs + kN * kChunk;              // [2][R][kN] state at chunk start
  float* A2s = carry + 2 * R * kN;              // [R][kN] A * log2(e)

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int j = lane & 15;
  const int r = 2 * warp + (lane >> 4);
  const int64_t b = blockIdx.y;
  const int64_t d0 = (int64_t)blockIdx.x * R;
  const int64_t d = d0 + r;
  const bool valid = d < p.Dch;
  const int64_t L = p.L;
  const int64_t row = b * p.Dch + (valid ? d : 0);

  for (int i = tid; i < R * kN; i += NT) {
    const int64_t dd = d0 + i / kN;
    carry[i] = 0.f;
    A2s[i] = dd < p.Dch ? p.A[dd * kN + i % kN] * kLog2e : 0.f;
  }
  const float Dd = (valid && p.D) ? p.D[d] : 0.f;
  const float bias = (valid && p.delta_bias) ? p.delta_bias[d] : 0.f;
  const T* urow = static_cast<const T*>(p.u) + row * L;
  const T* drow = static_cast<const T*>(p.delta) + row * L;
  const T* zrow = p.z ? static_cast<const T*>(p.z) + row * L : nullptr;
  T* yrow = y_out + row * L;
  const T* Bb = static_cast<const T*>(p.B) + b * kN * L;
  const T* Cb = static_cast<const T*>(p.C) + b * kN * L;

  int cur = 0;
  for (int64_t t0 = 0; t0 < L; t0 += kChunk, cur ^= 1) {
    __syncthreads();  // previous chunk done with Bs/Cs; carry writes visible
    stage_bc<Io, kVec>(Bb, Cb, L, t0, Bs, Cs, tid, NT);
    const int64_t ts = t0 + kT * j;
    float dl[kT], du[kT], y[kT], zz[kT];
    load_seg<Io, kVec>(urow, ts, L, valid, du);
    load_seg<Io, kVec>(drow, ts, L, valid, dl);
    load_seg<Io, kVec>(zrow, ts, L, valid && zrow != nullptr, zz);
    __syncthreads();

    float dsum = 0.f;
#pragma unroll
    for (int i = 0; i < kT; ++i) {
      const float x = dl[i] + bias;
      float dt = p.softplus ? softplus_f(x) : x;
      dt = (valid && ts + i < L) ? dt : 0.f;
      dl[i] = dt;
      y[i] = Dd * du[i];
      du[i] = dt * du[i];
      dsum += dt;
    }

#pragma unroll 1
    for (int n = 0; n < kN; ++n) {
      const float a2 = A2s[r * kN + n];
      const float hc = carry[(cur * R + r) * kN + n];
      float a[kT], bb[kT], v[kT];
      read_bc(Bs, n, j, v);
#pragma unroll
      for (int i = 0; i < kT; ++i) {
        a[i] = ex2f(dl[i] * a2);
        bb[i] = du[i] * v[i];
      }
      float S = bb[0];
#pragma unroll
      for (int i = 1; i < kT; ++i) S = fmaf(a[i], S, bb[i]);
      float P = ex2f(a2 * dsum);
      scan16_fwd(P, S, j);
      float Pe = __shfl_up_sync(0xffffffffu, P, 1, kRowLanes);
      float Se = __shfl_up_sync(0xffffffffu, S, 1, kRowLanes);
      if (j == 0) {
        Pe = 1.f;
        Se = 0.f;
      }
      float h = fmaf(Pe, hc, Se);
      read_bc(Cs, n, j, v);
#pragma unroll
      for (int i = 0; i < kT; ++i) {
        h = fmaf(a[i], h, bb[i]);
        y[i] = fmaf(v[i], h, y[i]);
      }
      if (j == kRowLanes - 1) carry[((cur ^ 1) * R + r) * kN + n] = h;
    }

    if (zrow) {
#pragma unroll
      for (int i = 0; i < kT; ++i) y[i] *= zz[i] * sigmoid_f(zz[i]);
    }
    store_seg<Io, kVec>(yrow, ts, L, valid, y);
  }
  if (h_last) {
    __syncthreads();
    if (valid) h_last[row * kN + j] = carry[(cur * R + r) * kN + j];
  }
}

template <typename Io, int W, bool kVec>
static cudaError_t launch_fwd_t(const ScanArgs& a, void* y, float* h_last, cudaStream_t s) {
  constexpr int R = 2 * W;
  const size_t smem = sizeof(float) * (2 * kN * kChunk + 3 * R * kN);
  auto kern = scan_fwd_kernel<Io, W, kVec>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((a.Dch + R - 1) / R), (unsigned)a.Bsz);
  kern<<<grid, W * 32, smem, s>>>(a, static_cast<typename Io::T*>(y), h_last);
  return cudaGetLastError();
}

cudaError_t launch_scan_fwd(const ScanArgs& a, void* y, float* h_last, cudaStream_t s) {
  constexpr int W = 8;
  if (a.dt == Dt::BF16) {
    const bool vec = (a.L % IoBf16::kVec) == 0;
    return vec ? launch_fwd_t<IoBf16, W, true>(a, y, h_last, s)
               : launch_fwd_t<IoBf16, W, false>(a, y, h_last, s);
  }
  const bool vec = (a.L % IoF32::kVec) == 0;
  return vec ? launch_fwd_t<IoF32, W, true>(a, y, h_last, s)
             : launch_fwd_t<IoF32, W, false>(a, y, h_last, s);
}

}  // namespace selscan

// Backward selective scan by recomputation.
//
// The official kernel's backward recomputes the forward's intermediates
// instead of storing them ("mamba.py" page, gittoolsai.com, performance
// section); the adjoint of the forward recurrence is a recurrence run in
// reverse time (the same page's TODO list: its parallel-scan backward runs the
// scan on time-flipped arrays).  With g = dL/dy, s = sigmoid(z):
//   yhat_t   = g_t z_t s_t                       (g_t without a gate)
//   dz_t     = g_t y_t s_t (1 + z_t (1 - s_t))   (y_t: pre-gate output)
//   lam_t[n] = yhat_t C_t[n] + a_{t+1}[n] lam_{t+1}[n]
//   du_t     = yhat_t D + delta_t sum_n lam_t[n] B_t[n]
//   ddelta_t = sum_n lam_t[n] (A[n] a_t[n] h_{t-1}[n] + B_t[n] u_t)
//   dA[n]   += sum lam_t[n] a_t[n] h_{t-1}[n] delta_t
//   dB_t[n] += lam_t[n] delta_t u_t,  dC_t[n] += yhat_t h_t[n]   (sums over d)
// with a_t h_{t-1} = h_t - b_t.
//
// Three kernels, all on the caller's stream:
//  1. bwd_states: the forward scan without outputs, storing for every
//     16-step lane segment its incoming state (workspace Hs).
//  2. bwd_main: chunks in reverse order; per state n: replay h from Hs,
//     reverse-fold the adjoint per lane, 16-lane reverse shuffle scan, replay
//     the adjoint and form all products.  dB/dC are summed over the CTA's rows
//     in shared memory and written as one partial per CTA (channel group);
//     dA/dD/dbias as one partial per (batch, channel).
//  3. bwd_reduce: sums the partials in a fixed order (deterministic results).
// The three stages are launched by launch_scan_bwd(phase = 0, 1, 2).
#include "common.cuh"
#include "launch.h"

namespace selscan {

namespace {

constexpr int kWf = 8;  // warps per CTA, state kernel
constexpr int kWb = 8;  // warps per CTA, main kernel

struct WsLayout {
  size_t hs, pbc, pa, pd, pbias, total;
  int64_t nchunks, groups;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline WsLayout ws_layout(int64_t Bsz, int64_t Dch, int64_t L) {
  WsLayout w;
  w.nchunks = (L + kChunk - 1) / kChunk;
  w.groups = (Dch + 2 * kWb - 1) / (2 * kWb);
  size_t off = 0;
  w.hs = off;
  off = align256(off + sizeof(float) * (size_t)(Bsz * Dch) * w.nchunks * kN * kRowLanes);
  w.pbc = off;
  off = align256(off + sizeof(float) * (size_t)w.groups * Bsz * 2 * kN * L);
  w.pa = off;
  off = align256(off + sizeof(float) * (size_t)(Bsz * Dch) * kN);
  w.pd = off;
  off = align256(off + sizeof(float) * (size_t)(Bsz * Dch));
  w.pbias = off;
  off = align256(off + sizeof(float) * (size_t)(Bsz * Dch));
  w.total = off;
  return w;
}

// ---------------------------------------------------------------------------
// 1. incoming state of every lane segment
// ---------------------------------------------------------------------------
template <typename Io, int W, bool kVec>
__global__ void __launch_bounds__(W * 32) bwd_states_kernel(ScanArgs p, float* __restrict__ Hs) {
  using T = typename Io::T;
  constexpr int R = 2 * W;
  constexpr int NT = W * 32;
  extern __shared__ float4 smem4[];
  float* Bs = reinterpret_cast<float*>(smem4);
  float* carry = Bs + kN * kChunk;  // [2][R][kN]
  float* A2s = carry + 2 * R * kN;  // [R][kN]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int j = lane & 15;
  const int r = 2 * warp + (lane >> 4);
  const int64_t b = blockIdx.y;
  const int64_t d0 = (int64_t)blockIdx.x * R;
  const int64_t d = d0 + r;
  const bool valid = d < p.Dch;
  const int64_t L = p.L;
  const int64_t row = b * p.Dch + (valid ? d : 0);
  const int64_t nchunks = (L + kChunk - 1) / kChunk;

  for (int i = tid; i < R * kN; i += NT) {
    const int64_t dd = d0 + i / kN;
    carry[i] = 0.f;
    A2s[i] = dd < p.Dch ? p.A[dd * kN + i % kN] * kLog2e : 0.f;
  }
  const float bias = (valid && p.delta_bias) ? p.delta_bias[d] : 0.f;
  const T* urow = static_cast<const T*>(p.u) + row * L;
  const T* drow = static_cast<const T*>(p.delta) + row * L;
  const T* Bb = static_cast<const T*>(p.B) + b * kN * L;

  int cur = 0;
  int64_t c = 0;
  for (int64_t t0 = 0; t0 < L; t0 += kChunk, cur ^= 1, ++c) {
    __syncthreads();
    // stage B only (C is not needed here); reuse the generic stager with C = B
    stage_bc<Io, kVec>(Bb, Bb, L, t0, Bs, Bs, tid, NT);
    const int64_t ts = t0 + kT * j;
    float dl[kT], du[kT];
    load_seg<Io, kVec>(urow, ts, L, valid, du);
    load_seg<Io, kVec>(drow, ts, L, valid, dl);
    __syncthreads();
    float dsum = 0.f;
#pragma unroll
    for (int i = 0; i < kT; ++i) {
      const float x = dl[i] + bias;
      float dt = p.softplus ? softplus_f(x) : x;
      dt = (valid && ts + i < L) ? dt : 0.f;
      dl[i] = dt;
      du[i] = dt * du[i];
      dsum += dt;
    }
    float* hs_out = Hs + ((row * nchunks + c) * kN) * kRowLanes + j;
#pragma unroll 1
    for (int n = 0; n < kN; ++n) {
      const float a2 = A2s[r * kN + n];
      const float hc = carry[(cur * R + r) * kN + n];
      float v[kT];
      read_bc(Bs, n, j, v);
      float S = 0.f;
#pragma unroll
      for (int i = 0; i < kT; ++i) S = fmaf(ex2f(dl[i] * a2), S, du[i] * v[i]);
      float P = ex2f(a2 * dsum);
      scan16_fwd(P, S, j);
      float Pe = __shfl_up_sync(0xffffffffu, P, 1, kRowLanes);
      float Se = __shfl_up_sync(0xffffffffu, S, 1, kRowLanes);
      if (j == 0) {
        Pe = 1.f;
        Se = 0.f;
      }
      if (valid) hs_out[n * kRowLanes] = fmaf(Pe, hc, Se);
      if (j == kRowLanes - 1) carry[((cur ^ 1) * R + r) * kN + n] = fmaf(P, hc, S);
    }
  }
}

// ---------------------------------------------------------------------------
// 2. reverse pass
// ---------------------------------------------------------------------------
template <typename Io, int W, bool kVec>
__global__ void __launch_bounds__(W * 32, 1)
    bwd_main_kernel(ScanArgs p, BwdOut o, const float* __restrict__ Hs, float* __restrict__ pBC,
                    float* __restrict__ pA, float* __restrict__ pD, float* __restrict__ pbias) {
  using T = typename Io::T;
  constexpr int R = 2 * W;
  constexpr int NT = W * 32;
  extern __shared__ float4 smem4[];
  float* Bs = reinterpret_cast<float*>(smem4);  // [kN][kChunk]
  float* Cs = Bs + kN * kChunk;                 // [kN][kChunk]
  float* red = Cs + kN * kChunk;                // [2 parity][W][2 (dB, dC)][kChunk]
  float* carry = red + 2 * W * 2 * kChunk;      // [2][R][kN] reverse carry
  float* A2s = carry + 2 * R * kN;              // [R][kN]
  float* Araw = A2s + R * kN;                   // [R][kN]
  float* dAs = Araw + R * kN;                   // [R][kN]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int j = lane & 15, half = lane >> 4;
  const int r = 2 * warp + half;
  const int64_t b = blockIdx.y;
  const int64_t g = blockIdx.x;
  const int64_t d0 = g * R;
  const int64_t d = d0 + r;
  const bool valid = d < p.Dch;
  const int64_t L = p.L;
  const int64_t Bsz = p.Bsz;
  const int64_t row = b * p.Dch + (valid ? d : 0);
  const int64_t nchunks = (L + kChunk - 1) / kChunk;

  for (int i = tid; i < R * kN; i += NT) {
    const int64_t dd = d0 + i / kN;
    const float av = dd < p.Dch ? p.A[dd * kN + i % kN] : 0.f;
    carry[i] = 0.f;
    A2s[i] = av * kLog2e;
    Araw[i] = av;
    dAs[i] = 0.f;
  }
  const float Dd = (valid && p.D) ? p.D[d] : 0.f;
  const float bias = (valid && p.delta_bias) ? p.delta_bias[d] : 0.f;
  const T* urow = static_cast<const T*>(p.u) + row * L;
  const T* drow = static_cast<const T*>(p.delta) + row * L;
  const T* zrow = p.z ? static_cast<const T*>(p.z) + row * L : nullptr;
  const T* grow = static_cast<const T*>(o.dy) + row * L;
  T* du_row = static_cast<T*>(o.du) + row * L;
  T* dd_row = static_cast<T*>(o.ddelta) + row * L;
  T* dz_row = o.dz ? static_cast<T*>(o.dz) + row * L : nullptr;
  const T* Bb = static_cast<const T*>(p.B) + b * kN * L;
  const T* Cb = static_cast<const T*>(p.C) + b * kN * L;

  float dD_acc = 0.f, dbias_acc = 0.f;
  int cur = 0;
  for (int64_t c = nchunks - 1; c >= 0; --c, cur ^= 1) {
    const int64_t t0 = c * kChunk;
    __syncthreads();
    stage_bc<Io, kVec>(Bb, Cb, L, t0, Bs, Cs, tid, NT);
    const int64_t ts = t0 + kT * j;
    float dl[kT], du[kT], yh[kT], yacc[kT], s1[kT], s2[kT];
    {
      float uu[kT], zz[kT], gg[kT];
      load_seg<Io, kVec>(urow, ts, L, valid, uu);
      load_seg<Io, kVec>(drow, ts, L, valid, dl);
      load_seg<Io, kVec>(zrow, ts, L, valid && zrow != nullptr, zz);
      load_seg<Io, kVec>(grow, ts, L, valid, gg);
#pragma unroll
      for (int i = 0; i < kT; ++i) {
        const float x = dl[i] + bias;
        float dt = p.softplus ? softplus_f(x) : x;
        dt = (valid && ts + i < L) ? dt : 0.f;
        dl[i] = dt;
        du[i] = dt * uu[i];
        yh[i] = zrow ? gg[i] * zz[i] * sigmoid_f(zz[i]) : gg[i];
        yacc[i] = Dd * uu[i];
        dD_acc = fmaf(yh[i], uu[i], dD_acc);
        s1[i] = 0.f;
        s2[i] = 0.f;
      }
    }
    float dsum = 0.f;
#pragma unroll
    for (int i = 0; i < kT; ++i) dsum += dl[i];
    const float* hs_in = Hs + ((row * nchunks + c) * kN) * kRowLanes + j;
    __syncthreads();

#pragma unroll 1
    for (int n = 0; n < kN; ++n) {
      const float a2 = A2s[r * kN + n];
      const float An = Araw[r * kN + n];
      const float rc = carry[(cur * R + r) * kN + n];
      float h = valid ? hs_in[n * kRowLanes] : 0.f;
      float a[kT], hh[kT], qq[kT], v[kT];
      read_bc(Bs, n, j, v);
      // forward replay from the stored segment state
#pragma unroll
      for (int i = 0; i < kT; ++i) {
        a[i] = ex2f(dl[i] * a2);
        qq[i] = a[i] * h;              // a_t h_{t-1}
        h = fmaf(du[i], v[i], qq[i]);  // h_t
        hh[i] = h;
      }
      // reverse fold of the adjoint within the segment (zero incoming)
      read_bc(Cs, n, j, v);
      float Lam = yh[kT - 1] * v[kT - 1];
#pragma unroll
      for (int i = kT - 2; i >= 0; --i) Lam = fmaf(a[i + 1], Lam, yh[i] * v[i]);
      float P = ex2f(a2 * dsum);
      float Q = a[0] * Lam;
      scan16_rev(P, Q, j);
      float Pe = __shfl_down_sync(0xffffffffu, P, 1, kRowLanes);
      float Qe = __shfl_down_sync(0xffffffffu, Q, 1, kRowLanes);
      if (j == kRowLanes - 1) {
        Pe = 1.f;
        Qe = 0.f;
      }
      const float rho_in = fmaf(Pe, rc, Qe);
      // products; dC, dB per time step, s1/s2/dA accumulations
      float dAn = 0.f;
      float dBv[kT], dCv[kT];
      float lam = 0.f;
#pragma unroll
      for (int i = kT - 1; i >= 0; --i) {
        const float mu = yh[i] * v[i];
        yacc[i] = fmaf(v[i], hh[i], yacc[i]);
        lam = (i == kT - 1) ? (mu + rho_in) : fmaf(a[i + 1], lam, mu);
        dCv[i] = yh[i] * hh[i];
        dBv[i] = lam * du[i];
        const float lq = lam * qq[i];
        s2[i] = fmaf(An, lq, s2[i]);
        dAn = fmaf(dl[i], lq, dAn);
        qq[i] = lam;  // keep lam_t for the B products below
      }
      if (j == 0) carry[((cur ^ 1) * R + r) * kN + n] = a[0] * qq[0];
      read_bc(Bs, n, j, v);
#pragma unroll
      for (int i = 0; i < kT; ++i) s1[i] = fmaf(qq[i], v[i], s1[i]);

      // dA: sum over the 16 lanes of the row
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1) dAn += __shfl_xor_sync(0xffffffffu, dAn, off);
      if (j == 0) dAs[r * kN + n] += dAn;

      // dB, dC: add the two rows of the warp, then sum over warps in smem
      float* slot = red + ((size_t)((n & 1) * W + warp) * 2) * kChunk;
#pragma unroll
      for (int i = 0; i < kT / 2; ++i) {
        const float sb = half ? dBv[i] : dBv[i + kT / 2];
        const float sc = half ? dCv[i] : dCv[i + kT / 2];
        const float rb = __shfl_xor_sync(0xffffffffu, sb, 16);
        const float rcv = __shfl_xor_sync(0xffffffffu, sc, 16);
        dBv[i] = (half ? dBv[i + kT / 2] : dBv[i]) + rb;
        dCv[i] = (half ? dCv[i + kT / 2] : dCv[i]) + rcv;
      }
      const int tl0 = kT * j + half * (kT / 2);
#pragma unroll
      for (int q4 = 0; q4 < kT / 8; ++q4) {
        *reinterpret_cast<float4*>(slot + tl0 + 4 * q4) =
            make_float4(dBv[4 * q4], dBv[4 * q4 + 1], dBv[4 * q4 + 2], dBv[4 * q4 + 3]);
        *reinterpret_cast<float4*>(slot + kChunk + tl0 + 4 * q4) =
            make_float4(dCv[4 * q4], dCv[4 * q4 + 1], dCv[4 * q4 + 2], dCv[4 * q4 + 3]);
      }
      __syncthreads();
      for (int i = tid; i < 2 * kChunk; i += NT) {
        const int q = i / kChunk, tl = i % kChunk;
        const float* col = red + ((size_t)((n & 1) * W) * 2 + q) * kChunk + tl;
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) acc += col[(size_t)w * 2 * kChunk];
        if (t0 + tl < L) pBC[(((g * Bsz + b) * 2 + q) * kN + n) * L + t0 + tl] = acc;
      }
    }

    // per-time-step outputs
    {
      float uu[kT], dr[kT], zz[kT], gg[kT], o1[kT], o2[kT], o3[kT];
      load_seg<Io, kVec>(urow, ts, L, valid, uu);
      load_seg<Io, kVec>(drow, ts, L, valid, dr);
      load_seg<Io, kVec>(zrow, ts, L, valid && zrow != nullptr, zz);
      load_seg<Io, kVec>(grow, ts, L, valid, gg);
#pragma unroll
      for (int i = 0; i < kT; ++i) {
        o1[i] = fmaf(yh[i], Dd, dl[i] * s1[i]);  // du
        const float ddt = fmaf(uu[i], s1[i], s2[i]);
        const float ddr = p.softplus ? ddt * sigmoid_f(dr[i] + bias) : ddt;
        o2[i] = ddr;
        dbias_acc += (valid && ts + i < L) ? ddr : 0.f;
        if (zrow) {
          const float s = sigmoid_f(zz[i]);
          o3[i] = gg[i] * yacc[i] * s * fmaf(zz[i], 1.f - s, 1.f);
        } else {
          o3[i] = 0.f;
        }
      }
      store_seg<Io, kVec>(du_row, ts, L, valid, o1);
      store_seg<Io, kVec>(dd_row, ts, L, valid, o2);
      if (dz_row) store_seg<Io, kVec>(dz_row, ts, L, valid, o3);
    }
  }

#pragma unroll
  for (int off = 8; off >= 1; off >>= 1) {
    dD_acc += __shfl_xor_sync(0xffffffffu, dD_acc, off);
    dbias_acc += __shfl_xor_sync(0xffffffffu, dbias_acc, off);
  }
  __syncthreads();
  if (valid) {
    if (j == 0) {
      pD[row] = dD_acc;
      pbias[row] = dbias_acc;
    }
    pA[row * kN + j] = dAs[r * kN + j];
  }
}

// ---------------------------------------------------------------------------
// 3. fixed-order reduction of the partials
// ---------------------------------------------------------------------------
__global__ void bwd_reduce_bc_kernel(const float* __restrict__ pBC, int64_t groups, int64_t Bsz,
                                     int64_t L, float* __restrict__ dB, float* __restrict__ dC) {
  const int64_t per = Bsz * kN * L;  // elements of dB (and of dC)
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= 2 * per) return;
  const int64_t q = i / per, e = i % per;  // e = (b * kN + n) * L + t
  const int64_t b = e / (kN * L), nt = e % (kN * L);
  float acc = 0.f;
  for (int64_t g = 0; g < groups; ++g) acc += pBC[((g * Bsz + b) * 2 + q) * kN * L + nt];
  (q ? dC : dB)[e] = acc;
}

__global__ void bwd_reduce_param_kernel(const float* __restrict__ pA, const float* __restrict__ pD,
                                        const float* __restrict__ pbias, int64_t Bsz, int64_t Dch,
                                        float* __restrict__ dA, float* __restrict__ dD,
                                        float* __restrict__ dbias) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < Dch * kN) {
    float acc = 0.f;
    for (int64_t b = 0; b < Bsz; ++b) acc += pA[b * Dch * kN + i];
    dA[i] = acc;
  }
  if (i < Dch) {
    float a1 = 0.f, a2 = 0.f;
    for (int64_t b = 0; b < Bsz; ++b) {
      a1 += pD[b * Dch + i];
      a2 += pbias[b * Dch + i];
    }
    if (dD) dD[i] = a1;
    if (dbias) dbias[i] = a2;
  }
}

template <typename Io, bool kVec>
cudaError_t launch_bwd_t(int phase, const ScanArgs& a, const BwdOut& o, void* ws, cudaStream_t s) {
  const WsLayout w = ws_layout(a.Bsz, a.Dch, a.L);
  char* base = static_cast<char*>(ws);
  float* Hs = reinterpret_cast<float*>(base + w.hs);
  float* pBC = reinterpret_cast<float*>(base + w.pbc);
  float* pA = reinterpret_cast<float*>(base + w.pa);
  float* pD = reinterpret_cast<float*>(base + w.pd);
  float* pbias = reinterpret_cast<float*>(base + w.pbias);
  cudaError_t e;
  if (phase == 0) {
    constexpr int R = 2 * kWf;
    const size_t smem = sizeof(float) * (kN * kChunk + 3 * R * kN);
    auto kern = bwd_states_kernel<Io, kWf, kVec>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((a.Dch + R - 1) / R), (unsigned)a.Bsz);
    kern<<<grid, kWf * 32, smem, s>>>(a, Hs);
    return cudaGetLastError();
  }
  if (phase == 1) {
    constexpr int R = 2 * kWb;
    const size_t smem =
        sizeof(float) * (2 * kN * kChunk + 2 * kWb * 2 * kChunk + 2 * R * kN + 3 * R * kN);
    auto kern = bwd_main_kernel<Io, kWb, kVec>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)w.groups, (unsigned)a.Bsz);
    kern<<<grid, kWb * 32, smem, s>>>(a, o, Hs, pBC, pA, pD, pbias);
    return cudaGetLastError();
  }
  const int64_t n = 2 * a.Bsz * kN * a.L;
  bwd_reduce_bc_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(pBC, w.groups, a.Bsz, a.L,
                                                                     o.dB, o.dC);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t m = a.Dch * kN;
  bwd_reduce_param_kernel<<<(unsigned)((m + 255) / 256), 256, 0, s>>>(
      pA, pD, pbias, a.Bsz, a.Dch, o.dA, o.dD, o.ddelta_bias);
  return cudaGetLastError();
}

}  // namespace

size_t bwd_workspace_bytes(int64_t Bsz, int64_t Dch, int64_t L) {
  return ws_layout(Bsz, Dch, L).total;
}

cudaError_t launch_scan_bwd(int phase, const ScanArgs& a, const BwdOut& o, void* ws,
                            cudaStream_t s) {
  if (a.dt == Dt::BF16) {
    return (a.L % IoBf16::kVec) == 0 ? launch_bwd_t<IoBf16, true>(phase, a, o, ws, s)
                                     : launch_bwd_t<IoBf16, false>(phase, a, o, ws, s);
  }
  return (a.L % IoF32::kVec) == 0 ? launch_bwd_t<IoF32, true>(phase, a, o, ws, s)
                                  : launch_bwd_t<IoF32, false>(phase, a, o, ws, s);
}

}  // namespace selscan

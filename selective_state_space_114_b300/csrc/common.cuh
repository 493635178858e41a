// Device-side building blocks shared by the selective-scan kernels.
//
// Thread layout used by the scan kernels: a warp holds two (batch, channel)
// rows, one per half-warp; lane j of a half-warp owns the kT consecutive
// time steps [t0 + kT*j, t0 + kT*j + kT) of the current chunk, so a chunk is
// kChunk = 16 * kT steps of each row.  The state recurrence
//   h_t = a_t h_{t-1} + b_t
// is evaluated per state n in three stages: a lane-local fold of its kT
// steps, a 16-lane shuffle scan over the per-lane affine maps (P, S) with
// (P1, S1) o (P2, S2) = (P1 P2, P2 S1 + S2), and a lane-local replay from
// the lane's incoming state.  The per-lane product P of the decays a_t is
// exp2(A_n log2(e) * sum_t delta_t), one MUFU op per lane and state.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace selscan {

constexpr int kN = 16;        // state size (d_state)
constexpr int kT = 16;        // time steps owned by one lane per chunk
constexpr int kRowLanes = 16; // lanes per row
constexpr int kChunk = kT * kRowLanes;  // 256 time steps per chunk
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// MUFU wrappers (approximate, flush-to-zero).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// softplus(x) = log(1 + e^x) in the overflow-free form max(x, 0) + log1p(e^-|x|).
// log1pf keeps full float accuracy when e^-|x| is small (delta ~ 1e-4 .. 1e-1).
__device__ __forceinline__ float softplus_f(float x) {
  return fmaxf(x, 0.f) + log1pf(ex2f(-fabsf(x) * kLog2e));
}

__device__ __forceinline__ float rcpf_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// logistic sigmoid 1 / (1 + e^-x)
__device__ __forceinline__ float sigmoid_f(float x) {
  return rcpf_approx(1.f + ex2f(-x * kLog2e));
}

// ---------------------------------------------------------------------------
// I/O element types.
// ---------------------------------------------------------------------------
struct IoF32 {
  using T = float;
  static constexpr int kVec = 4;  // elements per 16-byte vector
  __device__ __forceinline__ static float to_f(T v) { return v; }
  __device__ __forceinline__ static T from_f(float v) { return v; }
};

struct IoBf16 {
  using T = uint16_t;  // bf16 bit pattern
  static constexpr int kVec = 8;
  __device__ __forceinline__ static float to_f(T v) { return __uint_as_float((uint32_t)v << 16); }
  __device__ __forceinline__ static T from_f(float v) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  }
};

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void stg_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void unpack_bf16x8(uint4 w, float* f) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(ws[i] << 16);
    f[2 * i + 1] = __uint_as_float(ws[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Load kT consecutive elements row[t], t in [t, t + kT), as float; elements
// at or past L (or all of them when !valid) read as 0.  kVec: the caller
// guarantees 16-byte alignment of row + t whenever t + kT <= L.
template <typename Io, bool kVec>
__device__ __forceinline__ void load_seg(const typename Io::T* row, int64_t t, int64_t L,
                                         bool valid, float (&v)[kT]) {
  if (!valid) {
#pragma unroll
    for (int i = 0; i < kT; ++i) v[i] = 0.f;
    return;
  }
  if (kVec && t + kT <= L) {
    if constexpr (Io::kVec == 8) {
#pragma unroll
      for (int q = 0; q < kT / 8; ++q) unpack_bf16x8(ldg_nc_v4(row + t + 8 * q), v + 8 * q);
    } else {
#pragma unroll
      for (int q = 0; q < kT / 4; ++q) {
        uint4 w = ldg_nc_v4(row + t + 4 * q);
        v[4 * q] = __uint_as_float(w.x);
        v[4 * q + 1] = __uint_as_float(w.y);
        v[4 * q + 2] = __uint_as_float(w.z);
        v[4 * q + 3] = __uint_as_float(w.w);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < kT; ++i) v[i] = (t + i < L) ? Io::to_f(__ldg(row + t + i)) : 0.f;
  }
}

// Store kT values to row[t .. t + kT) (only the elements below L).
template <typename Io, bool kVec>
__device__ __forceinline__ void store_seg(typename Io::T* row, int64_t t, int64_t L, bool valid,
                                          const float (&v)[kT]) {
  if (!valid) return;
  if (kVec && t + kT <= L) {
    if constexpr (Io::kVec == 8) {
#pragma unroll
      for (int q = 0; q < kT / 8; ++q) {
        uint4 w;
        w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
        w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
        w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
        w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
        stg_v4(row + t + 8 * q, w);
      }
    } else {
#pragma unroll
      for (int q = 0; q < kT / 4; ++q) {
        uint4 w = make_uint4(__float_as_uint(v[4 * q]), __float_as_uint(v[4 * q + 1]),
                             __float_as_uint(v[4 * q + 2]), __float_as_uint(v[4 * q + 3]));
        stg_v4(row + t + 4 * q, w);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < kT; ++i)
      if (t + i < L) row[t + i] = Io::from_f(v[i]);
  }
}

// ---------------------------------------------------------------------------
// B / C chunk staging.  Shared layout per state row n (kChunk floats): the
// k-th float4 of lane j's kT-step segment sits at float4 slot k*16 + j, so
// that a half-warp's 128-bit reads of slot k are 256 contiguous bytes.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int bc_slot(int tl) {  // tl: time offset within chunk
  const int j = tl / kT, k = (tl % kT) >> 2;
  return ((k * kRowLanes + j) << 2) + (tl & 3);
}

// Stage B[b][n][t0 .. t0+kChunk) and C likewise (n < kN) into Bs/Cs
// ([kN][kChunk] floats, slot-permuted), zero past L.  All nthr threads call.
template <typename Io, bool kVec>
__device__ __forceinline__ void stage_bc(const typename Io::T* __restrict__ Bb,
                                         const typename Io::T* __restrict__ Cb, int64_t L,
                                         int64_t t0, float* Bs, float* Cs, int tid, int nthr) {
  if (kVec) {
    constexpr int V = Io::kVec;
    constexpr int vecs_per_row = kChunk / V;
    constexpr int total = 2 * kN * vecs_per_row;
    for (int i = tid; i < total; i += nthr) {
      const int which = i / (kN * vecs_per_row);
      const int rem = i % (kN * vecs_per_row);
      const int n = rem / vecs_per_row;
      const int tl = (rem % vecs_per_row) * V;
      const typename Io::T* src = (which ? Cb : Bb) + (int64_t)n * L + t0 + tl;
      float* dst = (which ? Cs : Bs) + n * kChunk;
      float f[V];
      if (t0 + tl + V <= L) {
        uint4 w = ldg_nc_v4(src);
        if constexpr (V == 8) {
          unpack_bf16x8(w, f);
        } else {
          f[0] = __uint_as_float(w.x);
          f[1] = __uint_as_float(w.y);
          f[2] = __uint_as_float(w.z);
          f[3] = __uint_as_float(w.w);
        }
      } else {
#pragma unroll
        for (int e = 0; e < V; ++e) f[e] = (t0 + tl + e < L) ? Io::to_f(src[e]) : 0.f;
      }
#pragma unroll
      for (int g = 0; g < V / 4; ++g)
        *reinterpret_cast<float4*>(dst + bc_slot(tl + 4 * g)) =
            make_float4(f[4 * g], f[4 * g + 1], f[4 * g + 2], f[4 * g + 3]);
    }
  } else {
    const int total = 2 * kN * kChunk;
    for (int i = tid; i < total; i += nthr) {
      const int which = i / (kN * kChunk);
      const int rem = i % (kN * kChunk);
      const int n = rem / kChunk, tl = rem % kChunk;
      const typename Io::T* src = (which ? Cb : Bb) + (int64_t)n * L + t0 + tl;
      float* dst = (which ? Cs : Bs) + n * kChunk;
      dst[bc_slot(tl)] = (t0 + tl < L) ? Io::to_f(*src) : 0.f;
    }
  }
}

// Read lane j's kT values of state row n from a staged buffer.
__device__ __forceinline__ void read_bc(const float* S, int n, int j, float (&v)[kT]) {
  const float4* p = reinterpret_cast<const float4*>(S + n * kChunk);
#pragma unroll
  for (int k = 0; k < kT / 4; ++k) {
    float4 q = p[k * kRowLanes + j];
    v[4 * k] = q.x;
    v[4 * k + 1] = q.y;
    v[4 * k + 2] = q.z;
    v[4 * k + 3] = q.w;
  }
}

// Inclusive scan over the 16 lanes of each half-warp of affine maps
// x -> P x + S, earlier lanes applied first.
__device__ __forceinline__ void scan16_fwd(float& P, float& S, int j) {
#pragma unroll
  for (int off = 1; off < kRowLanes; off <<= 1) {
    const float Pp = __shfl_up_sync(0xffffffffu, P, off, kRowLanes);
    const float Sp = __shfl_up_sync(0xffffffffu, S, off, kRowLanes);
    if (j >= off) {
      S = fmaf(P, Sp, S);
      P = P * Pp;
    }
  }
}

// Same, with later lanes applied first (reverse time).
__device__ __forceinline__ void scan16_rev(float& P, float& S, int j) {
#pragma unroll
  for (int off = 1; off < kRowLanes; off <<= 1) {
    const float Pn = __shfl_down_sync(0xffffffffu, P, off, kRowLanes);
    const float Sn = __shfl_down_sync(0xffffffffu, S, off, kRowLanes);
    if (j + off < kRowLanes) {
      S = fmaf(P, Sn, S);
      P = P * Pn;
    }
  }
}

}  // namespace selscan

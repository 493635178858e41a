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
#include <cuda_fp16.h>
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

// ---------------------------------------------------------------------------
// I/O element types: the element type T, the elements per 16-byte vector
// kVec, scalar conversions, and the conversion of one 16-byte vector to and
// from kVec floats (round to nearest even on the way out).
// ---------------------------------------------------------------------------
struct IoF32 {
  using T = float;
  static constexpr int kVec = 4;
  __device__ __forceinline__ static float to_f(T v) { return v; }
  __device__ __forceinline__ static T from_f(float v) { return v; }
  __device__ __forceinline__ static void unpack(uint4 w, float* f) {
    f[0] = __uint_as_float(w.x);
    f[1] = __uint_as_float(w.y);
    f[2] = __uint_as_float(w.z);
    f[3] = __uint_as_float(w.w);
  }
  __device__ __forceinline__ static uint4 pack(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
};

struct IoBf16 {
  using T = uint16_t;  // bf16 bit pattern
  static constexpr int kVec = 8;
  __device__ __forceinline__ static float to_f(T v) { return __uint_as_float((uint32_t)v << 16); }
  __device__ __forceinline__ static T from_f(float v) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  }
  __device__ __forceinline__ static void unpack(uint4 w, float* f) { unpack_bf16x8(w, f); }
  __device__ __forceinline__ static uint4 pack(const float* f) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
  }
};

struct IoF16 {
  using T = uint16_t;  // IEEE binary16 bit pattern
  static constexpr int kVec = 8;
  __device__ __forceinline__ static float to_f(T v) { return __half2float(__ushort_as_half(v)); }
  __device__ __forceinline__ static T from_f(float v) { return __half_as_ushort(__float2half_rn(v)); }
  __device__ __forceinline__ static void unpack(uint4 w, float* f) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&ws[i]));
      f[2 * i] = v.x;
      f[2 * i + 1] = v.y;
    }
  }
  __device__ __forceinline__ static uint4 pack(const float* f) {
    uint32_t r[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 v = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
      r[i] = *reinterpret_cast<const uint32_t*>(&v);
    }
    return make_uint4(r[0], r[1], r[2], r[3]);
  }
};

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
    constexpr int V = Io::kVec;
#pragma unroll
    for (int q = 0; q < kT / V; ++q) Io::unpack(ldg_nc_v4(row + t + V * q), v + V * q);
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
    constexpr int V = Io::kVec;
#pragma unroll
    for (int q = 0; q < kT / V; ++q) stg_v4(row + t + V * q, Io::pack(v + V * q));
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
        Io::unpack(ldg_nc_v4(src), f);
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

// ===========================================================================
// Programmatic dependent launch.  Every kernel of the library is launched
// with programmatic stream serialization (launch_pdl), so that it may be
// scheduled while the previous kernel of the stream finishes.  It starts
// with pdl_wait, which waits for that kernel to complete and its memory to be
// visible, and calls pdl_trigger once its main work is done, which lets the
// next kernel be scheduled as this one drains.  Only launch latency and block
// scheduling overlap, never a memory access; triggering at the end rather
// than the start keeps the next kernel's blocks from occupying SMs while
// this one still computes.
// ===========================================================================
namespace selscan {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

}  // namespace selscan

// ===========================================================================
// Building blocks of the paired-state kernels.
//
// Two states (n, n+1) travel together in a float2 and are updated by one
// packed instruction (sm_100+ f32x2 arithmetic: two IEEE fp32 operations,
// round-to-nearest, per instruction), which halves the issue slots of the
// state recurrences.
// ===========================================================================
namespace selscan {

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float lg2f_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// softplus(x) = max(x, 0) + log1p(w), w = e^-|x| in (0, 1].
// log1p(w): for w <= 1/32 the Mercator series w - w^2/2 + w^3/3 - w^4/4 + w^5/5
// (truncation error below w^6/6, i.e. < 2e-10 relative); above, ln2 * log2(1 + w),
// whose rounding of 1 + w costs at most ~2e-6 relative there.  One MUFU ex2 and
// one MUFU lg2; accurate where the steps of a selective scan live (x << 0).
__device__ __forceinline__ float softplus_fast(float x) {
  const float w = ex2f(-fabsf(x) * kLog2e);
  float s = fmaf(w, 0.2f, -0.25f);
  s = fmaf(w, s, 0.33333334f);
  s = fmaf(w, s, -0.5f);
  s = fmaf(w, s, 1.f);
  s *= w;
  const float l = lg2f_approx(1.f + w) * 0.69314718f;
  return fmaxf(x, 0.f) + (w <= 0.03125f ? s : l);
}

// Inclusive scan of the affine maps h -> P h + S on two states at once over
// the RL segments of a row, earlier segments first.  The row's lanes are
// lane0 + STRIDE * j, j = 0 .. RL-1 (STRIDE = 2: two rows interleaved in a
// warp; STRIDE = 1 with RL-lane shuffle segments otherwise).
template <int RL, int STRIDE>
__device__ __forceinline__ void scan_pair_fwd(float2& P, float2& S, int j) {
#pragma unroll
  for (int off = 1; off < RL; off <<= 1) {
    float2 Pp, Sp;
    constexpr int Wd = STRIDE == 1 ? RL : 32;
    Pp.x = __shfl_up_sync(0xffffffffu, P.x, STRIDE * off, Wd);
    Pp.y = __shfl_up_sync(0xffffffffu, P.y, STRIDE * off, Wd);
    Sp.x = __shfl_up_sync(0xffffffffu, S.x, STRIDE * off, Wd);
    Sp.y = __shfl_up_sync(0xffffffffu, S.y, STRIDE * off, Wd);
    if (j >= off) {
      S = fma2(P, Sp, S);
      P = mul2(P, Pp);
    }
  }
}

// Same with later segments applied first (the reverse-time adjoint recurrence).
template <int RL, int STRIDE>
__device__ __forceinline__ void scan_pair_rev(float2& P, float2& S, int j) {
#pragma unroll
  for (int off = 1; off < RL; off <<= 1) {
    float2 Pn, Sn;
    constexpr int Wd = STRIDE == 1 ? RL : 32;
    Pn.x = __shfl_down_sync(0xffffffffu, P.x, STRIDE * off, Wd);
    Pn.y = __shfl_down_sync(0xffffffffu, P.y, STRIDE * off, Wd);
    Sn.x = __shfl_down_sync(0xffffffffu, S.x, STRIDE * off, Wd);
    Sn.y = __shfl_down_sync(0xffffffffu, S.y, STRIDE * off, Wd);
    if (j + off < RL) {
      S = fma2(P, Sn, S);
      P = mul2(P, Pn);
    }
  }
}

// ---------------------------------------------------------------------------
// Asynchronous global -> shared copies (cp.async, 16 bytes; the bytes past
// src_bytes are zero-filled and not read).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc, int src_bytes) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem_dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gsrc),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// Wait until at most N committed groups (the newest ones) are still in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait_depth() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Wait until at most one committed group (the newest) is still in flight.
__device__ __forceinline__ void cp_async_wait_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// ---------------------------------------------------------------------------
// B / C chunk staging for the paired kernels.
//
// Raw copy: raw[2][kN][CH] elements of the I/O type (B rows then C rows of
// the chunk [t0, t0 + CH) of one batch), filled by cp.async; steps at or
// past L are zero.  Requires L % Io::kVec == 0 (16-byte aligned rows).
//
// Pair layout: float4 slot ((w * 8 + q) * (KT / 2) + k) * RL + j holds
// (X[2q][t], X[2q+1][t], X[2q][t+1], X[2q+1][t+1]) with t = KT j + 2 k and
// X = B (w = 0) or C (w = 1): lane j of a row reads its KT steps of the
// state pair q as KT/2 conflict-free 128-bit loads.
// ---------------------------------------------------------------------------
template <typename Io, int CH, int NS = kN>
__device__ __forceinline__ void issue_raw_bc(const typename Io::T* __restrict__ Bb,
                                             const typename Io::T* __restrict__ Cb, int64_t L,
                                             int64_t t0, typename Io::T* raw, int tid, int nthr) {
  using T = typename Io::T;
  constexpr int V = Io::kVec;  // elements per 16 bytes
  constexpr int per_row = CH / V;
  constexpr int total = 2 * NS * per_row;
  for (int i = tid; i < total; i += nthr) {
    const int w = i / (NS * per_row);
    const int rem = i - w * NS * per_row;
    const int n = rem / per_row;
    const int tl = (rem - n * per_row) * V;
    const int64_t t = t0 + tl;
    const T* row = (w ? Cb : Bb) + (int64_t)n * L;
    const bool in = t < L;  // whole vector in or out: L % V == 0
    cp_async16(raw + (w * NS + n) * CH + tl, in ? (const void*)(row + t) : (const void*)row,
               in ? 16 : 0);
  }
}

template <typename Io, int CH, int KT, int RL, int NS = kN>
__device__ __forceinline__ void raw_to_pairs(const typename Io::T* raw, float4* pairs, int tid,
                                             int nthr) {
  constexpr int items = 2 * (NS / 2) * (CH / 8);  // (w, q, octet of steps)
  constexpr int m = KT / 8;                         // octets per lane segment
  static_assert(CH / 8 == RL * m, "chunk = RL segments of KT steps");
  for (int i = tid; i < items; i += nthr) {
    // consecutive threads -> consecutive segments j at the same k: the four
    // 16-byte stores of a quarter-warp fill one contiguous 128-byte line
    const int x = i % (CH / 8);
    const int o = m * (x % RL) + x / RL;
    const int wq = i / (CH / 8);  // w * NS / 2 + q
    const int w = wq / (NS / 2), q = wq % (NS / 2);
    const typename Io::T* r0 = raw + (w * NS + 2 * q) * CH + 8 * o;
    const typename Io::T* r1 = r0 + CH;
    float v0[8], v1[8];
#pragma unroll
    for (int h = 0; h < 8 / Io::kVec; ++h) {
      Io::unpack(*reinterpret_cast<const uint4*>(r0 + Io::kVec * h), v0 + Io::kVec * h);
      Io::unpack(*reinterpret_cast<const uint4*>(r1 + Io::kVec * h), v1 + Io::kVec * h);
    }
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int t = 8 * o + 2 * s;
      const int j = t / KT, k = (t % KT) / 2;
      pairs[(wq * (KT / 2) + k) * RL + j] = make_float4(v0[2 * s], v1[2 * s], v0[2 * s + 1], v1[2 * s + 1]);
    }
  }
}

// Scalar (any L) version: read B/C of the chunk straight into the pair layout.
template <typename Io, int CH, int KT, int RL, int NS = kN>
__device__ __forceinline__ void load_pairs_scalar(const typename Io::T* __restrict__ Bb,
                                                  const typename Io::T* __restrict__ Cb, int64_t L,
                                                  int64_t t0, float4* pairs, int tid, int nthr) {
  constexpr int items = 2 * (NS / 2) * (CH / 2);  // (w, q, step pair)
  for (int i = tid; i < items; i += nthr) {
    const int k2 = i % (CH / 2);
    const int wq = i / (CH / 2);
    const int w = wq / (NS / 2), q = wq % (NS / 2);
    const int t = 2 * k2;
    const typename Io::T* r0 = (w ? Cb : Bb) + (int64_t)(2 * q) * L;
    const typename Io::T* r1 = r0 + L;
    const int64_t ta = t0 + t, tb = ta + 1;
    const float a0 = ta < L ? Io::to_f(r0[ta]) : 0.f, a1 = ta < L ? Io::to_f(r1[ta]) : 0.f;
    const float b0 = tb < L ? Io::to_f(r0[tb]) : 0.f, b1 = tb < L ? Io::to_f(r1[tb]) : 0.f;
    const int j = t / KT, k = (t % KT) / 2;
    pairs[(wq * (KT / 2) + k) * RL + j] = make_float4(a0, a1, b0, b1);
  }
}

// Load KT consecutive elements starting at t (KT % Io::kVec == 0) as float,
// zero at or past L.  kVec: L % Io::kVec == 0, so each 16-byte vector is
// wholly inside or outside [0, L).
template <typename Io, int KT, bool kVec>
__device__ __forceinline__ void load_kt(const typename Io::T* row, int64_t t, int64_t L, bool valid,
                                        float (&v)[KT]) {
  constexpr int V = Io::kVec;
  if (kVec) {
#pragma unroll
    for (int q = 0; q < KT / V; ++q) {
      const bool in = valid && (t + V * q < L);
      Io::unpack(in ? ldg_nc_v4(row + t + V * q) : make_uint4(0, 0, 0, 0), v + V * q);
    }
  } else {
#pragma unroll
    for (int i = 0; i < KT; ++i) v[i] = (valid && t + i < L) ? Io::to_f(row[t + i]) : 0.f;
  }
}

// Raw (undecoded) vector loads, for prefetching into registers.
template <typename Io, int KT>
struct RawSeg {
  uint4 w[KT / Io::kVec];
};

template <typename Io, int KT>
__device__ __forceinline__ void load_raw(const typename Io::T* row, int64_t t, int64_t L,
                                         bool valid, RawSeg<Io, KT>& r) {
  constexpr int V = Io::kVec;
#pragma unroll
  for (int q = 0; q < KT / V; ++q) {
    const bool in = valid && (t + V * q < L);
    r.w[q] = in ? ldg_nc_v4(row + t + V * q) : make_uint4(0, 0, 0, 0);
  }
}

template <typename Io, int KT>
__device__ __forceinline__ void decode_raw(const RawSeg<Io, KT>& r, float (&v)[KT]) {
  constexpr int V = Io::kVec;
#pragma unroll
  for (int q = 0; q < KT / V; ++q) Io::unpack(r.w[q], v + V * q);
}

// Store KT values at row[t ..) (elements below L only).
template <typename Io, int KT, bool kVec>
__device__ __forceinline__ void store_kt(typename Io::T* row, int64_t t, int64_t L, bool valid,
                                         const float (&v)[KT]) {
  if (!valid) return;
  constexpr int V = Io::kVec;
  if (kVec) {
#pragma unroll
    for (int q = 0; q < KT / V; ++q) {
      if (t + V * q >= L) continue;
      stg_v4(row + t + V * q, Io::pack(v + V * q));
    }
  } else {
#pragma unroll
    for (int i = 0; i < KT; ++i)
      if (t + i < L) row[t + i] = Io::from_f(v[i]);
  }
}

}  // namespace selscan

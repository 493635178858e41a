// Forward selective scan: discretisation, state recurrence, contraction with
// C, D skip and silu gate fused in one pass; the state never leaves the SM.
//
// Fusion and on-chip state follow the "hardware-aware" scan described on the
// "mamba.py" page (gittoolsai.com, performance section: the state lives only
// in fast memory, cutting HBM traffic by O(N)); the recurrence is the
// sequential loop of the "PyTorch 한 파일에서의 Mamba 구현" thread
// (news.hada.io, topic 12448), evaluated here as a chunked parallel scan.
//
// Three kernels.  scan_fwd_rows_kernel (at the end) walks each row in time
// order with the states split over a quad of lanes; it serves workloads with
// many rows whose byte length is a multiple of 16.  The two chunked kernels
// split the sequence of a row across lanes instead: scan_fwd_pair_kernel for
// rows of 16-byte multiples, scan_fwd_kernel, the element-wise version of
// the same scheme, for any other L.  Chunked scheme -- grid: x = channel groups of
// R = 2W rows, y = batch.  Each warp holds two rows; the lanes of a row
// split the current chunk into consecutive segments (see common.cuh).  The
// CTA stages B and C of its batch for the chunk once in shared memory (as
// float) and every row reuses them.  The state crossing chunk boundaries
// lives in shared memory (carry), so a CTA walks the whole sequence with no
// second pass.
#include "common.cuh"
#include "launch.h"

namespace selscan {

template <typename Io, int W, bool kVec>
__global__ void __launch_bounds__(W * 32)
    scan_fwd_kernel(ScanArgs p, typename Io::T* __restrict__ y_out, float* __restrict__ h_last) {
  pdl_wait();
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
    carry[i] = (p.h0 && dd < p.Dch) ? p.h0[(b * p.Dch + dd) * kN + i % kN] : 0.f;
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
  pdl_trigger();  // the main work is done: the next kernel may be scheduled
  if (h_last) {
    __syncthreads();
    if (valid) h_last[row * kN + j] = carry[(cur * R + r) * kN + j];
  }
}

// ---------------------------------------------------------------------------
// Paired-state kernel (rows whose length is a multiple of the 16-byte vector).
//
// RL = 16 lanes per row, KT steps per lane, two rows per warp in adjacent
// lanes (lane = 2 j + row), so that both rows' 128-bit reads of the shared
// B / C tiles, identical addresses, are served once; every state update
// handles the pair of states (2q, 2q+1) with
// one packed f32x2 instruction, B and C arrive by cp.async one chunk ahead
// (double-buffered raw copy, converted once per CTA into the pair layout),
// and u / delta of the next chunk are prefetched into registers while the
// current chunk is scanned.
// ---------------------------------------------------------------------------
template <typename Io, int W, int KT>
struct FwdPairCfg {
  static constexpr int RL = 16;
  static constexpr int R = 2 * W;
  static constexpr int NT = W * 32;
  static constexpr int CH = KT * RL;
  static constexpr size_t raw_bytes = 2ull * kN * CH * sizeof(typename Io::T);
  static constexpr size_t pair_bytes = 2ull * kN * CH * sizeof(float);
  // raw[2] | pairs | carry[2][R][kN] | A2[R][kN]
  static constexpr size_t smem = 2 * raw_bytes + pair_bytes + sizeof(float) * 3 * R * kN;
};

template <typename Io, int W, int KT>
__global__ void __launch_bounds__(W * 32)
    scan_fwd_pair_kernel(ScanArgs p, typename Io::T* __restrict__ y_out, float* __restrict__ h_last) {
  pdl_wait();
  using T = typename Io::T;
  using Cfg = FwdPairCfg<Io, W, KT>;
  constexpr int RL = Cfg::RL, R = Cfg::R, NT = Cfg::NT, CH = Cfg::CH;
  extern __shared__ float4 smem4[];
  T* raw0 = reinterpret_cast<T*>(smem4);
  T* raw1 = reinterpret_cast<T*>(reinterpret_cast<char*>(smem4) + Cfg::raw_bytes);
  float4* pairs = reinterpret_cast<float4*>(reinterpret_cast<char*>(smem4) + 2 * Cfg::raw_bytes);
  float* carry = reinterpret_cast<float*>(reinterpret_cast<char*>(pairs) + Cfg::pair_bytes);
  float* A2s = carry + 2 * R * kN;
  const float4* Bp = pairs;
  const float4* Cp = pairs + kN / 2 * (KT / 2) * RL;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int j = lane >> 1;
  const int r = 2 * warp + (lane & 1);
  const int64_t b = blockIdx.y;
  const int64_t d0 = (int64_t)blockIdx.x * R;
  const int64_t d = d0 + r;
  const bool valid = d < p.Dch;
  const int64_t L = p.L;
  const int64_t row = b * p.Dch + (valid ? d : 0);

  for (int i = tid; i < R * kN; i += NT) {
    const int64_t dd = d0 + i / kN;
    carry[i] = (p.h0 && dd < p.Dch) ? p.h0[(b * p.Dch + dd) * kN + i % kN] : 0.f;
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
  static_assert(RL == 16, "two interleaved rows of 16 segments per warp");

  // prologue: chunk 0's B/C copy and u/delta registers
  issue_raw_bc<Io, CH>(Bb, Cb, L, 0, raw0, tid, NT);
  cp_async_commit();
  RawSeg<Io, KT> ru, rd;
  load_raw<Io, KT>(urow, KT * j, L, valid, ru);
  load_raw<Io, KT>(drow, KT * j, L, valid, rd);

  int cur = 0;
  for (int64_t t0 = 0; t0 < L; t0 += CH, cur ^= 1) {
    cp_async_wait_all();
    __syncthreads();  // raw[cur] landed for all threads; pairs free; carry visible
    raw_to_pairs<Io, CH, KT, RL>(cur ? raw1 : raw0, pairs, tid, NT);
    if (t0 + CH < L) issue_raw_bc<Io, CH>(Bb, Cb, L, t0 + CH, cur ? raw0 : raw1, tid, NT);
    cp_async_commit();
    __syncthreads();  // pairs ready

    const int64_t ts = t0 + KT * j;
    float dl[KT], du[KT], y[KT];
    decode_raw<Io, KT>(ru, du);
    decode_raw<Io, KT>(rd, dl);
    RawSeg<Io, KT> rz;
    load_raw<Io, KT>(zrow, ts, L, valid && zrow != nullptr, rz);
    load_raw<Io, KT>(urow, ts + CH, L, valid, ru);  // next chunk
    load_raw<Io, KT>(drow, ts + CH, L, valid, rd);

    float dsum = 0.f;
#pragma unroll
    for (int i = 0; i < KT; ++i) {
      const float x = dl[i] + bias;
      float dt = p.softplus ? softplus_fast(x) : x;
      dt = (valid && ts + i < L) ? dt : 0.f;
      dl[i] = dt;
      y[i] = Dd * du[i];
      du[i] = dt * du[i];
      dsum += dt;
    }

#pragma unroll 1
    for (int q = 0; q < kN / 2; ++q) {
      const float2 a2 = *reinterpret_cast<const float2*>(A2s + r * kN + 2 * q);
      const float2 hc = *reinterpret_cast<const float2*>(carry + (cur * R + r) * kN + 2 * q);
      const float4* bq = Bp + q * (KT / 2) * RL + j;
      const float4* cq = Cp + q * (KT / 2) * RL + j;
      float2 a[KT], bb[KT], hout;
#pragma unroll
      for (int k = 0; k < KT / 2; ++k) {
        const float2 dd = make_float2(dl[2 * k], dl[2 * k + 1]);
        const float2 e0 = mul2(dd, make_float2(a2.x, a2.x));
        const float2 e1 = mul2(dd, make_float2(a2.y, a2.y));
        a[2 * k] = make_float2(ex2f(e0.x), ex2f(e1.x));
        a[2 * k + 1] = make_float2(ex2f(e0.y), ex2f(e1.y));
        const float4 v = bq[k * RL];
        bb[2 * k] = make_float2(du[2 * k] * v.x, du[2 * k] * v.y);
        bb[2 * k + 1] = make_float2(du[2 * k + 1] * v.z, du[2 * k + 1] * v.w);
      }
      float2 S = bb[0];
#pragma unroll
      for (int i = 1; i < KT; ++i) S = fma2(a[i], S, bb[i]);
      const float2 ps = mul2(make_float2(dsum, dsum), a2);
      float2 P = make_float2(ex2f(ps.x), ex2f(ps.y));
      scan_pair_fwd<RL, 2>(P, S, j);
      hout = fma2(P, hc, S);  // state after this lane's segment
      float2 h;
      h.x = __shfl_up_sync(0xffffffffu, hout.x, 2);
      h.y = __shfl_up_sync(0xffffffffu, hout.y, 2);
      if (j == 0) h = hc;
#pragma unroll
      for (int k = 0; k < KT / 2; ++k) {
        const float4 c = cq[k * RL];
        h = fma2(a[2 * k], h, bb[2 * k]);
        y[2 * k] = fmaf(c.y, h.y, fmaf(c.x, h.x, y[2 * k]));
        h = fma2(a[2 * k + 1], h, bb[2 * k + 1]);
        y[2 * k + 1] = fmaf(c.w, h.y, fmaf(c.z, h.x, y[2 * k + 1]));
      }
      if (j == RL - 1) *reinterpret_cast<float2*>(carry + ((cur ^ 1) * R + r) * kN + 2 * q) = hout;
    }

    if (zrow) {
      float zz[KT];
      decode_raw<Io, KT>(rz, zz);
#pragma unroll
      for (int i = 0; i < KT; ++i) y[i] *= zz[i] * sigmoid_f(zz[i]);
    }
    store_kt<Io, KT, true>(yrow, ts, L, valid, y);
  }
  cp_async_wait_all();
  pdl_trigger();  // the main work is done: the next kernel may be scheduled
  if (h_last) {
    __syncthreads();
    if (valid) h_last[row * kN + j] = carry[(cur * R + r) * kN + j];
  }
}

// ---------------------------------------------------------------------------
// Row-sequential kernel (every state size; with 16 states, rows whose length
// is a multiple of the 16-byte vector and enough rows to occupy every SM).
//
// The recurrence of a row is walked in time order by a quad of lanes, each
// lane holding NS / 4 of the NS states in registers for the whole sequence,
// so every h_t is formed exactly once (the chunked kernels form it twice: a
// fold of the chunk and a replay from the carried prefix).  A CTA takes R
// rows of one batch through the sequence in tiles of T steps, three phases
// per tile:
//   A  element-parallel: delta -> dt = softplus(delta + bias) and dt*u into
//      shared memory; B and C of the tile converted once to float [t][n]
//      (all R rows share them);
//   B  row quads: T steps of the recurrence; per step each lane adds the
//      C.h terms of its states and writes that partial to shared memory
//      (four steps per 128-bit store);
//   C  element-parallel: y = sum of the four partials + D u, times silu(z),
//      stored as 16-byte vectors.
// Phase C of a tile shares the barrier interval of the next tile's phase A.
// kVec (rows of 16-byte multiples): B/C tiles arrive by cp.async one tile
// ahead, and u and delta of the next tile and z of the current one are
// loaded into registers during phase B.  Otherwise every load is an
// element-wise load checked against L, issued in the phase that uses it.
// Steps at or past L and rows past Dch get dt = 0 (the state stays put).
// ---------------------------------------------------------------------------
template <typename Io, int R, int T, int NR, int NS>
struct FwdRowsCfg {
  using E = typename Io::T;
  static constexpr int NT = 4 * R / NR;          // threads: a quad per NR rows
  static constexpr int SPL = NS / 4;             // states per lane
  static constexpr int V = Io::kVec;             // elements per 16-byte vector
  static constexpr int VPR = T / V;              // vectors of a row in a tile
  static constexpr int NV = R * VPR / NT;        // vectors per thread, phases A/C
  static constexpr int RAWB = T * (int)sizeof(E) + 16;  // raw B/C row bytes (padded)
  static constexpr int CF_OFF = NS * T + 16;     // C tile offset from B tile (floats)
  static constexpr int DDS = 2 * T + 4;          // (dt, dt*u) row stride (floats)
  static constexpr int YPS = 4 * T;              // partial row stride (floats, 128-byte rows)
  static constexpr size_t raw_bytes = 2ull * 2 * NS * RAWB;
  static constexpr size_t smem =
      raw_bytes + sizeof(float) * ((size_t)CF_OFF + NS * T + (size_t)R * DDS + (size_t)R * YPS);
  static_assert(NV >= 1 && R * VPR == NV * NT, "whole vectors per thread");
  static_assert(T % 8 == 0 && (RAWB % 16) == 0 && R % (8 * NR) == 0, "tile shape");
  static_assert(NS % 8 == 0 && NS <= 64, "state pairs per lane");
};

// Position of 16-byte chunk c (the partials of steps 4 (c / 4) .. + 3 from
// state group c % 4) in partial row r.  Within each 128-byte line the chunks
// are permuted by row so that both access patterns are conflict-free: phase B
// (eight consecutive rows, one chunk) and phase C (two consecutive rows, the
// four chunks of a step group rotated by the reading lane).
__device__ __forceinline__ int ypos(int r, int c) {
  return (c & ~7) | ((((c & 7) + 4 * (r & 1)) & 7) ^ ((r >> 1) & 3));
}

// SPL consecutive floats of shared memory (16-byte aligned when SPL % 4 == 0,
// else 8-byte aligned) as SPL / 2 float2.
template <int SPL>
__device__ __forceinline__ void lds_states(const float* p, float2 (&v)[SPL / 2]) {
  if constexpr (SPL % 4 == 0) {
#pragma unroll
    for (int c = 0; c < SPL / 4; ++c) {
      const float4 w = reinterpret_cast<const float4*>(p)[c];
      v[2 * c] = make_float2(w.x, w.y);
      v[2 * c + 1] = make_float2(w.z, w.w);
    }
  } else {
#pragma unroll
    for (int c = 0; c < SPL / 2; ++c) v[c] = reinterpret_cast<const float2*>(p)[c];
  }
}

template <typename Io, int R, int T, int NR, int NS, bool kVec, bool kSave>
__global__ void __launch_bounds__(4 * R / NR)
    scan_fwd_rows_kernel(ScanArgs p, typename Io::T* __restrict__ y_out, float* __restrict__ h_last,
                         float* __restrict__ h_chunks) {
  static_assert(kScanChunk % T == 0, "chunks of whole tiles");
  pdl_wait();
  using E = typename Io::T;
  using Cfg = FwdRowsCfg<Io, R, T, NR, NS>;
  constexpr int NT = Cfg::NT, V = Cfg::V, VPR = Cfg::VPR, NV = Cfg::NV, SPL = Cfg::SPL;
  constexpr int RAWE = Cfg::RAWB / (int)sizeof(E);  // raw row stride in elements
  extern __shared__ float4 smem4[];
  char* base = reinterpret_cast<char*>(smem4);
  E* raw = reinterpret_cast<E*>(base);  // [2 buffers][2 * NS rows][RAWE]
  float* Bf = reinterpret_cast<float*>(base + Cfg::raw_bytes);
  float* Cf = Bf + Cfg::CF_OFF;
  float* dd = Cf + NS * T;  // [R][DDS]
  float* yp = dd + R * Cfg::DDS;  // [R][YPS]

  const int tid = threadIdx.x;
  const int64_t b = blockIdx.y, L = p.L, Dch = p.Dch;
  const int64_t d0 = (int64_t)blockIdx.x * R;
  const E* Bb = static_cast<const E*>(p.B) + b * NS * L;
  const E* Cb = static_cast<const E*>(p.C) + b * NS * L;

  // recurrence lane: rows qr + j R / NR (j < NR), states SPL qk .. SPL qk + SPL - 1.
  // The four lanes of a row sit one per quarter-warp (lanes l, l + 8, l + 16,
  // l + 24 of a warp), so that each quarter-warp reads a single address of the
  // B / C tile: a 128-bit load then takes two shared-memory wavefronts, where
  // four lanes per row side by side (the same address in every quarter-warp)
  // take four.
  const int qr = (tid >> 5) * 8 + (tid & 7), qk = (tid >> 3) & 3;
  float2 A2[NR][SPL / 2], h[NR][SPL / 2];
#pragma unroll
  for (int j = 0; j < NR; ++j) {
    const int64_t qd = d0 + qr + j * (R / NR);
    const bool ok = qd < Dch;
    const int64_t hrow = b * Dch + (ok ? qd : 0);
#pragma unroll
    for (int c = 0; c < SPL / 2; ++c) {
      const int n = SPL * qk + 2 * c;
      const float2 a = ok ? *reinterpret_cast<const float2*>(p.A + qd * NS + n)
                          : make_float2(0.f, 0.f);
      A2[j][c] = make_float2(a.x * kLog2e, a.y * kLog2e);
      h[j][c] = (ok && p.h0) ? *reinterpret_cast<const float2*>(p.h0 + hrow * NS + n)
                             : make_float2(0.f, 0.f);
    }
  }

  // element lanes: vector m covers row er[m], steps es[m] * V .. + V of a tile
  int er[NV], es[NV];
  bool ev[NV];
  float ebias[NV], eD[NV];
  const E* eu[NV];
  const E* edl[NV];
  const E* ez[NV];
  E* ey[NV];
#pragma unroll
  for (int m = 0; m < NV; ++m) {
    const int v = tid + NT * m;
    er[m] = v / VPR;
    es[m] = v % VPR;
    const int64_t d = d0 + er[m];
    ev[m] = d < Dch;
    const int64_t row = b * Dch + (ev[m] ? d : 0);
    ebias[m] = (ev[m] && p.delta_bias) ? p.delta_bias[d] : 0.f;
    eD[m] = (ev[m] && p.D) ? p.D[d] : 0.f;
    // row bases (element-wise path) or the lane's first vector (kVec)
    const int64_t off = row * L + (kVec ? es[m] * V : 0);
    eu[m] = static_cast<const E*>(p.u) + off;
    edl[m] = static_cast<const E*>(p.delta) + off;
    ez[m] = p.z ? static_cast<const E*>(p.z) + off : nullptr;
    ey[m] = y_out + off;
  }
  const uint4 zero4 = make_uint4(0, 0, 0, 0);

  auto issue_bc = [&](int64_t t0, E* dst) {
    for (int i = tid; i < 2 * NS * VPR; i += NT) {
      const int rr = i / VPR, s = i % VPR;  // rr = w * NS + n
      const E* src = (rr < NS ? Bb + (int64_t)rr * L : Cb + (int64_t)(rr - NS) * L);
      const int64_t t = t0 + s * V;
      const bool in = t < L;
      cp_async16(dst + rr * RAWE + s * V, in ? (const void*)(src + t) : (const void*)src,
                 in ? 16 : 0);
    }
  };

  uint4 ru[NV], rd[NV], rz[NV], ru_cur[NV];
  if constexpr (kVec) {
    issue_bc(0, raw);
    cp_async_commit();
#pragma unroll
    for (int m = 0; m < NV; ++m) {
      const bool in = ev[m] && es[m] * V < L;
      ru[m] = in ? ldg_nc_v4(eu[m]) : zero4;
      rd[m] = in ? ldg_nc_v4(edl[m]) : zero4;
      rz[m] = zero4;
      ru_cur[m] = zero4;
    }
  }

  for (int64_t t0 = 0, i = 0;; t0 += T, ++i) {
    if constexpr (kVec) cp_async_wait_all();
    __syncthreads();  // tile i's B/C landed; phase B of tile i-1 done

    // ---- phase C of tile i-1
    if (t0 > 0) {
      const int64_t tp = t0 - T;
#pragma unroll
      for (int m = 0; m < NV; ++m) {
        const int64_t t = tp + es[m] * V;
        if (!ev[m] || t >= L) continue;
        const int rot = (V == 8 ? es[m] : es[m] >> 1) & 3;  // bank-conflict-free order
        const float4* prow = reinterpret_cast<const float4*>(yp + er[m] * Cfg::YPS);
        float y[V], u[V], zz[V];
#pragma unroll
        for (int hh = 0; hh < V / 4; ++hh) {
          const int g = es[m] * (V / 4) + hh;
          float2 lo = make_float2(0.f, 0.f), hi = lo;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const float4 q = prow[ypos(er[m], 4 * g + ((kk + rot) & 3))];
            lo = add2(lo, make_float2(q.x, q.y));
            hi = add2(hi, make_float2(q.z, q.w));
          }
          y[4 * hh] = lo.x;
          y[4 * hh + 1] = lo.y;
          y[4 * hh + 2] = hi.x;
          y[4 * hh + 3] = hi.y;
        }
        if constexpr (kVec) {
          Io::unpack(ru_cur[m], u);
          if (ez[m]) Io::unpack(rz[m], zz);
        } else {
          load_kt<Io, V, false>(eu[m], t, L, true, u);
          load_kt<Io, V, false>(ez[m], t, L, ez[m] != nullptr, zz);
        }
#pragma unroll
        for (int e = 0; e < V; ++e) y[e] = fmaf(eD[m], u[e], y[e]);
        if (ez[m]) {
#pragma unroll
          for (int e = 0; e < V; ++e) y[e] *= zz[e] * sigmoid_f(zz[e]);
        }
        if constexpr (kVec)
          stg_v4(ey[m] + tp, Io::pack(y));
        else
          store_kt<Io, V, false>(ey[m], t, L, true, y);
      }
    }
    if (t0 >= L) break;

    // ---- phase A of tile i
    if constexpr (kVec) {
      const E* rb = raw + (i & 1) * (2 * NS * RAWE);
      for (int it = tid; it < 2 * NS * VPR; it += NT) {
        const int rr = it % (2 * NS), ts = it / (2 * NS);  // rr = w * NS + n
        float f[V];
        Io::unpack(*reinterpret_cast<const uint4*>(rb + rr * RAWE + ts * V), f);
        float* X = rr < NS ? Bf + rr : Cf + (rr - NS);
#pragma unroll
        for (int e = 0; e < V; ++e) X[(ts * V + e) * NS] = f[e];
      }
      if (t0 + T < L) issue_bc(t0 + T, raw + ((i + 1) & 1) * (2 * NS * RAWE));
      cp_async_commit();
    } else {
      for (int it = tid; it < 2 * NS * T; it += NT) {
        const int rr = it / T, tt = it % T;  // consecutive threads: consecutive steps
        const int64_t t = t0 + tt;
        const E* src = rr < NS ? Bb + (int64_t)rr * L : Cb + (int64_t)(rr - NS) * L;
        float* X = rr < NS ? Bf + rr : Cf + (rr - NS);
        X[tt * NS] = t < L ? Io::to_f(src[t]) : 0.f;
      }
    }
#pragma unroll
    for (int m = 0; m < NV; ++m) {
      const int64_t t = t0 + es[m] * V;
      const bool in = ev[m] && t < L;
      float u[V], dl[V];
      if constexpr (kVec) {
        Io::unpack(ru[m], u);
        Io::unpack(rd[m], dl);
      } else {
        load_kt<Io, V, false>(eu[m], t, L, ev[m], u);
        load_kt<Io, V, false>(edl[m], t, L, ev[m], dl);
      }
      float q[2 * V];
#pragma unroll
      for (int e = 0; e < V; ++e) {
        const float x = dl[e] + ebias[m];
        float dt = p.softplus ? softplus_fast(x) : x;
        dt = (in && (kVec || t + e < L)) ? dt : 0.f;
        q[2 * e] = dt;
        q[2 * e + 1] = dt * u[e];
      }
      float4* dst = reinterpret_cast<float4*>(dd + er[m] * Cfg::DDS + 2 * es[m] * V);
#pragma unroll
      for (int c = 0; c < V / 2; ++c)
        dst[c] = make_float4(q[4 * c], q[4 * c + 1], q[4 * c + 2], q[4 * c + 3]);
      if constexpr (kVec) {
        // registers for phase C of this tile and phase A of the next one
        ru_cur[m] = ru[m];
        rz[m] = (in && ez[m]) ? ldg_nc_v4(ez[m] + t0) : zero4;
        const bool nin = ev[m] && t + T < L;
        ru[m] = nin ? ldg_nc_v4(eu[m] + t0 + T) : zero4;
        rd[m] = nin ? ldg_nc_v4(edl[m] + t0 + T) : zero4;
      }
    }
    __syncthreads();  // (dt, dt*u) and the B/C tile ready; phase C of tile i-1 done

    // ---- phase B of tile i
    if (kSave && t0 % kScanChunk == 0) {
      // the state entering chunk t0 / kScanChunk (the backward's chunk states)
      const int64_t nch = (L + kScanChunk - 1) / kScanChunk, c = t0 / kScanChunk;
#pragma unroll
      for (int j = 0; j < NR; ++j) {
        const int64_t qd = d0 + qr + j * (R / NR);
        if (qd < Dch) {
          float* dst = h_chunks + ((b * Dch + qd) * nch + c) * NS + SPL * qk;
          if constexpr (SPL % 4 == 0) {
#pragma unroll
            for (int c4 = 0; c4 < SPL / 4; ++c4)
              reinterpret_cast<float4*>(dst)[c4] = make_float4(
                  h[j][2 * c4].x, h[j][2 * c4].y, h[j][2 * c4 + 1].x, h[j][2 * c4 + 1].y);
          } else {
            *reinterpret_cast<float2*>(dst) = h[j][0];
          }
        }
      }
    }
    {
      const float* Bq = Bf + SPL * qk;
      const float* Cq = Cf + SPL * qk;
#pragma unroll 2
      for (int g = 0; g < T / 4; ++g) {
        float dts[NR][4], dus[NR][4], yv[NR][4];
#pragma unroll
        for (int j = 0; j < NR; ++j) {
          const float4* d4 = reinterpret_cast<const float4*>(dd + (qr + j * (R / NR)) * Cfg::DDS);
          const float4 q0 = d4[2 * g], q1 = d4[2 * g + 1];
          dts[j][0] = q0.x, dts[j][1] = q0.z, dts[j][2] = q1.x, dts[j][3] = q1.z;
          dus[j][0] = q0.y, dus[j][1] = q0.w, dus[j][2] = q1.y, dus[j][3] = q1.w;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int t = 4 * g + e;
          float2 bv[SPL / 2], cv[SPL / 2];
          lds_states<SPL>(Bq + t * NS, bv);
          lds_states<SPL>(Cq + t * NS, cv);
#pragma unroll
          for (int j = 0; j < NR; ++j) {
            const float2 dt2 = make_float2(dts[j][e], dts[j][e]);
            const float2 du2 = make_float2(dus[j][e], dus[j][e]);
            float2 yy = make_float2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < SPL / 2; ++c) {
              const float2 ee = mul2(dt2, A2[j][c]);
              const float2 a = make_float2(ex2f(ee.x), ex2f(ee.y));
              h[j][c] = fma2(a, h[j][c], mul2(du2, bv[c]));
              yy = c ? fma2(cv[c], h[j][c], yy) : mul2(cv[c], h[j][c]);
            }
            yv[j][e] = yy.x + yy.y;
          }
        }
#pragma unroll
        for (int j = 0; j < NR; ++j)
          reinterpret_cast<float4*>(yp + (qr + j * (R / NR)) * Cfg::YPS)[ypos(qr + j * (R / NR), 4 * g + qk)] =
              make_float4(yv[j][0], yv[j][1], yv[j][2], yv[j][3]);
      }
    }
  }
  pdl_trigger();  // the main work is done: the next kernel may be scheduled
  if (h_last) {
#pragma unroll
    for (int j = 0; j < NR; ++j) {
      const int64_t qd = d0 + qr + j * (R / NR);
      if (qd < Dch) {
#pragma unroll
        for (int c = 0; c < SPL / 2; ++c)
          *reinterpret_cast<float2*>(h_last + (b * Dch + qd) * NS + SPL * qk + 2 * c) = h[j][c];
      }
    }
  }
}

template <typename Io, int R, int T, int NR, int NS, bool kVec>
static cudaError_t launch_fwd_rows(const ScanArgs& a, void* y, float* h_last, cudaStream_t s,
                                   float* h_chunks) {
  using Cfg = FwdRowsCfg<Io, R, T, NR, NS>;
  auto kern = h_chunks ? scan_fwd_rows_kernel<Io, R, T, NR, NS, kVec, true>
                       : scan_fwd_rows_kernel<Io, R, T, NR, NS, kVec, false>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((a.Dch + R - 1) / R), (unsigned)a.Bsz);
  return launch_pdl(kern, grid, dim3(Cfg::NT), Cfg::smem, s, a, static_cast<typename Io::T*>(y),
                    h_last, h_chunks);
}

template <typename Io, int W, int KT>
static cudaError_t launch_fwd_pair(const ScanArgs& a, void* y, float* h_last, cudaStream_t s) {
  using Cfg = FwdPairCfg<Io, W, KT>;
  auto kern = scan_fwd_pair_kernel<Io, W, KT>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((a.Dch + Cfg::R - 1) / Cfg::R), (unsigned)a.Bsz);
  return launch_pdl(kern, grid, dim3(W * 32), Cfg::smem, s, a, static_cast<typename Io::T*>(y),
                    h_last);
}

template <typename Io, int W, bool kVec>
static cudaError_t launch_fwd_t(const ScanArgs& a, void* y, float* h_last, cudaStream_t s) {
  constexpr int R = 2 * W;
  const size_t smem = sizeof(float) * (2 * kN * kChunk + 3 * R * kN);
  auto kern = scan_fwd_kernel<Io, W, kVec>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((a.Dch + R - 1) / R), (unsigned)a.Bsz);
  return launch_pdl(kern, grid, dim3(W * 32), smem, s, a, static_cast<typename Io::T*>(y), h_last);
}

// Rows of 16-byte multiples: with at least 8192 rows (enough quads of lanes to
// occupy every SM) the row-sequential kernel, 32 channels per CTA, one row
// per quad for 16-bit I/O and two for fp32 (measured fastest: bf16 8 x 1536
// x 2048, fp32 8 x 2048 x 2048); with fewer rows the chunked paired kernel
// (bf16 / fp16: 4 warps, 16 steps per lane; fp32: 8 warps, 8 steps per
// lane), which splits the sequence across lanes.  Other lengths take the
// element-wise kernel.
// State sizes other than 16 always take the row-sequential kernel (32
// channels per CTA, one row per quad), with element-wise loads when the rows
// are not 16-byte multiples.
constexpr int64_t kRowsKernelMinRows = 8192;

template <typename Io, int NS>
static cudaError_t launch_fwd_ns(const ScanArgs& a, void* y, float* h_last, cudaStream_t s,
                                 float* hc) {
  if (a.L % Io::kVec == 0) return launch_fwd_rows<Io, 32, 32, 1, NS, true>(a, y, h_last, s, hc);
  return launch_fwd_rows<Io, 32, 32, 1, NS, false>(a, y, h_last, s, hc);
}

template <typename Io>
static cudaError_t launch_fwd_other_n(const ScanArgs& a, void* y, float* h_last, cudaStream_t s,
                                      float* hc) {
  switch (a.N) {
    case 8: return launch_fwd_ns<Io, 8>(a, y, h_last, s, hc);
    case 32: return launch_fwd_ns<Io, 32>(a, y, h_last, s, hc);
    case 64: return launch_fwd_ns<Io, 64>(a, y, h_last, s, hc);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_scan_fwd(const ScanArgs& a, void* y, float* h_last, cudaStream_t s,
                            float* hc) {
  if (a.N != kN) {
    if (a.dt == Dt::BF16) return launch_fwd_other_n<IoBf16>(a, y, h_last, s, hc);
    if (a.dt == Dt::F16) return launch_fwd_other_n<IoF16>(a, y, h_last, s, hc);
    return launch_fwd_other_n<IoF32>(a, y, h_last, s, hc);
  }
  const bool many_rows = a.Bsz * a.Dch >= kRowsKernelMinRows;
  // the chunked kernels cannot write the chunk states
  const bool rows = many_rows && a.L % (a.dt == Dt::F32 ? IoF32::kVec : IoBf16::kVec) == 0;
  if (hc && !rows) return cudaErrorNotSupported;
  if (a.dt == Dt::BF16) {
    if (a.L % IoBf16::kVec == 0)
      return many_rows ? launch_fwd_rows<IoBf16, 32, 32, 1, 16, true>(a, y, h_last, s, hc)
                       : launch_fwd_pair<IoBf16, 4, 16>(a, y, h_last, s);
    return launch_fwd_t<IoBf16, 8, false>(a, y, h_last, s);
  }
  if (a.dt == Dt::F16) {
    if (a.L % IoF16::kVec == 0)
      return many_rows ? launch_fwd_rows<IoF16, 32, 32, 1, 16, true>(a, y, h_last, s, hc)
                       : launch_fwd_pair<IoF16, 4, 16>(a, y, h_last, s);
    return launch_fwd_t<IoF16, 8, false>(a, y, h_last, s);
  }
  if (a.L % IoF32::kVec == 0)
    return many_rows ? launch_fwd_rows<IoF32, 32, 32, 2, 16, true>(a, y, h_last, s, hc)
                     : launch_fwd_pair<IoF32, 8, 8>(a, y, h_last, s);
  return launch_fwd_t<IoF32, 8, false>(a, y, h_last, s);
}

}  // namespace selscan

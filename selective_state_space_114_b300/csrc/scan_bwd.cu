// Backward selective scan by recomputation, chunk-parallel.
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
//
// The sequence is cut into chunks of kBwdChunk steps that are processed
// independently once the state entering each chunk (forward) and the adjoint
// entering it from the later chunk (reverse) are known:
//  stage 0a  bwd_summary: one thread per (row, chunk, group of up to 16
//            states) walks the chunk in time order with the group's states in
//            registers (no cross-lane traffic) and
//            records the chunk's affine summaries: S = state at the chunk end
//            from a zero start, Q = sum_t (prod_{k<=t} a_k) yhat_t C_t (the
//            adjoint carry it sends back from a zero incoming carry), and
//            sum_t delta_t (the decay over the chunk is exp(A sum delta)).
//  stage 0b  bwd_carry: per (row, state), a walk over the chunks turns the
//            summaries into the true incoming state h_in[c] and the incoming
//            adjoint carry rho_in[c] = a lam at the first step of chunk c+1.
//  stage 1   bwd_main: per (batch, chunk, block of 64 or 128 rows): per state pair,
//            forward fold / 16-lane scan / replay for h, reverse fold / scan /
//            replay for lam, and all products.  dB and dC are summed over the
//            block's rows in shared memory (fixed order) and written as one
//            partial per (batch, row block); dA, dD, dbias as one partial per
//            (row, chunk).
//  stage 2   bwd_reduce: fixed-order sums of the partials (results are
//            bitwise reproducible).
#include <type_traits>

#include "common.cuh"
#include "launch.h"

namespace selscan {

namespace {

constexpr int kKTb = 8;                    // steps per lane (main kernel)
constexpr int kRLb = 16;                   // lanes per row
constexpr int kBwdChunk = kKTb * kRLb;     // 128 steps per chunk
static_assert(kBwdChunk == kScanChunk, "the forward's chunk states use the backward's chunks");

// What the chunk-summary stage computes: both summaries; the state ones
// alone (the chunk states for a forward that cannot write them); the adjoint
// ones alone (the chunk states were saved by the forward).
enum SumMode : int { kSumBoth = 0, kSumS = 1, kSumQ = 2 };
// Rows per CTA of the main kernel (one dB/dC partial each).  16-bit I/O: 64,
// so that the bench layer's 3072 CTAs fill 6.9 waves of three CTAs per SM
// (128 rows: 3.5 waves, 5% slower with the tail); fp32 (two CTAs per SM,
// more waves already): 128, which writes half the partials.
constexpr int kRowBlockMin = 64;
template <typename Io>
__host__ __device__ constexpr int row_block() {
  return std::is_same<Io, IoF32>::value ? 128 : 64;
}
constexpr int kSumThreads = 128;           // rows per CTA (summary kernel)
constexpr int kSumDepth = 3;               // input blocks in flight (summary kernel)

struct WsLayout {
  size_t sumS, sumQ, dsum, pbc, pa, pd, pbias, total;
  int64_t nchunks, blocks;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline WsLayout ws_layout(int64_t Bsz, int64_t Dch, int64_t L, int64_t N) {
  WsLayout w;
  w.nchunks = (L + kBwdChunk - 1) / kBwdChunk;
  w.blocks = (Dch + kRowBlockMin - 1) / kRowBlockMin;  // partials sized for the smallest block
  const size_t rc = (size_t)(Bsz * Dch) * w.nchunks;  // (row, chunk) pairs
  size_t off = 0;
  w.sumS = off;  off = align256(off + sizeof(float) * rc * N);
  w.sumQ = off;  off = align256(off + sizeof(float) * rc * N);
  w.dsum = off;  off = align256(off + sizeof(float) * rc);
  w.pbc = off;   off = align256(off + sizeof(float) * (size_t)(Bsz * w.blocks) * 2 * N * L);
  w.pa = off;    off = align256(off + sizeof(float) * rc * N);
  w.pd = off;    off = align256(off + sizeof(float) * rc);
  w.pbias = off; off = align256(off + sizeof(float) * rc);
  w.total = off;
  return w;
}

// The discretised step delta = softplus(raw + bias) (or the raw sum).
__device__ __forceinline__ float step_delta(float raw, float bias, int softplus) {
  const float x = raw + bias;
  return softplus ? softplus_fast(x) : x;
}

// ---------------------------------------------------------------------------
// 0a. chunk summaries
// ---------------------------------------------------------------------------
// NS states in groups of SG = min(NS, 16): grid z = NS / SG, each thread
// holds the SG states of its group (states SG z .. SG z + SG - 1).
// Registers capped for four CTAs per SM (128): 5% faster than three with
// bf16 I/O, the same with fp32.  The adjoint-only mode with 16-bit I/O fits
// in 95 registers and runs five CTAs per SM (6 µs less on the Mamba-130M
// layer; six gained nothing more).  MODE (SumMode) drops the state or the
// adjoint summaries, their inputs, their shared-memory tile and their stores.
template <typename Io, int MODE>
constexpr int sum_min_blocks() {
  return (MODE == kSumQ && sizeof(typename Io::T) == 2) ? 5 : 4;
}

template <typename Io, bool kVec, int NS, int MODE>
__global__ void __launch_bounds__(kSumThreads, sum_min_blocks<Io, MODE>())
    bwd_summary_kernel(ScanArgs p, BwdOut o, int64_t nrb, float* __restrict__ sumS,
                       float* __restrict__ sumQ, float* __restrict__ dsum_out) {
  pdl_wait();
  constexpr bool kS = MODE != kSumQ, kQ = MODE != kSumS;
  using T = typename Io::T;
  constexpr int CH = kBwdChunk;
  constexpr int SG = NS < 16 ? NS : 16;
  extern __shared__ float4 smem4[];
  // the B and / or C tiles the mode uses, [t][n of the group], then the ring
  float* sB = reinterpret_cast<float*>(smem4);
  float* sC = sB + (kS ? CH * SG : 0);
  uint4* ring = reinterpret_cast<uint4*>(sC + (kQ ? CH * SG : 0));  // input ring (16-byte rows only)
  const int tid = threadIdx.x;
  const int n0 = SG * blockIdx.z;
  const int64_t c = blockIdx.x / nrb;
  const int64_t rb = blockIdx.x - c * nrb;
  const int64_t b = blockIdx.y;
  const int64_t d = rb * kSumThreads + tid;
  const bool valid = d < p.Dch;
  const int64_t L = p.L, t0 = c * CH;
  const int64_t nch = (L + CH - 1) / CH;
  const int64_t row = b * p.Dch + (valid ? d : 0);

  // stage B, C of (b, chunk) transposed to [t][n]
  const T* Bb = static_cast<const T*>(p.B) + (b * NS + n0) * L;
  const T* Cb = static_cast<const T*>(p.C) + (b * NS + n0) * L;
  constexpr int w_lo = kS ? 0 : 1, w_hi = kQ ? 2 : 1;  // B (w = 0) and / or C (w = 1)
  for (int i = tid; i < (w_hi - w_lo) * SG * (CH / 8); i += kSumThreads) {
    // consecutive threads -> consecutive states n: the transposed [t][n]
    // stores of a warp land in two 64-byte runs
    const int n = i % SG;
    const int wo = i / SG;
    const int o = wo % (CH / 8), w = w_lo + wo / (CH / 8);
    const T* src = (w ? Cb : Bb) + (int64_t)n * L + t0 + 8 * o;
    float v[8];
    load_kt<Io, 8, kVec>(src, 0, L - t0 - 8 * o, true, v);
    float* dst = (w ? sC : sB) + 8 * o * SG + n;
#pragma unroll
    for (int s = 0; s < 8; ++s) dst[s * SG] = v[s];
  }
  __syncthreads();
  if (!valid) return;

  float A2[SG];
#pragma unroll
  for (int n = 0; n < SG; ++n) A2[n] = p.A[d * NS + n0 + n] * kLog2e;
  const float bias = p.delta_bias ? p.delta_bias[d] : 0.f;
  // the inputs a mode does not use are not read (they load as zeros)
  const T* urow = kS ? static_cast<const T*>(p.u) + row * L : nullptr;
  const T* drow = static_cast<const T*>(p.delta) + row * L;
  const T* zrow = (kQ && p.z) ? static_cast<const T*>(p.z) + row * L : nullptr;
  const T* grow = kQ ? static_cast<const T*>(o.dy) + row * L : nullptr;

  float2 S[SG / 2], Q[SG / 2], cp[SG / 2];
#pragma unroll
  for (int q = 0; q < SG / 2; ++q) {
    S[q] = make_float2(0.f, 0.f);
    Q[q] = make_float2(0.f, 0.f);
    cp[q] = make_float2(1.f, 1.f);
  }
  float dsum = 0.f;
  // 8-step blocks.  With 16-byte rows each thread keeps the inputs of the next
  // kSumDepth - 1 blocks in flight (cp.async into a per-thread ring in shared
  // memory, [slot][tensor][vector][thread] 16-byte units).
  constexpr int VPB = 8 / Io::kVec;  // 16-byte vectors per tensor per block
  auto issue_block = [&](int tb) {
    uint4* slot = ring + ((tb / 8) % kSumDepth) * 4 * VPB * kSumThreads;
    const T* src[4] = {urow, drow, zrow, grow};
#pragma unroll
    for (int w = 0; w < 4; ++w)
#pragma unroll
      for (int v = 0; v < VPB; ++v) {
        const int64_t t = t0 + tb + Io::kVec * v;
        const bool in = tb < CH && src[w] != nullptr && t < L;
        cp_async16(slot + (w * VPB + v) * kSumThreads + tid,
                   in ? (const void*)(src[w] + t) : (const void*)drow, in ? 16 : 0);
      }
  };
  if (kVec) {
#pragma unroll
    for (int k = 0; k < kSumDepth - 1; ++k) {
      issue_block(8 * k);
      cp_async_commit();
    }
  }
#pragma unroll 1
  for (int tb = 0; tb < CH; tb += 8) {
    const int64_t t = t0 + tb;
    float uu[8], dd[8], zz[8], gg[8];
    if (kVec) {
      issue_block(tb + 8 * (kSumDepth - 1));
      cp_async_commit();
      cp_async_wait_depth<kSumDepth - 1>();  // block tb has landed
      const uint4* slot = ring + ((tb / 8) % kSumDepth) * 4 * VPB * kSumThreads + tid;
      RawSeg<Io, 8> r;
#pragma unroll
      for (int v = 0; v < VPB; ++v) r.w[v] = slot[(0 * VPB + v) * kSumThreads];
      decode_raw<Io, 8>(r, uu);
#pragma unroll
      for (int v = 0; v < VPB; ++v) r.w[v] = slot[(1 * VPB + v) * kSumThreads];
      decode_raw<Io, 8>(r, dd);
#pragma unroll
      for (int v = 0; v < VPB; ++v) r.w[v] = slot[(2 * VPB + v) * kSumThreads];
      decode_raw<Io, 8>(r, zz);
#pragma unroll
      for (int v = 0; v < VPB; ++v) r.w[v] = slot[(3 * VPB + v) * kSumThreads];
      decode_raw<Io, 8>(r, gg);
    } else {
      load_kt<Io, 8, kVec>(urow, t, L, urow != nullptr, uu);
      load_kt<Io, 8, kVec>(drow, t, L, true, dd);
      load_kt<Io, 8, kVec>(zrow, t, L, zrow != nullptr, zz);
      load_kt<Io, 8, kVec>(grow, t, L, grow != nullptr, gg);
    }
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const bool in = t + s < L;
      const float dt = in ? step_delta(dd[s], bias, p.softplus) : 0.f;
      const float dtu = kS ? dt * uu[s] : 0.f;
      const float yh = !kQ ? 0.f : (zrow ? gg[s] * zz[s] * sigmoid_f(zz[s]) : gg[s]);
      dsum += dt;
      const float4* bq = reinterpret_cast<const float4*>(sB + (tb + s) * SG);
      const float4* cq = reinterpret_cast<const float4*>(sC + (tb + s) * SG);
#pragma unroll
      for (int k = 0; k < SG / 4; ++k) {
        const float4 bv = kS ? bq[k] : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 cv = kQ ? cq[k] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int q = 2 * k + h;
          const float2 A2q = make_float2(A2[2 * q], A2[2 * q + 1]);
          if (kS) {
            const float2 e = mul2(make_float2(dt, dt), A2q);
            const float2 a = make_float2(ex2f(e.x), ex2f(e.y));
            const float2 bp = h ? make_float2(bv.z, bv.w) : make_float2(bv.x, bv.y);
            S[q] = fma2(a, S[q], mul2(make_float2(dtu, dtu), bp));
            if (kQ) cp[q] = mul2(cp[q], a);
          } else {
            // adjoint summaries alone: the decay from the chunk start as one
            // exponential of the running sum of delta, not a running product
            const float2 e = mul2(make_float2(dsum, dsum), A2q);
            cp[q] = make_float2(ex2f(e.x), ex2f(e.y));
          }
          if (kQ) {
            const float2 cc = h ? make_float2(cv.z, cv.w) : make_float2(cv.x, cv.y);
            Q[q] = fma2(cp[q], mul2(make_float2(yh, yh), cc), Q[q]);
          }
        }
      }
    }
  }
  pdl_trigger();  // the main work is done: the next kernel may be scheduled
  const size_t rc = (size_t)row * nch + c;
  float4* so = reinterpret_cast<float4*>(sumS + rc * NS + n0);
  float4* qo = reinterpret_cast<float4*>(sumQ + rc * NS + n0);
#pragma unroll
  for (int k = 0; k < SG / 4; ++k) {
    if (kS) so[k] = make_float4(S[2 * k].x, S[2 * k].y, S[2 * k + 1].x, S[2 * k + 1].y);
    if (kQ) qo[k] = make_float4(Q[2 * k].x, Q[2 * k].y, Q[2 * k + 1].x, Q[2 * k + 1].y);
  }
  if (n0 == 0) dsum_out[rc] = dsum;
}

// ---------------------------------------------------------------------------
// 0b. chunk carries: sumS[row][c] <- h entering chunk c; sumQ[row][c] <- the
//     adjoint carry entering chunk c from chunk c+1 (zero for the last).
// ---------------------------------------------------------------------------
template <int NS, int MODE>
__global__ void bwd_carry_kernel(const float* __restrict__ A, int64_t Bsz, int64_t Dch,
                                 int64_t nch, float* __restrict__ sumS, float* __restrict__ sumQ,
                                 const float* __restrict__ dsum) {
  pdl_wait();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= Bsz * Dch * NS) return;
  const int64_t row = i / NS;
  const int n = (int)(i % NS);
  const int64_t d = row % Dch;
  const float a2 = A[d * NS + n] * kLog2e;
  float h = 0.f;
  for (int64_t c = 0; c < nch && MODE != kSumQ; ++c) {
    const size_t rc = (size_t)row * nch + c;
    const float P = ex2f(a2 * dsum[rc]);
    const float s = sumS[rc * NS + n];
    sumS[rc * NS + n] = h;
    h = fmaf(P, h, s);
  }
  float rho = 0.f;
  for (int64_t c = nch - 1; c >= 0 && MODE != kSumS; --c) {
    const size_t rc = (size_t)row * nch + c;
    const float P = ex2f(a2 * dsum[rc]);
    const float qv = sumQ[rc * NS + n];
    sumQ[rc * NS + n] = rho;
    rho = fmaf(P, rho, qv);
  }
  pdl_trigger();  // the main work is done: the next kernel may be scheduled
}

// ---------------------------------------------------------------------------
// 1. main reverse pass
//
// Lane layout: the two rows of a warp sit in adjacent lanes (lane = 2 j + rs,
// j = 0..15 the time segment, rs the row), so the 128-bit reads of the B / C
// pair layout, identical for both rows, are served once per lane pair.
// Per state pair the lane runs: forward and reverse folds and their
// 16-segment scans (interleaved), the forward replay (h_t, qq_t = a_t h_{t-1},
// pre-gate output, dC terms), the reverse replay (lam_t, dB terms, the du /
// ddelta sums over states, dA terms).  Every row of a pass writes its dB / dC
// terms to its own slot; after a barrier the CTA's threads sum the pass's
// rows' slots into the block accumulator.
// ---------------------------------------------------------------------------
template <int W, typename T, int kSlotBufs, int NS>
struct MainSmem {
  static constexpr int KT = kKTb, RL = kRLb, CH = kBwdChunk, R = 2 * W;
  static constexpr size_t pairs = sizeof(float4) * 2 * (NS / 2) * (KT / 2) * RL;  // B, C
  static constexpr size_t slot_row = 2 * CH * 2 + 4;  // [dB,dC][CH][2 states] floats, padded
                                                      // so the two rows of a warp use other banks
  static constexpr size_t slots = sizeof(float) * kSlotBufs * R * slot_row;  // [buffer][row]
  static constexpr size_t acc = sizeof(float) * 2 * NS * CH;            // [dB,dC][q][CH][2]
  static constexpr size_t dA = sizeof(float) * R * NS * RL;             // [row][n][j]
  static constexpr size_t params = sizeof(float) * 4 * R * NS;          // A2, A, h_in, rho_in
  // u, delta, z, dy segments of a pass, [buffer][tensor][vector][thread] 16-byte units
  static constexpr size_t ins = 2ull * 4 * KT * sizeof(T) * (W * 32);
  static constexpr size_t total = pairs + slots + acc + dA + params + ins;
};

// Copy the KT-step segments of u, delta, z, dy of one row into the lane's
// slots of an input buffer (cp.async; zeros for an invalid row, for steps at
// or past L and for an absent z).  Rows of 16-byte multiples only.
template <typename Io, int KT, int NT>
__device__ __forceinline__ void issue_row_inputs(const ScanArgs& p, const void* dy, int64_t row,
                                                 bool valid, int64_t ts, int64_t L, uint4* buf,
                                                 int tid) {
  using T = typename Io::T;
  constexpr int V = Io::kVec, VPL = KT / V;
  const T* src[4] = {static_cast<const T*>(p.u) + row * L, static_cast<const T*>(p.delta) + row * L,
                     p.z ? static_cast<const T*>(p.z) + row * L : nullptr,
                     static_cast<const T*>(dy) + row * L};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
      const int64_t t = ts + V * v;
      const bool in = valid && src[w] != nullptr && t < L;
      cp_async16(buf + (w * VPL + v) * NT + tid, in ? (const void*)(src[w] + t) : (const void*)src[0],
                 in ? 16 : 0);
    }
  }
}

template <typename Io, int KT, int NT>
__device__ __forceinline__ void read_row_input(const uint4* buf, int w, int tid, float (&v)[KT]) {
  constexpr int V = Io::kVec, VPL = KT / V;
  RawSeg<Io, KT> r;
#pragma unroll
  for (int k = 0; k < VPL; ++k) r.w[k] = buf[(w * VPL + k) * NT + tid];
  decode_raw<Io, KT>(r, v);
}

// KT steps of a state pair, stored as [step][state]: two steps per float4.
// The lane's KT / 2 float4 are rotated by sw (slot_swizzle) so that the eight
// lanes of a quarter-warp (four segments j, two rows) hit eight different
// 16-byte bank groups.
template <int KT>
__device__ __forceinline__ void store_steps(float* dst, const float2 (&v)[KT], int sw) {
#pragma unroll
  for (int i = 0; i < KT; i += 2) {
    const int k = ((i >> 1) + sw) & (KT / 2 - 1);
    *reinterpret_cast<float4*>(dst + 4 * k) = make_float4(v[i].x, v[i].y, v[i + 1].x, v[i + 1].y);
  }
}

__device__ __forceinline__ int slot_swizzle(int j) { return 2 * ((j >> 1) & 1); }

// One state pair q of one row: forward fold / scan / replay, reverse fold /
// scan / replay and the products.  Accumulates the per-step sums over states
// (pre-gate output, sum lam B, sum A lam a h) in the row's registers, stores
// the row's dB and dC terms of the pair at dB_lo / dC_lo (state 2q, state 2q+1
// at +CH) and the lane's dA terms of the two states at dA_lo[0], dA_lo[RL].
template <int KT, int RL, int CH, int NS, bool kKeepB, bool kSyncSlots>
__device__ __forceinline__ void bwd_state_pair(
    int q, int j, int r, bool valid, const float* A2s, const float* Ars, const float* hin_row,
    const float* rin_row, const float4* Bp, const float4* Cp, const float (&dl)[KT],
    const float2 (&du2)[KT], const float2 (&yh2)[KT], float dsum, float2 (&yacc2)[KT],
    float2 (&s12)[KT], float2 (&s22)[KT], float* dB_lo, float* dC_lo, float* dA_lo) {
    const float2 a2 = *reinterpret_cast<const float2*>(A2s + r * NS + 2 * q);
    const float2 Ar = *reinterpret_cast<const float2*>(Ars + r * NS + 2 * q);
    const float2 hc = valid ? *reinterpret_cast<const float2*>(hin_row + 2 * q) : make_float2(0.f, 0.f);
    const float2 rcar = valid ? *reinterpret_cast<const float2*>(rin_row + 2 * q) : make_float2(0.f, 0.f);
    const float4* bq = Bp + q * (KT / 2) * RL + j;
    const float4* cq = Cp + q * (KT / 2) * RL + j;

    float2 a[KT], bb[KT], mu[KT];
    // kKeepB: the lane's B steps stay in registers from the prep to the
    // reverse replay (one shared-memory read instead of two)
    float4 Bk[KT / 2];
    if (kKeepB) {
#pragma unroll
      for (int k = 0; k < KT / 2; ++k) Bk[k] = bq[k * RL];
    }
#pragma unroll
    for (int k = 0; k < KT / 2; ++k) {
      const float2 dd = make_float2(dl[2 * k], dl[2 * k + 1]);
      const float2 e0 = mul2(dd, make_float2(a2.x, a2.x));
      const float2 e1 = mul2(dd, make_float2(a2.y, a2.y));
      a[2 * k] = make_float2(ex2f(e0.x), ex2f(e1.x));
      a[2 * k + 1] = make_float2(ex2f(e0.y), ex2f(e1.y));
      const float4 v = kKeepB ? Bk[k] : bq[k * RL];
      bb[2 * k] = mul2(du2[2 * k], make_float2(v.x, v.y));
      bb[2 * k + 1] = mul2(du2[2 * k + 1], make_float2(v.z, v.w));
      const float4 cv = cq[k * RL];
      mu[2 * k] = mul2(yh2[2 * k], make_float2(cv.x, cv.y));
      mu[2 * k + 1] = mul2(yh2[2 * k + 1], make_float2(cv.z, cv.w));
    }
    const float2 ps = mul2(make_float2(dsum, dsum), a2);
    const float2 Pseg = make_float2(ex2f(ps.x), ex2f(ps.y));

    // The reverse fold needs only the decays and mu, not h: both folds and
    // both segment scans run interleaved (two independent chains).
    float2 S = bb[0], Lam = mu[KT - 1];
#pragma unroll
    for (int k = 0; k < KT - 1; ++k) {
      S = fma2(a[k + 1], S, bb[k + 1]);
      Lam = fma2(a[KT - 1 - k], Lam, mu[KT - 2 - k]);
    }
    float2 Qs = mul2(a[0], Lam);
    float2 Pf = Pseg, Pr = Pseg;
#pragma unroll
    for (int off = 1; off < RL; off <<= 1) {
      float2 Pp, Sp, Pn, Sn;
      Pp.x = __shfl_up_sync(0xffffffffu, Pf.x, 2 * off);
      Pp.y = __shfl_up_sync(0xffffffffu, Pf.y, 2 * off);
      Sp.x = __shfl_up_sync(0xffffffffu, S.x, 2 * off);
      Sp.y = __shfl_up_sync(0xffffffffu, S.y, 2 * off);
      Pn.x = __shfl_down_sync(0xffffffffu, Pr.x, 2 * off);
      Pn.y = __shfl_down_sync(0xffffffffu, Pr.y, 2 * off);
      Sn.x = __shfl_down_sync(0xffffffffu, Qs.x, 2 * off);
      Sn.y = __shfl_down_sync(0xffffffffu, Qs.y, 2 * off);
      if (j >= off) {
        S = fma2(Pf, Sp, S);
        Pf = mul2(Pf, Pp);
      }
      if (j + off < RL) {
        Qs = fma2(Pr, Sn, Qs);
        Pr = mul2(Pr, Pn);
      }
    }
    const float2 hout = fma2(Pf, hc, S);
    const float2 rout = fma2(Pr, rcar, Qs);
    float2 h, rin;
    h.x = __shfl_up_sync(0xffffffffu, hout.x, 2);
    h.y = __shfl_up_sync(0xffffffffu, hout.y, 2);
    rin.x = __shfl_down_sync(0xffffffffu, rout.x, 2);
    rin.y = __shfl_down_sync(0xffffffffu, rout.y, 2);
    if (j == 0) h = hc;
    if (j == RL - 1) rin = rcar;

    // forward replay: h_t, qq_t = a_t h_{t-1}, pre-gate output, dC terms
    float2 qq[KT];
#pragma unroll
    for (int k = 0; k < KT / 2; ++k) {
      const float4 cv = cq[k * RL];
      const float2 c0 = make_float2(cv.x, cv.y), c1 = make_float2(cv.z, cv.w);
      qq[2 * k] = mul2(a[2 * k], h);
      h = add2(qq[2 * k], bb[2 * k]);
      yacc2[2 * k] = fma2(c0, h, yacc2[2 * k]);
      bb[2 * k] = mul2(yh2[2 * k], h);  // dC term (bb is free now)
      qq[2 * k + 1] = mul2(a[2 * k + 1], h);
      h = add2(qq[2 * k + 1], bb[2 * k + 1]);
      yacc2[2 * k + 1] = fma2(c1, h, yacc2[2 * k + 1]);
      bb[2 * k + 1] = mul2(yh2[2 * k + 1], h);
    }
    // kSyncSlots (one slot buffer): the previous pair's cross-row sum must
    // have read the slots before they are written again; waiting only here
    // lets that sum overlap the folds, scans and forward replay above
    if (kSyncSlots) __syncthreads();
    store_steps<KT>(dC_lo, bb, slot_swizzle(j));

    // reverse replay: lam_t and the products
    float2 lam = add2(mu[KT - 1], rin);
    float2 dA2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = KT / 2 - 1; k >= 0; --k) {
      const float4 bv = kKeepB ? Bk[k] : bq[k * RL];
#pragma unroll
      for (int e = 1; e >= 0; --e) {
        const int i = 2 * k + e;
        if (i < KT - 1) lam = fma2(a[i + 1], lam, mu[i]);
        const float2 bp = e ? make_float2(bv.z, bv.w) : make_float2(bv.x, bv.y);
        bb[i] = mul2(du2[i], lam);  // dB term
        s12[i] = fma2(bp, lam, s12[i]);
        const float2 lq = mul2(lam, qq[i]);
        s22[i] = fma2(Ar, lq, s22[i]);
        dA2 = fma2(make_float2(dl[i], dl[i]), lq, dA2);
      }
    }
    store_steps<KT>(dB_lo, bb, slot_swizzle(j));
    dA_lo[0] = dA2.x;   // state 2q
  dA_lo[RL] = dA2.y;  // state 2q + 1

}

template <typename Io, bool kVec, int W, int kMinBlocks, int kSlotBufs, int NS, bool kKeepB>
__global__ void __launch_bounds__(W * 32, kMinBlocks)
    bwd_main_kernel(ScanArgs p, BwdOut o, int64_t nrb, const float* __restrict__ Hin,
                    const float* __restrict__ Rin, float* __restrict__ pBC,
                    float* __restrict__ pA, float* __restrict__ pD, float* __restrict__ pbias) {
  pdl_wait();
  using T = typename Io::T;
  using Sm = MainSmem<W, T, kSlotBufs, NS>;
  constexpr int KT = kKTb, RL = kRLb, CH = kBwdChunk, R = 2 * W, NT = W * 32;
  constexpr int RB = row_block<Io>();
  constexpr int kPasses = RB / R;
  constexpr int SR = (int)Sm::slot_row;
  extern __shared__ float4 smem4[];
  char* sm = reinterpret_cast<char*>(smem4);
  float4* pairs = reinterpret_cast<float4*>(sm);
  float* slots = reinterpret_cast<float*>(sm + Sm::pairs);
  float* acc = reinterpret_cast<float*>(sm + Sm::pairs + Sm::slots);
  float* dAs = reinterpret_cast<float*>(sm + Sm::pairs + Sm::slots + Sm::acc);
  float* A2s = reinterpret_cast<float*>(sm + Sm::pairs + Sm::slots + Sm::acc + Sm::dA);
  float* Ars = A2s + R * NS;
  float* Hs = Ars + R * NS;   // [row][n] state entering the chunk
  float* Rs = Hs + R * NS;    // [row][n] adjoint carry entering the chunk
  uint4* ins = reinterpret_cast<uint4*>(sm + Sm::pairs + Sm::slots + Sm::acc + Sm::dA + Sm::params);
  constexpr int kInsBuf = (int)(Sm::ins / 2 / sizeof(uint4));  // uint4 per buffer
  const float4* Bp = pairs;
  const float4* Cp = pairs + (NS / 2) * (KT / 2) * RL;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int j = lane >> 1, rs = lane & 1;
  const int r = 2 * warp + rs;
  const int64_t c = blockIdx.x / nrb;
  const int64_t g = blockIdx.x - c * nrb;
  const int64_t b = blockIdx.y;
  const int64_t L = p.L, t0 = c * CH;
  const int64_t nch = (L + CH - 1) / CH;
  const T* Bb = static_cast<const T*>(p.B) + b * NS * L;
  const T* Cb = static_cast<const T*>(p.C) + b * NS * L;

  if (kVec) {
    // one-shot copy of the chunk's B / C, staged raw in the accumulator area
    T* raw = reinterpret_cast<T*>(acc);
    static_assert(2 * NS * CH * sizeof(T) <= Sm::acc, "raw staging must fit");
    issue_raw_bc<Io, CH, NS>(Bb, Cb, L, t0, raw, tid, NT);
    cp_async_commit();
    {
      const int64_t d = g * RB + r;
      issue_row_inputs<Io, KT, NT>(p, o.dy, b * p.Dch + (d < p.Dch ? d : 0), d < p.Dch,
                                   t0 + KT * j, L, ins, tid);
    }
    cp_async_commit();
    cp_async_wait_one();  // B / C landed (the inputs may still be in flight)
    __syncthreads();
    raw_to_pairs<Io, CH, KT, RL, NS>(raw, pairs, tid, NT);
    __syncthreads();
  } else {
    load_pairs_scalar<Io, CH, KT, RL, NS>(Bb, Cb, L, t0, pairs, tid, NT);
  }
  for (int i = tid; i < 2 * NS * CH; i += NT) acc[i] = 0.f;

  const int64_t ts = t0 + KT * j;
  float* my_slot0 = slots + (size_t)r * SR + 2 * KT * j;  // + buffer * R * SR
  // cross-row sum assignment: thread -> four consecutive floats of [dB,dC][2][CH]
  const int sum_e = 4 * tid;                      // element of the row slot
  const int sum_wh = sum_e / (2 * CH);            // 0: dB, 1: dC
  const int sum_st = sum_e % (2 * CH);            // (step, state) within the tensor
  // where store_steps put that float4: segment js, rotated position
  const int sum_js = (sum_st / 4) / (KT / 2);
  const int sum_phys = sum_wh * 2 * CH +
                       4 * (sum_js * (KT / 2) + (((sum_st / 4) % (KT / 2) + slot_swizzle(sum_js)) & (KT / 2 - 1)));
  static_assert(KT == 8, "the slot swizzle assumes four float4 per lane segment");
  static_assert(4 * NT >= 2 * 2 * CH, "one float4 of the row slot per summing thread");

#pragma unroll 1
  for (int pass = 0; pass < kPasses; ++pass) {
    const int64_t d0 = g * RB + pass * R;
    if (d0 >= p.Dch) break;  // uniform over the CTA
    const int64_t d = d0 + r;
    const bool valid = d < p.Dch;
    const int64_t row = b * p.Dch + (valid ? d : 0);
    __syncthreads();  // previous pass done with the per-pass buffers
    for (int i = tid; i < R * NS; i += NT) {
      const int64_t dd = d0 + i / NS;
      const bool ok = dd < p.Dch;
      const float av = ok ? p.A[dd * NS + i % NS] : 0.f;
      A2s[i] = av * kLog2e;
      Ars[i] = av;
      const size_t rci = ((size_t)(b * p.Dch + (ok ? dd : 0)) * nch + c) * NS + i % NS;
      Hs[i] = ok ? Hin[rci] : 0.f;
      Rs[i] = ok ? Rin[rci] : 0.f;
    }
    __syncthreads();

    const float Dd = (valid && p.D) ? p.D[d] : 0.f;
    const float bias = (valid && p.delta_bias) ? p.delta_bias[d] : 0.f;
    const T* urow = static_cast<const T*>(p.u) + row * L;
    const T* drow = static_cast<const T*>(p.delta) + row * L;
    const T* zrow = p.z ? static_cast<const T*>(p.z) + row * L : nullptr;
    const T* grow = static_cast<const T*>(o.dy) + row * L;
    const size_t rc = (size_t)row * nch + c;
    const float* hin_row = Hs + r * NS;
    const float* rin_row = Rs + r * NS;

    const uint4* inb = ins + (pass & 1) * kInsBuf;  // this pass's inputs (16-byte rows)
    if (kVec) {
      // next pass's inputs go in flight now; this pass's have landed after the wait
      const int64_t dn = d + R;
      if (pass + 1 < kPasses && d0 + R < p.Dch)
        issue_row_inputs<Io, KT, NT>(p, o.dy, b * p.Dch + (dn < p.Dch ? dn : 0), dn < p.Dch, ts,
                                     L, ins + ((pass + 1) & 1) * kInsBuf, tid);
      cp_async_commit();
      cp_async_wait_one();
    }
    float dl[KT];
    float2 du2[KT], yh2[KT], yacc2[KT], s12[KT], s22[KT];
    float dD_acc = 0.f, dsum = 0.f;
    {
      float uu[KT], zz[KT], gg[KT];
      if (kVec) {
        read_row_input<Io, KT, NT>(inb, 0, tid, uu);
        read_row_input<Io, KT, NT>(inb, 1, tid, dl);
        read_row_input<Io, KT, NT>(inb, 2, tid, zz);
        read_row_input<Io, KT, NT>(inb, 3, tid, gg);
      } else {
        load_kt<Io, KT, kVec>(urow, ts, L, valid, uu);
        load_kt<Io, KT, kVec>(drow, ts, L, valid, dl);
        load_kt<Io, KT, kVec>(zrow, ts, L, valid && zrow != nullptr, zz);
        load_kt<Io, KT, kVec>(grow, ts, L, valid, gg);
      }
#pragma unroll
      for (int i = 0; i < KT; ++i) {
        const bool in = valid && ts + i < L;
        const float dt = in ? step_delta(dl[i], bias, p.softplus) : 0.f;
        const float yh = in ? (zrow ? gg[i] * zz[i] * sigmoid_f(zz[i]) : gg[i]) : 0.f;
        dl[i] = dt;
        du2[i] = make_float2(dt * uu[i], dt * uu[i]);
        yh2[i] = make_float2(yh, yh);
        yacc2[i] = make_float2(Dd * uu[i], 0.f);
        s12[i] = make_float2(0.f, 0.f);
        s22[i] = make_float2(0.f, 0.f);
        dD_acc = fmaf(yh, uu[i], dD_acc);
        dsum += dt;
      }
    }

#pragma unroll 1
    for (int q = 0; q < NS / 2; ++q) {
      const int sb = kSlotBufs == 2 ? (q & 1) : 0;
      float* slot = my_slot0 + (size_t)sb * R * SR;
      bwd_state_pair<KT, RL, CH, NS, kKeepB, kSlotBufs == 1>(q, j, r, valid, A2s, Ars, hin_row, rin_row, Bp, Cp, dl, du2,
                                     yh2, dsum, yacc2, s12, s22, slot, slot + 2 * CH,
                                     dAs + (r * NS + 2 * q) * RL + j);

      // dB / dC of this state pair: sum the rows' slots into the accumulator
      __syncthreads();
      if (tid < 2 * 2 * CH / 4) {
        const float* base = slots + (size_t)sb * R * SR + sum_phys;
        float4 v = *reinterpret_cast<const float4*>(base);
        float2 lo = make_float2(v.x, v.y), hi = make_float2(v.z, v.w);
#pragma unroll
        for (int rr = 1; rr < R; ++rr) {
          v = *reinterpret_cast<const float4*>(base + (size_t)rr * SR);
          lo = add2(lo, make_float2(v.x, v.y));
          hi = add2(hi, make_float2(v.z, v.w));
        }
        float4* ap = reinterpret_cast<float4*>(acc + ((size_t)sum_wh * (NS / 2) + q) * 2 * CH + sum_st);
        v = *ap;
        lo = add2(lo, make_float2(v.x, v.y));
        hi = add2(hi, make_float2(v.z, v.w));
        *ap = make_float4(lo.x, lo.y, hi.x, hi.y);
      }
    }

    // per-time-step outputs
    {
      float uu[KT], dr[KT], zz[KT], gg[KT], o1[KT], o2[KT], o3[KT];
      if (kVec) {
        read_row_input<Io, KT, NT>(inb, 0, tid, uu);
        read_row_input<Io, KT, NT>(inb, 1, tid, dr);
        read_row_input<Io, KT, NT>(inb, 2, tid, zz);
        read_row_input<Io, KT, NT>(inb, 3, tid, gg);
      } else {
        load_kt<Io, KT, kVec>(urow, ts, L, valid, uu);
        load_kt<Io, KT, kVec>(drow, ts, L, valid, dr);
        load_kt<Io, KT, kVec>(zrow, ts, L, valid && zrow != nullptr, zz);
        load_kt<Io, KT, kVec>(grow, ts, L, valid, gg);
      }
      float dbias_acc = 0.f;
#pragma unroll
      for (int i = 0; i < KT; ++i) {
        const float s1 = s12[i].x + s12[i].y;
        const float s2 = s22[i].x + s22[i].y;
        const float yacc = yacc2[i].x + yacc2[i].y;
        o1[i] = fmaf(yh2[i].x, Dd, dl[i] * s1);  // du
        const float ddt = fmaf(uu[i], s1, s2);
        const float ddr = p.softplus ? ddt * sigmoid_f(dr[i] + bias) : ddt;
        o2[i] = ddr;
        dbias_acc += (valid && ts + i < L) ? ddr : 0.f;
        if (zrow) {
          const float s = sigmoid_f(zz[i]);
          o3[i] = gg[i] * yacc * s * fmaf(zz[i], 1.f - s, 1.f);
        } else {
          o3[i] = 0.f;
        }
      }
      store_kt<Io, KT, kVec>(static_cast<T*>(o.du) + row * L, ts, L, valid, o1);
      store_kt<Io, KT, kVec>(static_cast<T*>(o.ddelta) + row * L, ts, L, valid, o2);
      if (o.dz) store_kt<Io, KT, kVec>(static_cast<T*>(o.dz) + row * L, ts, L, valid, o3);
#pragma unroll
      for (int off = 2; off < 32; off <<= 1) {  // the row's 16 lanes (same parity)
        dD_acc += __shfl_xor_sync(0xffffffffu, dD_acc, off);
        dbias_acc += __shfl_xor_sync(0xffffffffu, dbias_acc, off);
      }
      if (valid && j == 0) {
        pD[rc] = dD_acc;
        pbias[rc] = dbias_acc;
      }
    }
    // dA of the pass's rows: thread -> (row, state), sum over the 16 segments
    __syncthreads();
    for (int i = tid; i < R * NS; i += NT) {
      const int rr = i / NS, n = i % NS;
      const int64_t dd = d0 + rr;
      const float4* src = reinterpret_cast<const float4*>(dAs + (rr * NS + n) * RL);
      float sd = 0.f;
#pragma unroll
      for (int k4 = 0; k4 < RL / 4; ++k4) {
        const float4 v = src[k4];
        sd += (v.x + v.y) + (v.z + v.w);
      }
      if (dd < p.Dch) pA[((size_t)(b * p.Dch + dd) * nch + c) * NS + n] = sd;
    }
  }
  __syncthreads();
  pdl_trigger();  // the main work is done: the next kernel may be scheduled
  // this block's dB / dC partial for the chunk
  float* out = pBC + ((size_t)(b * nrb + g) * 2) * NS * L;
  for (int i = tid; i < 2 * NS * CH; i += NT) {
    const int whn = i / CH, tt = i % CH;  // (wh * NS + n, t)
    const int wh = whn / NS, n = whn % NS;
    if (t0 + tt < L) out[(size_t)whn * L + t0 + tt] = acc[((wh * (NS / 2) + n / 2) * CH + tt) * 2 + (n & 1)];
  }
}

// ---------------------------------------------------------------------------
// 2. fixed-order reduction of the partials
// ---------------------------------------------------------------------------
template <int NS>
__global__ void bwd_reduce_bc_kernel(const float* __restrict__ pBC, int64_t nrb, int64_t Bsz,
                                     int64_t L, float* __restrict__ dB, float* __restrict__ dC) {
  pdl_wait();
  const int64_t per = Bsz * NS * L;  // elements of dB (and of dC)
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= 2 * per) return;
  const int64_t wh = i / per, e = i % per;  // e = (b * NS + n) * L + t
  const int64_t b = e / (NS * L), nt = e % (NS * L);
  float acc = 0.f;
  for (int64_t g = 0; g < nrb; ++g) acc += pBC[((b * nrb + g) * 2 + wh) * NS * L + nt];
  (wh ? dC : dB)[e] = acc;
  pdl_trigger();  // the main work is done: the next kernel may be scheduled
}

// One CTA per channel d.  Thread (g, n), g = 0..7, sums the chunk partials of
// batches g, g + 8, g + 16, ... (batch, then chunk order); the eight group
// sums are then added in order of g.  Fixed order: bitwise reproducible.
constexpr int kParamGroups = 8;
template <int NS>
__global__ void __launch_bounds__(kParamGroups * NS)
    bwd_reduce_param_kernel(const float* __restrict__ pA, const float* __restrict__ pD,
                            const float* __restrict__ pbias, int64_t Bsz, int64_t Dch,
                            int64_t nch, float* __restrict__ dA, float* __restrict__ dD,
                            float* __restrict__ dbias) {
  pdl_wait();
  __shared__ float sA[kParamGroups * NS], sD[kParamGroups], sB[kParamGroups];
  const int64_t d = blockIdx.x;
  const int tid = threadIdx.x, n = tid % NS, gq = tid / NS;
  float acc = 0.f, a1 = 0.f, a2 = 0.f;
  for (int64_t b = gq; b < Bsz; b += kParamGroups) {
    const int64_t rc0 = (b * Dch + d) * nch;
    const float* src = pA + rc0 * NS + n;
#pragma unroll 8
    for (int64_t c = 0; c < nch; ++c) acc += src[c * NS];
    if (n == 0) {
#pragma unroll 8
      for (int64_t c = 0; c < nch; ++c) {
        a1 += pD[rc0 + c];
        a2 += pbias[rc0 + c];
      }
    }
  }
  sA[tid] = acc;
  if (n == 0) {
    sD[gq] = a1;
    sB[gq] = a2;
  }
  __syncthreads();
  if (tid < NS) {
    float t = 0.f;
#pragma unroll
    for (int g = 0; g < kParamGroups; ++g) t += sA[g * NS + tid];
    dA[d * NS + tid] = t;
  }
  if (tid == 0) {
    float t1 = 0.f, t2 = 0.f;
#pragma unroll
    for (int g = 0; g < kParamGroups; ++g) {
      t1 += sD[g];
      t2 += sB[g];
    }
    if (dD) dD[d] = t1;
    if (dbias) dbias[d] = t2;
  }
  pdl_trigger();  // the main work is done: the next kernel may be scheduled
}

template <typename Io, bool kVec, int W, int kMinBlocks, int kSlotBufs, int NS, bool kKeepB>
cudaError_t launch_main(const ScanArgs& a, const BwdOut& o, const WsLayout& w, float* sumS,
                        float* sumQ, float* pBC, float* pA, float* pD, float* pbias,
                        cudaStream_t s) {
  using Sm = MainSmem<W, typename Io::T, kSlotBufs, NS>;
  auto kern = bwd_main_kernel<Io, kVec, W, kMinBlocks, kSlotBufs, NS, kKeepB>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Sm::total);
  if (e != cudaSuccess) return e;
  const int64_t nrb = (a.Dch + row_block<Io>() - 1) / row_block<Io>();
  dim3 grid((unsigned)(nrb * w.nchunks), (unsigned)a.Bsz);
  return launch_pdl(kern, grid, dim3(W * 32), Sm::total, s, a, o, nrb, sumS, sumQ, pBC, pA, pD,
                    pbias);
}

template <typename Io, bool kVec, int NS>
cudaError_t launch_bwd_t(int phase, const ScanArgs& a, const BwdOut& o, void* ws, cudaStream_t s) {
  const WsLayout w = ws_layout(a.Bsz, a.Dch, a.L, NS);
  char* base = static_cast<char*>(ws);
  float* sumS = reinterpret_cast<float*>(base + w.sumS);
  float* sumQ = reinterpret_cast<float*>(base + w.sumQ);
  float* dsum = reinterpret_cast<float*>(base + w.dsum);
  float* pBC = reinterpret_cast<float*>(base + w.pbc);
  float* pA = reinterpret_cast<float*>(base + w.pa);
  float* pD = reinterpret_cast<float*>(base + w.pd);
  float* pbias = reinterpret_cast<float*>(base + w.pbias);
  cudaError_t e;
  if (phase == kBwdStates || phase == kBwdAdjointStates || phase == kBwdChunkStates) {
    constexpr int SG = NS < 16 ? NS : 16;  // states per summary thread
    const int64_t nrb = (a.Dch + kSumThreads - 1) / kSumThreads;
    dim3 grid((unsigned)(nrb * w.nchunks), (unsigned)a.Bsz, (unsigned)(NS / SG));
    // one B or C tile per summary the mode makes, plus the input ring
    auto smem_for = [&](int tiles) {
      return sizeof(float) * tiles * kBwdChunk * SG +
             (kVec ? sizeof(uint4) * kSumDepth * 4 * (8 / Io::kVec) * kSumThreads : 0);
    };
    const int64_t n = a.Bsz * a.Dch * NS;
    const dim3 cgrid((unsigned)((n + 255) / 256));
    auto run = [&](auto kern, auto carry, int tiles) -> cudaError_t {
      const size_t smem = smem_for(tiles);
      cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (r != cudaSuccess) return r;
      r = launch_pdl(kern, grid, dim3(kSumThreads), smem, s, a, o, nrb, sumS, sumQ, dsum);
      if (r != cudaSuccess) return r;
      return launch_pdl(carry, cgrid, dim3(256), 0, s, a.A, a.Bsz, a.Dch, w.nchunks, sumS, sumQ,
                        dsum);
    };
    if (phase == kBwdStates)
      return run(bwd_summary_kernel<Io, kVec, NS, kSumBoth>, bwd_carry_kernel<NS, kSumBoth>, 2);
    if (phase == kBwdAdjointStates)
      return run(bwd_summary_kernel<Io, kVec, NS, kSumQ>, bwd_carry_kernel<NS, kSumQ>, 1);
    return run(bwd_summary_kernel<Io, kVec, NS, kSumS>, bwd_carry_kernel<NS, kSumS>, 1);
  }
  if (phase == kBwdReverse) {
    // 16-bit I/O: 4 warps per CTA, registers capped for three CTAs per SM
    // (168 used), one dB/dC slot buffer so that three CTAs also fit in
    // shared memory with 16 states: 12 warps per SM (measured fastest of
    // 8/12 warps, 1/2 buffers).  fp32 I/O: two CTAs per SM with B kept in
    // registers and two slot buffers (one barrier fewer per state pair),
    // measured 6% faster there and 10% slower for bf16.  Larger state
    // sizes fit fewer CTAs per SM.
    if constexpr (std::is_same<Io, IoF32>::value && NS <= 32)  // 64 states: no room for two buffers
      return launch_main<Io, kVec, 4, 2, 2, NS, true>(a, o, w, sumS, sumQ, pBC, pA, pD, pbias, s);
    else
      return launch_main<Io, kVec, 4, 3, 1, NS, false>(a, o, w, sumS, sumQ, pBC, pA, pD, pbias, s);
  }
  const int64_t n = 2 * a.Bsz * NS * a.L;
  const int64_t nrb = (a.Dch + row_block<Io>() - 1) / row_block<Io>();
  e = launch_pdl(bwd_reduce_bc_kernel<NS>, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s,
                 (const float*)pBC, nrb, a.Bsz, a.L, o.dB, o.dC);
  if (e != cudaSuccess) return e;
  return launch_pdl(bwd_reduce_param_kernel<NS>, dim3((unsigned)a.Dch), dim3(kParamGroups * NS), 0,
                    s, (const float*)pA, (const float*)pD, (const float*)pbias, a.Bsz, a.Dch,
                    w.nchunks, o.dA, o.dD, o.ddelta_bias);
}

template <typename Io, int NS>
cudaError_t launch_bwd_ns(int phase, const ScanArgs& a, const BwdOut& o, void* ws,
                          cudaStream_t s) {
  return (a.L % Io::kVec) == 0 ? launch_bwd_t<Io, true, NS>(phase, a, o, ws, s)
                               : launch_bwd_t<Io, false, NS>(phase, a, o, ws, s);
}

template <typename Io>
cudaError_t launch_bwd_io(int phase, const ScanArgs& a, const BwdOut& o, void* ws,
                          cudaStream_t s) {
  switch (a.N) {
    case 8: return launch_bwd_ns<Io, 8>(phase, a, o, ws, s);
    case 16: return launch_bwd_ns<Io, 16>(phase, a, o, ws, s);
    case 32: return launch_bwd_ns<Io, 32>(phase, a, o, ws, s);
    case 64: return launch_bwd_ns<Io, 64>(phase, a, o, ws, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

size_t bwd_workspace_bytes(int64_t Bsz, int64_t Dch, int64_t L, int64_t N) {
  return ws_layout(Bsz, Dch, L, N).total;
}

size_t bwd_chunk_states_offset(int64_t Bsz, int64_t Dch, int64_t L, int64_t N) {
  return ws_layout(Bsz, Dch, L, N).sumS;  // after the carries: h entering each chunk
}

cudaError_t launch_scan_bwd(int phase, const ScanArgs& a, const BwdOut& o, void* ws,
                            cudaStream_t s) {
  if (a.dt == Dt::BF16) return launch_bwd_io<IoBf16>(phase, a, o, ws, s);
  if (a.dt == Dt::F16) return launch_bwd_io<IoF16>(phase, a, o, ws, s);
  return launch_bwd_io<IoF32>(phase, a, o, ws, s);
}

}  // namespace selscan

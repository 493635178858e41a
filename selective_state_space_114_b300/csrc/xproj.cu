// Input projection of the selective scan on the 5th-generation tensor cores:
//   xdbl[t][m]  = sum_k Wx[m][k] u[k][t]      (m < R + 2N; x_proj, no bias)
//   delta[d][t] = sum_r Wdt[d][r] xdbl[t][r]  (r < R;      dt_proj without its
//                                              bias, which the scan adds)
//   B[n][t] = xdbl[t][R + n],  C[n][t] = xdbl[t][R + N + n]
// per batch, u and delta [Dch][L], B and C [N][L] (time innermost).  The
// comment thread of "PyTorch 한 파일에서의 Mamba 구현" (news.hada.io, topic
// 12448) notes that x_proj has no bias, so the two projections compose into
// one; here they run back to back inside one kernel and xdbl never leaves the
// SM, so the kernel reads u once and writes delta, B, C once (HBM-bound)
// instead of multiplying by the merged Dch x Dch weight (12x the flops).
//
// One CTA (8 warps) per tile of 128 tokens of one batch; one elected thread
// issues tcgen05.mma (kind::f16, fp32 accumulators in tensor memory):
//   GEMM 1  M = 128 tokens, N = R + 2N (padded to 16), K = Dch in chunks of
//           128 channels.  A = u^T: the chunk [128 channels][128 tokens] is
//           copied by cp.async, then transposed into the K-major core-matrix
//           layout with ldmatrix.trans; B = Wx, K-major as stored.  A ring
//           of stages (two with dt_rank 48 and 16 states; one when the
//           weight tile is large) keeps the copy of the next chunk in
//           flight while the MMAs of the current one run.
//   epilogue 1  tcgen05.ld: B and C columns to global memory; the R dt
//           columns rounded to the I/O type into shared memory (GEMM 2's A).
//   GEMM 2  M = 128, N = 128 channels per step, K = R (padded to 16); B =
//           Wdt rows of the step, K-major as stored.  Two Wdt buffers and two
//           accumulators: the epilogue of step s-1 (delta stores) runs while
//           the MMAs of step s execute and the rows of step s+1 arrive.
// Operand tiles use the no-swizzle K-major canonical layout: core matrices of
// 8 rows x 16 bytes, [K group][row group] order (leading byte offset = the
// K-group stride, stride byte offset = 128 bytes).
// Every mbarrier wait is bounded: on timeout the kernel counts a failure,
// waits (bounded) for its own MMAs, frees its tensor memory and returns.
#include <type_traits>

#include "common.cuh"
#include "launch.h"

namespace selscan {

__device__ int g_xproj_wait_failures = 0;

namespace {

constexpr int kXpThreads = 256;  // 8 warps: two per tensor-memory lane quarter
constexpr int kTokTile = 128;          // tokens per CTA (MMA M)
constexpr int kKc = 128;               // channels per GEMM-1 chunk (64: 10% slower)
constexpr int kN2 = 128;               // delta channels per GEMM-2 step (MMA N)
constexpr int kStageRowB = 2 * kTokTile + 16;  // u staging row bytes (padded)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemCol2 = 256;    // GEMM-2 accumulator columns
constexpr uint32_t kWaitIters = 1u << 20;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Wait for the completion of the mbarrier phase with the given parity;
// false after `polls` polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          uint32_t polls = kWaitIters) {
  const uint32_t a = smem_u32(bar);
  for (uint32_t i = 0; i < polls; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(a), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  return false;
}

// Shared-memory matrix descriptor: no swizzle, K-major canonical layout.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version of the 5th-generation tensor cores
  return d;                // base offset 0, relative leading offset, no swizzle
}

// Instruction descriptor, kind::f16: fp32 accumulator, A and B both bf16 or
// both fp16, both K-major, shape M x N.
__host__ __device__ constexpr uint32_t instr_desc(int M, int N, bool bf16) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 16 consecutive fp32 accumulator columns of this thread's lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 64 consecutive fp32 accumulator columns of this thread's lane.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t saddr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(saddr));
}

// Byte offset of element (row, k) in a K-major core-matrix tile with `rows`
// rows (a multiple of 8): [k / 8][row / 8][row % 8][k % 8], 2-byte elements.
__device__ __forceinline__ uint32_t cm_off(int row, int k, int rows) {
  return (uint32_t)((((k >> 3) * (rows >> 3) + (row >> 3)) << 7) + ((row & 7) << 4) +
                    ((k & 7) << 1));
}

struct XpLayout {
  int M1p, Rp, S;  // padded GEMM-1 N, padded dt_rank, GEMM-1 pipeline stages
  size_t stage_bytes, a2, b2, total;
};

constexpr size_t kXpSmemBudget = 200 * 1024;

// GEMM-1 stage s: [u chunk, natural layout][A tile][Wx tile] at s * stage_bytes.
// GEMM 2 reuses the region: A2 at 0, two B2 buffers after it.
__host__ __device__ inline XpLayout xp_layout(int R, int N) {
  XpLayout s;
  s.M1p = ((R + 2 * N) + 15) / 16 * 16;
  s.Rp = (R + 15) / 16 * 16;
  s.stage_bytes = (size_t)kKc * kStageRowB + (size_t)kTokTile * kKc * 2 + (size_t)s.M1p * kKc * 2;
  s.S = (int)(kXpSmemBudget / s.stage_bytes);
  if (s.S > 4) s.S = 4;
  const size_t g1 = (size_t)s.S * s.stage_bytes;
  s.a2 = 0;
  s.b2 = (size_t)kTokTile * s.Rp * 2;
  const size_t g2 = s.b2 + 2 * (size_t)kN2 * s.Rp * 2;
  s.total = (g1 > g2 ? g1 : g2);
  return s;
}

template <typename Io>
__global__ void __launch_bounds__(kXpThreads, 1) xproj_kernel(XprojArgs p) {
  using T = typename Io::T;
  constexpr bool kBf16 = std::is_same<Io, IoBf16>::value;
  extern __shared__ __align__(1024) unsigned char xsm[];
  __shared__ uint64_t bar1, bar2[2], bar_never;
  __shared__ uint32_t tmem_slot;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int R = (int)p.R, Nn = (int)p.N, M1 = R + 2 * Nn;
  const int64_t Dch = p.Dch, L = p.L;
  const XpLayout lay = xp_layout(R, Nn);
  const int M1p = lay.M1p, Rp = lay.Rp, S = lay.S;
  const int64_t tiles_per_b = (L + kTokTile - 1) / kTokTile;
  const int64_t b = blockIdx.x / tiles_per_b;
  const int64_t t0 = (blockIdx.x - b * tiles_per_b) * kTokTile;
  const T* ub = static_cast<const T*>(p.u) + b * Dch * L;
  const T* Wx = static_cast<const T*>(p.Wx);
  const T* Wdt = static_cast<const T*>(p.Wdt);

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    mbar_init(&bar1, 1);
    mbar_init(&bar2[0], 1);
    mbar_init(&bar2[1], 1);
    mbar_init(&bar_never, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  uint32_t ph1 = 0, ph2[2] = {0, 0};  // completed waits per barrier
  uint32_t c1 = 0, c2[2] = {0, 0};    // commits issued per barrier (thread 0)
  bool failed = false;

  auto stage_of = [&](int st) { return xsm + (size_t)st * lay.stage_bytes; };
  auto aop_of = [&](int st) { return stage_of(st) + (size_t)kKc * kStageRowB; };
  auto bop_of = [&](int st) { return aop_of(st) + (size_t)kTokTile * kKc * 2; };

  // cp.async of GEMM-1 chunk kc (channels kc * kKc ..) into stage st
  auto issue_chunk = [&](int kc, int st) {
    const int64_t k0 = (int64_t)kc * kKc;
    unsigned char* sg = stage_of(st);
    for (int i = tid; i < kKc * (kTokTile / 8); i += kXpThreads) {
      const int c = i / (kTokTile / 8), v = i % (kTokTile / 8);
      const int64_t k = k0 + c, t = t0 + 8 * v;
      const bool in = k < Dch && t < L;
      cp_async16(sg + c * kStageRowB + v * 16, in ? (const void*)(ub + k * L + t) : (const void*)ub,
                 in ? 16 : 0);
    }
    unsigned char* bo = bop_of(st);
    for (int i = tid; i < M1p * (kKc / 8); i += kXpThreads) {
      const int m = i / (kKc / 8), kg = i % (kKc / 8);
      const int64_t k = k0 + 8 * kg;
      const bool in = m < M1 && k < Dch;
      cp_async16(bo + cm_off(m, 8 * kg, M1p), in ? (const void*)(Wx + (int64_t)m * Dch + k)
                                                  : (const void*)Wx,
                 in ? 16 : 0);
    }
  };

  // ---------------- GEMM 1: S-stage cp.async ring ----------------
  const int nK = (int)((Dch + kKc - 1) / kKc);
  const uint32_t id1 = instr_desc(kTokTile, M1p, kBf16);
  for (int k = 0; k < S - 1; ++k) {  // one commit group per chunk (empty past the end)
    if (k < nK) issue_chunk(k, k);
    cp_async_commit();
  }
  for (int kc = 0; kc < nK; ++kc) {
    const int st = kc % S;
    if (kc >= 1) {  // the MMAs of chunk kc-1 are done: stage (kc-1) % S is free
      if (!failed && !mbar_wait(&bar1, ph1 & 1)) failed = true;
      ++ph1;
    }
    if (kc + S - 1 < nK) issue_chunk(kc + S - 1, (kc + S - 1) % S);
    cp_async_commit();
    // at most S-1 groups newer than chunk kc's may stay in flight
    if (S == 4)
      cp_async_wait_depth<3>();
    else if (S == 3)
      cp_async_wait_depth<2>();
    else if (S == 2)
      cp_async_wait_depth<1>();
    else
      cp_async_wait_all();
    failed = __syncthreads_or(failed);  // chunk kc staged by every thread
    // transpose u [kKc channels][128 tokens] into A core matrices (row = token)
    {
      const uint32_t sg = smem_u32(stage_of(st));
      unsigned char* ao = aop_of(st);
      // 16 token groups x kKc / 8 channel groups of core matrices, four per
      // ldmatrix (matrix m of the instruction = token group rg0 + m)
#pragma unroll
      for (int q = 0; q < kKc / 16; ++q) {
        const int idx = warp * (kKc / 16) + q;  // (kg, rg0 / 4)
        const int kg = idx >> 2, rg0 = (idx & 3) * 4;
        const int m = lane >> 3, i = lane & 7;
        uint32_t r[4];
        ldsm_x4_trans(sg + (uint32_t)((8 * kg + i) * kStageRowB + (rg0 + m) * 16), r);
#pragma unroll
        for (int mm = 0; mm < 4; ++mm) {
          const uint32_t off = (uint32_t)(((kg * (kTokTile / 8) + rg0 + mm) << 7) +
                                          ((lane >> 2) << 4) + ((lane & 3) << 2));
          *reinterpret_cast<uint32_t*>(ao + off) = r[mm];
        }
      }
    }
    fence_async_smem();
    __syncthreads();  // A and B tiles of chunk kc visible to the tensor core
    if (tid == 0 && !failed) {
      tc_fence_after();
      const uint32_t a0 = smem_u32(aop_of(st)), b0 = smem_u32(bop_of(st));
#pragma unroll
      for (int j = 0; j < kKc / 16; ++j) {
        const uint64_t ad = smem_desc(a0 + j * 2 * (kTokTile / 8) * 128, (kTokTile / 8) * 128, 128);
        const uint64_t bd = smem_desc(b0 + j * 2 * (M1p / 8) * 128, (M1p / 8) * 128, 128);
        mma_f16(tmem, ad, bd, id1, (kc > 0 || j > 0) ? 1u : 0u);
      }
      mma_commit(&bar1);
      ++c1;
    }
  }
  if (!failed && !mbar_wait(&bar1, ph1 & 1)) failed = true;
  ++ph1;
  // test hook: a wait on a barrier nothing arrives at, which must give up
  // (the MMAs issued so far complete normally; the drain below waits for them)
  if (p.test_stuck_wait && !failed && !mbar_wait(&bar_never, 0, 64)) failed = true;
  cp_async_wait_all();  // the trailing empty groups
  failed = __syncthreads_or(failed);
  tc_fence_after();

  // ---------------- epilogue 1 ----------------
  // warp w reads tensor-memory lanes 32 (w % 4) .. (its quarter) and the
  // column half w / 4 of every 32 columns
  const int quarter = warp & 3, half = warp >> 2;
  const int row = quarter * 32 + lane;  // token of this thread's accumulator lane
  const uint32_t tlane = (uint32_t)(quarter * 32) << 16;
  const int64_t t = t0 + row;
  const bool tok_in = t < L;
  unsigned char* a2 = xsm + lay.a2;
  if (!failed) {
    T* Bo = static_cast<T*>(p.B) + b * Nn * L;
    T* Co = static_cast<T*>(p.C) + b * Nn * L;
    for (int c0 = 16 * half; c0 < M1p; c0 += 32) {
      float v[16];
      tmem_ld16(tmem + tlane + (uint32_t)c0, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int m = c0 + i;
        if (m < R) {
          *reinterpret_cast<T*>(a2 + cm_off(row, m, kTokTile)) = Io::from_f(v[i]);
        } else if (m < R + Nn) {
          if (tok_in) Bo[(int64_t)(m - R) * L + t] = Io::from_f(v[i]);
        } else if (m < M1) {
          if (tok_in) Co[(int64_t)(m - R - Nn) * L + t] = Io::from_f(v[i]);
        }
      }
    }
    if (half == 0)
      for (int m = R; m < Rp; ++m)  // zero K padding of GEMM 2's A
        *reinterpret_cast<T*>(a2 + cm_off(row, m, kTokTile)) = Io::from_f(0.f);
  }

  // ---------------- GEMM 2: double-buffered Wdt steps and accumulators ----------------
  // Step s: Wdt rows d0 = 128 s .. into B2[s % 2], MMA into tensor-memory
  // columns kTmemCol2 + 128 (s % 2), committed to bar2[s % 2]; the epilogue
  // of step s-1 runs while the MMA of step s executes.
  const uint32_t id2 = instr_desc(kTokTile, kN2, kBf16);
  T* dout = static_cast<T*>(p.delta) + b * Dch * L;
  const int nS = (int)((Dch + kN2 - 1) / kN2);
  auto b2_of = [&](int buf) { return xsm + lay.b2 + (size_t)buf * kN2 * Rp * 2; };
  auto issue_wdt = [&](int s2) {
    unsigned char* dst = b2_of(s2 & 1);
    const int64_t d0 = (int64_t)s2 * kN2;
    for (int i = tid; i < kN2 * (Rp / 8); i += kXpThreads) {
      const int dd = i / (Rp / 8), kg = i % (Rp / 8);
      const int64_t d = d0 + dd;
      const bool in = d < Dch && 8 * kg < R;
      cp_async16(dst + cm_off(dd, 8 * kg, kN2), in ? (const void*)(Wdt + d * R + 8 * kg)
                                                    : (const void*)Wdt,
                 in ? 16 : 0);
    }
  };
  auto epilogue2 = [&](int s2) {  // this warp's 64 of the step's 128 channels
    const int64_t dbeg = (int64_t)s2 * kN2 + (kN2 / 2) * half;
    const uint32_t col = kTmemCol2 + (uint32_t)((s2 & 1) * kN2 + (kN2 / 2) * half);
    const bool full = dbeg + kN2 / 2 <= Dch;
    T* dp = dout + dbeg * L + t;
    float v[kN2 / 2];
    tmem_ld64(tmem + tlane + col, v);  // one load, one wait for the warp's 64 columns
    if (tok_in) {
      if (full) {
#pragma unroll
        for (int i = 0; i < kN2 / 2; ++i) dp[(int64_t)i * L] = Io::from_f(v[i]);
      } else {
#pragma unroll
        for (int i = 0; i < kN2 / 2; ++i)
          if (dbeg + i < Dch) dp[(int64_t)i * L] = Io::from_f(v[i]);
      }
    }
  };
  if (!failed) {
    issue_wdt(0);
    cp_async_commit();
  }
  for (int s2 = 0; s2 < nS && !failed; ++s2) {
    if (s2 >= 1) {  // the MMAs of step s2-1 are done: B2[(s2+1) % 2] is free
      const int pb = (s2 - 1) & 1;
      if (!mbar_wait(&bar2[pb], ph2[pb] & 1)) failed = true;
      ++ph2[pb];
    }
    if (s2 + 1 < nS) issue_wdt(s2 + 1);
    cp_async_commit();
    cp_async_wait_one();  // step s2's Wdt rows landed
    fence_async_smem();
    tc_fence_before();
    failed = __syncthreads_or(failed);  // B2[s2 % 2] and A2 visible; epilogue of step s2-2 done
    if (failed) break;
    tc_fence_after();
    if (tid == 0) {
      const uint32_t a0 = smem_u32(a2), b0 = smem_u32(b2_of(s2 & 1));
      const uint32_t dcol = tmem + kTmemCol2 + (uint32_t)((s2 & 1) * kN2);
      for (int j = 0; j < Rp / 16; ++j) {
        const uint64_t ad = smem_desc(a0 + j * 2 * (kTokTile / 8) * 128, (kTokTile / 8) * 128, 128);
        const uint64_t bd = smem_desc(b0 + j * 2 * (kN2 / 8) * 128, (kN2 / 8) * 128, 128);
        mma_f16(dcol, ad, bd, id2, j > 0 ? 1u : 0u);
      }
      mma_commit(&bar2[s2 & 1]);
      ++c2[s2 & 1];
    }
    if (s2 >= 1) epilogue2(s2 - 1);  // overlaps the MMAs of step s2
  }
  if (!failed && nS >= 1) {
    const int pb = (nS - 1) & 1;
    if (!mbar_wait(&bar2[pb], ph2[pb] & 1)) failed = true;
    ++ph2[pb];
    failed = __syncthreads_or(failed);
    tc_fence_after();
    if (!failed) epilogue2(nS - 1);
  }
  cp_async_wait_all();

  if (failed) {
    if (tid == 0) {
      atomicAdd(&g_xproj_wait_failures, 1);
      if (p.err) atomicOr(p.err, kErrXprojTimeout);
      // the CTA's MMAs may still be in flight: wait (bounded) for the last
      // commit on each barrier
      if (c1) mbar_wait(&bar1, (c1 - 1) & 1);
      if (c2[0]) mbar_wait(&bar2[0], (c2[0] - 1) & 1);
      if (c2[1]) mbar_wait(&bar2[1], (c2[1] - 1) & 1);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

}  // namespace

size_t xproj_smem_bytes(int64_t R, int64_t N) { return xp_layout((int)R, (int)N).total; }

cudaError_t launch_xproj(const XprojArgs& a, cudaStream_t s) {
  const size_t smem = xp_layout((int)a.R, (int)a.N).total;
  const int64_t tiles = a.Bsz * ((a.L + kTokTile - 1) / kTokTile);
  cudaError_t e;
  if (a.dt == Dt::BF16) {
    e = cudaFuncSetAttribute(xproj_kernel<IoBf16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    xproj_kernel<IoBf16><<<(unsigned)tiles, kXpThreads, smem, s>>>(a);
  } else {
    e = cudaFuncSetAttribute(xproj_kernel<IoF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    xproj_kernel<IoF16><<<(unsigned)tiles, kXpThreads, smem, s>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t xproj_wait_failures(int* out) {
  return cudaMemcpyFromSymbol(out, g_xproj_wait_failures, sizeof(int));
}

}  // namespace selscan

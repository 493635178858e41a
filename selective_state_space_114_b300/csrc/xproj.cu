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
// One CTA (8 warps) per tile of 128 tokens of one batch and part of the
// delta channels (with few tiles, each tile's channels are split over two or
// more CTAs, which repeat GEMM 1: its u reads are then served by L2).  The
// CTA allocates 256 tensor-memory columns, so two CTAs share an SM.  One
// elected thread issues tcgen05.mma (kind::f16, fp32 accumulators in tensor
// memory):
//   GEMM 1  M = 128 tokens, N = R + 2N (padded to 16), K = Dch in chunks of
//           64 channels, accumulated in columns 0 ...  Both operands arrive
//           by TMA in 128-byte rows with the 128-byte swizzle, which the
//           tensor core reads as is: A = u^T as two boxes of 64 tokens x 64
//           channels (MN-major: token-contiguous rows, one per channel),
//           B = Wx as one box of 64 channels x R + 2N rows (K-major).  A ring
//           of stages with full / empty mbarriers: warp 0 issues the loads,
//           warp 1 the MMAs, each MMA batch committing its stage's empty
//           barrier.
//   epilogue 1  tcgen05.ld: B and C columns to global memory (by the first
//           CTA of the tile); the R dt columns rounded to the I/O type into
//           shared memory (GEMM 2's B).
//   GEMM 2  delta^T: M = 128 channels per step, N = 128 tokens, K = R (padded
//           to 16); A = Wdt rows of the step, K-major as stored; B = the dt
//           columns of xdbl.  A tensor-memory lane is then a channel and its
//           columns consecutive tokens: each warp writes its 32 channels x 64
//           tokens as 128-byte rows (128-byte swizzle) into shared memory,
//           and one lane stores the box by TMA.  A ring of two to four Wdt
//           buffers (rows of up to three later steps in flight; as many as
//           keep two CTAs per SM) and two accumulators
//           (columns 0 .. 255, free once epilogue 1 has read GEMM 1's): the
//           epilogue of step s-1 (delta stores) runs while the MMAs of step s
//           execute.
// GEMM 2's operands (Wdt rows, and the dt columns written by epilogue 1) use the
// no-swizzle K-major canonical layout: core matrices of 8 rows x 16 bytes,
// [K group][row group] order (leading byte offset = the K-group stride,
// stride byte offset = 128 bytes).  GEMM 1's operands use the 128-byte
// swizzle: 8-row atoms of 1024 bytes, the 16-byte chunks of row r stored at
// chunk position c ^ (r % 8) (as the TMA writes them).
// Every mbarrier wait is bounded: on timeout the kernel counts a failure,
// waits (bounded) for its own TMA loads and MMAs, frees its tensor memory and
// returns.
#include <cuda.h>

#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "launch.h"

namespace selscan {

__device__ int g_xproj_wait_failures = 0;

namespace {

constexpr int kXpThreads = 256;  // 8 warps: two per tensor-memory lane quarter
constexpr int kTokTile = 128;          // tokens per CTA (MMA M)
constexpr int kKc = 64;                // channels per GEMM-1 chunk
constexpr int kN2 = 128;               // delta channels per GEMM-2 step (MMA N)
constexpr uint32_t kTmemCols = 256;    // GEMM 1 (R + 2N <= 256), then GEMM 2 (2 x 128)
constexpr uint32_t kTmemCol2 = 0;      // GEMM-2 accumulator columns
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

// Shared-memory matrix descriptor: start address, leading and stride byte
// offsets, layout type (0: no swizzle, 2: 128-byte swizzle; swizzled tiles
// start on 1024-byte boundaries, so the base offset is 0).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t layout = 0) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version of the 5th-generation tensor cores
  d |= (uint64_t)(layout & 7u) << 61;
  return d;
}
constexpr uint32_t kSw128 = 2;

// Instruction descriptor, kind::f16: fp32 accumulator, A and B both bf16 or
// both fp16, B K-major, A K-major or (a_mn) MN-major, shape M x N.
__host__ __device__ constexpr uint32_t instr_desc(int M, int N, bool bf16, bool a_mn = false) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((a_mn ? 1u : 0u) << 15) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// TMA tile store from shared memory (bulk group of the issuing thread);
// parts of the box outside the tensor are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y,
                                             int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(map),
      "r"(x), "r"(y), "r"(z), "r"(smem_u32(src))
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// none of this thread's store groups still reading shared memory
__device__ __forceinline__ void bulk_wait_read_0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// TMA tile loads (box at element coordinates, x innermost; x a multiple of
// 64 here) that complete the transaction count of `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
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

// Byte offset of element (row, k) in a K-major core-matrix tile with `rows`
// rows (a multiple of 8): [k / 8][row / 8][row % 8][k % 8], 2-byte elements.
__device__ __forceinline__ uint32_t cm_off(int row, int k, int rows) {
  return (uint32_t)((((k >> 3) * (rows >> 3) + (row >> 3)) << 7) + ((row & 7) << 4) +
                    ((k & 7) << 1));
}

struct XpLayout {
  int M1p, Rp, S;  // padded GEMM-1 N, padded dt_rank, GEMM-1 pipeline stages
  int W;           // GEMM-2 weight buffers
  size_t stage_bytes, a2, b2, ostage, total;
};
constexpr size_t kOutBox = 32 * 128;  // one warp's delta box: 32 channels x 64 tokens
constexpr int kWdtBufsMax = 4;        // GEMM-2 weight ring

constexpr size_t kXpSmemBudget = 110 * 1024;  // two CTAs per SM
constexpr size_t kXpSmemFloor = 80 * 1024;    // three CTAs (240 KB) never fit

constexpr int kXpMaxStages = 4;

// GEMM-1 stage s: [A tile: two 64-token halves][Wx tile] at s * stage_bytes
// (every part a multiple of 1024 bytes).
// GEMM 2 reuses the region: the tile's dt columns (a2) at 0, the Wdt ring
// (b2) after it, then the warps' delta boxes (ostage).
__host__ __device__ inline XpLayout xp_layout(int R, int N) {
  XpLayout s;
  s.M1p = ((R + 2 * N) + 15) / 16 * 16;
  s.Rp = (R + 15) / 16 * 16;
  s.stage_bytes = (size_t)kTokTile * kKc * 2 + (size_t)s.M1p * kKc * 2;
  s.S = (int)(kXpSmemBudget / s.stage_bytes);
  if (s.S > kXpMaxStages) s.S = kXpMaxStages;
  const size_t g1 = (size_t)s.S * s.stage_bytes;
  s.a2 = 0;
  s.b2 = (size_t)kTokTile * s.Rp * 2;
  // the weight ring: up to four buffers while two CTAs still fit per SM
  // (large dt_rank: two), then one delta box per warp (1024-byte aligned)
  const size_t wdt = (size_t)kN2 * s.Rp * 2;
  const size_t fixed = s.b2 + 1024 + (kXpThreads / 32) * kOutBox;
  s.W = fixed + 2 * wdt <= kXpSmemBudget ? (int)((kXpSmemBudget - fixed) / wdt) : 2;
  if (s.W > kWdtBufsMax) s.W = kWdtBufsMax;
  s.ostage = (s.b2 + (size_t)s.W * wdt + 1023) & ~(size_t)1023;
  const size_t g2 = s.ostage + (kXpThreads / 32) * kOutBox;
  s.total = (g1 > g2 ? g1 : g2);
  // at most two CTAs per SM: two 256-column tensor-memory allocations fill
  // the SM's 512 columns, so a third CTA must not fit by shared memory
  if (s.total < kXpSmemFloor) s.total = kXpSmemFloor;
  return s;
}

template <typename Io>
__global__ void __launch_bounds__(kXpThreads, 2)
    xproj_kernel(XprojArgs p, int split, const __grid_constant__ CUtensorMap map_u,
                 const __grid_constant__ CUtensorMap map_wx,
                 const __grid_constant__ CUtensorMap map_d) {
  pdl_wait();
  using T = typename Io::T;
  constexpr bool kBf16 = std::is_same<Io, IoBf16>::value;
  extern __shared__ __align__(1024) unsigned char xsm[];
  __shared__ uint64_t bar1, bar2[2], bar_never, full[kXpMaxStages], empty[kXpMaxStages];
  __shared__ uint32_t tmem_slot;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int R = (int)p.R, Nn = (int)p.N, M1 = R + 2 * Nn;
  const int64_t Dch = p.Dch, L = p.L;
  const XpLayout lay = xp_layout(R, Nn);
  const int M1p = lay.M1p, Rp = lay.Rp, S = lay.S, W = lay.W;
  const int64_t tiles_per_b = (L + kTokTile - 1) / kTokTile;
  const int64_t tile = blockIdx.x / split;
  const int part = (int)(blockIdx.x - tile * split);  // which share of the delta channels
  const int64_t b = tile / tiles_per_b;
  const int64_t t0 = (tile - b * tiles_per_b) * kTokTile;
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
    for (int i = 0; i < kXpMaxStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
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
  // the swizzled tiles need 1024-byte alignment: refuse (as a failure) otherwise
  bool failed = (smem_u32(xsm) & 1023u) != 0;

  auto aop_of = [&](int st) { return xsm + (size_t)st * lay.stage_bytes; };
  auto bop_of = [&](int st) { return aop_of(st) + (size_t)kTokTile * kKc * 2; };

  // ---------------- GEMM 1: TMA ring, warp 0 loads, warp 1 issues ----------------
  const int nK = (int)((Dch + kKc - 1) / kKc);
  const uint32_t id1 = instr_desc(kTokTile, M1p, kBf16, true);
  const uint32_t tx_bytes = (uint32_t)lay.stage_bytes;
  uint32_t loads[kXpMaxStages] = {0, 0, 0, 0};   // TMA loads issued per stage (warp 0)
  uint32_t frees[kXpMaxStages] = {0, 0, 0, 0};   // empty-barrier commits per stage (warp 1)
  if (warp == 0) {
    for (int kc = 0; kc < nK && !failed; ++kc) {
      const int st = kc % S;
      if (kc >= S) {  // the MMAs that read this stage's previous chunk are done
        const bool ok = mbar_wait(&empty[st], (uint32_t)((kc / S) - 1) & 1u);
        if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&full[st], tx_bytes);
        tma_load_3d(aop_of(st), &map_u, (int)t0, kc * kKc, (int)b, &full[st]);
        tma_load_3d(aop_of(st) + 64 * kKc * 2, &map_u, (int)t0 + 64, kc * kKc, (int)b, &full[st]);
        tma_load_2d(bop_of(st), &map_wx, kc * kKc, 0, &full[st]);
      }
      ++loads[st];
      __syncwarp();
    }
  } else if (warp == 1) {
    for (int kc = 0; kc < nK && !failed; ++kc) {
      const int st = kc % S;
      const bool ok = mbar_wait(&full[st], (uint32_t)(kc / S) & 1u);
      if (!__all_sync(0xffffffffu, ok)) { failed = true; break; }
      tc_fence_after();
      if (lane == 0) {
        const uint32_t a0 = smem_u32(aop_of(st)), b0 = smem_u32(bop_of(st));
#pragma unroll
        for (int j = 0; j < kKc / 16; ++j) {
          // A (MN-major): 16 channels = two 8-row atoms (2048 bytes) per MMA;
          // the two 64-token halves kKc * 128 bytes apart.  B (K-major): 16
          // channels = 32 bytes into each 128-byte row; 8-row groups 1024
          // bytes apart.
          const uint64_t ad = smem_desc(a0 + j * 2048, kKc * 128, 1024, kSw128);
          const uint64_t bd = smem_desc(b0 + j * 32, 16, 1024, kSw128);
          mma_f16(tmem, ad, bd, id1, (kc > 0 || j > 0) ? 1u : 0u);
        }
        mma_commit(&empty[st]);  // frees the stage once these MMAs complete
      }
      ++frees[st];
      __syncwarp();
    }
    if (!failed) {
      if (lane == 0) mma_commit(&bar1);  // all of GEMM 1 complete
      c1 = 1;
    }
  }
  failed = __syncthreads_or(failed);
  if (!failed && !mbar_wait(&bar1, 0)) failed = true;
  ++ph1;
  // test hook: a wait on a barrier nothing arrives at, which must give up
  // (the MMAs issued so far complete normally; the drain below waits for them)
  if (p.test_stuck_wait && !failed && !mbar_wait(&bar_never, 0, 64)) failed = true;
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
          if (tok_in && part == 0) Bo[(int64_t)(m - R) * L + t] = Io::from_f(v[i]);
        } else if (m < M1) {
          if (tok_in && part == 0) Co[(int64_t)(m - R - Nn) * L + t] = Io::from_f(v[i]);
        }
      }
    }
    if (half == 0)
      for (int m = R; m < Rp; ++m)  // zero K padding of GEMM 2's B
        *reinterpret_cast<T*>(a2 + cm_off(row, m, kTokTile)) = Io::from_f(0.f);
  }

  // ---------------- GEMM 2: double-buffered Wdt steps and accumulators ----------------
  // Step s: Wdt rows d0 = 128 s .. into B2[s % 2], MMA into tensor-memory
  // columns kTmemCol2 + 128 (s % 2), committed to bar2[s % 2]; the epilogue
  // of step s-1 runs while the MMA of step s executes.
  const uint32_t id2 = instr_desc(kN2, kTokTile, kBf16);
  const int nS_all = (int)((Dch + kN2 - 1) / kN2);
  const int sb = (int)((int64_t)part * nS_all / split);
  const int nS = (int)((int64_t)(part + 1) * nS_all / split) - sb;  // this CTA's steps
  auto b2_of = [&](int buf) { return xsm + lay.b2 + (size_t)buf * kN2 * Rp * 2; };
  auto issue_wdt = [&](int s2) {  // local step s2 (global sb + s2)
    unsigned char* dst = b2_of(s2 % W);
    const int64_t d0 = (int64_t)(sb + s2) * kN2;
    for (int i = tid; i < kN2 * (Rp / 8); i += kXpThreads) {
      const int dd = i / (Rp / 8), kg = i % (Rp / 8);
      const int64_t d = d0 + dd;
      const bool in = d < Dch && 8 * kg < R;
      cp_async16(dst + cm_off(dd, 8 * kg, kN2), in ? (const void*)(Wdt + d * R + 8 * kg)
                                                    : (const void*)Wdt,
                 in ? 16 : 0);
    }
  };
  auto epilogue2 = [&](int s2) {  // channels 32 quarter .., tokens 64 half ..
    const uint32_t col = kTmemCol2 + (uint32_t)((s2 & 1) * kN2 + 64 * half);
    float v[64];
    tmem_ld64(tmem + tlane + col, v);  // one load, one wait for the warp's 64 columns
    unsigned char* ob = xsm + lay.ostage + (size_t)warp * kOutBox;
    if (lane == 0) bulk_wait_read_0();  // the box's previous store has read it
    __syncwarp();
    // row = this lane's channel; its 16-byte chunk i at position i ^ (row % 8)
#pragma unroll
    for (int i = 0; i < 8; ++i)
      *reinterpret_cast<uint4*>(ob + lane * 128 + ((i ^ (lane & 7)) << 4)) = Io::pack(v + 8 * i);
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(&map_d, ob, (int)(t0 + 64 * half), (sb + s2) * kN2 + quarter * 32, (int)b);
      bulk_commit();
    }
  };
  if (!failed && nS >= 1) {
    for (int k = 0; k < W - 1; ++k) {  // one commit group per step (empty past the end)
      if (k < nS) issue_wdt(k);
      cp_async_commit();
    }
  }
  for (int s2 = 0; s2 < nS && !failed; ++s2) {
    if (s2 >= 1) {  // the MMAs of step s2-1 are done: its Wdt buffer is free
      const int pb = (s2 - 1) & 1;
      if (!mbar_wait(&bar2[pb], ph2[pb] & 1)) failed = true;
      ++ph2[pb];
    }
    if (s2 + W - 1 < nS) issue_wdt(s2 + W - 1);
    cp_async_commit();
    // step s2's Wdt rows landed (at most W - 1 later groups in flight)
    if (W == 4)
      cp_async_wait_depth<3>();
    else if (W == 3)
      cp_async_wait_depth<2>();
    else
      cp_async_wait_depth<1>();
    fence_async_smem();
    tc_fence_before();
    failed = __syncthreads_or(failed);  // its buffer and a2 visible; epilogue of step s2-2 done
    if (failed) break;
    tc_fence_after();
    if (tid == 0) {
      const uint32_t a0 = smem_u32(a2), b0 = smem_u32(b2_of(s2 % W));
      const uint32_t dcol = tmem + kTmemCol2 + (uint32_t)((s2 & 1) * kN2);
      for (int j = 0; j < Rp / 16; ++j) {
        // A = the step's Wdt rows (channels), B = the tile's dt columns (tokens)
        const uint64_t ad = smem_desc(b0 + j * 2 * (kN2 / 8) * 128, (kN2 / 8) * 128, 128);
        const uint64_t bd = smem_desc(a0 + j * 2 * (kTokTile / 8) * 128, (kTokTile / 8) * 128, 128);
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
  if (lane == 0) bulk_wait_all();  // the warp's delta stores are complete
  pdl_trigger();  // the main work is done: the next kernel may be scheduled

  if (failed) {
    // wait (bounded) for everything this CTA issued, so that no copy writes
    // and no MMA reads its memory after it
    if (tid == 0) {  // TMA loads and GEMM-2 commits
      atomicAdd(&g_xproj_wait_failures, 1);
      if (p.err) atomicOr(p.err, kErrXprojTimeout);
      for (int st = 0; st < S; ++st)
        if (loads[st]) mbar_wait(&full[st], (loads[st] - 1) & 1);
      if (c2[0]) mbar_wait(&bar2[0], (c2[0] - 1) & 1);
      if (c2[1]) mbar_wait(&bar2[1], (c2[1] - 1) & 1);
    }
    if (tid == 32) {  // GEMM-1 commits
      for (int st = 0; st < S; ++st)
        if (frees[st]) mbar_wait(&empty[st], (frees[st] - 1) & 1);
      if (c1) mbar_wait(&bar1, 0);
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

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point (the
// library links the runtime only).
cudaError_t encode_tiled(CUtensorMap* map, CUtensorMapDataType type, int rank, const void* base,
                         const cuuint64_t* dims, const cuuint64_t* strides_bytes,
                         const cuuint32_t* box) {
  static std::mutex mu;
  static EncodeTiledFn fn = nullptr;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!fn) {
      void* f = nullptr;
      cudaDriverEntryPointQueryResult q;
      const cudaError_t e =
          cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess) return e;
      if (q != cudaDriverEntryPointSuccess || !f) return cudaErrorNotSupported;
      fn = reinterpret_cast<EncodeTiledFn>(f);
    }
  }
  cuuint32_t elem_strides[5] = {1, 1, 1, 1, 1};
  const CUresult r = fn(map, type, (cuuint32_t)rank, const_cast<void*>(base), dims, strides_bytes,
                        box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_xproj(const XprojArgs& a, cudaStream_t s) {
  const XpLayout lay = xp_layout((int)a.R, (int)a.N);
  const size_t smem = lay.total;
  const int64_t tiles = a.Bsz * ((a.L + kTokTile - 1) / kTokTile);
  // split the delta channels of each tile over up to 2 x SMs / tiles CTAs
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 148;
  const int64_t steps = (a.Dch + kN2 - 1) / kN2;
  int64_t split = (2 * (int64_t)sms) / (tiles > 0 ? tiles : 1);
  split = split < 1 ? 1 : (split > steps ? steps : split);
  const unsigned grid = (unsigned)(tiles * split);
  // u as (token, channel, batch), boxes of 64 tokens x kKc channels; Wx as
  // (channel, row), boxes of kKc channels x M1p rows; both 128-byte rows
  // with the 128-byte swizzle.  Out-of-range elements read as 0.
  const CUtensorMapDataType ty =
      a.dt == Dt::BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap mu_, mwx;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)a.L, (cuuint64_t)a.Dch, (cuuint64_t)a.Bsz};
    const cuuint64_t strides[2] = {(cuuint64_t)a.L * 2, (cuuint64_t)(a.Dch * a.L * 2)};
    const cuuint32_t box[3] = {64, (cuuint32_t)kKc, 1};
    const cudaError_t e = encode_tiled(&mu_, ty, 3, a.u, dims, strides, box);
    if (e != cudaSuccess) return e;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)a.Dch, (cuuint64_t)(a.R + 2 * a.N)};
    const cuuint64_t strides[1] = {(cuuint64_t)a.Dch * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kKc, (cuuint32_t)lay.M1p};
    const cudaError_t e = encode_tiled(&mwx, ty, 2, a.Wx, dims, strides, box);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap md;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)a.L, (cuuint64_t)a.Dch, (cuuint64_t)a.Bsz};
    const cuuint64_t strides[2] = {(cuuint64_t)a.L * 2, (cuuint64_t)(a.Dch * a.L * 2)};
    const cuuint32_t box[3] = {64, 32, 1};
    const cudaError_t e = encode_tiled(&md, ty, 3, a.delta, dims, strides, box);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e;
  if (a.dt == Dt::BF16) {
    e = cudaFuncSetAttribute(xproj_kernel<IoBf16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(xproj_kernel<IoBf16>, dim3(grid), dim3(kXpThreads), smem, s, a, (int)split,
                      mu_, mwx, md);
  } else {
    e = cudaFuncSetAttribute(xproj_kernel<IoF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(xproj_kernel<IoF16>, dim3(grid), dim3(kXpThreads), smem, s, a, (int)split,
                      mu_, mwx, md);
  }
}

cudaError_t xproj_wait_failures(int* out) {
  return cudaMemcpyFromSymbol(out, g_xproj_wait_failures, sizeof(int));
}

}  // namespace selscan

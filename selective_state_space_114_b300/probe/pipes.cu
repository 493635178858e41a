// Pipe-rate microbenchmark for the roofline denominators of the scan kernels.
//
// Each test runs one CTA per SM (the dynamic shared-memory request keeps a
// second one off the SM) of W warps; every thread issues a fixed number of
// independent operations of one kind, unrolled, and the CTA reads the SM
// cycle counter around the loop.  The rate reported is operations (lane
// results) per SM clock, or for the shared-memory tests the SM clocks one
// warp-wide access takes when accesses of that pattern are issued back to
// back (the shared-memory pipe delivers one 128-byte wavefront per clock, so
// this is the wavefront count of the pattern).  Every loop has a fixed trip
// count: nothing waits on anything but the CTA's own barriers.
//
// C ABI:
//   int ssp_run(int test, int warps, int iters, double* clocks_per_cta, double* rate)
// returns 0 on success, a CUDA error code otherwise.  rate = lane results per
// SM clock (tests 0..5) or SM clocks per warp-wide access (tests 16..).
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr int kChains = 8;   // independent dependency chains per thread (ALU tests)
constexpr int kUnroll = 16;  // accesses per loop trip (shared-memory tests)
constexpr int kSmemBytes = 160 * 1024;

enum Test {
  T_EX2 = 0, T_LG2 = 1, T_RCP = 2, T_FFMA = 3, T_FFMA2 = 4, T_SHFL = 5,
  // 2 FFMA2 + 1 SHFL + 1 EX2 per chain step: 4 instructions of three pipes
  T_MIX = 6,
  // shared-memory access patterns (float4 index per lane within a 512-byte window)
  L128_UNIFORM = 16,   // all lanes one address
  L128_QUAD = 17,      // lane & 3: four addresses, lanes congruent mod 4 share
  L128_MOD8 = 18,      // lane & 7: eight addresses, lanes congruent mod 8 share
  L128_PAIR = 19,      // lane >> 1: sixteen addresses, adjacent pairs share
  L128_DIV4 = 20,      // lane >> 2: eight addresses, adjacent quads share
  L128_DIV8 = 21,      // lane >> 3: four addresses, adjacent octets share
  L128_DISTINCT = 22,  // lane: 32 addresses (512 contiguous bytes)
  L64_UNIFORM = 23,    // 8-byte load, all lanes one address
  L64_DISTINCT = 24,   // 8-byte load, 32 contiguous addresses
  L32_UNIFORM = 25,    // 4-byte load, all lanes one address
  L32_DISTINCT = 26,   // 4-byte load, 32 contiguous addresses
  S128_DISTINCT = 27,  // 16-byte store, 32 contiguous addresses
  L128_HALFU = 28,     // lane >> 4: two addresses (one per half-warp)
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm volatile("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp(float x) {
  float y;
  asm volatile("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float ffma(float a, float b, float c) {
  float d;
  asm volatile("fma.rn.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm volatile("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ float shfl(float x, int m) {
  float y;
  asm volatile("shfl.sync.bfly.b32 %0, %1, %2, 0x1f, 0xffffffff;" : "=f"(y) : "f"(x), "r"(m));
  return y;
}

template <int T>
__global__ void __launch_bounds__(1024) alu_kernel(int iters, long long* cyc, float* sink) {
  const int tid = threadIdx.x;
  float x[kChains];
  uint64_t x2[kChains];
#pragma unroll
  for (int k = 0; k < kChains; ++k) {
    x[k] = 0.25f + 1e-3f * (tid + k);
    x2[k] = ((uint64_t)__float_as_uint(x[k]) << 32) | __float_as_uint(x[k] + 0.5f);
  }
  const uint64_t m2 = ((uint64_t)__float_as_uint(0.999f) << 32) | __float_as_uint(0.998f);
  const uint64_t c2 = ((uint64_t)__float_as_uint(1e-3f) << 32) | __float_as_uint(2e-3f);
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int k = 0; k < kChains; ++k) {
      if (T == T_EX2) x[k] = ex2(x[k]);
      if (T == T_LG2) x[k] = lg2(x[k]);
      if (T == T_RCP) x[k] = rcp(x[k] + 1.f);
      if (T == T_FFMA) x[k] = ffma(x[k], 0.999f, 1e-3f);
      if (T == T_FFMA2) x2[k] = ffma2(x2[k], m2, c2);
      if (T == T_SHFL) x[k] = shfl(x[k], 1 + (k & 15));
      if (T == T_MIX) {
        x2[k] = ffma2(ffma2(x2[k], m2, c2), m2, c2);
        x[k] = ex2(shfl(x[k], 1 + (k & 15)));
      }
    }
  }
  __syncthreads();
  const long long t1 = clock64();
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < kChains; ++k) s += x[k] + __uint_as_float((uint32_t)x2[k]);
  if (s == 12345.f) sink[tid] = s;  // keeps the chains live
  if (tid == 0) cyc[blockIdx.x] = t1 - t0;
}

template <int T>
__device__ __forceinline__ int lane_slot(int lane) {
  switch (T) {
    case L128_UNIFORM: case L64_UNIFORM: case L32_UNIFORM: return 0;
    case L128_QUAD: return lane & 3;
    case L128_MOD8: return lane & 7;
    case L128_PAIR: return lane >> 1;
    case L128_DIV4: return lane >> 2;
    case L128_DIV8: return lane >> 3;
    case L128_HALFU: return lane >> 4;
    default: return lane;
  }
}

template <int T>
__global__ void __launch_bounds__(1024) smem_kernel(int iters, long long* cyc, unsigned* sink) {
  extern __shared__ uint4 sm[];
  const int tid = threadIdx.x, lane = tid & 31;
  for (int i = tid; i < kSmemBytes / 16; i += blockDim.x) sm[i] = make_uint4(i, 2 * i, 3 * i, 4 * i);
  __syncthreads();
  constexpr int bytes = (T == L64_UNIFORM || T == L64_DISTINCT) ? 8
                        : (T == L32_UNIFORM || T == L32_DISTINCT) ? 4 : 16;
  // each access of a trip reads a different 1 KiB block; trips rotate over 4
  // groups of 16 blocks (64 KiB in all, inside the 160 KiB allocation)
  const unsigned base = (unsigned)__cvta_generic_to_shared(sm) + lane_slot<T>(lane) * bytes;
  unsigned acc = 0;
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
    const unsigned b = base + (it & 3) * (kUnroll * 1024);
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      if (bytes == 16) {
        if (T == S128_DISTINCT) {
          asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(b + k * 1024), "r"(acc + k) : "memory");
        } else {
          unsigned v0, v1, v2, v3;
          asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3)
                       : "r"(b + k * 1024));
          acc += (v0 ^ v1) + (v2 ^ v3);  // every word live: the load stays 128-bit
        }
      } else if (bytes == 8) {
        unsigned v0, v1;
        asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v0), "=r"(v1) : "r"(b + k * 1024));
        acc += v0 ^ v1;
      } else {
        unsigned v0;
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v0) : "r"(b + k * 1024));
        acc += v0;
      }
    }
  }
  __syncthreads();
  const long long t1 = clock64();
  if (acc == 0xdeadbeefu) sink[tid] = acc;
  if (tid == 0) cyc[blockIdx.x] = t1 - t0;
}

template <typename S>
cudaError_t launch(void (*kern)(int, long long*, S*), int ctas, int warps, int iters,
                   long long* cyc, S* sink) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<ctas, warps * 32, kSmemBytes>>>(iters, cyc, sink);
  return cudaGetLastError();
}

}  // namespace

extern "C" int ssp_run(int test, int warps, int iters, double* clocks_per_cta, double* rate) {
  if (warps < 1 || warps > 32 || iters < 1 || iters > (1 << 20)) return (int)cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return (int)e;
  long long* cyc = nullptr;
  void* sink = nullptr;
  if ((e = cudaMalloc(&cyc, sizeof(long long) * sms)) != cudaSuccess) return (int)e;
  if ((e = cudaMalloc(&sink, 4 * 32 * warps)) != cudaSuccess) {
    cudaFree(cyc);
    return (int)e;
  }
  switch (test) {
#define ALU(t) case t: e = launch(alu_kernel<t>, sms, warps, iters, cyc, (float*)sink); break;
    ALU(T_EX2) ALU(T_LG2) ALU(T_RCP) ALU(T_FFMA) ALU(T_FFMA2) ALU(T_SHFL) ALU(T_MIX)
#undef ALU
#define SM(t) case t: e = launch(smem_kernel<t>, sms, warps, iters, cyc, (unsigned*)sink); break;
    SM(L128_UNIFORM) SM(L128_QUAD) SM(L128_MOD8) SM(L128_PAIR) SM(L128_DIV4) SM(L128_DIV8)
    SM(L128_DISTINCT) SM(L64_UNIFORM) SM(L64_DISTINCT) SM(L32_UNIFORM) SM(L32_DISTINCT)
    SM(S128_DISTINCT) SM(L128_HALFU)
#undef SM
    default: e = cudaErrorInvalidValue;
  }
  long long host[1024];
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e == cudaSuccess && sms <= 1024)
    e = cudaMemcpy(host, cyc, sizeof(long long) * sms, cudaMemcpyDeviceToHost);
  cudaFree(cyc);
  cudaFree(sink);
  if (e != cudaSuccess) return (int)e;
  // median over the CTAs (one per SM)
  for (int i = 1; i < sms; ++i)
    for (int k = i; k > 0 && host[k] < host[k - 1]; --k) {
      const long long t = host[k];
      host[k] = host[k - 1];
      host[k - 1] = t;
    }
  const double c = (double)host[sms / 2];
  *clocks_per_cta = c;
  const double ops = (double)warps * iters * (test < 16 ? 32.0 * kChains * (test == T_FFMA2 ? 2 : 1)
                                                        : (double)kUnroll);
  *rate = test < 16 ? ops / c : c / ops;
  return 0;
}

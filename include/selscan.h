/*
 * selscan.h -- C ABI of libselscan, the selective scan of the Mamba
 * selective state-space layer on NVIDIA B300 (sm_103a).
 *
 * The operation (per batch b, channel d, state n; time t = 0 .. L-1):
 *
 *   delta_t  = softplus(delta_raw_t + delta_bias_d)   (raw sum if softplus == 0)
 *   h_t[n]   = exp(delta_t * A_d[n]) * h_{t-1}[n] + delta_t * B_t[n] * u_t,  h_{-1} = 0
 *   y_t      = (sum_n C_t[n] * h_t[n] + D_d * u_t) * silu(z_t)
 *
 * Where it comes from: the selective SSM layer of Mamba ("Mamba SSM 架构",
 * toolpotion.ai: the layer of section 3 / algorithm 2 of the Mamba paper;
 * "Mamba 7.9.1", lpnh.cn, section 2.2: the SSM parameters become functions
 * of the input), evaluated as the sequential recurrence quoted in the
 * "PyTorch 한 파일에서의 Mamba 구현" thread (news.hada.io, topic 12448: the
 * state update with deltaA and deltaB_u, then the contraction with C over
 * the state dimension).  The pages name deltaA and deltaB_u but do not print
 * them; this library reads them as exp(delta*A) and delta*B*u.  The fused,
 * "hardware-aware" evaluation (state kept on chip, backward by recomputation)
 * is described on the "mamba.py" page (gittoolsai.com), performance section.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The
 *     library allocates no memory.  The only state it keeps between calls
 *     is the static scratch of ss_scan_bwd_noalloc and the failure counter
 *     of ss_xproj_wait_failures.
 *   - Layouts are row-major with time innermost (no strides):
 *       u, delta, z, y, du, ddelta, dz, dy : [Bsz][Dch][L]   (I/O dtype)
 *       B, C                               : [Bsz][N][L]     (I/O dtype)
 *       dB, dC                             : [Bsz][N][L]     float32
 *       A, dA                              : [Dch][N]        float32
 *       D, delta_bias, dD, ddelta_bias     : [Dch]           float32
 *       h, h_last                          : [Bsz][Dch][N]   float32
 *     The I/O dtype (ss_dtype) is float32, bf16 or fp16 (16-bit patterns);
 *     arithmetic is float32 throughout, the state h is always float32.
 *   - Every pointer must be 16-byte aligned (SS_ERR_ALIGN otherwise).  The
 *     scan, step and conv1d entry points accept any L >= 0: rows whose byte
 *     length is a multiple of 16 take the vectorised path, other L a slower
 *     element-wise path.  ss_xproj has its own shape rules (see its entry).
 *   - Optional inputs: D == NULL means D = 0, z == NULL means no gate,
 *     delta_bias == NULL means a zero bias.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  Arguments are checked before anything is launched; a
 *     rejected call launches nothing and writes nothing.  SS_ERR_CUDA reports
 *     a launch error (cudaGetLastError after the launch); faults during
 *     execution surface at the caller's next synchronisation.
 *   - Outputs are overwritten, never accumulated into.
 *   - N (the state size, d_state) is 8, 16, 32 or 64 for the scan and step
 *     entry points (SS_ERR_N_UNSUPPORTED otherwise).  N = 16 is the tuned
 *     configuration.
 *   - Bsz is at most 65535 for the scan and step entry points (SS_ERR_SHAPE
 *     otherwise): the batch index is a grid dimension.
 */
#ifndef SELSCAN_H_
#define SELSCAN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* ss_stream_t;

/* I/O element type.  SS_BF16 and SS_F16 arrays hold the 16-bit patterns
 * (bfloat16 / IEEE binary16); outputs in them are rounded to nearest even. */
typedef enum { SS_F32 = 0, SS_BF16 = 1, SS_F16 = 2 } ss_dtype;

typedef enum {
    SS_OK = 0,
    SS_ERR_NULL = 1,           /* a required pointer is NULL                      */
    SS_ERR_SHAPE = 2,          /* negative or too-large size                      */
    SS_ERR_DTYPE = 3,          /* unknown ss_dtype                                */
    SS_ERR_N_UNSUPPORTED = 4,  /* N not supported by the entry point (see above)  */
    SS_ERR_ALIGN = 5,          /* a pointer is not 16-byte aligned                */
    SS_ERR_WORKSPACE = 6,      /* workspace NULL/misaligned or smaller than needed */
    SS_ERR_CUDA = 7,           /* the CUDA runtime reported a launch error        */
    SS_ERR_SCRATCH_LIMIT = 8,  /* ss_scan_bwd_noalloc: problem needs more scratch
                                  than the library's static buffer holds          */
    SS_ERR_TIMEOUT = 9         /* a kernel's bounded wait on the hardware gave up
                                  (reported by ss_check_device_errors)            */
} ss_status;

/* Human-readable name of a status code (static string, never NULL). */
const char* ss_status_str(ss_status s);

/*
 * Device-side failures since the last check.  Kernels that wait on hardware
 * (ss_xproj waits on tensor-core completion barriers) bound every wait; a
 * wait that gives up sets a bit in a device error word, skips the rest of
 * its work (the outputs of that call are incomplete) and lets the kernel
 * finish.  This call synchronises stream, reads the word of the current
 * device, clears it and returns SS_ERR_TIMEOUT if any bit was set, SS_OK if
 * none, SS_ERR_CUDA if the copy itself failed.  The word is per device and
 * shared by all streams.
 */
ss_status ss_check_device_errors(ss_stream_t stream);

/* Library ABI version: major * 10000 + minor * 100 + patch. */
int ss_version(void);

/*
 * Forward selective scan.
 *   in : u, delta (delta_raw), z [Bsz][Dch][L]; B, C [Bsz][N][L]; A [Dch][N];
 *        D, delta_bias [Dch] (nullable, as are z); softplus: 0 or 1.
 *   out: y [Bsz][Dch][L] (I/O dtype);
 *        h_last [Bsz][Dch][N] float32 (nullable): the state after the last
 *        step (zeros when L == 0), to hand a sequence over to ss_step.
 * Zero-sized Bsz, Dch or L are valid (nothing but h_last is written).
 */
ss_status ss_scan_fwd(const void* u, const void* delta, const float* A, const void* B,
                      const void* C, const float* D, const void* z, const float* delta_bias,
                      int softplus, int64_t Bsz, int64_t Dch, int64_t L, int64_t N,
                      ss_dtype dtype, void* y, float* h_last, ss_stream_t stream);

/*
 * Forward selective scan continuing from a given state (chunked prefill, or a
 * sequence resumed after a previous scan or after decode steps): the scan of
 * ss_scan_fwd with h_{-1} = h0 instead of 0 ("mamba.py" page, step function of
 * the 2024-01-17 update and "Mamba 7.9.1", section 6.2: the recurrent form
 * carries the state from one token or segment to the next).
 *   h0 [Bsz][Dch][N] float32, nullable (NULL = zero state, i.e. ss_scan_fwd).
 *   h_last may be the same buffer as h0 (in-place update of a carried state);
 *   no other overlap between inputs and outputs is allowed.
 *   L == 0: h_last receives h0 (or zeros).
 * Everything else (arguments, layouts, checks, status) as ss_scan_fwd.
 * ss_scan_bwd is the backward of ss_scan_fwd, i.e. of a scan from h_{-1} = 0.
 */
ss_status ss_scan_fwd_from_state(const void* u, const void* delta, const float* A,
                                 const void* B, const void* C, const float* D, const void* z,
                                 const float* delta_bias, int softplus, const float* h0,
                                 int64_t Bsz, int64_t Dch, int64_t L, int64_t N, ss_dtype dtype,
                                 void* y, float* h_last, ss_stream_t stream);

/*
 * Bytes of device workspace ss_scan_bwd needs for these sizes (written to
 * *bytes; 0 is possible).  Pure host computation, no CUDA call.
 */
ss_status ss_scan_bwd_workspace_size(int64_t Bsz, int64_t Dch, int64_t L, int64_t N,
                                     ss_dtype dtype, size_t* bytes);

/*
 * Backward of ss_scan_fwd (zero initial state) for an upstream gradient dy
 * of y.  As the "mamba.py" page (gittoolsai.com, section 性能, performance)
 * describes for the hardware-aware scan, the backward recomputes the forward's
 * intermediate states instead of storing them; the adjoint recurrence runs in
 * reverse time (the same page's TODO list: the scan on time-flipped arrays).
 * The sequence is cut into 128-step chunks: the workspace holds, per (row,
 * chunk), the state entering the chunk and the adjoint carry entering it
 * from the later chunk (from a summary pass over every chunk), plus
 * per-block partial sums of dA, dB, dC, dD and ddelta_bias, reduced in a
 * fixed order, so reruns are bitwise identical.
 *   in : the forward's inputs, dy [Bsz][Dch][L] (I/O dtype),
 *        workspace (device, 16-byte aligned, >= ss_scan_bwd_workspace_size).
 *   out: du, ddelta (gradient of delta_raw), dz [Bsz][Dch][L] in the I/O
 *        dtype; dA [Dch][N], dB and dC [Bsz][N][L], dD and ddelta_bias
 *        [Dch] in float32.  dD / dz / ddelta_bias must be non-NULL exactly
 *        when D / z / delta_bias are.
 * The workspace contents on return are unspecified.
 */
ss_status ss_scan_bwd(const void* u, const void* delta, const float* A, const void* B,
                      const void* C, const float* D, const void* z, const float* delta_bias,
                      int softplus, const void* dy, int64_t Bsz, int64_t Dch, int64_t L,
                      int64_t N, ss_dtype dtype, void* du, void* ddelta, float* dA, float* dB,
                      float* dC, float* dD, void* dz, float* ddelta_bias, void* workspace,
                      size_t workspace_bytes, ss_stream_t stream);

/*
 * The three stages ss_scan_bwd runs, in this order, exposed for callers that
 * time them separately or interleave other work between them.  Each takes
 * exactly ss_scan_bwd's arguments and performs the same checks; calling the
 * three in order on one stream (same arguments, same workspace) is
 * ss_scan_bwd.
 *   ss_scan_bwd_states : the chunk summaries and carries: the state and the
 *                        adjoint carry entering every 128-step chunk, into
 *                        the workspace.
 *   ss_scan_bwd_reverse: the reverse-time pass; writes du, ddelta, dz and
 *                        the per-block partial sums of dA, dB, dC, dD,
 *                        ddelta_bias into the workspace.
 *   ss_scan_bwd_reduce : sums the partials in a fixed order into dA, dB,
 *                        dC, dD, ddelta_bias.
 */
ss_status ss_scan_bwd_states(const void* u, const void* delta, const float* A, const void* B,
                             const void* C, const float* D, const void* z,
                             const float* delta_bias, int softplus, const void* dy, int64_t Bsz,
                             int64_t Dch, int64_t L, int64_t N, ss_dtype dtype, void* du,
                             void* ddelta, float* dA, float* dB, float* dC, float* dD, void* dz,
                             float* ddelta_bias, void* workspace, size_t workspace_bytes,
                             ss_stream_t stream);
ss_status ss_scan_bwd_reverse(const void* u, const void* delta, const float* A, const void* B,
                              const void* C, const float* D, const void* z,
                              const float* delta_bias, int softplus, const void* dy,
                              int64_t Bsz, int64_t Dch, int64_t L, int64_t N, ss_dtype dtype,
                              void* du, void* ddelta, float* dA, float* dB, float* dC,
                              float* dD, void* dz, float* ddelta_bias, void* workspace,
                              size_t workspace_bytes, ss_stream_t stream);
ss_status ss_scan_bwd_reduce(const void* u, const void* delta, const float* A, const void* B,
                             const void* C, const float* D, const void* z,
                             const float* delta_bias, int softplus, const void* dy, int64_t Bsz,
                             int64_t Dch, int64_t L, int64_t N, ss_dtype dtype, void* du,
                             void* ddelta, float* dA, float* dB, float* dC, float* dD, void* dz,
                             float* ddelta_bias, void* workspace, size_t workspace_bytes,
                             ss_stream_t stream);

/*
 * Forward and backward with the chunk states kept in between (a training
 * step's forward followed by its backward on the same inputs).  The
 * backward above recomputes, in its first stage, the state entering each
 * 128-step chunk; the row-sequential forward kernel passes through those
 * states anyway.  ss_scan_fwd_save is ss_scan_fwd that also writes them into
 * a backward workspace (0.5 bytes of state per scanned element at N = 16:
 * the states at chunk boundaries, not the per-step states, which the
 * backward still recomputes).  ss_scan_bwd_saved is ss_scan_bwd for a
 * workspace so prepared: its first stage computes only the adjoint carries.
 *   ss_scan_fwd_save : ss_scan_fwd's arguments plus workspace and
 *                      workspace_bytes (device, 16-byte aligned, at least
 *                      ss_scan_bwd_workspace_size for the same sizes;
 *                      SS_ERR_WORKSPACE otherwise).  Shapes whose forward
 *                      runs the chunked kernels (few rows) get the chunk
 *                      states from the backward's state summaries, run
 *                      after the forward on the same stream.
 *   ss_scan_bwd_saved : ss_scan_bwd's arguments; the workspace must hold the
 *                      chunk states ss_scan_fwd_save wrote for the same u,
 *                      delta, A, B, delta_bias, softplus and sizes, with no
 *                      other use of that workspace in between (otherwise
 *                      the gradients are wrong; nothing detects it).
 *   ss_scan_bwd_states_saved : ss_scan_bwd_saved's first stage (then
 *                      ss_scan_bwd_reverse and ss_scan_bwd_reduce, as for
 *                      ss_scan_bwd_states).
 * Results equal ss_scan_fwd / ss_scan_bwd up to rounding: the chunk states
 * come from the forward's recurrence instead of the backward's summaries.
 */
ss_status ss_scan_fwd_save(const void* u, const void* delta, const float* A, const void* B,
                           const void* C, const float* D, const void* z,
                           const float* delta_bias, int softplus, int64_t Bsz, int64_t Dch,
                           int64_t L, int64_t N, ss_dtype dtype, void* y, float* h_last,
                           void* workspace, size_t workspace_bytes, ss_stream_t stream);
ss_status ss_scan_bwd_saved(const void* u, const void* delta, const float* A, const void* B,
                            const void* C, const float* D, const void* z,
                            const float* delta_bias, int softplus, const void* dy, int64_t Bsz,
                            int64_t Dch, int64_t L, int64_t N, ss_dtype dtype, void* du,
                            void* ddelta, float* dA, float* dB, float* dC, float* dD, void* dz,
                            float* ddelta_bias, void* workspace, size_t workspace_bytes,
                            ss_stream_t stream);
ss_status ss_scan_bwd_states_saved(const void* u, const void* delta, const float* A,
                                   const void* B, const void* C, const float* D, const void* z,
                                   const float* delta_bias, int softplus, const void* dy,
                                   int64_t Bsz, int64_t Dch, int64_t L, int64_t N,
                                   ss_dtype dtype, void* du, void* ddelta, float* dA, float* dB,
                                   float* dC, float* dD, void* dz, float* ddelta_bias,
                                   void* workspace, size_t workspace_bytes, ss_stream_t stream);

/*
 * One recurrent step (the "RNN form" used for token-by-token decoding;
 * "mamba.py" page, step function; "Mamba 7.9.1", section 6.2):
 *   in/out: h [Bsz][Dch][N] float32, updated in place;
 *   in : u_t, delta_t, z_t [Bsz][Dch]; B_t, C_t [Bsz][N] (I/O dtype);
 *        A [Dch][N]; D, delta_bias [Dch] (nullable, as is z_t).
 *   out: y_t [Bsz][Dch] (I/O dtype).
 * h must not alias any other argument.
 */
ss_status ss_step(float* h, const void* u_t, const void* delta_t, const float* A,
                  const void* B_t, const void* C_t, const float* D, const void* z_t,
                  const float* delta_bias, int softplus, int64_t Bsz, int64_t Dch, int64_t N,
                  ss_dtype dtype, void* y_t, ss_stream_t stream);

/*
 * Causal depthwise conv1d + silu, the step of the Mamba block that produces
 * the scan input u from the in-projection output x ("Mamba 7.9.1", section
 * 4.1: d_conv = 4; "mamba.py" page, resources: a plain Conv1d in the minimal
 * implementation):
 *   c_t = bias_d + sum_{k<K} w[d][k] x_{t-(K-1)+k}   (x_s = 0 for s < 0)
 *   u_t = c_t * sigmoid(c_t)                          (c_t when silu == 0)
 *   in : x [Bsz][Dch][L] (I/O dtype); w [Dch][K] float32; bias [Dch] float32
 *        (nullable = 0); K = kernel width, 1 .. 4 (SS_ERR_SHAPE otherwise).
 *   out: u [Bsz][Dch][L] (I/O dtype); must not overlap x.
 * Conventions as for the scan (device pointers, 16-byte alignment, async on
 * stream, checks before launch).
 */
ss_status ss_conv1d_silu_fwd(const void* x, const float* w, const float* bias, int silu,
                             int64_t Bsz, int64_t Dch, int64_t L, int64_t K, ss_dtype dtype,
                             void* u, ss_stream_t stream);

/*
 * Backward of ss_conv1d_silu_fwd for the upstream gradient du:
 *   gc_t = du_t silu'(c_t) (du_t when silu == 0);
 *   dx_s = sum_k w[d][k] gc_{s+(K-1)-k};  dw[d][k] = sum_{b,t} gc_t x_{t-(K-1)+k};
 *   dbias_d = sum_{b,t} gc_t.
 *   out: dx [Bsz][Dch][L] (I/O dtype); dw [Dch][K], dbias [Dch] float32 (dbias
 *        non-NULL iff bias non-NULL).  Sums over (b, t) in a fixed order:
 *        reruns are bitwise equal.  Empty Bsz or L: dw, dbias set to 0.
 */
ss_status ss_conv1d_silu_bwd(const void* x, const float* w, const float* bias, int silu,
                             const void* du, int64_t Bsz, int64_t Dch, int64_t L, int64_t K,
                             ss_dtype dtype, void* dx, float* dw, float* dbias,
                             ss_stream_t stream);

/*
 * Input projection that produces the scan's delta_raw, B and C from u
 * (x_proj, which has no bias, then dt_proj without its bias, which the scan
 * adds as delta_bias; "PyTorch 한 파일에서의 Mamba 구현", news.hada.io topic
 * 12448, comment thread on merging the two projections).  Per batch b, with
 * R = dt_rank and N states:
 *   xdbl[t][m]     = sum_k Wx[m][k] u[b][k][t]        (m < R + 2N)
 *   delta[b][d][t] = sum_r Wdt[d][r] xdbl[t][r]       (r < R)
 *   B[b][n][t] = xdbl[t][R + n],  C[b][n][t] = xdbl[t][R + N + n]
 *   in : u [Bsz][Dch][L]; Wx [R + 2N][Dch]; Wdt [Dch][R]; all SS_BF16 or all
 *        SS_F16 (SS_ERR_DTYPE otherwise); fp32 accumulation on the tensor
 *        cores; xdbl[.][r < R] is rounded to the I/O type before dt_proj.
 *   out: delta [Bsz][Dch][L]; B, C [Bsz][N][L] (I/O dtype).
 * Shapes: L, Dch and R multiples of 8, R >= 8, N >= 1, R + 2N <= 256
 * (SS_ERR_SHAPE otherwise).  Outputs must not overlap the inputs.
 * Conventions as for the scan (device pointers, 16-byte alignment, async on
 * stream, checks before launch).
 */
ss_status ss_xproj(const void* u, const void* Wx, const void* Wdt, int64_t Bsz, int64_t Dch,
                   int64_t L, int64_t R, int64_t N, ss_dtype dtype, void* delta, void* B, void* C,
                   ss_stream_t stream);

/*
 * Number of ss_xproj CTAs (since the library was loaded) whose bounded wait
 * for the tensor cores gave up; such a CTA leaves its outputs incomplete and
 * also sets the device error word that ss_check_device_errors reports.
 * Synchronous (device-to-host copy on the legacy stream); -1 on a CUDA error.
 */
int ss_xproj_wait_failures(void);

/*
 * Test hook for the timeout path: while on != 0, every ss_xproj CTA, after
 * its first GEMM, also waits (for 64 polls) on a barrier that nothing ever
 * completes, so that wait gives up and the CTA takes its failure path (the
 * tensor-core work already issued completes and is waited for; the outputs
 * are left unwritten).  Lets a test check that SS_ERR_TIMEOUT is reported
 * without faulting or hanging the device.  Off by default.
 */
void ss_debug_xproj_stuck_wait(int on);

/*
 * Backward scan for callers that cannot allocate device memory.
 *
 * The pages describe no counterpart of this entry point; it exists for
 * library users only.  Some callers cannot call cudaMalloc: a plugin running
 * inside a host application that owns every device allocation, or a
 * latency-critical loop that must never enter the allocator (which can
 * synchronise the device).  They can pass inputs and outputs but no
 * workspace.  This call is ss_scan_bwd with the workspace taken from a
 * scratch buffer compiled into the library: a static device array of
 * ss_scan_bwd_noalloc_max_scratch() bytes (32 MiB), which every GPU that
 * loads the library holds until the process exits.
 *   - Arguments, checks, outputs and results are those of ss_scan_bwd,
 *     without the workspace pair; its argument checks run first.
 *   - Then sizes whose ss_scan_bwd_workspace_size exceeds the buffer are
 *     rejected with SS_ERR_SCRATCH_LIMIT; nothing is launched.
 *   - The first call on a device looks up the buffer's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it.  With
 *     lazy module loading (the CUDA default) this lookup is what loads the
 *     library's device code and the buffer onto that device, so the first
 *     call does take device memory: make it at initialisation, outside
 *     allocation-sensitive code and before any stream capture starts.
 *   - The call allocates nothing (no cudaMalloc, cudaFree or allocating
 *     library routine).
 *   - All calls share the one buffer, which keeps the last call's contents;
 *     the kernels write every scratch word before reading it, so nothing is
 *     cleared.  Calls that overlap on the GPU (e.g. unordered streams) race
 *     on the buffer: order them.
 */
ss_status ss_scan_bwd_noalloc(const void* u, const void* delta, const float* A, const void* B,
                              const void* C, const float* D, const void* z,
                              const float* delta_bias, int softplus, const void* dy,
                              int64_t Bsz, int64_t Dch, int64_t L, int64_t N, ss_dtype dtype,
                              void* du, void* ddelta, float* dA, float* dB, float* dC,
                              float* dD, void* dz, float* ddelta_bias, ss_stream_t stream);

/* Size in bytes of the static scratch buffer ss_scan_bwd_noalloc uses. */
size_t ss_scan_bwd_noalloc_max_scratch(void);

#ifdef __cplusplus
}
#endif

#endif /* SELSCAN_H_ */

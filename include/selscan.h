/*
 * libselscan — the selective-scan forward of the Mamba selective state-space
 * model, and its one-token recurrent decode step, on an NVIDIA B300 (sm_103a).
 *
 * What is computed, for every batch b, channel d and state index n:
 *
 *   Δ_t   = softplus(δ_t + Δ_bias[d])          (or δ_t + Δ_bias[d] when delta_softplus == 0)
 *   Ā_t   = exp(Δ_t · A[d,n])
 *   h_t   = Ā_t · h_{t-1} + Δ_t · B[b,n,t] · u_t          (h_{-1} = h0, or 0)
 *   y_t   = Σ_n C[b,n,t] · h_t[n] + D[d] · u_t
 *   out_t = y_t · silu(z_t) = y_t · z_t / (1 + e^{-z_t})   (out_t = y_t when z is NULL)
 *
 * Sources (web pages on the Mamba selective SSM, cited by title and section):
 *  - "Mamba状态空间模型深度解析：挑战Transformer的下一代序列建模范式" §2.1 — the
 *    selective recurrence h_k = A·h_{k-1} + B(x_k)·x_k, y_k = C(x_k)·h_k with B,
 *    C and Δ functions of the input; §3.1 — the SiLU multiplicative gate.
 *  - "Mamba架构与SSM模型：高效序列建模技术解析" §2.1 — zero-order hold
 *    Ā = exp(ΔA); §2.2 — Δ = softplus(Linear(x) + param_Δ).  The Linear
 *    projection is upstream; its output is the `delta` argument here.
 *  - "Mamba: Linear-Time Sequence Modeling with Selective SSMs", "连续与离散SSM"
 *    — y = Cx + Du (the D skip); "选择性扫描要点" — the sequence is scanned in
 *    blocks whose end state is passed on as the next block's start state,
 *    which is exactly what h0 / h_last expose across calls.
 *  - "Mamba架构深度剖析：如何以线性时间重塑序列建模" §3 — recurrent (RNN-mode)
 *    inference with a constant-size state: selscan_step.
 * The input matrix is discretised as B̄ = Δ·B (not the exact zero-order-hold
 * form (ΔA)^{-1}(exp(ΔA) - I)·ΔB that the same §2.1 also prints).
 *
 * Conventions for every entry point:
 *  - All tensor arguments are DEVICE pointers (cudaMalloc'd, or pinned host
 *    memory mapped into the device address space) to contiguous row-major
 *    arrays, last index fastest.  The caller owns every buffer.
 *  - Scratch: selscan_fwd, selscan_fwd_ex and selscan_fwd_conv take stream-
 *    ordered scratch (cudaMallocAsync / cudaFreeAsync on `stream`) for the
 *    time blocks of problems with few rows (a few MB: block summaries and
 *    start states); if the memory pool cannot supply it the call returns
 *    SELSCAN_ERR_CUDA with cudaErrorMemoryAllocation and enqueues nothing
 *    else.  selscan_fwd_noalloc allocates nothing.
 *  - State kept between calls: cached device attributes and driver entry
 *    points; per host thread, the last CUDA error and launch count; per
 *    device, one word that a kernel sets when a bounded wait gives up
 *    (selscan_device_status) and selscan_fwd_noalloc's fixed scratch array.
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream).  A return of SELSCAN_OK means the work was
 *    enqueued; faults during execution surface at the caller's next
 *    synchronisation, as for any CUDA launch.
 *  - Arguments are checked on the host before anything is enqueued.  A bad
 *    argument returns an error status and enqueues nothing.  Each pointer must
 *    be device-accessible and lie, with its whole extent, inside one device
 *    allocation (checked with the driver's address-range query).
 *  - Element types: u, delta, z, B, C are `in_dtype` (fp32 or bf16); out is
 *    `out_dtype`; A, D, delta_bias, h0, h_last and the decode state are fp32.
 *  - Optional arguments may be NULL: D (treated as 0), z (no gate),
 *    delta_bias (0), h0 (zero start state), h_last (not written).
 *  - h_last may alias h0 (in-place carry).  No other output may overlap an
 *    input (SELSCAN_ERR_ALIAS).
 *  - Thread safety: calls from several host threads are safe; calls on the
 *    same stream run in order.  The one exception is selscan_fwd_noalloc:
 *    its calls share one scratch array, so calls whose work overlaps on the
 *    GPU race (see below).
 */
#ifndef SELSCAN_H_
#define SELSCAN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SELSCAN_ABI_VERSION 1
#define SELSCAN_MAX_DSTATE 16

typedef enum { SELSCAN_F32 = 0, SELSCAN_BF16 = 1 } selscan_dtype_t;

typedef enum {
  SELSCAN_OK = 0,
  SELSCAN_ERR_NULL = 1,        /* a required pointer (or the shape) is NULL */
  SELSCAN_ERR_SHAPE = 2,       /* negative size, dstate < 1, or a size product overflows */
  SELSCAN_ERR_ALIGN = 3,       /* a pointer is not aligned to its element size */
  SELSCAN_ERR_UNSUPPORTED = 4, /* dstate > SELSCAN_MAX_DSTATE or an unknown dtype */
  SELSCAN_ERR_CUDA = 5,        /* a CUDA call failed; see selscan_last_cuda_error() */
  SELSCAN_ERR_POINTER = 6,     /* a pointer is not device-accessible or its extent leaves its allocation */
  SELSCAN_ERR_ALIAS = 7,       /* an output overlaps an input (other than h_last == h0) */
  SELSCAN_ERR_SCRATCH = 8      /* the problem needs more scratch than the buffer it may use: selscan_fwd_noalloc's
                                  fixed array, or the workspace given to selscan_bwd */
} selscan_status_t;

/* Problem sizes.  For selscan_step, seqlen must be 1. */
typedef struct {
  int64_t batch;  /* B */
  int64_t dim;    /* D, the channel (d_inner) count */
  int64_t seqlen; /* L */
  int64_t dstate; /* N, 1 .. SELSCAN_MAX_DSTATE */
  selscan_dtype_t in_dtype;  /* type of u, delta, z, B, C */
  selscan_dtype_t out_dtype; /* type of out */
} selscan_shape_t;

/*
 * Selective-scan forward over a whole sequence.
 *
 *   u, delta, z : [B, D, L]  in_dtype     input, pre-softplus Δ, gate (z nullable)
 *   A           : [D, N]     fp32         diagonal state matrix (usually negative)
 *   B, C        : [B, N, L]  in_dtype     input-dependent input / output matrices,
 *                                         shared by all D channels of a batch row
 *   D           : [D]        fp32         skip weight (nullable)
 *   delta_bias  : [D]        fp32         added to delta before the softplus (nullable)
 *   delta_softplus : nonzero applies softplus to δ + Δ_bias
 *   h0          : [B, D, N]  fp32         start state (nullable: zeros)
 *   out         : [B, D, L]  out_dtype    gated output
 *   h_last      : [B, D, N]  fp32         state after the last step (nullable; may alias h0)
 *
 * Splitting a sequence into consecutive calls, each given the previous call's
 * h_last as h0, gives the same result as one call up to fp32 rounding.
 * L = 0 writes h_last = h0 (or zeros) and nothing else.
 */
selscan_status_t selscan_fwd(const selscan_shape_t* shape, const void* u, const void* delta, const float* A,
                             const void* B, const void* C, const float* D, const void* z,
                             const float* delta_bias, int delta_softplus, const float* h0, void* out,
                             float* h_last, void* stream);

/*
 * One recurrent decode step (the L = 1 case of the forward, done in place on
 * the state).  Shapes: u, delta, z, out [B, D]; B, C [B, N]; A [D, N];
 * D, delta_bias [D]; state [B, D, N] fp32, read as h_{t-1} and overwritten
 * with h_t.  shape->seqlen must be 1.  `state` must not overlap any input.
 */
selscan_status_t selscan_step(const selscan_shape_t* shape, const void* u, const void* delta, const float* A,
                              const void* B, const void* C, const float* D, const void* z,
                              const float* delta_bias, int delta_softplus, float* state, void* out,
                              void* stream);

/*
 * Selective-scan forward with options (flags, OR-ed):
 *
 *   SELSCAN_FLAG_REVERSE  scan from t = L-1 down to 0: h_t = Ā_t·h_{t+1} + B̄_t·u_t (h_L = h0),
 *                         y_t = Σ_n C[b,n,t]·h_t[n] + D[d]·u_t; h_last is the state after t = 0.
 *                         This is the backward direction of a bidirectional Mamba layer ("Mamba架构与
 *                         SSM模型：高效序列建模技术解析" §3.2 names a bidirectional option; "Mamba:
 *                         Linear-Time Sequence Modeling with Selective State Spaces" mentions
 *                         bidirectional use for DNA).
 *   SELSCAN_FLAG_ZOH      exact zero-order hold for the input matrix, B̄ = (exp(Δ·A) - 1)/A · B per
 *                         state (diagonal A; Δ·B at A = 0), instead of B̄ = Δ·B
 *                         ("Mamba架构与SSM模型：高效序列建模技术解析" §2.1 prints
 *                         B̄ = (ΔA)^{-1}(exp(ΔA) - I)·ΔB).
 *
 * Arguments, layouts, checks and errors are those of selscan_fwd.  flags = 0 computes exactly what
 * selscan_fwd computes.  Unknown flag bits return SELSCAN_ERR_UNSUPPORTED.  It runs the kernels
 * selscan_fwd runs (time blocks and their stream-ordered scratch for problems with few rows).
 */
#define SELSCAN_FLAG_REVERSE 1u
#define SELSCAN_FLAG_ZOH 2u
selscan_status_t selscan_fwd_ex(const selscan_shape_t* shape, const void* u, const void* delta, const float* A,
                                const void* B, const void* C, const float* D, const void* z,
                                const float* delta_bias, int delta_softplus, const float* h0, void* out,
                                float* h_last, unsigned flags, void* stream);

/*
 * Selective-scan forward with the block's convolution front computed in the kernel: u is not passed
 * but computed from x by a causal depthwise 1-D convolution of width 4 and SiLU,
 *
 *   u[b,d,t] = silu( conv_b[d] + Σ_{k=0}^{3} conv_w[d,k] · x[b,d,t-3+k] ),   x before t = 0 is 0,
 *
 * and the scan then runs on u as in selscan_fwd (the D skip uses u).  ("Mamba架构与SSM模型：高效序列
 * 建模技术解析" §3.2: d_conv = 4; "Mamba状态空间模型深度解析" §3.1: convolution then SiLU before the
 * SSM.)  This saves writing u to memory and reading it back.
 *
 *   x       : [B, D, L]  in_dtype   the convolution's input (in place of u)
 *   conv_w  : [D, 4]     fp32       taps; conv_w[d, 3] multiplies x_t, conv_w[d, 0] multiplies x_{t-3}
 *   conv_b  : [D]        fp32       bias (nullable: 0)
 *   flags   : 0 or SELSCAN_FLAG_ZOH (the front is causal: SELSCAN_FLAG_REVERSE is rejected with
 *             SELSCAN_ERR_UNSUPPORTED)
 * Every other argument, check and error is that of selscan_fwd.  A sequence split over calls
 * restarts the convolution from zero history at each call's first step.  It runs the kernels
 * selscan_fwd runs (time blocks and their stream-ordered scratch for problems with few rows).
 */
selscan_status_t selscan_fwd_conv(const selscan_shape_t* shape, const void* x, const float* conv_w,
                                  const float* conv_b, const void* delta, const float* A, const void* B,
                                  const void* C, const float* D, const void* z, const float* delta_bias,
                                  int delta_softplus, const float* h0, void* out, float* h_last, unsigned flags,
                                  void* stream);

/*
 * Selective-scan forward that allocates no memory at all: same arguments, layouts, validation and
 * result (within fp32 rounding) as selscan_fwd.  It is for callers that cannot call cudaMalloc or
 * cudaMallocAsync while they run, for example code that owns a fixed memory budget or that runs
 * inside a framework which forbids allocation during execution.  (selscan_fwd may take stream-ordered
 * scratch from the CUDA memory pool for problems with few rows, see below.)  The pages describe no
 * such entry point; it is an engineering addition.
 *
 * It runs the kernels selscan_fwd runs.  For problems with few rows they cut the sequence into time
 * blocks and keep, per block, a summary and a start state of every row:
 *   ((blocks - 1) * (N + 1) + blocks * N) * batch * dim floats.
 * These live in one fixed device array of SELSCAN_NOALLOC_SCRATCH_BYTES (8 MiB) inside the library,
 * reserved on every GPU that loads the library until the process exits.  A problem that would need
 * more returns SELSCAN_ERR_SCRATCH and enqueues nothing (the 1 x 1536 x 65536 x 16 case needs about
 * 2.4 MiB).  No part of the array has to start at zero: each call writes every entry it reads first.
 *
 * The first call on a device looks up the array's device address (once per device, with that
 * device current); make that first call before any stream capture.  Every call shares the one
 * array: calls whose work overlaps on the GPU (other streams, other host threads) race on it and
 * must be serialised by the caller.
 */
#define SELSCAN_NOALLOC_SCRATCH_BYTES (8u << 20)
selscan_status_t selscan_fwd_noalloc(const selscan_shape_t* shape, const void* u, const void* delta, const float* A,
                                     const void* B, const void* C, const float* D, const void* z,
                                     const float* delta_bias, int delta_softplus, const float* h0, void* out,
                                     float* h_last, void* stream);

/*
 * Gradients of selscan_fwd (the backward pass, for training): given dout = ∂loss/∂out and
 * dh_last = ∂loss/∂h_last, the gradients of the loss with respect to every input.  Reverse-mode
 * differentiation of the forward's recurrence, with g the gradient with respect to the state after the
 * step being undone (g = dh_last after the last step), for t from L-1 down to 0:
 *
 *   dy_t = dout_t · silu(z_t),      dz_t = dout_t · y_t · σ(z_t)·(1 + z_t·(1 - σ(z_t)))
 *   G[n] = g[n] + dy_t · C[b,n,t]
 *   dC[b,n,t] = Σ_d dy_t · h_t[n]          dB[b,n,t] = Σ_d G[n] · Δ_t · u_t
 *   du_t = dy_t · D[d] + Δ_t · Σ_n G[n]·B[b,n,t]
 *   dΔ_t = Σ_n G[n] · (B[b,n,t]·u_t + A[d,n]·Ā_t[n]·h_{t-1}[n]),   dδ_t = dΔ_t · σ(δ_t + Δ_bias[d])
 *   dA[d,n] += Σ_b Δ_t · G[n] · Ā_t[n] · h_{t-1}[n],    g[n] = G[n] · Ā_t[n]
 *   dD[d] = Σ_{b,t} dy_t · u_t,   dΔ_bias[d] = Σ_{b,t} dδ_t,   dh0 = g after t = 0
 *
 * (σ is the logistic function, the derivative of softplus; with delta_softplus == 0, dδ_t = dΔ_t.)
 * The forward's states are not stored: the call recomputes them, keeping only the state at the start
 * of every 16-step chunk in `workspace` — the recomputation that "Mamba状态空间模型深度解析：挑战
 * Transformer的下一代序列建模范式" §2.2 describes for training.  Where the forward's row-sequential
 * kernel can stage the rows (as selscan_fwd_ckpt requires) and needs no time blocks, that kernel forms
 * the checkpoints in a launch of its own before the backward; otherwise the backward kernel does.
 *
 *   u, delta, A, B, C, D, z, delta_bias, delta_softplus, h0 : the forward call's inputs (as selscan_fwd)
 *   dout        : [B, D, L]  out_dtype   ∂loss/∂out
 *   dh_last     : [B, D, N]  fp32        ∂loss/∂h_last (nullable: 0)
 *   du, ddelta  : [B, D, L]  in_dtype    ∂loss/∂u, ∂loss/∂delta (written)
 *   dz          : [B, D, L]  in_dtype    ∂loss/∂z (written; required when z is given, ignored otherwise)
 *   dA          : [D, N]     fp32        ∂loss/∂A (overwritten)
 *   dB, dC      : [B, N, L]  fp32        ∂loss/∂B, ∂loss/∂C (overwritten; fp32 whatever in_dtype is,
 *                                        since they are sums over the D channels)
 *   dD, ddelta_bias : [D]    fp32        (nullable: not computed; computed even when D or delta_bias is
 *                                        NULL, as the gradient at 0)
 *   dh0         : [B, D, N]  fp32        ∂loss/∂h0 (nullable; written also when h0 is NULL)
 *   workspace   : device memory of at least selscan_bwd_workspace_size(shape) bytes, 16-byte aligned,
 *                 used only while the call's work runs; NULL takes it from the CUDA memory pool of
 *                 `stream` (cudaMallocAsync / cudaFreeAsync) instead.  A smaller workspace_bytes returns
 *                 SELSCAN_ERR_SCRATCH.
 *
 * Accumulated gradients (dA, dB, dC, dD, ddelta_bias) are summed with floating-point atomics, so their
 * last bits may differ from run to run.  No output may overlap an input, another output or the
 * workspace.  The checks and errors are otherwise those of selscan_fwd; L = 0 or no rows writes zeros
 * to the accumulated gradients and dh0 = dh_last (or 0).
 */
selscan_status_t selscan_bwd(const selscan_shape_t* shape, const void* u, const void* delta, const float* A,
                             const void* B, const void* C, const float* D, const void* z,
                             const float* delta_bias, int delta_softplus, const float* h0, const void* dout,
                             const float* dh_last, void* du, void* ddelta, void* dz, float* dA, float* dB,
                             float* dC, float* dD, float* ddelta_bias, float* dh0, void* workspace,
                             size_t workspace_bytes, void* stream);

/* Bytes of workspace selscan_bwd needs for `shape` (0 for an invalid shape); enough for
 * selscan_bwd_ckpt too, which needs less (no checkpoints of its own). */
size_t selscan_bwd_workspace_size(const selscan_shape_t* shape);

/*
 * Training pair: a forward that keeps the state before every 16-step chunk, and a backward that reruns
 * chunks from those checkpoints instead of recomputing them with a forward pass of its own — the
 * checkpointed recomputation of "Mamba状态空间模型深度解析：挑战Transformer的下一代序列建模范式" §2.2,
 * with the forward's checkpoints kept.
 *
 * selscan_fwd_ckpt: selscan_fwd plus
 *   ckpt : [B, D, ceil(L/16), 16] fp32, written: ckpt[b,d,c,n] = the state h before step 16·c (h0 for
 *          c = 0); slots of states n >= N are left unwritten.  Required when there is work.
 * It needs the row-sequential kernel (every u, delta, z, B, C row 16-byte aligned: L a multiple of 8
 * for bf16, of 4 for fp32, and 16-byte aligned bases); otherwise it returns SELSCAN_ERR_UNSUPPORTED and
 * enqueues nothing.  The checkpoints cost 4 bytes of writes per element (64 bytes per row and chunk).
 *
 * selscan_bwd_ckpt: selscan_bwd with
 *   ckpt : the checkpoints selscan_fwd_ckpt wrote for the same u, delta, A, B, delta_bias,
 *          delta_softplus and h0 (read only; required when there is work).
 * Its workspace needs no checkpoint space (selscan_bwd_workspace_size is an upper bound).  Every other
 * argument, check and result is selscan_bwd's.
 */
selscan_status_t selscan_fwd_ckpt(const selscan_shape_t* shape, const void* u, const void* delta, const float* A,
                                  const void* B, const void* C, const float* D, const void* z,
                                  const float* delta_bias, int delta_softplus, const float* h0, void* out,
                                  float* h_last, float* ckpt, void* stream);
selscan_status_t selscan_bwd_ckpt(const selscan_shape_t* shape, const void* u, const void* delta, const float* A,
                                  const void* B, const void* C, const float* D, const void* z,
                                  const float* delta_bias, int delta_softplus, const float* h0, const void* dout,
                                  const float* dh_last, const float* ckpt, void* du, void* ddelta, void* dz,
                                  float* dA, float* dB, float* dC, float* dD, float* ddelta_bias, float* dh0,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* Human-readable name of a status code (static storage). */
const char* selscan_status_string(selscan_status_t status);

/* The cudaError_t of the last SELSCAN_ERR_CUDA returned on this host thread (0 if none). */
int selscan_last_cuda_error(void);

/*
 * Device-side status of earlier launches on the current device: 0 if every launch ran to completion,
 * 1 if a kernel gave up a bounded wait for one of its own asynchronous shared-memory copies (it then
 * stops early and leaves its outputs incomplete, instead of waiting forever).  `reset` != 0 clears
 * the word.  The read is a synchronous device-to-host copy: it waits for work already enqueued on
 * the legacy default stream.  Returns -1 if the read itself fails.
 */
int selscan_device_status(int reset);

/* SELSCAN_ABI_VERSION of the library that is loaded. */
int selscan_abi_version(void);

/*
 * The number of kernels that the last selscan_fwd, selscan_fwd_ex, selscan_fwd_conv,
 * selscan_fwd_noalloc, selscan_fwd_ckpt, selscan_bwd, selscan_bwd_ckpt or selscan_step call on this
 * host thread enqueued: 1 for a forward or backward run in one pass or a decode step, 3 for a forward
 * or backward run in time blocks (the summary pass, the carry pass and the scan), one more for a
 * selscan_bwd whose checkpoints come from a forward launch of their own (see selscan_bwd), 0 when the
 * call enqueued no kernel (an argument error, no rows, or an empty sequence, whose state is passed on
 * by a copy).
 * The pages have no counterpart; it lets a caller (or a benchmark) account for the
 * launches of its timed region.
 */
int selscan_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* SELSCAN_H_ */

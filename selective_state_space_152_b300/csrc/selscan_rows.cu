// Selective-scan forward for sm_103a: the row-sequential kernel with a warp-specialised copy pipeline.
//
// What it computes, per batch b, channel d and state n (see include/selscan.h):
//   Δ_t = softplus(δ_t + Δ_bias[d]),  Ā_t = exp(Δ_t A[d,n]),
//   h_t = Ā_t h_{t-1} + Δ_t B[b,n,t] u_t,  y_t = Σ_n C[b,n,t] h_t + D[d] u_t,  out_t = y_t silu(z_t)
// ("Mamba状态空间模型深度解析：挑战Transformer的下一代序列建模范式" §2.1 the selective recurrence, §3.1
//  the SiLU gate; "Mamba架构与SSM模型：高效序列建模技术解析" §2.1 Ā = exp(ΔA), §2.2
//  Δ = softplus(Linear(x) + param_Δ); "Mamba: Linear-Time Sequence Modeling with Selective SSMs",
//  连续与离散SSM, the D·u term).  This is the recurrent form run as written: every row (b, d) is walked
// from its first step to its last, so no step is computed twice and no partial scans are joined.
//
// Lanes.  Q lanes share a row; lane q owns the SPL = NS/Q states [q·SPL, (q+1)·SPL) and keeps them in
// SPL/2 float2 pairs, so the state update is one packed fp32x2 FMA per pair and step.  A warp holds
// RPW = 32/Q rows.  The exponent Δ·A·log2e is formed for two consecutive steps at once (one packed
// multiply of (Δ_t, Δ_t+1) by (A_n, A_n)), and each step costs per state pair: two ex2, one packed
// multiply for Δu·B, one packed FMA for the state and one packed FMA for C·h.
//
// Per chunk of kT steps a consumer warp
//   1. (Q > 1) computes Δ = softplus(δ + Δ_bias) and Δ·u once per (row, step) — each of the Q lanes
//      of a row takes kT/Q of the steps — into a warp-private shared buffer; with Q = 1 each lane does
//      its own row's steps in registers;
//   2. walks the kT steps in sub-blocks of kSB (the whole chunk when Q > 1), every lane accumulating the
//      partial y of its states;
//   3. after each sub-block adds the Q partial sums of a row through the warp buffer, each lane taking
//      kSB/Q of the steps, adds D·u, gates with silu(z) and stores its steps.
//
// Copy pipeline.  One producer warp per CTA issues the tensor-memory-accelerator copies of each chunk
// into one of S stages: u, δ, z of the CTA's rows as 2-D tiles [ROWS][kT] (64- or 128-byte swizzle)
// and the raw [N][kT] rows of B and C, which every row of the batch entry shares.  When a stage has
// landed the producer widens B and C to fp32 in a [t][n] layout (one 128-bit shared load then gives a
// lane four states of one step, read by all lanes at the same address) and signals the consumers; a
// stage is refilled once every consumer warp has released it.  Consumer warps never wait for each other.
//
// Time blocks.  When the rows alone cannot fill the GPU, the sequence is cut into blocks.  A summary
// pass (the same kernel with SUMMARY) runs every block but the last from a zero state and writes its
// end state and ΣΔ; a carry pass chains them, s ← exp(A·ΣΔ)·s + (zero-start end state), into the start
// state of every block; the scan pass then runs all blocks at once from their start states.  That is
// the blockwise scan whose end state seeds the next block ("Mamba: Linear-Time Sequence Modeling with
// Selective SSMs", 选择性扫描要点), with the blocks run side by side.
//
// Options: REV scans from the last step to the first (the backward direction of a bidirectional
// layer); ZOH uses the exact zero-order-hold input factor (exp(ΔA) - 1)/A·B instead of Δ·B
// ("Mamba架构与SSM模型：高效序列建模技术解析" §2.1); CONV computes u in the kernel from x by the block's
// causal depthwise convolution of width 4 and SiLU (§3.2 of the same page, d_conv = 4).
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "selscan_internal.cuh"

namespace selscan {

// Set by a kernel whose bounded wait gave up (read by selscan_device_status()).
__device__ int g_selscan_rows_error = 0;

// ---- the fixed scratch of selscan_fwd_noalloc ----------------------------------------------------------
//
// For callers that may not allocate memory while they run, the summaries and start states of the time
// blocks live in this array instead of stream-ordered scratch.  It is reserved on every GPU that loads
// the library, for the life of the process.  In host code the array's name stands for a host-side
// stand-in, not a device address, so its device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, and passed to the kernels.  Every call shares the
// array: work of calls that overlaps on the GPU races on it.
constexpr size_t kFixedScratchFloats = SELSCAN_NOALLOC_SCRATCH_BYTES / sizeof(float);
static __device__ __align__(256) float g_noalloc_scratch[kFixedScratchFloats];

namespace {
constexpr int kFixedMaxDevices = 64;
std::mutex g_fixed_mutex;
float* g_fixed_ptr[kFixedMaxDevices] = {};
}  // namespace

cudaError_t fixed_scratch(float** ptr, size_t* bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kFixedMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_fixed_mutex);
  if (!g_fixed_ptr[dev]) {
    void* a = nullptr;
    e = cudaGetSymbolAddress(&a, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_fixed_ptr[dev] = static_cast<float*>(a);
  }
  *ptr = g_fixed_ptr[dev];
  *bytes = kFixedScratchFloats * sizeof(float);
  return cudaSuccess;
}

namespace {

constexpr int kT = 32;  // steps per chunk
// Q > 1: Δ and Δu reach the Q lanes of a row as one 16-byte record per step pair from a warp buffer (1),
// or by shuffles from the lane that prepared them (0).
#ifndef SELSCAN_ROWS_DU_SMEM
#define SELSCAN_ROWS_DU_SMEM 1
#endif
// Q > 1: the row's Q partial sums of y meet through a warp buffer (1: each lane writes its partials, then
// reads the Q partials of the steps it stores) or by recursive halving with shuffles (0).
#ifndef SELSCAN_ROWS_YRED
#define SELSCAN_ROWS_YRED 1
#endif
// Q > 1: step pairs whose exponentials are formed ahead of the state update in progress.
#ifndef SELSCAN_ROWS_AHEAD
#define SELSCAN_ROWS_AHEAD 2
#endif
// Q > 1: the record of a step pair is read this many pairs before its exponentials are formed, so the
// shared-memory latency is not in the way of the exponent multiply.
#ifndef SELSCAN_ROWS_RECEARLY
#define SELSCAN_ROWS_RECEARLY 2
#endif
// Pause of the producer warp between polls of its two events, in nanoseconds.
#ifndef SELSCAN_ROWS_PSLEEP
#define SELSCAN_ROWS_PSLEEP 64
#endif
constexpr int kMaxWarps = 11;  // consumer warps per CTA (one producer warp more): 12 warps, up to 168 registers
constexpr int kMaxStages = 4;

template <int NS, int SPL, typename Tin, bool ZOH, bool CONV>
struct RowsGeom {
  static constexpr int Q = NS / SPL;   // lanes per row
  static constexpr int RPW = 32 / Q;   // rows per warp
  static constexpr int RB = kT * static_cast<int>(sizeof(Tin));  // bytes of one staged row of a chunk
  static constexpr CUtensorMapSwizzle kSwizzle = RB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  // Steps per sub-block: with several lanes per row the whole chunk, so that the row's partial sums of y
  // meet once per chunk (each meeting is a wait on shared memory the warp cannot hide; halving them
  // measured 3 % faster); with one lane per row, which keeps its inputs of a sub-block in registers, 16.
  static constexpr int SB = Q == 1 ? 16 : kT;
  static constexpr int NSB = kT / SB;  // sub-blocks per chunk
  static constexpr int EPS = SB / Q;   // steps per lane and sub-block that the lane prepares and stores
  static constexpr int TS = NS + 4;     // floats per step of the widened B, C tile
  // Warp-private buffer (Q > 1): per row and step pair the record (Δ_t, Δ_t+1, Δu_t, Δu_t+1), plus with ZOH
  // (u_t, u_t+1); rows padded by 16 bytes so that the 8 rows a quarter-warp reads fall in distinct banks.
  static constexpr int REC = (ZOH ? 6 : 4) * (kT / 2) + 4;  // floats per row
  static constexpr int REC_FLOATS = (Q > 1 && SELSCAN_ROWS_DU_SMEM) ? RPW * REC : 0;
  // y partials (Q > 1, SELSCAN_ROWS_YRED): [q][row][SB + 4]; the odd number of 16-byte units per row keeps
  // the 8 lanes of a quarter-warp in distinct banks both when they write and when they read.
  static constexpr int YS = SB + 4;
  static constexpr int Y_FLOATS = (Q > 1 && SELSCAN_ROWS_YRED) ? 32 * YS : 0;
  static constexpr int WARP_FLOATS = REC_FLOATS + Y_FLOATS;
  static_assert(NS % SPL == 0 && SPL % 4 == 0 && (Q == 1 || Q == 2 || Q == 4), "lanes per row");
  static_assert(RB == 64 || RB == 128, "staged rows of 64 or 128 bytes");
};

// Offsets of the dynamic shared memory of one CTA (W consumer warps, S stages), from a 1 KiB-aligned base.
struct RowsSmem {
  size_t tens, raw, tile, wbuf, bars, total;
};
template <class G, typename Tin, int NS>
__host__ __device__ inline RowsSmem rows_smem(int W, int S) {
  RowsSmem m;
  const size_t rows = static_cast<size_t>(W) * G::RPW;
  m.tens = (rows * G::RB + 1023) / 1024 * 1024;  // one tensor's tile, on a 1 KiB boundary (swizzle period)
  m.raw = static_cast<size_t>(S) * 3 * m.tens;
  m.tile = m.raw + static_cast<size_t>(S) * 2 * NS * kT * sizeof(Tin);
  m.wbuf = m.tile + static_cast<size_t>(S) * 2 * kT * G::TS * sizeof(float);
  m.bars = m.wbuf + static_cast<size_t>(W) * G::WARP_FLOATS * sizeof(float);
  m.total = m.bars + static_cast<size_t>(S) * 3 * sizeof(uint64_t) + 1024;  // + alignment slack
  return m;
}

// ---- device helpers --------------------------------------------------------------------------------

// The staged row of one tensor's tile [ROWS][RB bytes] that a lane reads, with its swizzle: the tile was
// written by a 2-D tensor copy with the RB-byte swizzle, so 16-byte chunk c of row r sits at chunk
// position c ^ (r mod 8) for 128-byte rows and c ^ ((r / 2) mod 4) for 64-byte rows (the tile starts
// on a 1 KiB boundary).
template <int RB>
__device__ __forceinline__ int stage_swizzle(int r) {
  return RB == 128 ? (r & 7) : ((r >> 1) & 3);
}

// NV consecutive staged inputs [e0, e0 + NV) of a staged row (see stage_swizzle).
template <typename Tin, int NV>
__device__ __forceinline__ void stage_load(float (&v)[NV], const unsigned char* __restrict__ row, int swz, int e0) {
  constexpr int PER = 16 / static_cast<int>(sizeof(Tin));
  if constexpr (NV * sizeof(Tin) >= 16) {
    static_assert(NV % PER == 0, "whole 16-byte chunks");
#pragma unroll
    for (int c = 0; c < NV / PER; c++) {
      const int chunk = e0 / PER + c;
      const uint4 w = *reinterpret_cast<const uint4*>(row + ((chunk ^ swz) << 4));
#pragma unroll
      for (int k = 0; k < PER; k++) v[c * PER + k] = elem_of(w, k, Tin());
    }
  } else {
    static_assert(NV * sizeof(Tin) == 8, "8-byte reads");
    const int chunk = e0 / PER, within = (e0 % PER) * static_cast<int>(sizeof(Tin));
    const uint2 w = *reinterpret_cast<const uint2*>(row + ((chunk ^ swz) << 4) + within);
    const uint4 w4 = make_uint4(w.x, w.y, 0u, 0u);
#pragma unroll
    for (int k = 0; k < NV; k++) v[k] = elem_of(w4, k, Tin());
  }
}

// NV outputs [t, t + NV) of a row: vector stores where the row is aligned and the steps lie inside L.
template <int NV>
__device__ __forceinline__ void store_out(void* __restrict__ out, int64_t row_off, int64_t t, int64_t L, bool vec,
                                          bool bf16, const float (&y)[NV]) {
  const bool whole = vec && t + NV <= L;
  if (!bf16) {
    float* o = static_cast<float*>(out) + row_off + t;
    if (whole) {
#pragma unroll
      for (int k = 0; k < NV / 4; k++)
        reinterpret_cast<float4*>(o)[k] = make_float4(y[4 * k], y[4 * k + 1], y[4 * k + 2], y[4 * k + 3]);
    } else {
#pragma unroll
      for (int k = 0; k < NV; k++)
        if (t + k < L) o[k] = y[k];
    }
    return;
  }
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out) + row_off + t;
  if (whole) {
    uint32_t w[NV / 2];
#pragma unroll
    for (int k = 0; k < NV / 2; k++)
      w[k] = out_bits(y[2 * k], __nv_bfloat16()) | (out_bits(y[2 * k + 1], __nv_bfloat16()) << 16);
    if constexpr (NV == 4) {
      *reinterpret_cast<uint2*>(o) = make_uint2(w[0], w[1]);
    } else {
#pragma unroll
      for (int k = 0; k < NV / 8; k++)
        reinterpret_cast<uint4*>(o)[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
    }
  } else {
#pragma unroll
    for (int k = 0; k < NV; k++)
      if (t + k < L) o[k] = __float2bfloat16_rn(y[k]);
  }
}

// Bounded wait on an mbarrier phase that also gives up when another warp of the CTA has raised the
// abort flag (checked every 256 polls).
__device__ __noinline__ bool wait_or_abort_slow(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                long long limit = kWaitLimit) {
  for (long long i = 0; i < limit; i++) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255) == 255 && *abort_flag) return false;
  }
  atomicExch(&g_selscan_rows_error, 1);
  *abort_flag = 1;
  return false;
}
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  return mbar_try_wait(bar, parity) || wait_or_abort_slow(bar, parity, abort_flag);
}

// Non-blocking test of an mbarrier phase.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// The exponentials of two consecutive steps (i, i+1) of one lane's SPL states: the exponent is formed for
// both steps at once per state, e_n = (Δ_i, Δ_i+1)·(A_n, A_n)·log2 e, and each 2^e is written straight
// into the (state 2p, state 2p+1) pair of its step, the operand layout of the packed state update.
template <int SPL>
__device__ __forceinline__ void expo_pair(float2 dd, const float2 (&A2d)[SPL], float2 (&e)[SPL], float2 (&a0)[SPL / 2],
                                          float2 (&a1)[SPL / 2]) {
#pragma unroll
  for (int n = 0; n < SPL; n++) e[n] = mul2s(dd, A2d[n]);
#pragma unroll
  for (int p = 0; p < SPL / 2; p++) {
    a0[p] = f2(ex2_approx(e[2 * p].x), ex2_approx(e[2 * p + 1].x));
    a1[p] = f2(ex2_approx(e[2 * p].y), ex2_approx(e[2 * p + 1].y));
  }
}

// The state update and readout of two consecutive steps (i, i+1), in scan order (i+1 first with REV),
// from their exponentials (a0: step i, a1: step i+1; e: the exponents, for ZOH).  du0/du1 = (Δu, Δu) of
// each step; u0/u1 = (u, u) (ZOH only); Bt/Ct: the widened tile rows of step i at this lane's states
// (step i+1 is TS floats further).  Writes the partial y = Σ C·h over the lane's states of each step
// (not in SUMMARY).
template <int SPL, int TS, bool REV, bool ZOH, bool SUMMARY>
__device__ __forceinline__ void update_pair(float2 (&h)[SPL / 2], const float2 (&IA)[SPL / 2], const float2 (&e)[SPL],
                                            const float2 (&a0)[SPL / 2], const float2 (&a1)[SPL / 2], float2 du0,
                                            float2 du1, float2 u0, float2 u1, const float* __restrict__ Bt,
                                            const float* __restrict__ Ct, float& y0, float& y1) {
  float2 yk[2];
#pragma unroll
  for (int kk = 0; kk < 2; kk++) {
    const int k = REV ? 1 - kk : kk;
    const float4* Bq = reinterpret_cast<const float4*>(Bt + k * TS);
    const float4* Cq = reinterpret_cast<const float4*>(Ct + k * TS);
    const float2 dup = k ? du1 : du0;
    float2 y2 = f2(0.f, 0.f);
#pragma unroll
    for (int g = 0; g < SPL / 4; g++) {
      const float4 bb = Bq[g];
      float4 cc = make_float4(0.f, 0.f, 0.f, 0.f);
      if (!SUMMARY) cc = Cq[g];
#pragma unroll
      for (int m = 0; m < 2; m++) {
        const int p = 2 * g + m;
        const float2 a = k ? a1[p] : a0[p];
        const float2 bpair = m ? f2(bb.z, bb.w) : f2(bb.x, bb.y);
        float2 fu = dup;
        if (ZOH) {
          const float2 ep = k ? f2(e[2 * p].y, e[2 * p + 1].y) : f2(e[2 * p].x, e[2 * p + 1].x);
          fu = zoh_factor2(dup, ep, a, mul2s(k ? u1 : u0, IA[p]));
        }
        h[p] = fma2s(a, h[p], mul2s(fu, bpair));
        if (!SUMMARY) y2 = fma2s(m ? f2(cc.z, cc.w) : f2(cc.x, cc.y), h[p], y2);
      }
    }
    yk[k] = y2;
  }
  if (!SUMMARY) {
    y0 = yk[0].x + yk[0].y;
    y1 = yk[1].x + yk[1].y;
  }
}

// One level of the reduce-scatter of a row's partial sums across its lanes: the lane whose partner bit is
// set keeps the upper half of v[0, LEN) and the other the lower half, each adding its partner's copy.
template <int LEN, int MASK, int NV>
__device__ __forceinline__ void halve_partials(float (&v)[NV], bool hi) {
#pragma unroll
  for (int m = 0; m < LEN / 2; m++) {
    const float send = hi ? v[m] : v[LEN / 2 + m];
    const float keep = hi ? v[LEN / 2 + m] : v[m];
    v[m] = keep + __shfl_xor_sync(kFull, send, MASK);
  }
}

// Δ and Δu of NV consecutive steps from t on: Δ = softplus(δ + bias) (SP) or δ + bias, and 0 at and
// past L (an identity step) when TAIL.
template <bool SP, bool TAIL, int NV>
__device__ __forceinline__ void deltas(const float (&xv)[NV], const float (&uv)[NV], float bias, int64_t t, int64_t L,
                                       float (&dl)[NV], float (&du)[NV]) {
#pragma unroll
  for (int i = 0; i < NV; i++) {
    const float x = xv[i] + bias;
    float d = SP ? softplus_fast(x) : x;
    if (TAIL && t + i >= L) d = 0.f;
    dl[i] = d;
    du[i] = d * uv[i];
  }
}
template <int NV>
__device__ __forceinline__ void deltas_any(bool sp, bool tail, const float (&xv)[NV], const float (&uv)[NV], float bias,
                                           int64_t t, int64_t L, float (&dl)[NV], float (&du)[NV]) {
  if (sp) {
    if (tail) deltas<true, true>(xv, uv, bias, t, L, dl, du);
    else deltas<true, false>(xv, uv, bias, t, L, dl, du);
  } else {
    if (tail) deltas<false, true>(xv, uv, bias, t, L, dl, du);
    else deltas<false, false>(xv, uv, bias, t, L, dl, du);
  }
}

// The causal convolution front of NV steps: u_i = silu(cb + w0·x_{i-3} + w1·x_{i-2} + w2·x_{i-1} + w3·x_i),
// with x3, x2, x1 the three inputs before the first step.  xv holds x on entry and u on return.
template <int NV>
__device__ __forceinline__ void conv_front(float (&xv)[NV], float x3, float x2, float x1, float cw0, float cw1,
                                           float cw2, float cw3, float cbias) {
  float a[NV];
#pragma unroll
  for (int i = 0; i < NV; i++) {
    const float xa = i >= 3 ? xv[i - 3] : (i == 0 ? x3 : (i == 1 ? x2 : x1));
    const float xb = i >= 2 ? xv[i - 2] : (i == 0 ? x2 : x1);
    const float xc = i >= 1 ? xv[i - 1] : x1;
    a[i] = fmaf(cw3, xv[i], fmaf(cw2, xc, fmaf(cw1, xb, fmaf(cw0, xa, cbias))));
  }
#pragma unroll
  for (int i = 0; i < NV; i++) xv[i] = silu_fast(a[i]);
}

// ---- the kernel -----------------------------------------------------------------------------------

// The lane's states before step t, if t starts a 16-step checkpoint chunk inside the sequence, into the
// checkpoints of selscan_fwd_ckpt: [row][t / 16][n0, n0 + SPL).
template <int SPL>
__device__ __forceinline__ void save_ckpt(const FwdParams& p, const float2 (&h)[SPL / 2], int64_t grow, int64_t t,
                                          bool row_ok, int n0) {
  if (!row_ok || t >= p.seqlen) return;
  float4* dst = reinterpret_cast<float4*>(p.ckpt + (grow * p.ckpt_chunks + t / 16) * 16 + n0);
#pragma unroll
  for (int k = 0; k < SPL / 4; k++) dst[k] = make_float4(h[2 * k].x, h[2 * k].y, h[2 * k + 1].x, h[2 * k + 1].y);
}

// CKPT: the plain forward scan that also keeps the state before every 16-step chunk (p.ckpt); with
// SUMMARY as well, the checkpoint pass: from the start state, keeping only the checkpoints (no C, y or
// outputs), the forward pass a backward reruns its chunks from.
template <int NS, int SPL, typename Tin, bool SUMMARY, bool REV, bool ZOH, bool CONV, bool CKPT = false>
__global__ void __launch_bounds__((kMaxWarps + 1) * 32, 1)
    selscan_fwd_rows_kernel(const FwdParams p, const __grid_constant__ TmaMaps maps) {
  static_assert(!(CONV && REV), "the convolution front is causal: forward direction only");
  static_assert(!CKPT || (!REV && !ZOH && !CONV), "checkpoints of the plain forward scan only");
  using G = RowsGeom<NS, SPL, Tin, ZOH, CONV>;
  constexpr int Q = G::Q, RPW = G::RPW, RB = G::RB, TS = G::TS, kSB = G::SB;
  const int W = p.warps, S = p.stages;
  const int ROWS = W * RPW;
  const RowsSmem sm = rows_smem<G, Tin, NS>(W, S);
  extern __shared__ __align__(128) unsigned char smem_dyn[];
  // (Offsetting the shared pointer itself keeps every derived pointer in the shared window.)
  unsigned char* base = smem_dyn + ((1024u - (smem_addr(smem_dyn) & 1023u)) & 1023u);
  unsigned char* udz = base;                                   // [S][3][tens]: u, δ, z tiles
  Tin* raw = reinterpret_cast<Tin*>(base + sm.raw);            // [S][2][NS][kT]: B, C as copied
  float* tile = reinterpret_cast<float*>(base + sm.tile);      // [S][2][kT][TS]: B, C widened
  float* wbuf = reinterpret_cast<float*>(base + sm.wbuf);      // [W][WARP_FLOATS]
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + sm.bars);  // [S][3]: copies landed, tile ready, released
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t b = blockIdx.y;
  const int kslot = blockIdx.z;                             // summary slot (SUMMARY) or time block
  const int kblk = (SUMMARY && REV) ? kslot + 1 : kslot;    // time block: steps [tbeg, tend)
  const int64_t L = p.seqlen;
  const int N = p.dstate;
  const int64_t tbeg = static_cast<int64_t>(kblk) * p.tblock;
  const int64_t tend = (tbeg + p.tblock) < L ? (tbeg + p.tblock) : L;
  const int64_t c_begin = tbeg / kT;  // tblock is a multiple of kT
  const int nchunks = static_cast<int>((tend - tbeg + kT - 1) / kT);
  const int64_t d0 = static_cast<int64_t>(blockIdx.x) * ROWS;
  const int64_t rows_total = p.batch * p.dim;
  auto chunk_t0 = [&](int ci) -> int64_t { return (REV ? c_begin + nchunks - 1 - ci : c_begin + ci) * kT; };

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < S; s++) {
      mbar_init(&bars[3 * s + 0], 1);
      mbar_init(&bars[3 * s + 1], 1);
      mbar_init(&bars[3 * s + 2], W);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  volatile int* abort_flag = &s_abort;

  // ---------------------------------------------------------------------------- producer warp
  if (warp == W) {
    const bool has_z = !SUMMARY && p.z != nullptr;
    const int ntens = has_z ? 3 : 2;
    const uint32_t bytes = static_cast<uint32_t>(ntens * ROWS * RB + (SUMMARY ? 1 : 2) * NS * kT * sizeof(Tin));
    const int row0 = static_cast<int>(b * p.dim + d0);
    const int brow = static_cast<int>(b * N);
    auto issue = [&](int ci, int s) {
      const int t0 = static_cast<int>(chunk_t0(ci));
      uint64_t* bar = &bars[3 * s];
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_expect_tx(bar, bytes);
      const CUtensorMap* m[3] = {&maps.u, &maps.delta, &maps.z};
      for (int k = 0; k < ntens; k++) tma_load_2d(udz + (static_cast<size_t>(s) * 3 + k) * sm.tens, m[k], t0, row0, bar);
      Tin* dst = raw + static_cast<size_t>(s) * 2 * NS * kT;
      tma_load_2d(dst, &maps.B, t0, brow, bar);
      if (!SUMMARY) tma_load_2d(dst + NS * kT, &maps.C, t0, brow, bar);
    };
    const int first = nchunks < S ? nchunks : S;
    if (lane == 0)
      for (int ci = 0; ci < first; ci++) issue(ci, ci);
    // Event loop: widen every chunk as soon as its copies have landed, and refill a stage as soon as every
    // consumer warp has released it; neither waits for the other.
    int next_widen = 0, next_issue = first;
    int ws = 0, wpar = 0;        // stage and phase of chunk next_widen
    int is = 0, ipar = 0;        // stage and phase of chunk next_issue - S (the stage's previous occupant)
    long long idle = 0;
    bool ok = true;
    while (next_widen < nchunks || next_issue < nchunks) {
      bool progress = false;
      if (next_widen < nchunks && next_widen < next_issue && mbar_test(&bars[3 * ws], static_cast<uint32_t>(wpar))) {
        // Widen B (and C) to fp32 [t][n], zeroing states >= N (their rows belong to the next batch entry).
        const Tin* rb = raw + static_cast<size_t>(ws) * 2 * NS * kT;
        float* tb = tile + static_cast<size_t>(ws) * 2 * kT * TS;
        constexpr int T4 = kT / 4, N4 = NS / 4;
        constexpr int UNITS = (SUMMARY ? 1 : 2) * N4 * T4;
        // Units with consecutive state quads in a quarter-warp: their 16-byte stores land in distinct banks
        // (TS = NS + 4 floats per step), where consecutive step quads would collide four ways.
        for (int unit = lane; unit < UNITS; unit += 32) {
          const int n4 = unit % N4, rest = unit / N4;
          const int t4 = rest % T4, tt = rest / T4;
          float v[4][4];
#pragma unroll
          for (int k = 0; k < 4; k++) {
            const Tin* src = rb + (tt * NS + n4 * 4 + k) * kT + t4 * 4;
            if (sizeof(Tin) == 2) {
              const uint2 w = *reinterpret_cast<const uint2*>(src);
              v[k][0] = __uint_as_float(w.x << 16);
              v[k][1] = __uint_as_float(w.x & 0xffff0000u);
              v[k][2] = __uint_as_float(w.y << 16);
              v[k][3] = __uint_as_float(w.y & 0xffff0000u);
            } else {
              const float4 w = *reinterpret_cast<const float4*>(src);
              v[k][0] = w.x;
              v[k][1] = w.y;
              v[k][2] = w.z;
              v[k][3] = w.w;
            }
            if (n4 * 4 + k >= N) v[k][0] = v[k][1] = v[k][2] = v[k][3] = 0.f;
          }
#pragma unroll
          for (int m = 0; m < 4; m++)
            *reinterpret_cast<float4*>(tb + (tt * kT + t4 * 4 + m) * TS + n4 * 4) =
                make_float4(v[0][m], v[1][m], v[2][m], v[3][m]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[3 * ws + 1]);
        next_widen++;
        if (++ws == S) {
          ws = 0;
          wpar ^= 1;
        }
        progress = true;
      }
      // The stage for chunk next_issue was last used by chunk next_issue - S, which must have been widened
      // (so the consumers could have it) and released by every consumer warp.
      if (next_issue < nchunks && next_issue - S < next_widen &&
          mbar_test(&bars[3 * is + 2], static_cast<uint32_t>(ipar))) {
        if (lane == 0) issue(next_issue, is);
        next_issue++;
        if (++is == S) {
          is = 0;
          ipar ^= 1;
        }
        progress = true;
      }
      __syncwarp();
      if (progress) {
        idle = 0;
      } else if (++idle > kIdleLimit || ((idle & 255) == 255 && *abort_flag)) {
        if (idle > kIdleLimit) atomicExch(&g_selscan_rows_error, 1);
        *abort_flag = 1;
        ok = false;
        break;
      } else {
        __nanosleep(SELSCAN_ROWS_PSLEEP);  // neither event yet: leave the issue slots to the consumer warps
      }
    }
    if (!ok && lane == 0) {
      // Let every copy still in flight land before the CTA's shared memory is released.
      for (int ci = next_widen; ci < next_issue; ci++) mbar_wait(&bars[3 * (ci % S)], static_cast<uint32_t>((ci / S) & 1));
    }
    return;
  }

  // ---------------------------------------------------------------------------- consumer warps
  const int r = lane % RPW;  // row of this lane within the warp
  const int q = lane / RPW;  // state group (scan, output) and step slice (prep) of this lane
  const int r_cta = warp * RPW + r;
  const int64_t d = d0 + r_cta;
  const bool row_ok = d < p.dim;
  const int64_t dd_ = row_ok ? d : 0;  // rows past `dim` compute on channel 0's parameters, never stored
  const int64_t grow = b * p.dim + d;
  const float bias = p.delta_bias ? p.delta_bias[dd_] : 0.f;
  const float Dd = p.D ? p.D[dd_] : 0.f;
  const bool softplus = p.delta_softplus != 0;
  const bool has_z = !SUMMARY && p.z != nullptr;
  const bool vec_out = p.vec_out != 0, out_bf16 = p.out_bf16 != 0;
  void* const out = p.out;
  // The common output case, with no per-store branches: a gate, fp32 vector stores, a live row.
  const bool fast = has_z && vec_out && !out_bf16 && row_ok;

  // This lane's states, in pairs: A·log2 e duplicated for the time-packed exponent, 1/A for ZOH, h.
  const int n0 = q * SPL;
  float2 A2d[SPL], IA[SPL / 2], h[SPL / 2];
#pragma unroll
  for (int n = 0; n < SPL; n++) {
    const float a = (n0 + n < N) ? p.A[dd_ * N + n0 + n] * kLog2e : 0.f;
    A2d[n] = f2(a, a);
  }
#pragma unroll
  for (int i = 0; i < SPL / 2; i++) {
    IA[i] = ZOH ? f2(kLog2e / A2d[2 * i].x, kLog2e / A2d[2 * i + 1].x) : f2(0.f, 0.f);
    float hh[2];
#pragma unroll
    for (int k = 0; k < 2; k++) {
      const int n = n0 + 2 * i + k;
      if ((SUMMARY && !CKPT) || n >= N || !row_ok)
        hh[k] = 0.f;
      else if (p.nblocks > 1)
        hh[k] = p.start[(static_cast<int64_t>(kblk) * rows_total + grow) * N + n];
      else
        hh[k] = p.h0 ? p.h0[grow * N + n] : 0.f;
    }
    h[i] = f2(hh[0], hh[1]);
  }
  // Convolution front: taps and bias of the row, and x before the block (history of the first chunk).
  float cw0 = 0.f, cw1 = 0.f, cw2 = 0.f, cw3 = 0.f, cbias = 0.f, xm3 = 0.f, xm2 = 0.f, xm1 = 0.f;
  if (CONV) {
    cw0 = p.conv_w[dd_ * 4 + 0];
    cw1 = p.conv_w[dd_ * 4 + 1];
    cw2 = p.conv_w[dd_ * 4 + 2];
    cw3 = p.conv_w[dd_ * 4 + 3];
    cbias = p.conv_b ? p.conv_b[dd_] : 0.f;
    const Tin* xrow = static_cast<const Tin*>(p.u) + (b * p.dim + dd_) * L;
    xm3 = tbeg >= 3 ? to_f32(xrow[tbeg - 3]) : 0.f;
    xm2 = tbeg >= 2 ? to_f32(xrow[tbeg - 2]) : 0.f;
    xm1 = tbeg >= 1 ? to_f32(xrow[tbeg - 1]) : 0.f;
  }

  float* const wrec = wbuf + static_cast<size_t>(warp) * G::WARP_FLOATS;  // this warp's records
  const int64_t row_off = (b * p.dim + dd_) * L;
  const int swz = stage_swizzle<RB>(r_cta);
  const size_t row_byte = static_cast<size_t>(r_cta) * RB;
  float sumD = 0.f;  // Σ Δ over this lane's prep steps of the block (SUMMARY)

  int s = 0;
  uint32_t par = 0;
  bool ok = true;
  for (int ci = 0; ci < nchunks; ci++) {
    const int64_t t0 = chunk_t0(ci);
    const bool tail = t0 + kT > L;
    if (!wait_or_abort(&bars[3 * s], par, abort_flag)) {
      ok = false;
      break;
    }
    const unsigned char* st_u = udz + static_cast<size_t>(s) * 3 * sm.tens + row_byte;  // this lane's staged rows
    const unsigned char* st_d = st_u + sm.tens;
    const unsigned char* st_z = st_d + sm.tens;
    const float* tB = tile + static_cast<size_t>(s) * 2 * kT * TS + n0;
    const float* tC = tB + kT * TS;

    // 1. (Q > 1) Δ, Δu and u of this lane's own steps of the chunk, {sb·kSB + q·EPS + m}: computed once
    //    per (row, step) and kept in registers.  They are also the steps whose outputs this lane stores.
    constexpr int NSB = G::NSB, EPS = G::EPS;
    float rdl[NSB * EPS], rdu[NSB * EPS], ru[NSB * EPS];
    if constexpr (Q > 1) {
      float xv[NSB][EPS], uv[NSB][EPS];
#pragma unroll
      for (int g = 0; g < NSB; g++) {
        stage_load<Tin, EPS>(xv[g], st_d, swz, g * kSB + q * EPS);
        stage_load<Tin, EPS>(uv[g], st_u, swz, g * kSB + q * EPS);
      }
      if constexpr (CONV) {
        // x before each of this lane's groups: the previous group of the row is lane q-1's group of the
        // same sub-block, or for q = 0 lane Q-1's group of the previous sub-block (or chunk).
        float h3[NSB], h2[NSB], h1[NSB];
#pragma unroll
        for (int g = 0; g < NSB; g++) {
          const float u3 = __shfl_up_sync(kFull, uv[g][EPS - 3], RPW), u2 = __shfl_up_sync(kFull, uv[g][EPS - 2], RPW),
                      u1 = __shfl_up_sync(kFull, uv[g][EPS - 1], RPW);
          float l3 = xm3, l2 = xm2, l1 = xm1;
          if (g > 0) {
            l3 = __shfl_sync(kFull, uv[g - 1][EPS - 3], (Q - 1) * RPW + r);
            l2 = __shfl_sync(kFull, uv[g - 1][EPS - 2], (Q - 1) * RPW + r);
            l1 = __shfl_sync(kFull, uv[g - 1][EPS - 1], (Q - 1) * RPW + r);
          }
          h3[g] = q ? u3 : l3;
          h2[g] = q ? u2 : l2;
          h1[g] = q ? u1 : l1;
        }
        // The row's last three x of this chunk, for its first group of the next chunk.
        xm3 = __shfl_sync(kFull, uv[NSB - 1][EPS - 3], (Q - 1) * RPW + r);
        xm2 = __shfl_sync(kFull, uv[NSB - 1][EPS - 2], (Q - 1) * RPW + r);
        xm1 = __shfl_sync(kFull, uv[NSB - 1][EPS - 1], (Q - 1) * RPW + r);
#pragma unroll
        for (int g = 0; g < NSB; g++) conv_front<EPS>(uv[g], h3[g], h2[g], h1[g], cw0, cw1, cw2, cw3, cbias);
      }
#pragma unroll
      for (int g = 0; g < NSB; g++) {
        float dl[EPS], du[EPS];
        deltas_any<EPS>(softplus, tail, xv[g], uv[g], bias, t0 + g * kSB + q * EPS, L, dl, du);
#pragma unroll
        for (int m = 0; m < EPS; m++) {
          rdl[g * EPS + m] = dl[m];
          rdu[g * EPS + m] = du[m];
          ru[g * EPS + m] = uv[g][m];
          if (SUMMARY) sumD += dl[m];
        }
      }
      if constexpr (SELSCAN_ROWS_DU_SMEM) {
        // Records of this lane's step pairs into the warp buffer (the previous chunk's readers are done: the
        // warp synchronised before releasing it).
        float* rec = wrec + r * G::REC;
#pragma unroll
        for (int g = 0; g < NSB; g++)
#pragma unroll
          for (int m = 0; m < EPS; m += 2) {
            const int pair = (g * kSB + q * EPS + m) / 2, k = g * EPS + m;
            reinterpret_cast<float4*>(rec)[pair] = make_float4(rdl[k], rdl[k + 1], rdu[k], rdu[k + 1]);
            if (ZOH) reinterpret_cast<float2*>(rec + 4 * (kT / 2))[pair] = f2(ru[k], ru[k + 1]);
          }
        __syncwarp();
      }
    }

    if (!wait_or_abort(&bars[3 * s + 1], par, abort_flag)) {
      ok = false;
      break;
    }

    // 2-3. The scan over the chunk, then the row's outputs of each sub-block.
    if constexpr (Q == 1) {
#pragma unroll
      for (int sbi = 0; sbi < kT / kSB; sbi++) {
        const int sb = REV ? kT / kSB - 1 - sbi : sbi;
        float yp[kSB];
        float xv[kSB], uv[kSB];
        stage_load<Tin, kSB>(xv, st_d, swz, sb * kSB);
        stage_load<Tin, kSB>(uv, st_u, swz, sb * kSB);
        if constexpr (CONV) {
          const float n3 = uv[kSB - 3], n2 = uv[kSB - 2], n1 = uv[kSB - 1];
          conv_front<kSB>(uv, xm3, xm2, xm1, cw0, cw1, cw2, cw3, cbias);
          xm3 = n3;
          xm2 = n2;
          xm1 = n1;
        }
        float dl[kSB], du[kSB];
        deltas_any<kSB>(softplus, tail, xv, uv, bias, t0 + sb * kSB, L, dl, du);
        if (SUMMARY) {
#pragma unroll
          for (int i = 0; i < kSB; i++) sumD += dl[i];
        }
        // The exponentials of each step pair are formed one pair ahead of its state update, so the
        // special-function unit's latency overlaps the previous pair's FMAs.
        float2 e[SPL], a0[SPL / 2], a1[SPL / 2];
        {
          const int i = REV ? kSB - 2 : 0;
          expo_pair<SPL>(f2(dl[i], dl[i + 1]), A2d, e, a0, a1);
        }
#pragma unroll
        for (int pi = 0; pi < kSB / 2; pi++) {
          const int pr = REV ? kSB / 2 - 1 - pi : pi;
          const int i = 2 * pr;
          if (CKPT && i % 16 == 0) save_ckpt<SPL>(p, h, grow, t0 + sb * kSB + i, row_ok, n0);
          float2 ne[SPL], na0[SPL / 2], na1[SPL / 2];
          if (pi + 1 < kSB / 2) {
            const int j = REV ? i - 2 : i + 2;
            expo_pair<SPL>(f2(dl[j], dl[j + 1]), A2d, ne, na0, na1);
          }
          update_pair<SPL, TS, REV, ZOH, SUMMARY>(h, IA, e, a0, a1, f2(du[i], du[i]), f2(du[i + 1], du[i + 1]),
                                                  f2(uv[i], uv[i]), f2(uv[i + 1], uv[i + 1]), tB + (sb * kSB + i) * TS,
                                                  tC + (sb * kSB + i) * TS, yp[i], yp[i + 1]);
          if (pi + 1 < kSB / 2) {
#pragma unroll
            for (int n = 0; n < SPL; n++) e[n] = ne[n];
#pragma unroll
            for (int q2 = 0; q2 < SPL / 2; q2++) {
              a0[q2] = na0[q2];
              a1[q2] = na1[q2];
            }
          }
        }
        if (!SUMMARY) {
          float zv[kSB];
          if (has_z) stage_load<Tin, kSB>(zv, st_z, swz, sb * kSB);
#pragma unroll
          for (int i = 0; i < kSB; i++) {
            float y = fmaf(Dd, uv[i], yp[i]);
            if (has_z) y *= silu_fast(zv[i]);
            yp[i] = y;
          }
          if (row_ok) store_out<kSB>(out, row_off, t0 + sb * kSB, L, vec_out, out_bf16, yp);
        }
      }
    } else {
      // Δ and Δu of a step pair come from the lane that prepared them: the row's record of the pair in the
      // warp buffer (Δ_t, Δ_t+1, Δu_t, Δu_t+1), or shuffles from lane (t / EPS) of the row.
      constexpr int P = kT / 2, PS = kSB / 2, AH = SELSCAN_ROWS_AHEAD;
      const float4* recs = reinterpret_cast<const float4*>(wrec + r * G::REC);
      const float2* urec = reinterpret_cast<const float2*>(wrec + r * G::REC + 4 * (kT / 2));
      auto record = [&](int gp) -> float4 {
        if constexpr (SELSCAN_ROWS_DU_SMEM) {
          return recs[gp];
        } else {
          const int tt = 2 * (gp % PS), src = (tt / EPS) * RPW + r, k = (gp / PS) * EPS + tt % EPS;
          return make_float4(__shfl_sync(kFull, rdl[k], src), __shfl_sync(kFull, rdl[k + 1], src),
                             __shfl_sync(kFull, rdu[k], src), __shfl_sync(kFull, rdu[k + 1], src));
        }
      };
      // The pairs in scan order g = 0 .. P-1 (pair gp = g, or P-1-g with REV).  The exponentials of pair g
      // are formed AH pairs ahead of its state update, across sub-block boundaries, so the special-function
      // unit's latency overlaps the FMAs of the pairs in between (only AH + 1 pairs are live at a time).
      float4 rq[P];
      float2 eq[P][SPL], a0q[P][SPL / 2], a1q[P][SPL / 2];
      constexpr int RE = SELSCAN_ROWS_RECEARLY;
      auto load_rec = [&](int g) { rq[g] = record(REV ? P - 1 - g : g); };
      auto start = [&](int g) {
        if (RE == 0) load_rec(g);
        expo_pair<SPL>(f2(rq[g].x, rq[g].y), A2d, eq[g], a0q[g], a1q[g]);
      };
      if (RE > 0) {
#pragma unroll
        for (int g = 0; g < AH + RE && g < P; g++) load_rec(g);
      }
#pragma unroll
      for (int g = 0; g < AH && g < P; g++) start(g);
      float yp[kSB];
#pragma unroll
      for (int g = 0; g < P; g++) {
        if (RE > 0 && g + AH + RE < P) load_rec(g + AH + RE);
        if (g + AH < P) start(g + AH);
        const int gp = REV ? P - 1 - g : g, sb = gp / PS, tt = 2 * (gp % PS);
        float u0 = 0.f, u1 = 0.f;
        if (ZOH) {
          if constexpr (SELSCAN_ROWS_DU_SMEM) {
            const float2 uu = urec[gp];
            u0 = uu.x;
            u1 = uu.y;
          } else {
            const int src = (tt / EPS) * RPW + r, k = sb * EPS + tt % EPS;
            u0 = __shfl_sync(kFull, ru[k], src);
            u1 = __shfl_sync(kFull, ru[k + 1], src);
          }
        }
        if (CKPT && (2 * gp) % 16 == 0) save_ckpt<SPL>(p, h, grow, t0 + 2 * gp, row_ok, n0);
        update_pair<SPL, TS, REV, ZOH, SUMMARY>(h, IA, eq[g], a0q[g], a1q[g], f2(rq[g].z, rq[g].z),
                                                f2(rq[g].w, rq[g].w), f2(u0, u0), f2(u1, u1), tB + 2 * gp * TS,
                                                tC + 2 * gp * TS, yp[tt], yp[tt + 1]);
        if (SUMMARY || (g + 1) % PS != 0) continue;
        // Sub-block sb is complete.  The row's Q partial sums of y meet: after it, lane q holds the full y of
        // steps [q·EPS, (q+1)·EPS) of the sub-block (the steps it prepared) in yp[0, EPS).
        if constexpr (SELSCAN_ROWS_YRED) {
          float* yb = wrec + G::REC_FLOATS;
          __syncwarp();  // the previous sub-block's partials have been read
          float4* mine = reinterpret_cast<float4*>(yb + (q * RPW + r) * G::YS);
#pragma unroll
          for (int c = 0; c < kSB / 4; c++) mine[c] = make_float4(yp[4 * c], yp[4 * c + 1], yp[4 * c + 2], yp[4 * c + 3]);
          __syncwarp();
          float2 acc[EPS / 2];
#pragma unroll
          for (int k = 0; k < EPS / 2; k++) acc[k] = f2(0.f, 0.f);
#pragma unroll
          for (int qq = 0; qq < Q; qq++) {
            const float4* src = reinterpret_cast<const float4*>(yb + (qq * RPW + r) * G::YS + q * EPS);
#pragma unroll
            for (int c = 0; c < EPS / 4; c++) {
              const float4 v = src[c];
              acc[2 * c] = add2s(acc[2 * c], f2(v.x, v.y));
              acc[2 * c + 1] = add2s(acc[2 * c + 1], f2(v.z, v.w));
            }
          }
#pragma unroll
          for (int k = 0; k < EPS / 2; k++) {
            yp[2 * k] = acc[k].x;
            yp[2 * k + 1] = acc[k].y;
          }
        } else if (Q == 4) {
          halve_partials<kSB, 2 * RPW>(yp, (q & 2) != 0);
          halve_partials<kSB / 2, RPW>(yp, (q & 1) != 0);
        } else {
          halve_partials<kSB, RPW>(yp, (q & 1) != 0);
        }
        const int e0 = sb * kSB + q * EPS;  // first output step of this lane, within the chunk
        float y[EPS];
#pragma unroll
        for (int m = 0; m < EPS; m++) y[m] = fmaf(Dd, ru[sb * EPS + m], yp[m]);
        if (fast && !tail) {  // gate present, fp32 vector stores, live row: no further branches
          float zv[EPS];
          stage_load<Tin, EPS>(zv, st_z, swz, e0);
          float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) + row_off + t0 + e0);
#pragma unroll
          for (int c = 0; c < EPS / 4; c++)
            o[c] = make_float4(y[4 * c] * silu_fast(zv[4 * c]), y[4 * c + 1] * silu_fast(zv[4 * c + 1]),
                               y[4 * c + 2] * silu_fast(zv[4 * c + 2]), y[4 * c + 3] * silu_fast(zv[4 * c + 3]));
        } else {
          if (has_z) {
            float zv[EPS];
            stage_load<Tin, EPS>(zv, st_z, swz, e0);
#pragma unroll
            for (int m = 0; m < EPS; m++) y[m] *= silu_fast(zv[m]);
          }
          if (row_ok) store_out<EPS>(out, row_off, t0 + e0, L, vec_out, out_bf16, y);
        }
      }
    }
    // Release the stage: this warp has read its u, δ, z tiles and the widened B, C.
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[3 * s + 2]);
    if (++s == S) {
      s = 0;
      par ^= 1;
    }
  }
  if (!ok) return;

  if (SUMMARY && CKPT) return;  // the checkpoint pass keeps nothing else
  if (SUMMARY) {
    // Each prep lane summed Δ over its slice of the block's steps; the row's Q lanes add them up.
#pragma unroll
    for (int o = RPW; o < 32; o <<= 1) sumD += __shfl_xor_sync(kFull, sumD, o);
    if (row_ok) {
      float* o = p.summ + (static_cast<int64_t>(kslot) * rows_total + grow) * (N + 1);
#pragma unroll
      for (int i = 0; i < SPL / 2; i++) {
        if (n0 + 2 * i < N) o[n0 + 2 * i] = h[i].x;
        if (n0 + 2 * i + 1 < N) o[n0 + 2 * i + 1] = h[i].y;
      }
      if (q == 0) o[N] = sumD;
    }
    return;
  }
  if (row_ok && p.h_last && kblk == (REV ? 0 : p.nblocks - 1)) {
#pragma unroll
    for (int i = 0; i < SPL / 2; i++) {
      if (n0 + 2 * i < N) p.h_last[grow * N + n0 + 2 * i] = h[i].x;
      if (n0 + 2 * i + 1 < N) p.h_last[grow * N + n0 + 2 * i + 1] = h[i].y;
    }
  }
}

// Start state of every time block from the block summaries, one thread per (row, state), in scan
// order: s ← 2^(A·log2e·ΣΔ)·s + (zero-start end state of the block).  The first block in scan order
// (block 0, or with REV block nblocks-1) starts from h0, which this pass copies into its slot, so the
// scan pass never reads h0 and may write h_last over it (in-place carry) while other blocks still run.
template <bool REV>
__global__ void __launch_bounds__(256) selscan_rows_carry_kernel(const FwdParams p) {
  const int64_t rows = p.batch * p.dim;
  const int N = p.dstate;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= rows * N) return;
  const int64_t grow = idx / N;
  const int n = static_cast<int>(idx - grow * N);
  const int64_t d = grow % p.dim;
  const float A2 = p.A[d * N + n] * kLog2e;
  float st = p.h0 ? p.h0[grow * N + n] : 0.f;
  const int first = REV ? p.nblocks - 1 : 0;
  p.start[(static_cast<int64_t>(first) * rows + grow) * N + n] = st;
  for (int k = 0; k < p.nblocks - 1; k++) {
    // Forward: summary slot k is block k and feeds block k+1.  Reverse: slot nblocks-2-k is block
    // nblocks-1-k and feeds block nblocks-2-k.
    const int slot = REV ? p.nblocks - 2 - k : k;
    const float* smv = p.summ + (static_cast<int64_t>(slot) * rows + grow) * (N + 1);
    st = fmaf(ex2_approx(A2 * smv[N]), st, smv[n]);
    p.start[(static_cast<int64_t>(REV ? slot : k + 1) * rows + grow) * N + n] = st;
  }
}

// ---- host side ------------------------------------------------------------------------------------

// Rough issue cost per element of the scan for each lane count (instructions of a lane-step times Q
// plus the per-element work); the summary pass costs about 0.7 of a scan.  Used only to rank plans.
// Relative time of one element of the scan for each lane count, at full occupancy (measured on B300 with
// 16 states: two lanes per row and four cost about the same per element, four a little more), and of one
// element of the summary pass relative to the scan (it reads no C, forms no y and stores nothing per step:
// measured 0.47 on the 65536-step workload).  Used only to rank plans.
double cost_per_element(int Q) { return Q == 1 ? 0.95 : Q == 2 ? 1.0 : 1.08; }
constexpr double kSummaryCost = 0.5;
constexpr double kFullWarps = 10.0;  // consumer warps per SM that keep it busy

struct RowsPlan {
  int warps = 1, stages = 2, nblocks = 1;
  int64_t tblock = 0;
  double cost = 1e300;
};

constexpr int64_t kMinTblock = 256;

// Choose warps per CTA and time blocks by the modelled time of the busiest SM over both passes.  An SM
// runs its CTAs in rounds of `resident` CTAs (its register, shared-memory and warp limits); a round takes
// tblock steps of its rows, but a round with fewer than kFullWarps consumer warps cannot hide the
// special-function and shared-memory latencies and takes as long as one with kFullWarps (measured on
// B300: 1 CTA of 11 warps per SM beats 2 CTAs of 6 warps whose third CTA runs alone).
RowsPlan plan_rows(const FwdParams& p, int rpw, int Q, int sms, int max_warps, int per_sm_cap[kMaxWarps + 1]) {
  RowsPlan best;
  const int64_t L = p.seqlen;
  const char* ew = getenv("SELSCAN_ROWS_WARPS");
  const char* eb = getenv("SELSCAN_TBLOCKS");
  const int force_w = ew ? atoi(ew) : 0, force_b = eb ? atoi(eb) : 0;
  static const int kBlocks[] = {1, 2, 3, 4, 5, 6, 8, 10, 12, 16, 20, 24, 32, 48, 64};
  for (int nb_try : kBlocks) {
    int nb_req = force_b > 0 ? force_b : nb_try;
    if (force_b > 0 && nb_try != 1) break;
    int64_t tb = nb_req <= 1 ? L : (L + nb_req - 1) / nb_req;
    tb = (tb + kT - 1) / kT * kT;
    if (nb_req > 1 && force_b <= 0 && tb < kMinTblock) continue;
    if (tb <= 0) tb = kT;
    const int nb = static_cast<int>((L + tb - 1) / tb);
    for (int W = max_warps; W >= 1; W--) {
      if (force_w > 0 && W != (force_w < max_warps ? force_w : max_warps)) continue;
      const int64_t cpb = (p.dim + static_cast<int64_t>(W) * rpw - 1) / (static_cast<int64_t>(W) * rpw);
      double cost = 0.0;
      for (int pass = 0; pass < (nb > 1 ? 2 : 1); pass++) {
        const int64_t blocks = pass == 0 ? nb : nb - 1;
        const int64_t ctas = cpb * p.batch * blocks;
        const int64_t per_sm = (ctas + sms - 1) / sms;
        const int64_t resident = per_sm_cap[W] > 0 ? per_sm_cap[W] : 1;
        double warp_rounds = 0.0;  // Σ over rounds of max(consumer warps in the round, kFullWarps)
        for (int64_t left = per_sm; left > 0; left -= resident) {
          const double w = static_cast<double>((left < resident ? left : resident) * W);
          warp_rounds += w > kFullWarps ? w : kFullWarps;
        }
        cost += warp_rounds * rpw * static_cast<double>(tb) * cost_per_element(Q) * (pass == 0 ? 1.0 : kSummaryCost);
      }
      if (cost < best.cost * 0.999) {
        best.cost = cost;
        best.warps = W;
        best.nblocks = nb;
        best.tblock = tb;
      }
    }
  }
  return best;
}

template <class G, typename Tin, int NS>
int stages_for(int W, size_t smem_max) {
  const char* e = getenv("SELSCAN_ROWS_STAGES");
  int S = e ? atoi(e) : 3;
  if (S < 2) S = 2;
  if (S > kMaxStages) S = kMaxStages;
  while (S > 2 && rows_smem<G, Tin, NS>(W, S).total > smem_max) S--;
  return rows_smem<G, Tin, NS>(W, S).total <= smem_max ? S : 0;
}

// Device attributes, cached per device.
struct DevInfo {
  int sms = 0, smem_max = 0, smem_sm = 0, regs_sm = 0;
};
DevInfo dev_info() {
  static std::mutex mu;
  static DevInfo cache[64];
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  DevInfo& di = cache[dev & 63];
  if (di.sms == 0) {
    cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&di.smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaDeviceGetAttribute(&di.smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    cudaDeviceGetAttribute(&di.regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev);
    if (di.sms <= 0) di.sms = 148;
    if (di.smem_max <= 0) di.smem_max = 227 * 1024;
    if (di.smem_sm <= 0) di.smem_sm = 228 * 1024;
    if (di.regs_sm <= 0) di.regs_sm = 65536;
  }
  return di;
}

// The scan kernel of one instantiation: with checkpoints (plain scans only; null for an option) or without.
template <int NS, int SPL, typename Tin, bool REV, bool ZOH, bool CONV>
auto scan_kernel(const FwdParams& p) -> decltype(&selscan_fwd_rows_kernel<NS, SPL, Tin, false, REV, ZOH, CONV>) {
  if (!p.ckpt) return selscan_fwd_rows_kernel<NS, SPL, Tin, false, REV, ZOH, CONV>;
  if constexpr (!REV && !ZOH && !CONV) {
    if (p.ckpt_only) return selscan_fwd_rows_kernel<NS, SPL, Tin, true, false, false, false, true>;
    return selscan_fwd_rows_kernel<NS, SPL, Tin, false, false, false, false, true>;
  }
  return nullptr;
}

// The plan of one instantiation: warps per CTA (within its shared-memory and register limits), pipeline
// stages and time blocks, with its estimated cost.
template <int NS, int SPL, typename Tin, bool REV, bool ZOH, bool CONV>
cudaError_t plan_cfg(const FwdParams& p, RowsPlan* out) {
  using G = RowsGeom<NS, SPL, Tin, ZOH, CONV>;
  const auto scan = scan_kernel<NS, SPL, Tin, REV, ZOH, CONV>(p);
  if (!scan) return cudaErrorInvalidValue;
  const DevInfo di = dev_info();
  // Largest W whose shared memory fits; CTAs per SM for every W (registers, shared memory, warps).
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, scan);
  if (e != cudaSuccess) return e;
  int cap[kMaxWarps + 1] = {0};
  int max_w = 0;
  // The dynamic shared memory leaves 1 KiB of the per-CTA limit for the kernel's static shared memory.
  const size_t dyn_max = static_cast<size_t>(di.smem_max) - 1024;
  for (int W = 1; W <= kMaxWarps && W * G::RPW <= 256; W++) {  // a tensor-copy box spans at most 256 rows
    const int S = stages_for<G, Tin, NS>(W, dyn_max);
    if (S == 0) break;
    max_w = W;
    const size_t smem = rows_smem<G, Tin, NS>(W, S).total;
    const int threads = (W + 1) * 32;
    int by_regs = di.regs_sm / (fa.numRegs > 0 ? fa.numRegs * threads : threads);
    int by_smem = static_cast<int>(static_cast<size_t>(di.smem_sm) / (smem + 1024));
    int by_warps = 64 / (W + 1);
    int c = by_regs < by_smem ? by_regs : by_smem;
    c = c < by_warps ? c : by_warps;
    cap[W] = c > 0 ? c : 1;
  }
  if (max_w == 0) return cudaErrorInvalidConfiguration;
  *out = plan_rows(p, G::RPW, G::Q, di.sms, max_w, cap);
  out->stages = stages_for<G, Tin, NS>(out->warps, dyn_max);
  return cudaSuccess;
}

template <int NS, int SPL, typename Tin, bool REV, bool ZOH, bool CONV>
cudaError_t launch_rows_cfg(const FwdParams& p_in, const RowsPlan& plan, cudaStream_t s, ScratchSource src,
                            bool* too_big) {
  using G = RowsGeom<NS, SPL, Tin, ZOH, CONV>;
  FwdParams p = p_in;
  const auto scan = scan_kernel<NS, SPL, Tin, REV, ZOH, CONV>(p);
  if (!scan) return cudaErrorInvalidValue;
  auto summary = selscan_fwd_rows_kernel<NS, SPL, Tin, true, REV, ZOH, CONV>;
  cudaError_t e = cudaSuccess;
  p.warps = plan.warps;
  p.stages = plan.stages;
  p.tblock = plan.tblock;
  p.nblocks = plan.nblocks;
  const size_t smem = rows_smem<G, Tin, NS>(p.warps, p.stages).total;
  const int ROWS = p.warps * G::RPW;

  TmaMaps maps;
  memset(&maps, 0, sizeof maps);
  const EncodeTiled enc = reinterpret_cast<EncodeTiled>(tensor_map_encoder());
  if (!enc) return cudaErrorNotSupported;
  const uint64_t rows = static_cast<uint64_t>(p.batch * p.dim), bc_rows = static_cast<uint64_t>(p.batch * p.dstate);
  const uint64_t L = static_cast<uint64_t>(p.seqlen);
  const bool ok = encode_2d<Tin>(enc, &maps.u, p.u, L, rows, kT, ROWS, G::kSwizzle) &&
                  encode_2d<Tin>(enc, &maps.delta, p.delta, L, rows, kT, ROWS, G::kSwizzle) &&
                  (!p.z || encode_2d<Tin>(enc, &maps.z, p.z, L, rows, kT, ROWS, G::kSwizzle)) &&
                  encode_2d<Tin>(enc, &maps.B, p.B, L, bc_rows, kT, NS, CU_TENSOR_MAP_SWIZZLE_NONE) &&
                  encode_2d<Tin>(enc, &maps.C, p.C, L, bc_rows, kT, NS, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (!ok) return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(scan, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(summary, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>((p.dim + ROWS - 1) / ROWS), static_cast<unsigned>(p.batch),
                  static_cast<unsigned>(p.nblocks));
  const int threads = (p.warps + 1) * 32;
  if (const char* dbg = getenv("SELSCAN_DEBUG_PLAN"); dbg && dbg[0] == '1')  // for tuning runs
    fprintf(stderr, "selscan rows plan: states/lane %d, lanes/row %d, warps %d, stages %d, time blocks %d x %lld, "
                    "grid %u x %u x %u, smem %zu, cost %.3g\n", SPL, G::Q, p.warps, p.stages, p.nblocks,
            static_cast<long long>(p.tblock), grid.x, grid.y, grid.z, smem, plan.cost);
  if (p.nblocks == 1) {
    scan<<<grid, threads, smem, s>>>(p, maps);
    count_launches(1);
    return cudaGetLastError();
  }
  const int64_t N = p.dstate;
  const size_t summ_floats = static_cast<size_t>(p.nblocks - 1) * rows * (N + 1);
  const size_t start_floats = static_cast<size_t>(p.nblocks) * rows * N;
  const size_t bytes = (summ_floats + start_floats) * sizeof(float);
  void* ws = nullptr;
  if (src == ScratchSource::Fixed) {
    float* fixed = nullptr;
    size_t cap_bytes = 0;
    e = fixed_scratch(&fixed, &cap_bytes);
    if (e != cudaSuccess) return e;
    if (bytes > cap_bytes) {
      *too_big = true;
      return cudaSuccess;
    }
    ws = fixed;
  } else {
    // Stream-ordered scratch, released on the same stream.  If the pool cannot supply it the call fails
    // with the allocation error (selscan_fwd_noalloc needs no allocation).
    e = cudaMallocAsync(&ws, bytes, s);
    if (e != cudaSuccess) return e;
  }
  p.summ = static_cast<float*>(ws);
  p.start = p.summ + summ_floats;
  const dim3 sgrid(grid.x, grid.y, grid.z - 1);
  summary<<<sgrid, threads, smem, s>>>(p, maps);
  e = cudaGetLastError();
  if (e == cudaSuccess) {
    const int64_t nthr = static_cast<int64_t>(rows) * N;
    selscan_rows_carry_kernel<REV><<<static_cast<unsigned>((nthr + 255) / 256), 256, 0, s>>>(p);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    scan<<<grid, threads, smem, s>>>(p, maps);
    e = cudaGetLastError();
  }
  count_launches(3);
  if (src == ScratchSource::Pool) {
    const cudaError_t ef = cudaFreeAsync(ws, s);
    if (e == cudaSuccess) e = ef;
  }
  return e;
}

// Plan and launch one instantiation.
template <int NS, int SPL, typename Tin, bool REV, bool ZOH, bool CONV>
cudaError_t run_rows(const FwdParams& p, cudaStream_t s, ScratchSource src, bool* too_big) {
  RowsPlan plan;
  cudaError_t e = plan_cfg<NS, SPL, Tin, REV, ZOH, CONV>(p, &plan);
  if (e != cudaSuccess) return e;
  return launch_rows_cfg<NS, SPL, Tin, REV, ZOH, CONV>(p, plan, s, src, too_big);
}

// For a plain scan with 8 or 16 states, two lanes per row (8 states each) or four (4 each): whichever plan
// the cost model ranks first (SELSCAN_ROWS_SPL=4|8 forces one).  Options use four lanes.
template <int NS, typename Tin>
cudaError_t run_plain(const FwdParams& p, cudaStream_t s, ScratchSource src, bool* too_big) {
  int force = 0;
  if (const char* e = getenv("SELSCAN_ROWS_SPL")) force = atoi(e);
  if (force == 4) return run_rows<NS, 4, Tin, false, false, false>(p, s, src, too_big);
  if (force == 8) return run_rows<NS, 8, Tin, false, false, false>(p, s, src, too_big);
  RowsPlan p4, p8;
  cudaError_t e = plan_cfg<NS, 4, Tin, false, false, false>(p, &p4);
  if (e != cudaSuccess) return e;
  e = plan_cfg<NS, 8, Tin, false, false, false>(p, &p8);
  if (e != cudaSuccess) return e;
  if (p8.cost < p4.cost) return launch_rows_cfg<NS, 8, Tin, false, false, false>(p, p8, s, src, too_big);
  return launch_rows_cfg<NS, 4, Tin, false, false, false>(p, p4, s, src, too_big);
}

template <typename Tin, bool REV, bool ZOH, bool CONV>
cudaError_t dispatch_rows(const FwdParams& p, cudaStream_t s, ScratchSource src, bool* too_big) {
  const int N = p.dstate;
  if (N <= 4) return run_rows<4, 4, Tin, REV, ZOH, CONV>(p, s, src, too_big);
  const bool plain = !REV && !ZOH && !CONV;
  if (N <= 8) {
    if (plain) return run_plain<8, Tin>(p, s, src, too_big);
    return run_rows<8, 4, Tin, REV, ZOH, CONV>(p, s, src, too_big);
  }
  if (plain) return run_plain<16, Tin>(p, s, src, too_big);
  return run_rows<16, 4, Tin, REV, ZOH, CONV>(p, s, src, too_big);
}

template <typename Tin>
cudaError_t dispatch_rows_opts(const FwdParams& p, const RowsOptions& o, cudaStream_t s, bool* too_big) {
  if (o.conv) return o.zoh ? dispatch_rows<Tin, false, true, true>(p, s, o.scratch, too_big)
                           : dispatch_rows<Tin, false, false, true>(p, s, o.scratch, too_big);
  if (o.reverse && o.zoh) return dispatch_rows<Tin, true, true, false>(p, s, o.scratch, too_big);
  if (o.reverse) return dispatch_rows<Tin, true, false, false>(p, s, o.scratch, too_big);
  if (o.zoh) return dispatch_rows<Tin, false, true, false>(p, s, o.scratch, too_big);
  return dispatch_rows<Tin, false, false, false>(p, s, o.scratch, too_big);
}

}  // namespace

bool rows_kernel_supports(const FwdParams& p, selscan_dtype_t in_dtype) {
  // Tensor copies need 16-byte aligned rows of every input and coordinates that fit in 32 bits.
  const uint64_t rows = static_cast<uint64_t>(p.batch * p.dim), bc_rows = static_cast<uint64_t>(p.batch * p.dstate);
  (void)in_dtype;
  return p.vec_stage && rows < (1ull << 31) && bc_rows < (1ull << 31) && p.seqlen < (1ll << 31) &&
         tensor_map_encoder() != nullptr;
}

cudaError_t launch_fwd_rows(const FwdParams& p_in, selscan_dtype_t in_dtype, selscan_dtype_t out_dtype,
                            const RowsOptions& o, cudaStream_t s, bool* too_big) {
  FwdParams p = p_in;
  p.out_bf16 = out_dtype == SELSCAN_BF16;
  bool tb = false;
  cudaError_t e = in_dtype == SELSCAN_F32 ? dispatch_rows_opts<float>(p, o, s, &tb)
                                          : dispatch_rows_opts<__nv_bfloat16>(p, o, s, &tb);
  if (too_big) *too_big = tb;
  return e;
}

namespace {

// The checkpoint pass with the plan the forward would take (two or four lanes per row by cost), when
// that plan needs no time blocks.
template <int NS, typename Tin>
cudaError_t ckpt_pass_ns(const FwdParams& p, cudaStream_t s, bool* launched) {
  RowsPlan p4;
  cudaError_t e = plan_cfg<NS, 4, Tin, false, false, false>(p, &p4);
  if (e != cudaSuccess) return e;
  if constexpr (NS >= 8) {
    RowsPlan p8;
    e = plan_cfg<NS, 8, Tin, false, false, false>(p, &p8);
    if (e != cudaSuccess) return e;
    if (p8.cost < p4.cost) {
      if (p8.nblocks > 1) return cudaSuccess;
      e = launch_rows_cfg<NS, 8, Tin, false, false, false>(p, p8, s, ScratchSource::Pool, nullptr);
      *launched = e == cudaSuccess;
      return e;
    }
  }
  if (p4.nblocks > 1) return cudaSuccess;
  e = launch_rows_cfg<NS, 4, Tin, false, false, false>(p, p4, s, ScratchSource::Pool, nullptr);
  *launched = e == cudaSuccess;
  return e;
}

template <typename Tin>
cudaError_t ckpt_pass(const FwdParams& p, cudaStream_t s, bool* launched) {
  if (p.dstate <= 4) return ckpt_pass_ns<4, Tin>(p, s, launched);
  if (p.dstate <= 8) return ckpt_pass_ns<8, Tin>(p, s, launched);
  return ckpt_pass_ns<16, Tin>(p, s, launched);
}

}  // namespace

cudaError_t launch_ckpt_pass(const FwdParams& p, selscan_dtype_t in_dtype, cudaStream_t s, bool* launched) {
  *launched = false;
  if (!p.ckpt || !p.ckpt_only || !rows_kernel_supports(p, in_dtype)) return cudaSuccess;
  return in_dtype == SELSCAN_F32 ? ckpt_pass<float>(p, s, launched) : ckpt_pass<__nv_bfloat16>(p, s, launched);
}

namespace {

// One CTA whose threads wait, with the bounded wait of the forward kernels, on an mbarrier phase that
// expects 16 bytes no copy will deliver (no copy is issued, so none is in flight when the waits give up).
__global__ void __launch_bounds__(32) selscan_wait_probe_kernel(long long polls, int* completed) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int s_abort;
  if (threadIdx.x == 0) {
    s_abort = 0;
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_expect_tx(&bar, 16);  // the phase's one arrival, with 16 bytes still to come
  __syncthreads();
  if (wait_or_abort_slow(&bar, 0, &s_abort, polls)) atomicAdd(completed, 1);
}

}  // namespace

cudaError_t probe_wait_timeout(long long polls, int* completed) {
  int* d = nullptr;
  cudaError_t e = cudaMalloc(&d, sizeof(int));
  if (e != cudaSuccess) return e;
  e = cudaMemset(d, 0, sizeof(int));
  if (e == cudaSuccess) {
    selscan_wait_probe_kernel<<<1, 32>>>(polls, d);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(completed, d, sizeof(int), cudaMemcpyDeviceToHost);
  cudaFree(d);
  return e;
}

cudaError_t read_rows_device_error(int* value, int reset) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_selscan_rows_error, sizeof(int));
  if (e == cudaSuccess && reset) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_selscan_rows_error, &zero, sizeof(int));
  }
  return e;
}

}  // namespace selscan

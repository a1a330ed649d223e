// Internal declarations shared by the libselscan CUDA sources (not part of the public ABI).
#pragma once

#include <cuda.h>  // CUtensorMap (declarations only: the library does not link libcuda)
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "selscan.h"

namespace selscan {

// Arguments of one selscan_fwd launch, already validated on the host.
struct FwdParams {
  int64_t batch, dim, seqlen;
  int dstate;
  const void* u;
  const void* delta;
  const void* z;  // nullable
  const void* B;
  const void* C;
  const float* A;
  const float* D;           // nullable
  const float* delta_bias;  // nullable
  const float* h0;          // nullable
  void* out;
  float* h_last;  // nullable
  int delta_softplus;
  int vec_in;   // u, delta, z rows may be read with 16-byte vectors
  int vec_out;  // out rows may be written with 16-byte vectors
  int vec_bc;   // B, C rows may be read with 16-byte vectors (and bulk-copied)
  int vec_stage;  // B, C and u, delta, z rows may all be bulk-copied
  int use_tma;    // set by a launcher: its kernel stages inputs with tensor copies
  // Time blocks of the sequential kernel (nblocks = 1: one pass over the whole sequence).  With
  // nblocks > 1 the sequence is cut into blocks of tblock steps (a multiple of 64): a summary pass
  // writes each block's zero-start end state and ΣΔ to `summ` ([nblocks-1][rows][N+1]), a carry pass
  // turns them into the start state of every block (`start`, [nblocks][rows][N]; block 0 starts
  // from h0), and the scan pass runs every block from its start state.
  int64_t tblock;
  int nblocks;
  float* summ;
  float* start;
  // Convolution front (selscan_fwd_conv): u = silu(conv_b + Σ_k conv_w[d,k]·x[t-3+k]); `u` then holds x.
  const float* conv_w;  // [D, 4]
  const float* conv_b;  // [D], nullable
  // Row-sequential kernel (selscan_rows.cu): consumer warps per CTA, pipeline stages, and the output
  // type (set by its launcher).
  int warps;
  int stages;
  int out_bf16;
  // Checkpoints (selscan_fwd_ckpt; nullable): the state before every 16-step chunk,
  // [rows][ckpt_chunks][16] fp32, written by the forward scan for the backward to rerun chunks from.
  float* ckpt;
  int64_t ckpt_chunks;
  // With ckpt: keep only the checkpoints (no out, h_last or gate): the backward's forward pass.
  int ckpt_only;
};

// Arguments of one selscan_step launch.
struct StepParams {
  int64_t batch, dim;
  int dstate;
  const void* u;
  const void* delta;
  const void* z;
  const void* B;
  const void* C;
  const float* A;
  const float* D;
  const float* delta_bias;
  float* state;
  void* out;
  int delta_softplus;
  int vec_state;  // state / A rows may be accessed as float4 (dstate % 4 == 0, 16-byte aligned)
  int vec_bc;     // B, C rows may be read four states at a time (bases aligned to 4 elements)
};

cudaError_t launch_fwd(const FwdParams& p, selscan_dtype_t in_dtype, selscan_dtype_t out_dtype, cudaStream_t s);

// Arguments of one selscan_bwd launch, already validated on the host.
struct BwdParams {
  int64_t batch, dim, seqlen;
  int dstate;
  const void* u;
  const void* delta;
  const void* z;  // nullable
  const void* B;
  const void* C;
  const float* A;
  const float* D;           // nullable
  const float* delta_bias;  // nullable
  const float* h0;          // nullable
  const void* dout;
  const float* dh_last;  // nullable
  void* du;
  void* ddelta;
  void* dz;  // required iff z is given
  float* dA;
  float* dB;
  float* dC;
  float* dD;           // nullable
  float* ddelta_bias;  // nullable
  float* dh0;          // nullable
  float* ckpt;         // the state at the start of every chunk, [rows][chunks][16]: in the workspace, or
  const float* ckpt_in;  // the forward's (selscan_fwd_ckpt; nullable), in which case phase 1 is skipped
  // Time blocks (nblocks > 1): blocks of tblock steps (a multiple of the chunk), their summaries
  // (zero-start end state and zero-end start gradient, [nblocks][rows][32]; ΣΔ, [nblocks][rows]) and
  // the carried start state and end gradient of every block ([nblocks][rows][16] each).
  int nblocks;
  int64_t tblock;
  float* summ;
  float* sumd;
  float* hstart;
  float* gend;
  int delta_softplus;
  int vec_in;    // u, delta, z may be read four steps at a time (8- or 16-byte loads)
  int vec_dout;  // dout may be read four steps at a time
  int vec_grad;  // du, ddelta, dz may be written four steps at a time (8- or 16-byte stores)
  int vec_dbc;   // dB, dC may take 16-byte atomic adds
};
// Bytes of the backward's workspace (chunk checkpoints, and the time blocks' summaries and carries when
// the problem has too few rows to fill the current device).
size_t bwd_workspace_bytes(int64_t batch, int64_t dim, int64_t seqlen, bool with_ckpt = true);
// The backward: zeroing of the accumulated gradients is the caller's; `workspace` (nullable: taken from
// the stream's memory pool) holds at least bwd_workspace_bytes.
cudaError_t launch_bwd(const BwdParams& p, selscan_dtype_t in_dtype, selscan_dtype_t dout_dtype, void* workspace,
                       cudaStream_t s);

// Tensor maps (2-D TMA descriptors) of one forward call: u, delta, z by rows of the CTA, B and C by the
// dstate rows of a batch entry.  Passed to the kernel as a __grid_constant__ parameter.
struct alignas(64) TmaMaps {
  CUtensorMap u, delta, z, B, C;
};
// cuTensorMapEncodeTiled, fetched through the runtime (nullptr if the driver does not provide it).
void* tensor_map_encoder();
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// A 2-D map of a row-major [rows][inner] tensor of Tin with box [box_rows][box_inner] (inner fastest).
// Boxes that reach past the tensor are zero-filled by the copy.
template <typename Tin>
inline bool encode_2d(EncodeTiled enc, CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                      uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * sizeof(Tin)};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = sizeof(Tin) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
cudaError_t launch_step(const StepParams& p, selscan_dtype_t in_dtype, selscan_dtype_t out_dtype, cudaStream_t s);
// The sequential forward kernel (rows-parallel, no scan) used by launch_fwd for many-row problems.
cudaError_t launch_fwd_seq(const FwdParams& p, selscan_dtype_t in_dtype, selscan_dtype_t out_dtype, cudaStream_t s);
// The sequential kernel in the reverse direction and/or with the exact zero-order-hold input matrix,
// or (conv) with the causal conv1d + SiLU front computing u from x.
cudaError_t launch_fwd_seq_ex(const FwdParams& p, selscan_dtype_t in_dtype, selscan_dtype_t out_dtype, bool reverse,
                              bool zoh, cudaStream_t s, bool conv = false);
// The sequential kernel with its time-block scratch in the library's fixed device array (no
// allocation).  Sets *too_big and enqueues nothing if the problem needs more than the array holds.
cudaError_t launch_fwd_seq_noalloc(const FwdParams& p, selscan_dtype_t in_dtype, selscan_dtype_t out_dtype,
                                   cudaStream_t s, bool* too_big);
// Kernels enqueued by the current entry-point call on this host thread (read by
// selscan_last_launch_count()); every launcher adds its launches.
void count_launches(int n);

// Read (and optionally clear) the device-side failure words set by a kernel's bounded wait.
cudaError_t read_device_error(int* value, int reset);
cudaError_t read_seq_device_error(int* value, int reset);
cudaError_t read_rows_device_error(int* value, int reset);
// Launch the bounded-wait probe (one CTA waiting on a phase that never completes, each wait giving up
// after `polls` polls) and synchronise; *completed = waits that saw the phase complete.
cudaError_t probe_wait_timeout(long long polls, int* completed);

// Where the time-block scratch of a forward call comes from: the CUDA memory pool of the call's stream
// (cudaMallocAsync / cudaFreeAsync), or the library's fixed device array (selscan_fwd_noalloc).
enum class ScratchSource { Pool, Fixed };
// Device address and size of the fixed array on the current device (looked up once per device).
cudaError_t fixed_scratch(float** ptr, size_t* bytes);

// Options of the row-sequential forward kernel (selscan_rows.cu).
struct RowsOptions {
  bool reverse = false;
  bool zoh = false;
  bool conv = false;
  ScratchSource scratch = ScratchSource::Pool;
};
// True when the row-sequential kernel can run the call: every input row 16-byte aligned for tensor
// copies (vec_stage) and sizes whose copy coordinates fit in 32 bits.
bool rows_kernel_supports(const FwdParams& p, selscan_dtype_t in_dtype);
// The row-sequential forward (time blocks chosen by the launcher).  With ScratchSource::Fixed it sets
// *too_big and enqueues nothing when the time blocks need more than the fixed array holds.
cudaError_t launch_fwd_rows(const FwdParams& p, selscan_dtype_t in_dtype, selscan_dtype_t out_dtype,
                            const RowsOptions& o, cudaStream_t s, bool* too_big);
// The backward's forward pass by the row-sequential kernel: only the checkpoints p.ckpt (p.ckpt_only set),
// in one pass over the sequence.  *launched is false, with nothing enqueued, when the rows cannot be staged
// by tensor copies or would need time blocks; the caller then forms the checkpoints itself.
cudaError_t launch_ckpt_pass(const FwdParams& p, selscan_dtype_t in_dtype, cudaStream_t s, bool* launched);

// ---------------------------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------------------------

constexpr float kLog2e = 1.4426950408889634f;

// 2^x on the special-function unit (approximate, flushes subnormal results to zero).
__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// softplus(x) = log(1 + e^x).  Above 20 the result equals x to within 2.1e-9 absolute.
__device__ __forceinline__ float softplus_f(float x) { return x > 20.f ? x : log1pf(__expf(x)); }

// silu(z) = z / (1 + e^{-z}); for z below about -88 the quotient underflows to -0.
__device__ __forceinline__ float silu_f(float z) { return __fdividef(z, 1.f + __expf(-z)); }

// ---- helpers shared by the forward kernels -------------------------------------------------------

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLn2 = 0.6931471805599453f;
// Polls of an mbarrier phase before a copy is declared lost.  Each mbarrier.try_wait that finds the phase
// incomplete suspends the thread for about 3.9 us on B300 (measured with selscan_probe_wait_timeout), so
// 2^18 polls give up after about one second, far beyond any copy's latency.
constexpr long long kWaitLimit = 1ll << 18;
// Idle rounds of a producer warp (a non-blocking test of its events and a 64 ns pause each, about
// 0.2 us) before it declares its pipeline stuck: also about one second.
constexpr long long kIdleLimit = 1ll << 22;

__device__ __forceinline__ float lg2_approx(float x) {
  float r;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// softplus(x) = max(x, 0) + log1p(e), e = exp(-|x|) ∈ (0, 1].
// For e ≥ 1/16, log1p(e) = log2(1 + e)·ln 2 on the special-function unit: 1 + e ≥ 1.0625 keeps the
// absolute error of lg2 small next to the result.  For e < 1/16 the Taylor series
// log1p(e) = e - e²/2 + e³/3 - e⁴/4 + ..., truncated after e⁴, errs by less than e⁵/5 ≤ 2e-7·e.
__device__ __forceinline__ float softplus_fast(float x) {
  const float e = ex2_approx(-fabsf(x) * kLog2e);
  const float big = lg2_approx(1.f + e) * kLn2;
  const float small = e * fmaf(e, fmaf(e, fmaf(e, -0.25f, 0.33333334f), -0.5f), 1.f);
  return fmaxf(x, 0.f) + (e >= 0.0625f ? big : small);
}

// silu(z) = z / (1 + e^{-z}); the reciprocal of +inf is 0, so very negative z gives -0.
__device__ __forceinline__ float silu_fast(float z) { return z * rcp_approx(1.f + ex2_approx(-z * kLog2e)); }

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// Element-wise fp32 arithmetic on float2 pairs as packed fp32x2 instructions (one instruction for two
// independent operations).
__device__ __forceinline__ float2 fma2s(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 mul2s(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 add2s(float2 a, float2 b) { return __fadd2_rn(a, b); }

// softplus(x) and its derivative σ(x) from one exponential: with e = exp(-|x|), softplus = max(x, 0) +
// log(1 + e) (as softplus_fast evaluates it) and σ(x) = 1/(1 + e) for x ≥ 0, e/(1 + e) for x < 0.
__device__ __forceinline__ void softplus_sigmoid(float x, float& sp, float& sg) {
  const float e = ex2_approx(-fabsf(x) * kLog2e);
  const float big = lg2_approx(1.f + e) * kLn2;
  const float small = e * fmaf(e, fmaf(e, fmaf(e, -0.25f, 0.33333334f), -0.5f), 1.f);
  sp = fmaxf(x, 0.f) + (e >= 0.0625f ? big : small);
  sg = (x >= 0.f ? 1.f : e) * rcp_approx(1.f + e);
}

// The input factor of a state pair at one step: Δu (B̄ = Δ·B), or with ZOH u·(Ā - 1)/A where
// |ΔA| >= 1/16 and Δu·φ(ΔA) below, φ(x) = (e^x - 1)/x = 1 + x/2 + x²/6 + x³/24 + ... truncated after x³
// (error below x⁴/120 < 1.3e-7 relative there, where Ā - 1 would lose its leading digits; at A = 0 it
// gives Δu, the limit).  The series is evaluated in the exponent e = x·log2 e itself, its coefficients
// scaled by powers of ln 2.  e: Δ·A·log2 e of the pair; a: its Ā; uia: u·(1/A) of the pair.
__device__ __forceinline__ float2 zoh_factor2(float2 du, float2 e, float2 a, float2 uia) {
  constexpr float c1 = kLn2 / 2.f, c2 = kLn2 * kLn2 / 6.f, c3 = kLn2 * kLn2 * kLn2 / 24.f;
  constexpr float kSmall = 0.0625f / kLn2;  // |ΔA| < 1/16 in units of e
  float2 phi = fma2s(e, f2(c3, c3), f2(c2, c2));
  phi = fma2s(e, phi, f2(c1, c1));
  phi = fma2s(e, phi, f2(1.f, 1.f));
  const float2 small = mul2s(du, phi);
  const float2 big = mul2s(add2s(a, f2(-1.f, -1.f)), uia);
  return f2(fabsf(e.x) < kSmall ? small.x : big.x, fabsf(e.y) < kSmall ? small.y : big.y);
}

// ---- raw lane segments: the 2H inputs of one lane, as 16-byte vectors per half -------------------
// Elements are unpacked with shifts and masks on 32-bit words (a bf16 is the top half of an fp32),
// never through a local array, so everything stays in registers.

__device__ __forceinline__ uint32_t word(const uint4& v, int w) {
  return w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w;
}
__device__ __forceinline__ float elem_of(const uint4& v, int k, float) { return __uint_as_float(word(v, k)); }
__device__ __forceinline__ float elem_of(const uint4& v, int k, __nv_bfloat16) {
  const uint32_t w = word(v, k >> 1);
  return __uint_as_float((k & 1) ? (w & 0xffff0000u) : (w << 16));
}
__device__ __forceinline__ uint32_t raw_bits(const float* p, int64_t i) { return __float_as_uint(p[i]); }
__device__ __forceinline__ uint32_t raw_bits(const __nv_bfloat16* p, int64_t i) {
  return reinterpret_cast<const unsigned short*>(p)[i];
}
__device__ __forceinline__ uint32_t out_bits(float v, float) { return __float_as_uint(v); }
__device__ __forceinline__ uint32_t out_bits(float v, __nv_bfloat16) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

template <typename T, int H>
struct Seg {
  static constexpr int kPerVec = 16 / sizeof(T);
  static constexpr int kVecs = H / kPerVec;
  static_assert(H % kPerVec == 0, "a half-segment must be whole 16-byte vectors");
  uint4 v[2][kVecs];
  __device__ __forceinline__ float get(int half, int i) const { return elem_of(v[half][i / kPerVec], i % kPerVec, T()); }
};

// Load steps [t, t+2H) of a row (length L) as two halves.  Steps at or past L read as 0.
template <typename T, int H>
__device__ __forceinline__ void load_seg(Seg<T, H>& s, const T* __restrict__ row, int64_t t, int64_t L, bool vec) {
  constexpr int kPerVec = Seg<T, H>::kPerVec;
  if (vec && t + 2 * H <= L) {
#pragma unroll
    for (int h = 0; h < 2; h++)
#pragma unroll
      for (int q = 0; q < Seg<T, H>::kVecs; q++)
        s.v[h][q] = __ldg(reinterpret_cast<const uint4*>(row + t + h * H) + q);
  } else {
#pragma unroll
    for (int h = 0; h < 2; h++)
#pragma unroll
      for (int q = 0; q < Seg<T, H>::kVecs; q++) {
        uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int k = 0; k < kPerVec; k++) {
          const int64_t tt = t + h * H + q * kPerVec + k;
          const uint32_t bits = tt < L ? raw_bits(row, tt) : 0u;
          if (sizeof(T) == 4) w[k] = bits;
          else w[k >> 1] |= (k & 1) ? (bits << 16) : bits;
        }
        s.v[h][q] = make_uint4(w[0], w[1], w[2], w[3]);
      }
  }
}

template <typename T, int H>
__device__ __forceinline__ void store_seg(T* __restrict__ row, int64_t t, int64_t L, bool vec, const float2 (&y)[H]) {
  constexpr int kPerVec = 16 / sizeof(T);
#pragma unroll
  for (int h = 0; h < 2; h++) {
    if (vec && t + 2 * H <= L) {
#pragma unroll
      for (int q = 0; q < H / kPerVec; q++) {
        uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int k = 0; k < kPerVec; k++) {
          const float2 v = y[q * kPerVec + k];
          const uint32_t bits = out_bits(h ? v.y : v.x, T());
          if (sizeof(T) == 4) w[k] = bits;
          else w[k >> 1] |= (k & 1) ? (bits << 16) : bits;
        }
        reinterpret_cast<uint4*>(row + t + h * H)[q] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < H; i++) {
        const int64_t tt = t + h * H + i;
        if (tt < L) row[tt] = from_f32<T>(h ? y[i].y : y[i].x);
      }
    }
  }
}

// ---- mbarrier / bulk-copy primitives ------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false if the phase did not complete within kWaitLimit polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (long long i = 0; i < kWaitLimit; i++)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
// 2-D tiled copy of the box at (x, y) (x: innermost coordinate, in elements) of a tensor map.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}


}  // namespace selscan

// Selective-scan forward for problems with many (batch, channel) rows: sequential in t, no scan.
//
// Same computation as the chunked kernel in selscan_fwd.cu (see include/selscan.h): per row (b, d)
// and state n, Δ_t = softplus(δ_t + Δ_bias[d]), h_t = exp(Δ_t A[d,n]) h_{t-1} + Δ_t B[b,n,t] u_t,
// y_t = Σ_n C[b,n,t] h_t + D[d] u_t, out_t = y_t silu(z_t)  ("Mamba状态空间模型深度解析" §2.1, §3.1;
// "Mamba架构与SSM模型：高效序列建模技术解析" §2.1, §2.2).  This is the recurrent form run directly:
// every lane walks its row from t = 0 to L-1, so no step is computed twice and no lanes have to be
// joined by a scan.  The parallelism comes from the rows: Q lanes share a row, each owning
// SPL = NS/Q of its states (Q = 2 for 16 states), and a warp holds 32/Q rows.
//
// Per step and lane, the states are taken in pairs (n, n+1) as float2:
//   Ā = 2^(Δ·(A_n, A_n+1)·log2 e),  h = Ā ⊙ h + Δu·(B_n, B_n+1),  y2 += (C_n, C_n+1) ⊙ h
// so the only dependency from one step to the next is one packed FMA per state pair; the
// exponentials of later steps are independent of the state and overlap with it.  The Q partial sums
// of y meet with a shuffle.
//
// Every input of a chunk of T steps is fetched by the tensor memory accelerator one chunk ahead (1-D
// bulk copies, one per row): the CTA's rows of u, δ and z, and the raw [n][t] rows of B and C.  B and C
// are then transposed once per CTA into a [t][n] fp32 tile, so that the B (or C) values of one step
// and one lane's states are one 128-bit shared load that every lane of a quarter-warp reads at the
// same address (a broadcast).  The u, δ, z rows are stored with a 16-byte pad per row so that the
// rows read by one quarter-warp fall in different bank groups.
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "selscan_internal.cuh"

namespace selscan {

// Set by a kernel whose bounded wait on a bulk copy gave up (read by selscan_device_status()).
__device__ int g_selscan_seq_error = 0;

namespace {

// Steps per chunk (32 or 64).  32 halves the shared memory of a CTA, so that 16 warps fit on an SM
// (measured faster on B300 for 1536 and 20480 rows of 16 states).
#ifndef SELSCAN_SEQ_T
#define SELSCAN_SEQ_T 32
#endif

template <int NS, int Q, int R, typename Tin>
struct SeqCfg {
  static constexpr int SPL = NS / Q;  // states per lane
  static constexpr int PAIRS = SPL / 2;
  static constexpr int RPW = 32 / Q;    // rows per warp
  static constexpr int ROWS = R * RPW;  // rows per CTA
  static constexpr int T = SELSCAN_SEQ_T;  // steps per chunk
  static constexpr int SB = 8;             // steps per sub-block
  static constexpr int TS = NS + 4;        // floats per step in the tile (padded: transposing stores spread over banks)
  // Stage rows of RB bytes (128, or 64 for 32 bf16 steps), written with the swizzle of that width.
  static constexpr int RB = T * static_cast<int>(sizeof(Tin)) < 128 ? T * static_cast<int>(sizeof(Tin)) : 128;
  static constexpr int EPR = RB / static_cast<int>(sizeof(Tin));  // inputs per stage row
  static constexpr int SUBT = T / EPR;                            // stage sub-tiles per tensor and chunk
  static constexpr CUtensorMapSwizzle kSwizzle = RB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  static constexpr int UDZ = 3 * T * ROWS;  // elements of one u, δ, z stage: [3][SUBT][ROWS][EPR]
  static constexpr int RAW = 2 * NS * T;    // raw elements of one chunk: B rows then C rows, [2][NS][T]
  static constexpr int TILE = 2 * T * TS;   // floats of one transposed tile: [2][T][TS]
  static constexpr size_t kUdzBytes = 2 * UDZ * sizeof(Tin);       // double-buffered
  static constexpr size_t kRawBytes = 2 * RAW * sizeof(Tin);       // double-buffered
  static constexpr size_t kTileBytes = 2 * TILE * sizeof(float);  // double-buffered
  // + 1 KiB so that the stage can start on a 1 KiB boundary (the 128-byte swizzle pattern repeats
  // every 8 rows of 128 bytes and is computed from the address).
  static constexpr size_t kSmem = 1024 + kUdzBytes + kRawBytes + kTileBytes + 2 * sizeof(uint64_t);
  static_assert(SPL >= 4 && SPL % 4 == 0, "each lane owns whole groups of 4 states");
  static_assert(RB == 128 || RB == 64, "stage rows of 64 or 128 bytes");
  static_assert((ROWS * RB) % 1024 == 0, "stage sub-tiles must keep 1 KiB alignment");
};

// 8 consecutive inputs of a row as 16-byte vectors.
template <typename T>
struct Vec8 {
  static constexpr int kPerVec = 16 / sizeof(T);
  static constexpr int kVecs = 8 / kPerVec;
  uint4 v[kVecs];
  __device__ __forceinline__ float get(int i) const { return elem_of(v[i / kPerVec], i % kPerVec, T()); }
};

template <typename T>
__device__ __forceinline__ void load8(Vec8<T>& s, const T* __restrict__ row, int64_t t, int64_t L, bool vec) {
  constexpr int kPerVec = Vec8<T>::kPerVec;
  if (vec && t + 8 <= L) {
#pragma unroll
    for (int q = 0; q < Vec8<T>::kVecs; q++) s.v[q] = __ldg(reinterpret_cast<const uint4*>(row + t) + q);
  } else {
#pragma unroll
    for (int q = 0; q < Vec8<T>::kVecs; q++) {
      uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int k = 0; k < kPerVec; k++) {
        const int64_t tt = t + q * kPerVec + k;
        const uint32_t bits = tt < L ? raw_bits(row, tt) : 0u;
        if (sizeof(T) == 4) w[k] = bits;
        else w[k >> 1] |= (k & 1) ? (bits << 16) : bits;
      }
      s.v[q] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

template <typename T>
__device__ __forceinline__ void store8(T* __restrict__ row, int64_t t, int64_t L, bool vec, const float (&y)[8]) {
  constexpr int kPerVec = 16 / sizeof(T);
  if (vec && t + 8 <= L) {
#pragma unroll
    for (int q = 0; q < 8 / kPerVec; q++) {
      uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int k = 0; k < kPerVec; k++) {
        const uint32_t bits = out_bits(y[q * kPerVec + k], T());
        if (sizeof(T) == 4) w[k] = bits;
        else w[k >> 1] |= (k & 1) ? (bits << 16) : bits;
      }
      reinterpret_cast<uint4*>(row + t)[q] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; i++)
      if (t + i < L) row[t + i] = from_f32<T>(y[i]);
  }
}

// 4 consecutive outputs [t, t+4) of a row (one 16-byte store for fp32, 8-byte for bf16).
template <typename T>
__device__ __forceinline__ void store4(T* __restrict__ row, int64_t t, int64_t L, bool vec, const float (&y)[4]) {
  if (vec && t + 4 <= L) {
    if (sizeof(T) == 4) {
      *reinterpret_cast<uint4*>(row + t) =
          make_uint4(out_bits(y[0], T()), out_bits(y[1], T()), out_bits(y[2], T()), out_bits(y[3], T()));
    } else {
      *reinterpret_cast<uint2*>(row + t) = make_uint2(out_bits(y[0], T()) | (out_bits(y[1], T()) << 16),
                                                      out_bits(y[2], T()) | (out_bits(y[3], T()) << 16));
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; i++)
      if (t + i < L) row[t + i] = from_f32<T>(y[i]);
  }
}

// 8 consecutive staged inputs [t, t+8) of CTA row r from a tensor's stage [SUBT][ROWS][RB bytes],
// written by a 2-D tensor copy with the RB-byte swizzle: 16-byte chunk c of stage row r sits at chunk
// position c ^ (r mod 8) for 128-byte rows, c ^ ((r / 2) mod 4) for 64-byte rows (each sub-tile starts
// on a 1 KiB boundary).  Steps past the end of the sequence were zero-filled by the copy.
template <typename T, int ROWS, int RB>
__device__ __forceinline__ void stage8(Vec8<T>& s, const unsigned char* __restrict__ stage, int r, int t) {
  constexpr int kPerVec = Vec8<T>::kPerVec, EPR = RB / static_cast<int>(sizeof(T));
  const int swz = RB == 128 ? (r & 7) : ((r >> 1) & 3);
#pragma unroll
  for (int q = 0; q < Vec8<T>::kVecs; q++) {
    const int e = t + q * kPerVec;
    const int sub = e / EPR, chunk = (e % EPR) / kPerVec;
    s.v[q] = *reinterpret_cast<const uint4*>(stage + (sub * ROWS + r) * RB + ((chunk ^ swz) << 4));
  }
}

// Transpose raw chunk rows [2][NS][T] (Tin) into the tile [2][T][TS] (fp32), zeroing states >= N and
// steps >= L.  Work unit: one tensor, 4 states, 4 steps (steps fastest across threads).
template <int NS, int Q, int R, typename Tin, bool MASK, int NT = 2>
__device__ __forceinline__ void transpose_chunk(const Tin* __restrict__ rb, float* __restrict__ tb, int tid,
                                                int64_t t0, int64_t L, int N) {
  using C = SeqCfg<NS, Q, R, Tin>;
  constexpr int T4 = C::T / 4, N4 = NS / 4, UNITS = NT * N4 * T4;  // NT = 1: B only
  for (int unit = tid; unit < UNITS; unit += R * 32) {
    const int t4 = unit % T4, rest = unit / T4;
    const int n4 = rest % N4, tt = rest / N4;
    float v[4][4];  // [state k][step m]
#pragma unroll
    for (int k = 0; k < 4; k++) {
      const Tin* src = rb + (tt * NS + n4 * 4 + k) * C::T + t4 * 4;
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
      if (MASK) {
#pragma unroll
        for (int m = 0; m < 4; m++)
          if (n4 * 4 + k >= N || t0 + t4 * 4 + m >= L) v[k][m] = 0.f;
      }
    }
#pragma unroll
    for (int m = 0; m < 4; m++)
      *reinterpret_cast<float4*>(tb + tt * C::T * C::TS + (t4 * 4 + m) * C::TS + n4 * 4) =
          make_float4(v[0][m], v[1][m], v[2][m], v[3][m]);
  }
}

#ifndef SELSCAN_SEQ_WARPS_PER_SM
#define SELSCAN_SEQ_WARPS_PER_SM 16
#endif

// The input-matrix factor of one state pair: Δ·u (the plain discretisation B̄ = Δ·B), or with ZOH the
// exact zero-order hold B̄ = (exp(ΔA) - 1)/A · B ("Mamba架构与SSM模型：高效序列建模技术解析" §2.1, for
// a diagonal A): u·(Ā - 1)/A where |ΔA| >= 1/16, and Δu·φ(ΔA) with the series
// φ(x) = (e^x - 1)/x = 1 + x/2 + x²/6 + x³/24 + x⁴/120 below (truncation error < 1.3e-9 there, where
// Ā - 1 would lose its leading digits).  At A = 0 the series gives Δu, the limit of the exact form.
template <bool ZOH>
__device__ __forceinline__ float2 input_factor(float2 du, float2 e, float2 ab, float2 inv_a, float uu) {
  if (!ZOH) return du;
  const float2 x = mul2s(e, f2(kLn2, kLn2));  // ΔA
  float2 phi = fma2s(x, f2(1.f / 120.f, 1.f / 120.f), f2(1.f / 24.f, 1.f / 24.f));
  phi = fma2s(x, phi, f2(1.f / 6.f, 1.f / 6.f));
  phi = fma2s(x, phi, f2(0.5f, 0.5f));
  phi = fma2s(x, phi, f2(1.f, 1.f));
  const float2 small = mul2s(du, phi);
  const float2 big = mul2s(add2s(ab, f2(-1.f, -1.f)), mul2s(inv_a, f2(uu, uu)));
  return f2(fabsf(x.x) < 0.0625f ? small.x : big.x, fabsf(x.y) < 0.0625f ? small.y : big.y);
}

// SUMMARY: the summary pass of a time-blocked run (no C, y, z or out; writes the block's
// zero-start end state and ΣΔ).  Otherwise the scan: time block blockIdx.z of the sequence, from h0
// (the first block in scan order) or from its start state.
// REV: the scan runs from t = L-1 down to 0 (the reverse direction of a bidirectional layer): chunks,
// sub-blocks and steps are taken in reverse order and h_last is the state after t = 0.  Time-block
// summaries then describe each block scanned backwards, for blocks 1 .. nblocks-1.
// ZOH: exact zero-order-hold input matrix (input_factor).
// CONV: the input u is computed in the kernel from x (passed as `u`) by the block's convolution front,
// u_t = silu(conv_b + Σ_{k<4} conv_w[k]·x_{t-3+k}) with x = 0 before t = 0 ("Mamba架构与SSM模型：
// 高效序列建模技术解析" §3.2, d_conv = 4; "Mamba状态空间模型深度解析" §3.1, convolution and SiLU
// before the SSM).  Each lane keeps the last three x of its row in registers; a time block reads
// the three before its first step from memory.  Forward direction only.
template <int NS, int Q, int R, typename Tin, typename Tout, bool FULLN, bool SOFTPLUS, bool SUMMARY, bool REV = false,
          bool ZOH = false, bool CONV = false>
__global__ void __launch_bounds__(R * 32, SELSCAN_SEQ_WARPS_PER_SM / R)
    selscan_fwd_seq_kernel(const FwdParams p, const __grid_constant__ TmaMaps maps) {
  static_assert(!(CONV && REV), "the convolution front is causal: forward direction only");
  using C = SeqCfg<NS, Q, R, Tin>;
  constexpr int T = C::T, SB = C::SB, TS = C::TS, SPL = C::SPL, PAIRS = C::PAIRS, RPW = C::RPW;
  extern __shared__ __align__(128) unsigned char smem_dyn[];
  // (Offsetting the shared pointer itself keeps every derived pointer in the shared window, so the
  // tile reads compile to shared loads rather than generic ones.)
  unsigned char* smem_base = smem_dyn + ((1024u - (smem_addr(smem_dyn) & 1023u)) & 1023u);
  unsigned char* udz = smem_base;                                           // [2 buffers][3][SUBT][ROWS][EPR]
  Tin* raw = reinterpret_cast<Tin*>(smem_base + C::kUdzBytes);              // [2 buffers][2][NS][T]
  float* tiles = reinterpret_cast<float*>(smem_base + C::kUdzBytes + C::kRawBytes);  // [2 buffers][2][T][TS]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_base + C::kUdzBytes + C::kRawBytes + C::kTileBytes);
  __shared__ int s_abort;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int q = lane / RPW;  // state group: states [q·SPL, (q+1)·SPL)
  const int rw = lane % RPW;
  const int64_t b = blockIdx.y;
  const int64_t d = static_cast<int64_t>(blockIdx.x) * C::ROWS + (tid >> 5) * RPW + rw;
  const bool row_ok = d < p.dim;
  const int N = FULLN ? NS : p.dstate;
  const int64_t L = p.seqlen;
  const int kslot = blockIdx.z;  // summary slot (summary pass) or time block (scan)
  const int kblk = (SUMMARY && REV) ? kslot + 1 : kslot;  // time block: steps [tbeg, tend)
  const int64_t tbeg = static_cast<int64_t>(kblk) * p.tblock;
  const int64_t tend = (tbeg + p.tblock) < L ? (tbeg + p.tblock) : L;
  const int64_t c_begin = tbeg / T;               // tblock is a multiple of T
  const int64_t nchunks = (tend - tbeg + T - 1) / T;
  const int64_t grow = b * p.dim + d;             // global row of this lane
  const int64_t rows_total = p.batch * p.dim;
  const Tin* __restrict__ Bsrc = static_cast<const Tin*>(p.B) + b * N * L;
  const Tin* __restrict__ Csrc = static_cast<const Tin*>(p.C) + b * N * L;
  const bool tma = p.use_tma;

  // Issue the five 2-D tensor copies of chunk c into buffer c & 1 (one thread): the B and C rows of
  // batch entry b, and the CTA's rows of u, δ, z.  Parts of a box past the end of a tensor are
  // zero-filled and still count towards the expected bytes.
  const int row0 = static_cast<int>(b * p.dim + static_cast<int64_t>(blockIdx.x) * C::ROWS);
  const int ntens = SUMMARY ? 2 : (p.z ? 3 : 2);  // u, δ (, z)
  // ci: chunk index within the time block in scan order (selects the buffer and the barrier phase).
  auto chunk_of = [&](int64_t ci) { return REV ? c_begin + nchunks - 1 - ci : c_begin + ci; };
  auto issue = [&](int64_t ci) {
    const int t0 = static_cast<int>(chunk_of(ci) * T);
    uint64_t* bar = &bars[ci & 1];
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_expect_tx(bar, static_cast<uint32_t>(((SUMMARY ? 1 : 2) * NS + ntens * C::ROWS) * T * sizeof(Tin)));
    Tin* dst = raw + (ci & 1) * C::RAW;
    tma_load_2d(dst, &maps.B, t0, static_cast<int>(b * N), bar);
    if (!SUMMARY) tma_load_2d(dst + NS * T, &maps.C, t0, static_cast<int>(b * N), bar);
    unsigned char* st = udz + (ci & 1) * (C::UDZ * sizeof(Tin));
    const CUtensorMap* m[3] = {&maps.u, &maps.delta, &maps.z};
    for (int k = 0; k < ntens; k++)
      for (int sub = 0; sub < C::SUBT; sub++)
        tma_load_2d(st + (k * C::SUBT + sub) * C::ROWS * C::RB, m[k], t0 + sub * C::EPR, row0, bar);
  };

  if (tid == 0) {
    s_abort = 0;
    if (tma) {
      mbar_init(&bars[0], 1);
      mbar_init(&bars[1], 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
  }
  __syncthreads();
  if (tma && tid == 0 && nchunks > 0) issue(0);

  // This lane's states, in pairs: state n0 + 2i and n0 + 2i + 1.
  const int n0 = q * SPL;
  float2 A2[PAIRS], h[PAIRS], IA[PAIRS];
#pragma unroll
  for (int i = 0; i < PAIRS; i++) {
    float a[2], hh[2];
#pragma unroll
    for (int k = 0; k < 2; k++) {
      const int n = n0 + 2 * i + k;
      const bool ok = row_ok && n < N;
      a[k] = ok ? p.A[d * N + n] * kLog2e : 0.f;
      if (SUMMARY)
        hh[k] = 0.f;
      else if (p.nblocks > 1)  // every block's start state, the first one's copied from h0 by the carry pass
        hh[k] = ok ? p.start[(kblk * rows_total + grow) * N + n] : 0.f;
      else
        hh[k] = (ok && p.h0) ? p.h0[grow * N + n] : 0.f;
    }
    A2[i] = f2(a[0], a[1]);
    h[i] = f2(hh[0], hh[1]);
    // 1/A for the zero-order-hold factor (inf at A = 0, where the series branch is taken).
    IA[i] = ZOH ? f2(kLog2e / a[0], kLog2e / a[1]) : f2(0.f, 0.f);
  }
  const float bias = (row_ok && p.delta_bias) ? p.delta_bias[d] : 0.f;
  const float Dd = (row_ok && p.D) ? p.D[d] : 0.f;
  // Rows past `dim` (tail of the last CTA) run on row 0's inputs so that every lane takes part in
  // the shuffles; only their stores are skipped.
  const int64_t row_off = (b * p.dim + (row_ok ? d : 0)) * L;
  const Tin* __restrict__ u_row = static_cast<const Tin*>(p.u) + row_off;
  const Tin* __restrict__ dl_row = static_cast<const Tin*>(p.delta) + row_off;
  const Tin* __restrict__ z_row = p.z ? static_cast<const Tin*>(p.z) + row_off : nullptr;
  Tout* __restrict__ o_row = static_cast<Tout*>(p.out) + row_off;
  const bool vec = p.vec_in && p.vec_out;
  // Convolution front: taps, bias and the x history (x_{t-3}, x_{t-2}, x_{t-1}) before the block.
  float cw0 = 0.f, cw1 = 0.f, cw2 = 0.f, cw3 = 0.f, cbias = 0.f, xm3 = 0.f, xm2 = 0.f, xm1 = 0.f;
  if (CONV) {
    const int64_t dd = row_ok ? d : 0;
    cw0 = p.conv_w[dd * 4 + 0];
    cw1 = p.conv_w[dd * 4 + 1];
    cw2 = p.conv_w[dd * 4 + 2];
    cw3 = p.conv_w[dd * 4 + 3];
    cbias = p.conv_b ? p.conv_b[dd] : 0.f;
    xm3 = tbeg >= 3 ? to_f32(u_row[tbeg - 3]) : 0.f;
    xm2 = tbeg >= 2 ? to_f32(u_row[tbeg - 2]) : 0.f;
    xm1 = tbeg >= 1 ? to_f32(u_row[tbeg - 1]) : 0.f;
  }

  float S = 0.f;  // Σ Δ over the block (summary pass)
  int64_t c = 0;  // chunk index within the time block
  for (; c < nchunks; c++) {
    const int64_t t0 = chunk_of(c) * T;
    const Tin* rb = raw + (c & 1) * C::RAW;
    float* tb = tiles + (c & 1) * C::TILE;
    const bool tail = t0 + T > L;
    if (tma) {
      if (!mbar_wait(&bars[c & 1], static_cast<uint32_t>((c >> 1) & 1))) s_abort = 1;
    } else {
      Tin* wb = raw + (c & 1) * C::RAW;
      for (int e = tid; e < C::RAW; e += R * 32) {
        const int rowi = e / T, tt = e - rowi * T;
        const int n = rowi < NS ? rowi : rowi - NS;
        const Tin* srcp = rowi < NS ? Bsrc : Csrc;
        wb[e] = (n < N && t0 + tt < L) ? srcp[n * L + t0 + tt] : from_f32<Tin>(0.f);
      }
      __syncthreads();
    }
    if (FULLN && !tail)
      transpose_chunk<NS, Q, R, Tin, false, SUMMARY ? 1 : 2>(rb, tb, tid, t0, L, N);
    else
      transpose_chunk<NS, Q, R, Tin, true, SUMMARY ? 1 : 2>(rb, tb, tid, t0, L, N);
    __syncthreads();  // tile c complete; every warp has finished chunk c-1
    if (s_abort) break;
    if (tma && tid == 0 && c + 1 < nchunks) issue(c + 1);

    const float* tB = tb + n0;
    const float* tC = tb + T * TS + n0;
    // This lane's row of the staged u, δ, z (rows past `dim` hold zeros or the next batch entry's
    // rows: computed on, never stored).
    const int r_cta = (tid >> 5) * RPW + rw;
    const unsigned char* su = udz + (c & 1) * (C::UDZ * sizeof(Tin));
    const unsigned char* sd = su + C::SUBT * C::ROWS * C::RB;
    const unsigned char* sz = sd + C::SUBT * C::ROWS * C::RB;
#pragma unroll 1
    for (int sbi = 0; sbi < T; sbi += SB) {
      const int sb = REV ? T - SB - sbi : sbi;
      const int64_t ts = t0 + sb;
      if (ts >= L) {
        if (REV) continue;  // sub-blocks past the end come first in reverse order
        break;
      }
      const bool full = !tail || ts + SB <= L;
      float dl[SB], du[SB], y[SB];
      float uval[SB];  // this sub-block's u (the D skip is added after the state loop)
      {
        Vec8<Tin> us, ds;
        if (tma) {
          stage8<Tin, C::ROWS, C::RB>(us, su, r_cta, sb);
          stage8<Tin, C::ROWS, C::RB>(ds, sd, r_cta, sb);
        } else {
          load8<Tin>(us, u_row, ts, L, vec && full);
          load8<Tin>(ds, dl_row, ts, L, vec && full);
        }
        if constexpr (CONV) {
          float xv[SB], a[SB];
#pragma unroll
          for (int i = 0; i < SB; i++) xv[i] = us.get(i);
#pragma unroll
          for (int i = 0; i < SB; i++) {
            const float x3 = i >= 3 ? xv[i - 3] : (i == 0 ? xm3 : (i == 1 ? xm2 : xm1));
            const float x2 = i >= 2 ? xv[i - 2] : (i == 0 ? xm2 : xm1);
            const float x1 = i >= 1 ? xv[i - 1] : xm1;
            a[i] = fmaf(cw3, xv[i], fmaf(cw2, x1, fmaf(cw1, x2, fmaf(cw0, x3, cbias))));
          }
          xm3 = xv[SB - 3];
          xm2 = xv[SB - 2];
          xm1 = xv[SB - 1];
          if constexpr (Q == 2) {
            // Each lane of the row applies SiLU to one half of the steps and the halves are swapped.
            constexpr int HB = SB / 2;
            float mine[HB], other[HB];
#pragma unroll
            for (int m = 0; m < HB; m++) mine[m] = silu_fast(q ? a[HB + m] : a[m]);
#pragma unroll
            for (int m = 0; m < HB; m++) other[m] = __shfl_xor_sync(kFull, mine[m], RPW);
#pragma unroll
            for (int i = 0; i < SB; i++) uval[i] = ((i < HB) == (q == 0)) ? mine[i % HB] : other[i % HB];
          } else {
#pragma unroll
            for (int i = 0; i < SB; i++) uval[i] = silu_fast(a[i]);
          }
        } else {
#pragma unroll
          for (int i = 0; i < SB; i++) uval[i] = us.get(i);
        }
        if constexpr (Q == 2) {
          // The row's two lanes each compute Δ for one half of the 8 steps (lane q: steps
          // [4q, 4q + 4)) and swap halves with a shuffle, so no softplus is computed twice.
          constexpr int HB = SB / 2;
          float mine[HB], other[HB];
#pragma unroll
          for (int m = 0; m < HB; m++) {
            const float x = (q ? ds.get(HB + m) : ds.get(m)) + bias;
            const float delta = SOFTPLUS ? softplus_fast(x) : x;
            mine[m] = (full || ts + q * HB + m < L) ? delta : 0.f;  // identity steps past the end
            if (SUMMARY) S += mine[m];
          }
#pragma unroll
          for (int m = 0; m < HB; m++) other[m] = __shfl_xor_sync(kFull, mine[m], RPW);
#pragma unroll
          for (int i = 0; i < SB; i++) {
            const int m = i % HB;
            dl[i] = ((i < HB) == (q == 0)) ? mine[m] : other[m];
            du[i] = dl[i] * uval[i];
          }
        } else {
          // Straight-line over the 8 steps (no branches), so their exponential/log chains overlap.
#pragma unroll
          for (int i = 0; i < SB; i++) {
            const float x = ds.get(i) + bias;
            float delta = SOFTPLUS ? softplus_fast(x) : x;
            delta = (full || ts + i < L) ? delta : 0.f;  // identity steps past the end
            const float uu = uval[i];
            dl[i] = delta;
            du[i] = delta * uu;
            y[i] = Dd * uu;
            if (SUMMARY) S += delta;
          }
        }
      }
      if constexpr (SUMMARY) {
        // The block's end state from a zero start: the state recurrence only.
#pragma unroll
        for (int ii = 0; ii < SB; ii++) {
          const int i = REV ? SB - 1 - ii : ii;
          const float2 dd = f2(dl[i], dl[i]), uu = f2(du[i], du[i]);
          const float4* bq = reinterpret_cast<const float4*>(tB + (sb + i) * TS);
#pragma unroll
          for (int g = 0; g < SPL / 4; g++) {
            const float4 bb = bq[g];
#pragma unroll
            for (int k = 0; k < 2; k++) {
              const int pi = 2 * g + k;
              const float2 e = mul2s(dd, A2[pi]);
              const float2 ab = f2(ex2_approx(e.x), ex2_approx(e.y));
              const float2 fu = input_factor<ZOH>(uu, e, ab, IA[pi], uval[i]);
              h[pi] = fma2s(ab, h[pi], mul2s(fu, k ? f2(bb.z, bb.w) : f2(bb.x, bb.y)));
            }
          }
        }
      } else {
      float part[SB];
#pragma unroll
      for (int ii = 0; ii < SB; ii++) {
        const int i = REV ? SB - 1 - ii : ii;
        const float2 dd = f2(dl[i], dl[i]), uu = f2(du[i], du[i]);
        const float4* bq = reinterpret_cast<const float4*>(tB + (sb + i) * TS);
        const float4* cq = reinterpret_cast<const float4*>(tC + (sb + i) * TS);
        float2 yp = f2(0.f, 0.f);
#pragma unroll
        for (int g = 0; g < SPL / 4; g++) {
          const float4 bb = bq[g], cc = cq[g];
#pragma unroll
          for (int k = 0; k < 2; k++) {
            const int pi = 2 * g + k;
            const float2 e = mul2s(dd, A2[pi]);
            const float2 ab = f2(ex2_approx(e.x), ex2_approx(e.y));
            const float2 fu = input_factor<ZOH>(uu, e, ab, IA[pi], uval[i]);
            h[pi] = fma2s(ab, h[pi], mul2s(fu, k ? f2(bb.z, bb.w) : f2(bb.x, bb.y)));
            yp = fma2s(k ? f2(cc.z, cc.w) : f2(cc.x, cc.y), h[pi], yp);
          }
        }
        part[i] = yp.x + yp.y;
      }
      if constexpr (Q == 2) {
        // Reduce-scatter of the two lanes' partial sums: lane q keeps steps [4q, 4q + 4), adds the
        // D skip, gates and stores them (4 shuffles instead of 8, and no silu computed twice).
        constexpr int HB = SB / 2;
        float yq[HB];
#pragma unroll
        for (int m = 0; m < HB; m++) {
          const float send = q ? part[m] : part[HB + m];
          const float keep = q ? part[HB + m] : part[m];
          yq[m] = keep + __shfl_xor_sync(kFull, send, RPW);
          const float uu = q ? uval[HB + m] : uval[m];
          yq[m] = fmaf(Dd, uu, yq[m]);
        }
        if (z_row) {
          Vec8<Tin> zs;
          if (tma) stage8<Tin, C::ROWS, C::RB>(zs, sz, r_cta, sb);
          else load8<Tin>(zs, z_row, ts, L, vec && full);
#pragma unroll
          for (int m = 0; m < HB; m++) yq[m] *= silu_fast(q ? zs.get(HB + m) : zs.get(m));
        }
        if (row_ok) store4<Tout>(o_row, ts + q * HB, L, vec && full, yq);
      } else {
        // The row's Q lanes each hold the sum over their states: add them up (8 independent shuffles).
#pragma unroll
        for (int o = RPW; o < 32; o <<= 1)
#pragma unroll
          for (int i = 0; i < SB; i++) part[i] += __shfl_xor_sync(kFull, part[i], o);
#pragma unroll
        for (int i = 0; i < SB; i++) y[i] += part[i];
        if (z_row) {
          Vec8<Tin> zs;
          if (tma) stage8<Tin, C::ROWS, C::RB>(zs, sz, r_cta, sb);
          else load8<Tin>(zs, z_row, ts, L, vec && full);
#pragma unroll
          for (int i = 0; i < SB; i++) y[i] *= silu_fast(zs.get(i));
        }
        if (row_ok && q == 0) store8<Tout>(o_row, ts, L, vec && full, y);
      }
      }  // scan (not summary)
    }
  }

  if (s_abort) {
    if (tid == 0) {
      atomicExch(&g_selscan_seq_error, 1);
      mbar_wait(&bars[c & 1], static_cast<uint32_t>((c >> 1) & 1));
    }
    return;
  }
  if (SUMMARY) {
    if constexpr (Q == 2) S += __shfl_xor_sync(kFull, S, RPW);  // each lane summed one half of the steps
    if (row_ok) {
      float* o = p.summ + (kslot * rows_total + grow) * (N + 1);
#pragma unroll
      for (int i = 0; i < PAIRS; i++)
#pragma unroll
        for (int k = 0; k < 2; k++) {
          const int n = n0 + 2 * i + k;
          if (n < N) o[n] = k ? h[i].y : h[i].x;
        }
      if (q == 0) o[N] = S;
    }
    return;
  }
  if (row_ok && p.h_last && kblk == (REV ? 0 : p.nblocks - 1)) {
#pragma unroll
    for (int i = 0; i < PAIRS; i++)
#pragma unroll
      for (int k = 0; k < 2; k++) {
        const int n = n0 + 2 * i + k;
        if (n < N) p.h_last[(b * p.dim + d) * N + n] = k ? h[i].y : h[i].x;
      }
  }
}

// Start state of every time block from the blocks' summaries: for each (row, state), in scan order,
// s ← 2^(A·log2e·ΣΔ) s + (zero-start end state of the block).  The first block in scan order starts
// from h0 (block 0, or with REV block nblocks-1, whose summaries sit in slots k-1 for blocks k >= 1).
template <bool REV = false>
__global__ void __launch_bounds__(256) selscan_carry_kernel(const FwdParams p) {
  const int64_t rows = p.batch * p.dim;
  const int N = p.dstate;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= rows * N) return;
  const int64_t grow = idx / N;
  const int n = static_cast<int>(idx - grow * N);
  const int64_t d = grow % p.dim;
  const float A2 = p.A[d * N + n] * kLog2e;
  float st = p.h0 ? p.h0[grow * N + n] : 0.f;
  // The first block in scan order starts from h0, copied into its slot: the scan pass then never reads
  // h0, which h_last may overwrite (in-place carry) while other blocks of the same launch still run.
  p.start[((REV ? p.nblocks - 1 : 0) * rows + grow) * N + n] = st;
#pragma unroll 8
  for (int k = 0; k < p.nblocks - 1; k++) {
    // Forward: summary slot k is block k and feeds block k+1.  Reverse: slot nblocks-2-k is block
    // nblocks-1-k and feeds block nblocks-2-k.
    const int slot = REV ? p.nblocks - 2 - k : k;
    const float* sm = p.summ + (slot * rows + grow) * (N + 1);
    st = fmaf(ex2_approx(A2 * sm[N]), st, sm[n]);
    p.start[((REV ? slot : k + 1) * rows + grow) * N + n] = st;
  }
}

// Time blocks for a problem whose rows alone do not fill the GPU: enough blocks that the scan's CTAs
// (row blocks x time blocks) fill the resident slots once, each block at least kMinTblock steps.
// SELSCAN_TBLOCKS=n forces n blocks (for tuning runs and tests).
constexpr int64_t kMinTblock = 512;
int64_t choose_tblock(const FwdParams& p, int64_t row_blocks, int slots) {
  const int64_t L = p.seqlen;
  int64_t nb = row_blocks >= slots ? 1 : slots / (row_blocks > 0 ? row_blocks : 1);
  if (const char* e = getenv("SELSCAN_TBLOCKS")) nb = atoi(e) > 0 ? atoi(e) : nb;
  if (nb <= 1) return L;
  int64_t tb = (L + nb - 1) / nb;
  tb = (tb + 63) / 64 * 64;  // whole chunks
  if (tb < kMinTblock) tb = kMinTblock;
  return tb;
}

// One forward call of the sequential kernel: one pass, or time blocks whose scratch comes from the
// stream's memory pool or (ScratchSource::Fixed, selscan_fwd_noalloc) the library's fixed array; with the
// fixed array *too_big is set and nothing enqueued when the blocks need more than it holds.
template <int NS, int Q, int R, typename Tin, typename Tout, bool FULLN, bool SOFTPLUS, bool REV = false,
          bool ZOH = false, bool CONV = false>
cudaError_t launch_seq_cfg(const FwdParams& p_in, cudaStream_t s, ScratchSource src = ScratchSource::Pool,
                           bool* too_big = nullptr) {
  using C = SeqCfg<NS, Q, R, Tin>;
  FwdParams p = p_in;
  TmaMaps maps;
  memset(&maps, 0, sizeof maps);
  // Tensor copies need 16-byte aligned rows (vec_stage) and coordinates that fit in 32 bits.
  const EncodeTiled enc = reinterpret_cast<EncodeTiled>(tensor_map_encoder());
  const uint64_t rows = static_cast<uint64_t>(p.batch * p.dim), bc_rows = static_cast<uint64_t>(p.batch * p.dstate);
  p.use_tma = p.vec_stage && enc && rows < (1ull << 31) && p.seqlen < (1ll << 31);
  if (p.use_tma) {
    const uint64_t L = static_cast<uint64_t>(p.seqlen);
    bool ok = encode_2d<Tin>(enc, &maps.u, p.u, L, rows, C::EPR, C::ROWS, C::kSwizzle) &&
              encode_2d<Tin>(enc, &maps.delta, p.delta, L, rows, C::EPR, C::ROWS, C::kSwizzle) &&
              (!p.z || encode_2d<Tin>(enc, &maps.z, p.z, L, rows, C::EPR, C::ROWS, C::kSwizzle)) &&
              encode_2d<Tin>(enc, &maps.B, p.B, L, bc_rows, C::T, NS, CU_TENSOR_MAP_SWIZZLE_NONE) &&
              encode_2d<Tin>(enc, &maps.C, p.C, L, bc_rows, C::T, NS, CU_TENSOR_MAP_SWIZZLE_NONE);
    p.use_tma = ok;
  }
  auto scan = selscan_fwd_seq_kernel<NS, Q, R, Tin, Tout, FULLN, SOFTPLUS, false, REV, ZOH, CONV>;
  auto summary = selscan_fwd_seq_kernel<NS, Q, R, Tin, float, FULLN, SOFTPLUS, true, REV, ZOH, CONV>;
  cudaError_t e = cudaFuncSetAttribute(scan, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::kSmem));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(summary, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::kSmem));
  if (e != cudaSuccess) return e;
  const int64_t row_blocks = ((p.dim + C::ROWS - 1) / C::ROWS) * p.batch;
  int per_sm = 0, sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, scan, R * 32, C::kSmem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  p.tblock = choose_tblock(p, row_blocks, sms * per_sm);
  p.nblocks = static_cast<int>((p.seqlen + p.tblock - 1) / p.tblock);
  const dim3 grid(static_cast<unsigned>((p.dim + C::ROWS - 1) / C::ROWS), static_cast<unsigned>(p.batch),
                  static_cast<unsigned>(p.nblocks));
  if (p.nblocks == 1) {
    scan<<<grid, R * 32, C::kSmem, s>>>(p, maps);
    count_launches(1);
    return cudaGetLastError();
  }
  const int64_t N = p.dstate;
  const size_t summ_floats = static_cast<size_t>(p.nblocks - 1) * rows * (N + 1);
  const size_t start_floats = static_cast<size_t>(p.nblocks) * rows * N;
  const size_t bytes = (summ_floats + start_floats) * sizeof(float);
  void* ws = nullptr;
  if (src == ScratchSource::Fixed) {
    // Every summary entry is written by the summary pass and every start entry by the carry pass before
    // it is read, so nothing in the array needs clearing.
    float* fixed = nullptr;
    size_t cap_bytes = 0;
    e = fixed_scratch(&fixed, &cap_bytes);
    if (e != cudaSuccess) return e;
    if (bytes > cap_bytes) {
      if (too_big) *too_big = true;
      return cudaSuccess;
    }
    ws = fixed;
  } else {
    // Stream-ordered scratch for the block summaries and start states, released on the same stream.  If
    // the pool cannot supply it the call fails with the allocation error (selscan_fwd_noalloc needs none).
    e = cudaMallocAsync(&ws, bytes, s);
    if (e != cudaSuccess) return e;
  }
  p.summ = static_cast<float*>(ws);
  p.start = p.summ + summ_floats;
  const dim3 sgrid(grid.x, grid.y, grid.z - 1);
  summary<<<sgrid, R * 32, C::kSmem, s>>>(p, maps);
  count_launches(1);
  e = cudaGetLastError();
  if (e == cudaSuccess) {
    const int64_t threads = static_cast<int64_t>(rows) * N;
    selscan_carry_kernel<REV><<<static_cast<unsigned>((threads + 255) / 256), 256, 0, s>>>(p);
    count_launches(1);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    scan<<<grid, R * 32, C::kSmem, s>>>(p, maps);
    count_launches(1);
    e = cudaGetLastError();
  }
  if (src == ScratchSource::Fixed) return e;
  const cudaError_t ef = cudaFreeAsync(ws, s);
  return e != cudaSuccess ? e : ef;
}

#ifndef SELSCAN_SEQ_R
#define SELSCAN_SEQ_R 4
#endif

template <typename Tin, typename Tout, bool SOFTPLUS>
cudaError_t dispatch_seq_sp(const FwdParams& p, cudaStream_t s) {
  constexpr int R = SELSCAN_SEQ_R;
  if (p.dstate == 16) return launch_seq_cfg<16, 2, R, Tin, Tout, true, SOFTPLUS>(p, s);
  if (p.dstate <= 4) return launch_seq_cfg<4, 1, R, Tin, Tout, false, SOFTPLUS>(p, s);
  if (p.dstate <= 8) return launch_seq_cfg<8, 2, R, Tin, Tout, false, SOFTPLUS>(p, s);
  return launch_seq_cfg<16, 2, R, Tin, Tout, false, SOFTPLUS>(p, s);
}

template <typename Tin, typename Tout>
cudaError_t dispatch_seq(const FwdParams& p, cudaStream_t s) {
  return p.delta_softplus ? dispatch_seq_sp<Tin, Tout, true>(p, s) : dispatch_seq_sp<Tin, Tout, false>(p, s);
}

template <typename Tin, typename Tout, bool SOFTPLUS, bool REV, bool ZOH, bool CONV = false>
cudaError_t dispatch_seq_ex_sp(const FwdParams& p, cudaStream_t s) {
  constexpr int R = SELSCAN_SEQ_R;
  if (p.dstate <= 4) return launch_seq_cfg<4, 1, R, Tin, Tout, false, SOFTPLUS, REV, ZOH, CONV>(p, s);
  if (p.dstate <= 8) return launch_seq_cfg<8, 2, R, Tin, Tout, false, SOFTPLUS, REV, ZOH, CONV>(p, s);
  if (CONV && p.dstate == 16) return launch_seq_cfg<16, 2, R, Tin, Tout, true, SOFTPLUS, REV, ZOH, CONV>(p, s);
  return launch_seq_cfg<16, 2, R, Tin, Tout, false, SOFTPLUS, REV, ZOH, CONV>(p, s);
}

template <typename Tin, typename Tout, bool REV, bool ZOH, bool CONV = false>
cudaError_t dispatch_seq_ex_flags(const FwdParams& p, cudaStream_t s) {
  return p.delta_softplus ? dispatch_seq_ex_sp<Tin, Tout, true, REV, ZOH, CONV>(p, s)
                          : dispatch_seq_ex_sp<Tin, Tout, false, REV, ZOH, CONV>(p, s);
}

template <typename Tin, typename Tout>
cudaError_t dispatch_seq_ex(const FwdParams& p, bool reverse, bool zoh, cudaStream_t s, bool conv) {
  if (conv) return zoh ? dispatch_seq_ex_flags<Tin, Tout, false, true, true>(p, s)
                       : dispatch_seq_ex_flags<Tin, Tout, false, false, true>(p, s);
  if (reverse && zoh) return dispatch_seq_ex_flags<Tin, Tout, true, true>(p, s);
  if (reverse) return dispatch_seq_ex_flags<Tin, Tout, true, false>(p, s);
  if (zoh) return dispatch_seq_ex_flags<Tin, Tout, false, true>(p, s);
  return dispatch_seq<Tin, Tout>(p, s);
}

}  // namespace

cudaError_t launch_fwd_seq_ex(const FwdParams& p, selscan_dtype_t in_dtype, selscan_dtype_t out_dtype, bool reverse,
                              bool zoh, cudaStream_t s, bool conv) {
  if (conv && reverse) return cudaErrorInvalidValue;  // the convolution front is causal
  if (in_dtype == SELSCAN_F32) {
    return out_dtype == SELSCAN_F32 ? dispatch_seq_ex<float, float>(p, reverse, zoh, s, conv)
                                    : dispatch_seq_ex<float, __nv_bfloat16>(p, reverse, zoh, s, conv);
  }
  return out_dtype == SELSCAN_F32 ? dispatch_seq_ex<__nv_bfloat16, float>(p, reverse, zoh, s, conv)
                                  : dispatch_seq_ex<__nv_bfloat16, __nv_bfloat16>(p, reverse, zoh, s, conv);
}

cudaError_t launch_fwd_seq(const FwdParams& p, selscan_dtype_t in_dtype, selscan_dtype_t out_dtype, cudaStream_t s) {
  if (in_dtype == SELSCAN_F32) {
    return out_dtype == SELSCAN_F32 ? dispatch_seq<float, float>(p, s) : dispatch_seq<float, __nv_bfloat16>(p, s);
  }
  return out_dtype == SELSCAN_F32 ? dispatch_seq<__nv_bfloat16, float>(p, s)
                                  : dispatch_seq<__nv_bfloat16, __nv_bfloat16>(p, s);
}

// ---- selscan_fwd_noalloc on rows that the row-sequential kernel cannot stage ------------------------

namespace {

template <typename Tin, typename Tout, bool SOFTPLUS>
cudaError_t dispatch_seq_noalloc_sp(const FwdParams& p, cudaStream_t s, bool* too_big) {
  constexpr int R = SELSCAN_SEQ_R;
  constexpr ScratchSource F = ScratchSource::Fixed;
  if (p.dstate == 16) return launch_seq_cfg<16, 2, R, Tin, Tout, true, SOFTPLUS>(p, s, F, too_big);
  if (p.dstate <= 4) return launch_seq_cfg<4, 1, R, Tin, Tout, false, SOFTPLUS>(p, s, F, too_big);
  if (p.dstate <= 8) return launch_seq_cfg<8, 2, R, Tin, Tout, false, SOFTPLUS>(p, s, F, too_big);
  return launch_seq_cfg<16, 2, R, Tin, Tout, false, SOFTPLUS>(p, s, F, too_big);
}

template <typename Tin, typename Tout>
cudaError_t dispatch_seq_noalloc(const FwdParams& p, cudaStream_t s, bool* too_big) {
  return p.delta_softplus ? dispatch_seq_noalloc_sp<Tin, Tout, true>(p, s, too_big)
                          : dispatch_seq_noalloc_sp<Tin, Tout, false>(p, s, too_big);
}

}  // namespace

cudaError_t launch_fwd_seq_noalloc(const FwdParams& p, selscan_dtype_t in_dtype, selscan_dtype_t out_dtype,
                                   cudaStream_t s, bool* too_big) {
  *too_big = false;
  if (in_dtype == SELSCAN_F32) {
    return out_dtype == SELSCAN_F32 ? dispatch_seq_noalloc<float, float>(p, s, too_big)
                                    : dispatch_seq_noalloc<float, __nv_bfloat16>(p, s, too_big);
  }
  return out_dtype == SELSCAN_F32 ? dispatch_seq_noalloc<__nv_bfloat16, float>(p, s, too_big)
                                  : dispatch_seq_noalloc<__nv_bfloat16, __nv_bfloat16>(p, s, too_big);
}

cudaError_t read_seq_device_error(int* value, int reset) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_selscan_seq_error, sizeof(int));
  if (e == cudaSuccess && reset) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_selscan_seq_error, &zero, sizeof(int));
  }
  return e;
}

}  // namespace selscan

// Selective-scan forward: fused chunked scan for sm_103a.
//
// Per row (b, d) and state n (see include/selscan.h):
//   Δ_t = softplus(δ_t + Δ_bias[d]),  Ā_t = exp(Δ_t A[d,n]),
//   h_t = Ā_t h_{t-1} + Δ_t B[b,n,t] u_t,  y_t = Σ_n C[b,n,t] h_t + D[d] u_t,  out_t = y_t silu(z_t)
// ("Mamba状态空间模型深度解析" §2.1 selective recurrence, §3.1 SiLU gate;
//  "Mamba架构与SSM模型：高效序列建模技术解析" §2.1 Ā = exp(ΔA), §2.2 Δ = softplus(·+param_Δ)).
//
// Decomposition.  A CTA owns one batch row b and ROWS = R·32/P consecutive channels.  P adjacent
// lanes share one channel; the sequence is cut into chunks of T = P·K steps and lane j of a channel
// owns the K steps [t0 + jK, t0 + jK + K) of each chunk, split into two halves ("sub-chains") of
// H = K/2 steps.  Every per-step quantity is held as a float2 (first-half step i, second-half
// step i), so each arithmetic instruction is one packed fp32x2 operation on two independent steps.
//
// For each state n a lane
//   1. forms Ā = 2^(Δ·A[d,n]·log2 e) and b = Δ·u·B for its 2H steps and folds each half into the
//      state it reaches from zero (pass 1),
//   2. joins its two halves and the P lanes of the channel with an inclusive shuffle scan under
//      the pair operator (a1, b1) ∘ (a2, b2) = (a2·a1, a2·b1 + b2)  — the "block scan with prefix
//      state" of "Mamba: Linear-Time Sequence Modeling with Selective SSMs", 选择性扫描要点,
//   3. takes its start state from the lane before it (lane 0: the carried state), reruns both
//      halves from their true start states and accumulates y += C·h (pass 2).
// The products of Ā over a half or a lane are 2^(A·log2e·ΣΔ), one exponential per state.
// The end state of the chunk is carried in registers into the next chunk, so long sequences never
// write their state to memory.
//
// Staging.  One thread issues the tensor-memory-accelerator copies of chunk c+1 while chunk c is
// computed (two buffers): u, δ and z of the CTA's channels as 2-D tiles [ROWS][T] with the 128-byte
// swizzle (each lane then reads its K steps as 16-byte shared loads), and the raw B, C rows of the
// batch entry.  Where the tensor copies cannot be used (rows not 16-byte aligned, channel blocks not
// a multiple of 8, or a chunk narrower than a 128-byte row) the lanes read u, δ, z from global
// memory and B, C come by 1-D bulk copies or plain loads.  B and C are shared by every channel of
// the CTA; they are widened once per CTA to fp32 in a layout where one 128-bit shared load yields
// the float2 pairs of two consecutive steps.  Steps past the end of the sequence get Δ = 0 and u = 0:
// the identity pair (1, 0), so a ragged last chunk needs no special case in the scan.
#include <cstdlib>
#include <cstring>

#include "selscan_internal.cuh"

namespace selscan {

// Set by a kernel whose bounded wait on a bulk copy gave up (read by selscan_device_status()).
__device__ int g_selscan_device_error = 0;

namespace {

// SELSCAN_STAGING=0 makes the chunked kernel read u, δ, z from global memory even where the tensor
// copies could be used (for tuning and for testing the direct path on aligned inputs).
bool staging_disabled() {
  const char* e = getenv("SELSCAN_STAGING");
  return e && e[0] == '0';
}

// ---- the kernel ----------------------------------------------------------------------------------

template <int NS, int P, int K, int R, typename Tin>
struct Cfg {
  static constexpr int H = K / 2;
  static constexpr int T = P * K;        // steps per chunk
  static constexpr int RPW = 32 / P;     // channels per warp
  static constexpr int ROWS = R * RPW;   // channels per CTA
  static constexpr int KP = K + 4;       // fp32 stride of one lane's K steps: an odd number of 16-byte
                                         // units, so the P lanes of a channel hit distinct bank groups
  static constexpr int SEG = P * KP;     // floats of one (tensor, n) row of the widened tile
  static constexpr int TILE = 2 * NS * SEG;  // floats of one widened B, C tile
  static constexpr int RAW = 2 * NS * T;     // raw elements of one chunk (B rows then C rows)
  static constexpr int UNITS = 2 * NS * P;   // widening work units per chunk (tensor, n, lane segment)
  static constexpr int UNITS_PER_THREAD = (UNITS + R * 32 - 1) / (R * 32);
  static constexpr int EPR = 128 / static_cast<int>(sizeof(Tin));  // inputs per 128-byte stage row
  // Tensor copies of u, δ, z need whole 128-byte stage rows and boxes of whole 1 KiB swizzle atoms.
  static constexpr bool kTmaShape = T % EPR == 0 && ROWS % 8 == 0;
  static constexpr int SUBT = kTmaShape ? T / EPR : 1;                  // boxes per tensor per chunk
  static constexpr int BCX = T < 128 ? T : 128;                         // steps per B / C box
  static constexpr int NB = T / BCX;                                    // B (and C) boxes per chunk
  static constexpr size_t kStageTensor = static_cast<size_t>(ROWS) * T * sizeof(Tin);
  static constexpr size_t kStageBytes = kTmaShape ? 2 * 3 * kStageTensor : 0;  // double-buffered u, δ, z
  static constexpr size_t kTileBytes = 2 * TILE * sizeof(float);  // double-buffered
  static constexpr size_t kRawBytes = 2 * RAW * sizeof(Tin);       // double-buffered
  static constexpr size_t kSmem = 1024 + kStageBytes + kTileBytes + kRawBytes + 2 * sizeof(uint64_t);
  static_assert(K % 4 == 0 && P >= 1 && P <= 32 && 32 % P == 0, "bad tile shape");
  static_assert(T % BCX == 0, "B, C boxes must tile the chunk");
};

// K consecutive inputs [e0, e0 + K) of stage row r of one tensor's stage [SUBT][ROWS][EPR], as two
// halves.  The stage was written by a 2-D tensor copy with the 128-byte swizzle: 16-byte chunk c of
// the stage row at byte offset 128·q sits at chunk position c ^ (q mod 8).
template <typename Tin, int H, int ROWS>
__device__ __forceinline__ void load_seg_stage(Seg<Tin, H>& s, const unsigned char* __restrict__ stage, int r,
                                               int e0) {
  constexpr int kPerVec = Seg<Tin, H>::kPerVec, EPR = 128 / static_cast<int>(sizeof(Tin));
#pragma unroll
  for (int h = 0; h < 2; h++)
#pragma unroll
    for (int q = 0; q < Seg<Tin, H>::kVecs; q++) {
      const int e = e0 + h * H + q * kPerVec;
      const int srow = (e / EPR) * ROWS + r, chunk = (e % EPR) / kPerVec;
      s.v[h][q] = *reinterpret_cast<const uint4*>(stage + srow * 128 + ((chunk ^ (srow & 7)) << 4));
    }
}

// Widen raw chunk c (raw buffer rb) into tile buffer tb.  MASK: zero steps at or past L and states
// at or past N (the raw buffer holds stale data there).  The raw chunk is [2 tensors][NB][NS][BCX]
// as written by the tensor copies (BOXED), else [2 tensors][NS][T].
template <int NS, int P, int K, int R, typename Tin, bool MASK, bool BOXED>
__device__ __forceinline__ void widen(const Tin* __restrict__ rb, float* __restrict__ tb, int tid, int64_t t0,
                                      int64_t L, int N) {
  using C = Cfg<NS, P, K, R, Tin>;
  constexpr int H = C::H;
  constexpr int BX = BOXED ? C::BCX : C::T;
#pragma unroll
  for (int k = 0; k < C::UNITS_PER_THREAD; k++) {
    const int unit = tid + k * R * 32;
    if (C::UNITS % (R * 32) != 0 && unit >= C::UNITS) break;
    const int s = unit % P, rowi = unit / P;  // rowi = tensor * NS + n
    Seg<Tin, H> rs;
    const int tensor = rowi / NS, n_raw = rowi % NS, box = (s * K) / BX, x = (s * K) % BX;
    const uint4* src = reinterpret_cast<const uint4*>(rb + tensor * NS * C::T + (box * NS + n_raw) * BX + x);
#pragma unroll
    for (int h = 0; h < 2; h++)
#pragma unroll
      for (int q = 0; q < Seg<Tin, H>::kVecs; q++) rs.v[h][q] = src[h * Seg<Tin, H>::kVecs + q];
    float2 w[H];
#pragma unroll
    for (int i = 0; i < H; i++) w[i] = f2(rs.get(0, i), rs.get(1, i));
    if (MASK) {
      const int n = rowi % NS;
      const int64_t tl = t0 + s * K;
#pragma unroll
      for (int i = 0; i < H; i++) {
        if (n >= N || tl + i >= L) w[i].x = 0.f;
        if (n >= N || tl + H + i >= L) w[i].y = 0.f;
      }
    }
    float4* dst = reinterpret_cast<float4*>(tb + rowi * C::SEG + s * C::KP);
#pragma unroll
    for (int q = 0; q < H / 2; q++) dst[q] = make_float4(w[2 * q].x, w[2 * q].y, w[2 * q + 1].x, w[2 * q + 1].y);
  }
}

// Per-channel values that persist across chunks, kept in shared memory (read once per state and
// chunk, as a broadcast to the channel's P lanes): A[d, n]·log2 e and the carried state.
template <int NS>
struct Carry {
  float* A2;     // [NS] of this lane's channel
  float* carry;  // [NS] state at the end of the previous chunk
};

// One chunk for one lane: inputs, then the states in groups of G, then the gated output.
// TAIL: the chunk runs past L or rows are not 16-byte aligned (masked, scalar-safe loads and stores).
// STAGED: u, δ, z come from the chunk's shared-memory stage [3][SUBT][ROWS][128 B] (row r_local,
// inputs [jK, jK + K)); otherwise from global memory.
template <int NS, int P, int K, int G, int ROWS, typename Tin, typename Tout, bool FULLN, bool TAIL, bool SOFTPLUS,
          bool STAGED>
__device__ __forceinline__ void compute_chunk(const FwdParams& p, Carry<NS>& cs, const float* __restrict__ tb,
                                              int j, int rw, int64_t ts, int64_t L, float bias, float Dd,
                                              const Tin* __restrict__ u_row, const Tin* __restrict__ dl_row,
                                              const Tin* __restrict__ z_row, Tout* __restrict__ o_row, bool row_ok,
                                              const unsigned char* __restrict__ stage, size_t stage_tensor,
                                              int r_local) {
  constexpr int H = K / 2, KP = K + 4, SEG = P * KP;
  const int N = FULLN ? NS : p.dstate;
  float2 dl[H], du[H], y[H];
  float S0 = 0.f, S1 = 0.f;  // Σ Δ over each half
  {
    Seg<Tin, H> us, ds;
    if (STAGED) {
      load_seg_stage<Tin, H, ROWS>(us, stage, r_local, j * K);
      load_seg_stage<Tin, H, ROWS>(ds, stage + stage_tensor, r_local, j * K);
    } else {
      load_seg<Tin, H>(us, u_row, ts, L, !TAIL);
      load_seg<Tin, H>(ds, dl_row, ts, L, !TAIL);
    }
    const float2 bias2 = f2(bias, bias), D2 = f2(Dd, Dd);
#pragma unroll
    for (int i = 0; i < H; i++) {
      const float2 x = add2s(f2(ds.get(0, i), ds.get(1, i)), bias2);
      float2 dd = SOFTPLUS ? f2(softplus_fast(x.x), softplus_fast(x.y)) : x;
      if (TAIL) {  // identity steps past the end
        dd.x = ts + i < L ? dd.x : 0.f;
        dd.y = ts + H + i < L ? dd.y : 0.f;
      }
      S0 += dd.x;
      S1 += dd.y;
      dl[i] = dd;
      const float2 uu = f2(us.get(0, i), us.get(1, i));
      du[i] = mul2s(dd, uu);
      y[i] = mul2s(D2, uu);
    }
  }

  const float* tB = tb + j * KP;
  const float* tC = tb + NS * SEG + j * KP;
#pragma unroll
  for (int n0 = 0; n0 < NS; n0 += G) {
    if (!FULLN && n0 >= N) break;
    float2 ab[G][H], bu[G][H], bagg[G];
    float a0[G], a1[G], a[G], bl[G];
    // Pass 1: Ā and Δ·u·B for every step; each half folded from a zero state.
#pragma unroll
    for (int g = 0; g < G; g++) {
      const int n = n0 + g;
      const float A2n = cs.A2[n];
      const float2 a2 = f2(A2n, A2n);
      const float4* bq = reinterpret_cast<const float4*>(tB + n * SEG);
      bagg[g] = f2(0.f, 0.f);
#pragma unroll
      for (int q = 0; q < H / 2; q++) {
        const float4 bb = bq[q];
#pragma unroll
        for (int k = 0; k < 2; k++) {
          const int i = 2 * q + k;
          const float2 e = mul2s(dl[i], a2);
          ab[g][i] = f2(ex2_approx(e.x), ex2_approx(e.y));
          bu[g][i] = mul2s(du[i], k ? f2(bb.z, bb.w) : f2(bb.x, bb.y));
          bagg[g] = fma2s(ab[g][i], bagg[g], bu[g][i]);
        }
      }
      // This lane's pair: the first half (a0, bagg.x) followed by the second half (a1, bagg.y).
      const float2 e01 = mul2s(a2, f2(S0, S1));
      a0[g] = ex2_approx(e01.x);
      a1[g] = ex2_approx(e01.y);
      a[g] = a0[g] * a1[g];
      bl[g] = fmaf(a1[g], bagg[g].x, bagg[g].y);
    }
    // Join the P lanes of the channel.  Lane j of a channel sits at warp lane j·RPW + rw, so the
    // lane holding the channel's previous segment is RPW lanes below.
    constexpr int RPW = 32 / P;
    float s0[G];
    if (P <= 4) {
      // Short chain: each lane's end state given the carried state, then P-1 hand-offs along the
      // segments; after hand-off k, segment k holds its true start and end states.
#pragma unroll
      for (int g = 0; g < G; g++) {
        const int n = n0 + g;
        const float cin = cs.carry[n];  // the channel's lanes all read it before any lane writes it
        float e = fmaf(a[g], cin, bl[g]);
        s0[g] = cin;
#pragma unroll
        for (int k = 1; k < P; k++) {
          const float prev = __shfl_up_sync(kFull, e, RPW);
          const bool mine = j == k;
          s0[g] = mine ? prev : s0[g];
          e = mine ? fmaf(a[g], prev, bl[g]) : e;
        }
        const float cout = P > 1 ? __shfl_sync(kFull, e, (P - 1) * RPW + rw) : e;
        if (j == 0) cs.carry[n] = cout;
      }
    } else {
      // Longer channels: inclusive scan of the lanes' (a, b) pairs in log2(P) levels, the G states
      // interleaved, then one hand-off of end states.
#pragma unroll
      for (int o = 1; o < P; o <<= 1) {
        const bool take = j >= o;
        float a_up[G], b_up[G];
#pragma unroll
        for (int g = 0; g < G; g++) {
          a_up[g] = __shfl_up_sync(kFull, a[g], o * RPW);
          b_up[g] = __shfl_up_sync(kFull, bl[g], o * RPW);
        }
#pragma unroll
        for (int g = 0; g < G; g++) {
          a_up[g] = take ? a_up[g] : 1.f;  // lanes without a predecessor at this distance combine with (1, 0)
          b_up[g] = take ? b_up[g] : 0.f;
          bl[g] = fmaf(a[g], b_up[g], bl[g]);
          a[g] *= a_up[g];
        }
      }
#pragma unroll
      for (int g = 0; g < G; g++) {
        const int n = n0 + g;
        const float cin = cs.carry[n];
        const float h_end = fmaf(a[g], cin, bl[g]);
        const float prev = __shfl_up_sync(kFull, h_end, RPW);
        s0[g] = j > 0 ? prev : cin;
        const float cout = __shfl_sync(kFull, h_end, (P - 1) * RPW + rw);
        if (j == 0) cs.carry[n] = cout;
      }
    }
    // Pass 2: rerun both halves from their true start states and read out C·h.
#pragma unroll
    for (int g = 0; g < G; g++) {
      const int n = n0 + g;
      float2 h = f2(s0[g], fmaf(a0[g], s0[g], bagg[g].x));
      const float4* cq = reinterpret_cast<const float4*>(tC + n * SEG);
#pragma unroll
      for (int q = 0; q < H / 2; q++) {
        const float4 cc = cq[q];
#pragma unroll
        for (int k = 0; k < 2; k++) {
          const int i = 2 * q + k;
          h = fma2s(ab[g][i], h, bu[g][i]);
          y[i] = fma2s(k ? f2(cc.z, cc.w) : f2(cc.x, cc.y), h, y[i]);
        }
      }
    }
  }

  if (z_row) {
    Seg<Tin, H> zs;
    if (STAGED)
      load_seg_stage<Tin, H, ROWS>(zs, stage + 2 * stage_tensor, r_local, j * K);
    else
      load_seg<Tin, H>(zs, z_row, ts, L, !TAIL);
#pragma unroll
    for (int i = 0; i < H; i++) y[i] = mul2s(y[i], f2(silu_fast(zs.get(0, i)), silu_fast(zs.get(1, i))));
  }
  if (row_ok) store_seg<Tout, H>(o_row, ts, L, !TAIL, y);
}

// Resident warps per SM the register budget is sized for (12 warps: at most 168 registers a thread).
#ifndef SELSCAN_WARPS_PER_SM
#define SELSCAN_WARPS_PER_SM 12
#endif

// STAGED: u, δ, z and B, C arrive by 2-D tensor copies (maps), else as described at the top.
template <int NS, int P, int K, int R, int G, typename Tin, typename Tout, bool FULLN, bool SOFTPLUS, bool STAGED>
__global__ void __launch_bounds__(R * 32, SELSCAN_WARPS_PER_SM / R)
    selscan_fwd_kernel(const FwdParams p, const __grid_constant__ TmaMaps maps) {
  using C = Cfg<NS, P, K, R, Tin>;
  constexpr int T = C::T;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  // The u, δ, z stage starts on a 1 KiB boundary (the period of the 128-byte swizzle).
  // (Offsetting the shared pointer itself keeps every derived pointer in the shared window, so the
  // tile reads compile to shared loads rather than generic ones.)
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  unsigned char* stage = smem;                                                  // [2 buffers][3][SUBT][ROWS][128 B]
  float* tiles = reinterpret_cast<float*>(smem + C::kStageBytes);               // [2 buffers][2][NS][P][KP]
  Tin* raw = reinterpret_cast<Tin*>(smem + C::kStageBytes + C::kTileBytes);     // [2 buffers][RAW]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStageBytes + C::kTileBytes + C::kRawBytes);
  __shared__ int s_abort;
  // Row stride NS + 1: the RPW channels of a quarter-warp reading state n hit distinct banks.
  __shared__ float s_A2[C::ROWS][NS + 1], s_carry[C::ROWS][NS + 1];

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  // Segment-major lanes: lane = j·RPW + rw, so the RPW channels of a warp that read the same time
  // segment share one quarter-warp (a broadcast shared load) when P <= 8.
  const int rw = lane % C::RPW;
  const int j = lane / C::RPW;  // segment of this lane within its channel
  const int r_local = (tid >> 5) * C::RPW + rw;
  const int64_t b = blockIdx.y;
  const int64_t d0 = static_cast<int64_t>(blockIdx.x) * C::ROWS;
  const int64_t d = d0 + r_local;
  const bool row_ok = d < p.dim;
  const int N = FULLN ? NS : p.dstate;
  const int64_t L = p.seqlen;
  const int64_t nchunks = (L + T - 1) / T;
  const Tin* __restrict__ Bsrc = static_cast<const Tin*>(p.B) + b * N * L;
  const Tin* __restrict__ Csrc = static_cast<const Tin*>(p.C) + b * N * L;
  const bool bulk = STAGED || p.vec_bc;  // chunks arrive by asynchronous copies (else plain loads)
  const bool has_z = p.z != nullptr;

  // Issue the copies of chunk c into buffer c & 1 (one thread).
  auto issue = [&](int64_t c) {
    const int64_t t0 = c * T;
    Tin* dst = raw + (c & 1) * C::RAW;
    uint64_t* bar = &bars[c & 1];
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (STAGED) {
      // Whole boxes always land (zero-filled past the tensor), so the byte count is fixed.
      const uint32_t bytes = static_cast<uint32_t>((has_z ? 3 : 2) * C::kStageTensor +
                                                   2 * C::NB * NS * C::BCX * sizeof(Tin));
      mbar_expect_tx(bar, bytes);
      unsigned char* st = stage + (c & 1) * 3 * C::kStageTensor;
      const int x0 = static_cast<int>(t0), y0 = static_cast<int>(b * p.dim + d0);
      const CUtensorMap* m[3] = {&maps.u, &maps.delta, &maps.z};
#pragma unroll
      for (int k = 0; k < 3; k++) {
        if (k == 2 && !has_z) break;
#pragma unroll
        for (int sub = 0; sub < C::SUBT; sub++)
          tma_load_2d(st + k * C::kStageTensor + sub * C::ROWS * 128, m[k], x0 + sub * C::EPR, y0, bar);
      }
      const int yb = static_cast<int>(b * N);
#pragma unroll
      for (int box = 0; box < C::NB; box++) {
        tma_load_2d(dst + box * NS * C::BCX, &maps.B, x0 + box * C::BCX, yb, bar);
        tma_load_2d(dst + NS * T + box * NS * C::BCX, &maps.C, x0 + box * C::BCX, yb, bar);
      }
    } else {
      const int64_t len = (L - t0) < T ? (L - t0) : T;
      const uint32_t bytes = static_cast<uint32_t>(len * sizeof(Tin));
      mbar_expect_tx(bar, 2u * N * bytes);
      for (int n = 0; n < N; n++) {
        bulk_copy_g2s(dst + n * T, Bsrc + n * L + t0, bytes, bar);
        bulk_copy_g2s(dst + (NS + n) * T, Csrc + n * L + t0, bytes, bar);
      }
    }
  };

  if (tid == 0) {
    s_abort = 0;
    if (bulk) {
      mbar_init(&bars[0], 1);
      mbar_init(&bars[1], 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
  }
  __syncthreads();
  if (bulk && tid == 0 && nchunks > 0) issue(0);

  Carry<NS> cs{s_A2[r_local], s_carry[r_local]};
  if (j == 0) {
#pragma unroll
    for (int n = 0; n < NS; n++) {
      const bool ok = row_ok && n < N;
      cs.A2[n] = ok ? p.A[d * N + n] * kLog2e : 0.f;
      cs.carry[n] = (ok && p.h0) ? p.h0[(b * p.dim + d) * N + n] : 0.f;
    }
  }
  // (the chunk loop's first barrier orders these writes before any read)
  const float bias = (row_ok && p.delta_bias) ? p.delta_bias[d] : 0.f;
  const float Dd = (row_ok && p.D) ? p.D[d] : 0.f;
  // Channels past `dim` (tail of the last CTA) run the scan on channel 0's inputs (or, staged, on
  // whatever rows the tile holds there) so that every lane takes part in the warp shuffles; only
  // their stores are skipped.
  const int64_t row_off = (b * p.dim + (row_ok ? d : 0)) * L;
  const Tin* __restrict__ u_row = static_cast<const Tin*>(p.u) + row_off;
  const Tin* __restrict__ dl_row = static_cast<const Tin*>(p.delta) + row_off;
  const Tin* __restrict__ z_row = has_z ? static_cast<const Tin*>(p.z) + row_off : nullptr;
  Tout* __restrict__ o_row = static_cast<Tout*>(p.out) + row_off;

  int64_t c = 0;
  for (; c < nchunks; c++) {
    const int64_t t0 = c * T;
    const Tin* rb = raw + (c & 1) * C::RAW;
    float* tb = tiles + (c & 1) * C::TILE;
    const bool tail = t0 + T > L;
    if (bulk) {
      if (!mbar_wait(&bars[c & 1], static_cast<uint32_t>((c >> 1) & 1))) s_abort = 1;
    } else {
      // Unaligned or ragged B, C rows: every thread loads part of the raw chunk directly.
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
      widen<NS, P, K, R, Tin, false, STAGED>(rb, tb, tid, t0, L, N);
    else
      widen<NS, P, K, R, Tin, true, STAGED>(rb, tb, tid, t0, L, N);
    // Tile c is complete, and every warp has finished chunk c-1 (whose buffers the next copy reuses).
    __syncthreads();
    if (s_abort) break;
    if (bulk && tid == 0 && c + 1 < nchunks) issue(c + 1);

    const int64_t ts = t0 + static_cast<int64_t>(j) * K;  // this lane's first step
    const unsigned char* st = stage + (c & 1) * 3 * C::kStageTensor;
    if (!tail && p.vec_in && p.vec_out)
      compute_chunk<NS, P, K, G, C::ROWS, Tin, Tout, FULLN, false, SOFTPLUS, STAGED>(
          p, cs, tb, j, rw, ts, L, bias, Dd, u_row, dl_row, z_row, o_row, row_ok, st, C::kStageTensor, r_local);
    else
      compute_chunk<NS, P, K, G, C::ROWS, Tin, Tout, FULLN, true, SOFTPLUS, STAGED>(
          p, cs, tb, j, rw, ts, L, bias, Dd, u_row, dl_row, z_row, o_row, row_ok, st, C::kStageTensor, r_local);
  }

  if (s_abort) {
    // Chunk c's copy did not complete in time (chunk c+1 was never issued).  Record the failure and
    // give that copy one more bounded wait, so it does not land after the CTA's shared memory is
    // released.
    if (tid == 0) {
      atomicExch(&g_selscan_device_error, 1);
      mbar_wait(&bars[c & 1], static_cast<uint32_t>((c >> 1) & 1));
    }
    return;
  }
  if (row_ok && p.h_last) {
#pragma unroll
    for (int n = 0; n < NS; n++)
      if (n < N && j == P - 1) p.h_last[(b * p.dim + d) * N + n] = cs.carry[n];
  }
}

size_t smem_bytes(int NS, int P, size_t in_bytes);

template <int NS, int P, int K, int R, int G, typename Tin, typename Tout, bool FULLN, bool STAGED>
cudaError_t launch_kernel(const FwdParams& p, const TmaMaps& maps, cudaStream_t s) {
  using C = Cfg<NS, P, K, R, Tin>;
  if (smem_bytes(NS, P, sizeof(Tin)) != C::kSmem) return cudaErrorInvalidConfiguration;  // estimate out of step
  auto kern = p.delta_softplus ? selscan_fwd_kernel<NS, P, K, R, G, Tin, Tout, FULLN, true, STAGED>
                               : selscan_fwd_kernel<NS, P, K, R, G, Tin, Tout, FULLN, false, STAGED>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::kSmem));
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>((p.dim + C::ROWS - 1) / C::ROWS), static_cast<unsigned>(p.batch));
  kern<<<grid, R * 32, C::kSmem, s>>>(p, maps);
  count_launches(1);
  return cudaGetLastError();
}

// The staged kernel when the shape allows tensor copies and the maps encode, else the direct one.
template <int NS, int P, int K, int R, int G, typename Tin, typename Tout, bool FULLN>
cudaError_t launch_cfg(const FwdParams& p, cudaStream_t s) {
  using C = Cfg<NS, P, K, R, Tin>;
  TmaMaps maps;
  memset(&maps, 0, sizeof maps);
  if constexpr (C::kTmaShape) {
    const EncodeTiled enc = reinterpret_cast<EncodeTiled>(tensor_map_encoder());
    const uint64_t rows = static_cast<uint64_t>(p.batch * p.dim), bc_rows = static_cast<uint64_t>(p.batch * p.dstate);
    const uint64_t L = static_cast<uint64_t>(p.seqlen);
    bool ok = enc && p.vec_stage && p.vec_in && rows < (1ull << 31) && bc_rows < (1ull << 31) && L < (1ull << 31);
    ok = ok && encode_2d<Tin>(enc, &maps.u, p.u, L, rows, C::EPR, C::ROWS, CU_TENSOR_MAP_SWIZZLE_128B) &&
         encode_2d<Tin>(enc, &maps.delta, p.delta, L, rows, C::EPR, C::ROWS, CU_TENSOR_MAP_SWIZZLE_128B) &&
         (!p.z || encode_2d<Tin>(enc, &maps.z, p.z, L, rows, C::EPR, C::ROWS, CU_TENSOR_MAP_SWIZZLE_128B)) &&
         encode_2d<Tin>(enc, &maps.B, p.B, L, bc_rows, C::BCX, NS, CU_TENSOR_MAP_SWIZZLE_NONE) &&
         encode_2d<Tin>(enc, &maps.C, p.C, L, bc_rows, C::BCX, NS, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (ok && !staging_disabled()) return launch_kernel<NS, P, K, R, G, Tin, Tout, FULLN, true>(p, maps, s);
  }
  return launch_kernel<NS, P, K, R, G, Tin, Tout, FULLN, false>(p, maps, s);
}

// Warps per CTA for each lane count: enough channels per CTA (32·R/P) to amortise the per-chunk
// widening of B and C, few enough CTAs per channel block to balance the SMs.
#ifndef SELSCAN_R_P2
#define SELSCAN_R_P2 2
#endif
#ifndef SELSCAN_R_P4
#define SELSCAN_R_P4 4
#endif
#ifndef SELSCAN_R_P8
#define SELSCAN_R_P8 4
#endif
#ifndef SELSCAN_R_P16
#define SELSCAN_R_P16 4
#endif
#ifndef SELSCAN_R_P32
#define SELSCAN_R_P32 4
#endif
#ifndef SELSCAN_G
#define SELSCAN_G 2
#endif
#ifndef SELSCAN_K
#define SELSCAN_K 16
#endif
constexpr int kK = SELSCAN_K;  // steps per lane-segment

// Warps of one CTA of the chunked kernel for P lanes per channel (the table above).
constexpr int warps_per_cta_for(int P) {
  return P == 2 ? SELSCAN_R_P2 : P == 4 ? SELSCAN_R_P4 : P == 8 ? SELSCAN_R_P8 : P == 16 ? SELSCAN_R_P16 : SELSCAN_R_P32;
}

// Dynamic shared memory of the kernel for NS states and P lanes (Cfg::kSmem, evaluated at run time).
size_t smem_bytes(int NS, int P, size_t in_bytes) {
  const size_t T = static_cast<size_t>(P) * kK, EPR = 128 / in_bytes;
  const size_t rows = static_cast<size_t>(warps_per_cta_for(P)) * (32 / P);
  const bool tma_shape = T % EPR == 0 && rows % 8 == 0;
  const size_t stage = tma_shape ? 2 * 3 * rows * T * in_bytes : 0;
  return 1024 + stage + 2 * 2 * NS * P * (kK + 4) * sizeof(float) + 2 * 2 * NS * T * in_bytes + 2 * sizeof(uint64_t);
}

// Lanes per channel: as few as keep enough warps in flight (each extra lane adds scan work), more
// when channels are scarce, and no more than the shared-memory tile allows.
int pick_lanes(const FwdParams& p, int NS, size_t in_bytes) {
  static int sms = 0, smem_max = 0;
  if (sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (sms <= 0) sms = 148;
    if (smem_max <= 0) smem_max = 48 * 1024;
  }
  // Lane counts measured fastest on B300 for 16 states, by the number of (batch, channel) rows:
  // 20480 and 12288 rows -> 4 lanes, 1536 -> 16.  Fewer lanes mean less scan work per step but
  // fewer warps; the thresholds sit between the measured shapes.
  const int64_t rows = p.batch * p.dim;
  int P = rows >= 4096 ? 4 : rows >= 512 ? 16 : 32;
  (void)sms;
  // SELSCAN_LANES (2, 4, 8, 16 or 32) overrides the choice; for tuning runs only.
  if (const char* e = getenv("SELSCAN_LANES")) {
    const int v = atoi(e);
    if (v == 2 || v == 4 || v == 8 || v == 16 || v == 32) P = v;
  }
  const size_t static_smem = 8 * 1024;  // s_A2, s_carry and the abort flag, with margin
  while (P > 2 && smem_bytes(NS, P, in_bytes) + static_smem > static_cast<size_t>(smem_max)) P /= 2;
  return P;
}

template <int NS, bool FULLN, typename Tin, typename Tout>
cudaError_t dispatch_p(const FwdParams& p, cudaStream_t s) {
  constexpr int G = SELSCAN_G;
  switch (pick_lanes(p, NS, sizeof(Tin))) {
    case 2: return launch_cfg<NS, 2, kK, SELSCAN_R_P2, G, Tin, Tout, FULLN>(p, s);
    case 4: return launch_cfg<NS, 4, kK, SELSCAN_R_P4, G, Tin, Tout, FULLN>(p, s);
    case 8: return launch_cfg<NS, 8, kK, SELSCAN_R_P8, G, Tin, Tout, FULLN>(p, s);
    case 16: return launch_cfg<NS, 16, kK, SELSCAN_R_P16, G, Tin, Tout, FULLN>(p, s);
    default: return launch_cfg<NS, 32, kK, SELSCAN_R_P32, G, Tin, Tout, FULLN>(p, s);
  }
}

template <typename Tin, typename Tout>
cudaError_t dispatch_ns(const FwdParams& p, cudaStream_t s) {
  if (p.dstate == 16) return dispatch_p<16, true, Tin, Tout>(p, s);
  if (p.dstate <= 4) return dispatch_p<4, false, Tin, Tout>(p, s);
  if (p.dstate <= 8) return dispatch_p<8, false, Tin, Tout>(p, s);
  return dispatch_p<16, false, Tin, Tout>(p, s);
}

}  // namespace

// The sequential kernel when the rows alone fill the GPU with its two lanes per row (16384 rows and
// more), or when they are too few for the chunked scan (below 4096: the sequential kernel then cuts the
// sequence into time blocks joined by a summary and a carry pass); the chunked scan in between.
// Measured on B300 with 16 states: 20480 rows 576 us (sequential) vs 606 us (chunked); 12288 rows
// 207 us vs 187 us; 1536 rows 899 us (time blocks) vs 1865 us.
// SELSCAN_KERNEL=seq|chunk overrides the choice (for tuning runs and tests).
bool use_sequential(const FwdParams& p) {
  if (const char* e = getenv("SELSCAN_KERNEL")) {
    if (e[0] == 's') return true;
    if (e[0] == 'c') return false;
  }
  const int64_t rows = p.batch * p.dim;
  return rows < 4096 || rows >= 16384;
}

// The row-sequential kernel (selscan_rows.cu) wherever its tensor copies can stage the inputs; the
// older kernels otherwise.  SELSCAN_KERNEL=rows|seq|chunk forces one (for tuning runs and tests).
cudaError_t launch_fwd(const FwdParams& p, selscan_dtype_t in_dtype, selscan_dtype_t out_dtype, cudaStream_t s) {
  const char* k = getenv("SELSCAN_KERNEL");
  if ((!k || k[0] == 'r') && rows_kernel_supports(p, in_dtype))
    return launch_fwd_rows(p, in_dtype, out_dtype, RowsOptions{}, s, nullptr);
  if (use_sequential(p)) return launch_fwd_seq(p, in_dtype, out_dtype, s);
  if (in_dtype == SELSCAN_F32) {
    return out_dtype == SELSCAN_F32 ? dispatch_ns<float, float>(p, s) : dispatch_ns<float, __nv_bfloat16>(p, s);
  }
  return out_dtype == SELSCAN_F32 ? dispatch_ns<__nv_bfloat16, float>(p, s)
                                  : dispatch_ns<__nv_bfloat16, __nv_bfloat16>(p, s);
}

cudaError_t read_device_error(int* value, int reset) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_selscan_device_error, sizeof(int));
  if (e == cudaSuccess && reset) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_selscan_device_error, &zero, sizeof(int));
  }
  return e;
}

}  // namespace selscan

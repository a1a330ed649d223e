// Gradients of the selective-scan forward (the backward pass) for sm_103a.
//
// The forward (include/selscan.h): Δ_t = softplus(x_t), x_t = δ_t + Δ_bias[d], Ā_t = exp(Δ_t A[d,n]),
// h_t = Ā_t h_{t-1} + Δ_t B[b,n,t] u_t, y_t = Σ_n C[b,n,t] h_t + D[d] u_t, out_t = y_t silu(z_t)
// ("Mamba状态空间模型深度解析：挑战Transformer的下一代序列建模范式" §2.1, §3.1; "Mamba架构与SSM模型：
// 高效序列建模技术解析" §2.1, §2.2).  Reverse-mode differentiation runs the recurrence backwards with
// g, the gradient with respect to the state after the step being undone (g = dh_last after the last step):
//   dy_t = dout_t silu(z_t),   dz_t = dout_t y_t σ(z_t)(1 + z_t(1 - σ(z_t))),   G_n = g_n + dy_t C_t[n]
//   dC_t[n] += dy_t h_t[n],    dB_t[n] += G_n Δ_t u_t,    du_t = dy_t D + Δ_t Σ_n G_n B_t[n]
//   dΔ_t = Σ_n G_n (B_t[n] u_t + A_n Ā_t[n] h_{t-1}[n]),  dA_n += Δ_t G_n Ā_t[n] h_{t-1}[n]
//   g_n ← G_n Ā_t[n],   dδ_t = dΔ_t σ(x_t) (softplus' = σ),  dΔ_bias += dδ_t,  dD += dy_t u_t,  dh0 = g.
// The states are recomputed, not stored by the forward: the recomputation the pages describe for
// training ("Mamba状态空间模型深度解析" §2.2).  Phase 1 runs the forward and keeps only the state at the
// start of every chunk of kBT steps (checkpoints, in the call's workspace); phase 2 takes the chunks
// from last to first, reruns each one from its checkpoint keeping its states in shared memory, and
// sweeps it backwards.
//
// Decomposition: a CTA owns kRows channels of one batch entry; 4 lanes share a row, lane q owning
// states [4q, 4q+4) as two float2 pairs (packed fp32x2 arithmetic), lane = 8q + r, so the 8 rows of a
// warp that read one state group read the same B, C values (shared-memory broadcast).  Lane q also owns
// steps [4q, 4q+4) of every chunk: it loads their inputs, forms Δ, Δu, σ(x), σ(z) and dy once, hands
// Δ, Δu and dy to the row's other lanes (by shuffles in phase 1, as records in shared memory in phase 2),
// keeps the row sums of its own steps as the sweep passes them, and after the sweep forms and stores
// those steps' du, dδ and dz, all lanes at once.  The next
// chunk's inputs are loaded into registers while the current one is computed.  The row's lanes add
// their partial sums over states (y, Σ G B, Σ A G Ā h) with two shuffles.  dB and dC are sums over the
// channels of a batch entry: per step a warp adds up its 8 rows' contributions by recursive halving (7
// shuffles leave lane 8q + r holding the sum of value r of {dB of states 4q..4q+3, dC of states
// 4q..4q+3}), the CTA adds its warps in shared memory at the end of the chunk, and one 16-byte atomic add
// per (tensor, state, 4 steps) goes to global memory.  dA, dD and dΔ_bias are summed in registers over
// the sequence and added with one atomic per row and value.
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <type_traits>

#include "selscan_internal.cuh"

namespace selscan {
namespace {

constexpr int kBT = 16;         // steps per chunk (checkpoint interval)
constexpr int kBW = 4;          // warps per CTA
constexpr int kRows = kBW * 8;  // channels per CTA
constexpr int kNS = 16;         // states per row held by the 4 lanes (lanes mask states >= N)
constexpr int kThreads = kBW * 32;
constexpr int kTS = kNS + 4;  // floats per step of the B, C tile: the stagers' column writes spread over banks

// The chunk loops of phase 2 run in groups of kU steps, unrolled within a group and not across groups:
// fully unrolled 16-step loops hoist enough loads to spill at the 168 registers that three CTAs per SM
// allow (four CTAs, at 128 registers, and two, at 255, both measured slower).
constexpr int kU = 4;          // a multiple of 4: a group holds whole step quads
constexpr int kMinBlocks = 3;  // resident CTAs per SM the registers are sized for

struct BwdSmem {
  float bc[2][kBT][kTS];     // B, C of the chunk, [step][state]
  float h[kBW][kBT][32][4];  // per warp: h_{t-1} of every step of the chunk, per lane
  float red[kBW][kBT][32];   // per warp and step: the 8-row sums of dB, dC (lane 8q + r: value r)
  float4 rec[kBW][kBT][8];   // per warp, step and row: (Δ, Δu, dy, 0) from the lane that prepared the step
};

__device__ __forceinline__ float row_sum(float v) {
  v += __shfl_xor_sync(kFull, v, 8);
  v += __shfl_xor_sync(kFull, v, 16);
  return v;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
}

// The raw bits of a lane's four steps of one row: 8 bytes of bf16 or 16 bytes of fp32.
template <typename T>
struct Quad {
  uint32_t w[sizeof(T)];  // 2 words (bf16) or 4 words (fp32)
};

// Load steps [t, t + n) of a row (n = 0..4; zeros past n): one 8- or 16-byte load when all four exist
// and the row is aligned for it.
template <typename T>
__device__ __forceinline__ Quad<T> load_quad(const T* __restrict__ src, int n, bool vec) {
  Quad<T> qd;
  if (vec && n == 4) {
    if constexpr (sizeof(T) == 2) {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(src));
      qd.w[0] = v.x;
      qd.w[1] = v.y;
    } else {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(src));
      qd.w[0] = v.x;
      qd.w[1] = v.y;
      qd.w[2] = v.z;
      qd.w[3] = v.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < static_cast<int>(sizeof(T)); k++) qd.w[k] = 0u;
#pragma unroll
    for (int k = 0; k < 4; k++) {
      if (k >= n) break;
      if constexpr (sizeof(T) == 2) {
        const uint32_t b = __bfloat16_as_ushort(src[k]);
        qd.w[k >> 1] |= (k & 1) ? (b << 16) : b;
      } else {
        qd.w[k] = __float_as_uint(src[k]);
      }
    }
  }
  return qd;
}

template <typename T>
__device__ __forceinline__ float quad_at(const Quad<T>& qd, int k) {
  if constexpr (sizeof(T) == 2) {
    const uint32_t w = qd.w[k >> 1];
    return __uint_as_float((k & 1) ? (w & 0xffff0000u) : (w << 16));
  } else {
    return __uint_as_float(qd.w[k]);
  }
}

// `n` (1..4) consecutive values of one row; one 8- or 16-byte store when all four are written and
// the destination is aligned.
template <typename T>
__device__ __forceinline__ void store4(T* dst, int n, bool vec, const float (&v)[4]) {
  if (vec && n == 4) {
    if constexpr (sizeof(T) == 2) {
      *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
    } else {
      *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 4; k++)
      if (k < n) dst[k] = from_f32<T>(v[k]);
  }
}

// Values of step quad q of a chunk of len steps that exist (0..4).
__device__ __forceinline__ int quad_len(int len, int q) {
  const int n = len - 4 * q;
  return n < 0 ? 0 : (n > 4 ? 4 : n);
}

// Steps in chunk c of a sequence of L steps.
__device__ __forceinline__ int chunk_len(int64_t L, int c) {
  const int64_t left = L - static_cast<int64_t>(c) * kBT;
  return static_cast<int>(left < kBT ? left : kBT);
}

// The B (and C) values of a chunk that thread tid stages: element e = tid + kThreads·j of the
// [tensor][state][step] chunk, j = 0, 1 for B and 2, 3 for C.  Zero past N and past the chunk.
template <typename Tin, int NT>
struct BCStage {
  float v[2 * NT];
  __device__ __forceinline__ void load(const BwdParams& p, int64_t b, int c) {
    const int len = chunk_len(p.seqlen, c);
    const int64_t t0 = static_cast<int64_t>(c) * kBT;
#pragma unroll
    for (int j = 0; j < 2 * NT; j++) {
      const int e = static_cast<int>(threadIdx.x) + kThreads * j;
      const int tensor = e / (kBT * kNS), n = (e / kBT) % kNS, tt = e % kBT;
      float x = 0.f;
      if (n < p.dstate && tt < len)
        x = to_f32(static_cast<const Tin*>(tensor ? p.C : p.B)[(b * p.dstate + n) * p.seqlen + t0 + tt]);
      v[j] = x;
    }
  }
  __device__ __forceinline__ void store(BwdSmem& sm) const {
#pragma unroll
    for (int j = 0; j < 2 * NT; j++) {
      const int e = static_cast<int>(threadIdx.x) + kThreads * j;
      sm.bc[e / (kBT * kNS)][e % kBT][(e / kBT) % kNS] = v[j];
    }
  }
};
static_assert(2 * kThreads == kBT * kNS, "two B values and two C values per thread and chunk");

// Broadcast step i's value from the lane of the row that prepared it (lane 8·(i / 4) + r).
__device__ __forceinline__ float from_prep(const float (&v)[4], int i, int r) {
  return __shfl_sync(kFull, v[i & 3], (i >> 2) * 8 + r);
}

template <typename Tin, typename Tg>
__global__ void __launch_bounds__(kThreads, kMinBlocks) selscan_bwd_kernel(const BwdParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  BwdSmem& sm = *reinterpret_cast<BwdSmem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane & 7, q = lane >> 3;
  const int64_t b = blockIdx.y;
  const int64_t d = static_cast<int64_t>(blockIdx.x) * kRows + warp * 8 + r;
  const bool row_ok = d < p.dim;
  const int64_t dd = row_ok ? d : 0;  // rows past D read channel 0's inputs with dout = 0 and write nothing
  const int64_t grow = b * p.dim + dd;
  const int64_t L = p.seqlen;
  const int N = p.dstate;
  const int nchunks = static_cast<int>((L + kBT - 1) / kBT);
  // This CTA's time block: chunks [cb, ce).
  const int kb = blockIdx.z;
  const int cpb = static_cast<int>(p.tblock / kBT);
  const int cb = kb * cpb, ce = cb + cpb < nchunks ? cb + cpb : nchunks;
  const int64_t rows = p.batch * p.dim;
  const float bias = p.delta_bias ? p.delta_bias[dd] : 0.f;
  const float Dd = p.D ? p.D[dd] : 0.f;
  const bool softplus = p.delta_softplus != 0;
  const Tin* u_row = static_cast<const Tin*>(p.u) + grow * L + 4 * q;
  const Tin* x_row = static_cast<const Tin*>(p.delta) + grow * L + 4 * q;
  const Tin* z_row = p.z ? static_cast<const Tin*>(p.z) + grow * L + 4 * q : nullptr;
  const Tg* go_row = static_cast<const Tg*>(p.dout) + grow * L + 4 * q;
  // The block's start state: h0 for one block, else the carried start state.
  const float* hs = p.nblocks > 1 ? p.hstart + (static_cast<int64_t>(kb) * rows + grow) * kNS : nullptr;
  // This lane's states as pairs: A·log2 e (exponent), A (dΔ), h.
  float2 A2[2], Ar[2], h[2];
#pragma unroll
  for (int k = 0; k < 2; k++) {
    const int n = 4 * q + 2 * k;
    const float a0 = n < N ? p.A[dd * N + n] : 0.f, a1 = n + 1 < N ? p.A[dd * N + n + 1] : 0.f;
    Ar[k] = f2(a0, a1);
    A2[k] = f2(a0 * kLog2e, a1 * kLog2e);
    if (hs) {
      h[k] = f2(row_ok && n < N ? hs[n] : 0.f, row_ok && n + 1 < N ? hs[n + 1] : 0.f);
    } else {
      const bool has = row_ok && p.h0;
      h[k] = f2(has && n < N ? p.h0[grow * N + n] : 0.f, has && n + 1 < N ? p.h0[grow * N + n + 1] : 0.f);
    }
  }
  float4* ck = reinterpret_cast<float4*>(p.ckpt) + grow * nchunks * (kNS / 4) + q;
  // The checkpoints phase 2 reruns chunks from: the forward's (phase 1 skipped), or phase 1's.
  const float4* ckr = p.ckpt_in ? reinterpret_cast<const float4*>(p.ckpt_in) + grow * nchunks * (kNS / 4) + q : ck;

  // ---- phase 1: the forward, keeping the state at the start of every chunk --------------------------
  if (!p.ckpt_in) {
    BCStage<Tin, 1> bs;
    bs.load(p, b, cb);
    const int64_t o0 = static_cast<int64_t>(cb) * kBT;
    Quad<Tin> uq = load_quad(u_row + o0, quad_len(chunk_len(L, cb), q), p.vec_in);
    Quad<Tin> xq = load_quad(x_row + o0, quad_len(chunk_len(L, cb), q), p.vec_in);
    for (int c = cb; c < ce; c++) {
      const int len = chunk_len(L, c);
      __syncthreads();  // the previous chunk's B has been read
      bs.store(sm);
      if (row_ok) ck[static_cast<int64_t>(c) * (kNS / 4)] = make_float4(h[0].x, h[0].y, h[1].x, h[1].y);
      // This lane's steps: Δ and Δu (zero past the chunk: an identity step).
      float dlq[4], duq[4];
#pragma unroll
      for (int m = 0; m < 4; m++) {
        const float x = quad_at(xq, m) + bias;
        const float dl = softplus ? softplus_fast(x) : x;
        const bool in = 4 * q + m < len;
        dlq[m] = in ? dl : 0.f;
        duq[m] = in ? dl * quad_at(uq, m) : 0.f;
      }
      if (c + 1 < ce) {  // the next chunk's inputs, in flight during this one
        const int nlen = chunk_len(L, c + 1);
        bs.load(p, b, c + 1);
        uq = load_quad(u_row + static_cast<int64_t>(c + 1) * kBT, quad_len(nlen, q), p.vec_in);
        xq = load_quad(x_row + static_cast<int64_t>(c + 1) * kBT, quad_len(nlen, q), p.vec_in);
      }
      __syncthreads();
      // Whole chunks (all but possibly the last) run without per-step bounds checks.
      auto scan = [&](auto whole) {
#pragma unroll
        for (int i = 0; i < kBT; i++) {
          if (!decltype(whole)::value && i >= len) break;
          const float dl = from_prep(dlq, i, r), du = from_prep(duq, i, r);
          const float4 Bv = *reinterpret_cast<const float4*>(&sm.bc[0][i][4 * q]);
          const float2 d2 = f2(dl, dl), du2 = f2(du, du);
          const float2 e0 = mul2s(d2, A2[0]), e1 = mul2s(d2, A2[1]);
          const float2 a0 = f2(ex2_approx(e0.x), ex2_approx(e0.y)), a1 = f2(ex2_approx(e1.x), ex2_approx(e1.y));
          h[0] = fma2s(a0, h[0], mul2s(du2, f2(Bv.x, Bv.y)));
          h[1] = fma2s(a1, h[1], mul2s(du2, f2(Bv.z, Bv.w)));
        }
      };
      if (len == kBT)
        scan(std::true_type{});
      else
        scan(std::false_type{});
    }
  }

  // ---- phase 2: the chunks from last to first ----------------------------------------------------------
  // The gradient with respect to the block's end state: dh_last for one block, else the carried one.
  const float* ge = p.nblocks > 1 ? p.gend + (static_cast<int64_t>(kb) * rows + grow) * kNS : nullptr;
  float2 g[2], dA[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
  for (int k = 0; k < 2; k++) {
    const int n = 4 * q + 2 * k;
    if (ge) {
      g[k] = f2(row_ok && n < N ? ge[n] : 0.f, row_ok && n + 1 < N ? ge[n + 1] : 0.f);
    } else {
      const bool has = row_ok && p.dh_last;
      g[k] = f2(has && n < N ? p.dh_last[grow * N + n] : 0.f, has && n + 1 < N ? p.dh_last[grow * N + n + 1] : 0.f);
    }
  }
  float dD = 0.f, dbias = 0.f;  // over this lane's steps
  const bool has_z = p.z != nullptr;
  const bool b2 = r & 4, b1 = r & 2, b0 = r & 1;
  BCStage<Tin, 2> bs;
  bs.load(p, b, ce - 1);
  Quad<Tin> uq, xq, zq;
  Quad<Tg> gq;
  {
    const int n0 = quad_len(chunk_len(L, ce - 1), q);
    const int64_t o = static_cast<int64_t>(ce - 1) * kBT;
    uq = load_quad(u_row + o, n0, p.vec_in);
    xq = load_quad(x_row + o, n0, p.vec_in);
    if (has_z) zq = load_quad(z_row + o, n0, p.vec_in);
    gq = load_quad(go_row + o, n0, p.vec_dout);
  }
  // (Rows past D have no checkpoints: channel 0's belong to its own row.  Their dout is 0, so every
  // contribution they make is 0 whatever their states are.)
  const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c = ce - 1; c >= cb; c--) {
    const int64_t t0 = static_cast<int64_t>(c) * kBT;
    const int len = chunk_len(L, c);
    const int nq = quad_len(len, q);
    __syncthreads();  // the previous chunk's B, C and dB/dC sums have been read
    bs.store(sm);
    float4 c4 = row_ok ? ckr[static_cast<int64_t>(c) * (kNS / 4)] : zero4;
    // (A forward with fewer than 16 states leaves the slots of states >= N unwritten.)
    if (4 * q + 0 >= N) c4.x = 0.f;
    if (4 * q + 1 >= N) c4.y = 0.f;
    if (4 * q + 2 >= N) c4.z = 0.f;
    if (4 * q + 3 >= N) c4.w = 0.f;
    float2 hc[2] = {f2(c4.x, c4.y), f2(c4.z, c4.w)};
    // This lane's steps: Δ, Δu, σ(x), dy and the factor of y in dz (zero past the chunk).
    float dlq[4], duq[4], sgq[4], dyq[4], fzq[4], uqv[4];
#pragma unroll
    for (int m = 0; m < 4; m++) {
      const bool in = m < nq;
      const float x = quad_at(xq, m) + bias, uu = quad_at(uq, m);
      float dl = x, sg = 1.f;
      if (softplus) softplus_sigmoid(x, dl, sg);
      const float go = row_ok ? quad_at(gq, m) : 0.f;
      float dy = go, fz = 0.f;
      if (has_z) {
        const float zz = quad_at(zq, m);
        const float sz = rcp_approx(1.f + ex2_approx(-zz * kLog2e));
        dy = go * zz * sz;
        fz = go * sz * fmaf(zz, 1.f - sz, 1.f);
      }
      dlq[m] = in ? dl : 0.f;
      duq[m] = in ? dl * uu : 0.f;
      sgq[m] = sg;
      dyq[m] = in ? dy : 0.f;
      fzq[m] = fz;
      uqv[m] = uu;
    }
    // The row's lanes read these steps' Δ, Δu and dy from the records (the previous chunk's readers are
    // done: the CTA synchronised above).
#pragma unroll
    for (int m = 0; m < 4; m++) sm.rec[warp][4 * q + m][r] = make_float4(dlq[m], duq[m], dyq[m], 0.f);
    if (c > cb) {  // the next chunk (in scan order: the previous one in time), in flight during this one
      const int n1 = quad_len(chunk_len(L, c - 1), q);
      const int64_t o = static_cast<int64_t>(c - 1) * kBT;
      bs.load(p, b, c - 1);
      uq = load_quad(u_row + o, n1, p.vec_in);
      xq = load_quad(x_row + o, n1, p.vec_in);
      if (has_z) zq = load_quad(z_row + o, n1, p.vec_in);
      gq = load_quad(go_row + o, n1, p.vec_dout);
    }
    __syncthreads();
    // Whole chunks (all but possibly the first) run without per-step bounds checks.
    auto rerun_and_sweep = [&](auto whole) {
      constexpr bool W = decltype(whole)::value;
      // Rerun the chunk from its checkpoint: h_{t-1} of every step to shared memory, y for dz.  The steps
      // run in quads (qd: the quad, prepared by lane qd of the row; k: the step within it).
      float yq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
      for (int o = 0; o < kBT / kU; o++) {
#pragma unroll
        for (int k = 0; k < kU; k++) {
          const int i = kU * o + k, qd = i >> 2;
          if (!W && i >= len) continue;
          const float4 rc = sm.rec[warp][i][r];
          const float dl = rc.x, du = rc.y;
          *reinterpret_cast<float4*>(sm.h[warp][i][lane]) = make_float4(hc[0].x, hc[0].y, hc[1].x, hc[1].y);
          const float4 Bv = *reinterpret_cast<const float4*>(&sm.bc[0][i][4 * q]);
          const float2 d2 = f2(dl, dl), du2 = f2(du, du);
          const float2 e0 = mul2s(d2, A2[0]), e1 = mul2s(d2, A2[1]);
          const float2 a0 = f2(ex2_approx(e0.x), ex2_approx(e0.y)), a1 = f2(ex2_approx(e1.x), ex2_approx(e1.y));
          hc[0] = fma2s(a0, hc[0], mul2s(du2, f2(Bv.x, Bv.y)));
          hc[1] = fma2s(a1, hc[1], mul2s(du2, f2(Bv.z, Bv.w)));
          if (has_z) {
            const float4 Cv = *reinterpret_cast<const float4*>(&sm.bc[1][i][4 * q]);
            const float2 yp2 = fma2s(f2(Cv.z, Cv.w), hc[1], mul2s(f2(Cv.x, Cv.y), hc[0]));
            const float y = row_sum(yp2.x + yp2.y);
            if (qd == q) yq[k & 3] = y;  // kept by the lane that prepared the step
          }
        }
      }
      if (has_z && row_ok && nq > 0) {
        float dzs[4];
#pragma unroll
        for (int m = 0; m < 4; m++) dzs[m] = fmaf(Dd, uqv[m], yq[m]) * fzq[m];
        store4(static_cast<Tin*>(p.dz) + grow * L + t0 + 4 * q, nq, p.vec_grad, dzs);
      }
      __syncwarp();
      // The reverse sweep of the chunk; hn holds h_t (the state after the step being undone).
      float2 hn[2] = {hc[0], hc[1]};
      // Σ_n G B and Σ_n A G Ā h of the steps this lane prepared (zero for steps past the chunk).
      float Sq[4] = {0.f, 0.f, 0.f, 0.f}, Tq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
      for (int o = kBT / kU - 1; o >= 0; o--) {
#pragma unroll
        for (int k = kU - 1; k >= 0; k--) {
          const int i = kU * o + k, qd = i >> 2;
          if (!W && i >= len) continue;
          const float4 hp4 = *reinterpret_cast<const float4*>(sm.h[warp][i][lane]);
          const float4 Bv = *reinterpret_cast<const float4*>(&sm.bc[0][i][4 * q]);
          const float4 Cv = *reinterpret_cast<const float4*>(&sm.bc[1][i][4 * q]);
          const float2 hp[2] = {f2(hp4.x, hp4.y), f2(hp4.z, hp4.w)};
          const float2 B2[2] = {f2(Bv.x, Bv.y), f2(Bv.z, Bv.w)}, C2[2] = {f2(Cv.x, Cv.y), f2(Cv.z, Cv.w)};
          const float4 rc = sm.rec[warp][i][r];
          const float dl = rc.x, du = rc.y, dy = rc.z;
          const float2 d2 = f2(dl, dl), dy2 = f2(dy, dy), du2 = f2(du, du);
          float2 sGB = f2(0.f, 0.f), sAGw = f2(0.f, 0.f), vB[2], vC[2];
#pragma unroll
          for (int j = 0; j < 2; j++) {
            const float2 e = mul2s(d2, A2[j]);
            const float2 ab = f2(ex2_approx(e.x), ex2_approx(e.y));
            const float2 G = fma2s(dy2, C2[j], g[j]);
            const float2 t = mul2s(G, mul2s(ab, hp[j]));  // G Ā h_{t-1}
            vB[j] = mul2s(G, du2);                        // this row's dB
            vC[j] = mul2s(dy2, hn[j]);                    // this row's dC
            sGB = fma2s(G, B2[j], sGB);
            sAGw = fma2s(Ar[j], t, sAGw);
            dA[j] = fma2s(t, d2, dA[j]);
            g[j] = mul2s(G, ab);
            hn[j] = hp[j];
          }
          // dB, dC: the sum over the warp's 8 rows by recursive halving; lane 8q + r ends with value r of
          // {dB of states 4q..4q+3, dC of states 4q..4q+3}.
          const float v[8] = {vB[0].x, vB[0].y, vB[1].x, vB[1].y, vC[0].x, vC[0].y, vC[1].x, vC[1].y};
          float w4[4], w2[2];
#pragma unroll
          for (int j = 0; j < 4; j++) {
            const float send = b2 ? v[j] : v[4 + j];
            w4[j] = (b2 ? v[4 + j] : v[j]) + __shfl_xor_sync(kFull, send, 4);
          }
#pragma unroll
          for (int j = 0; j < 2; j++) {
            const float send = b1 ? w4[j] : w4[2 + j];
            w2[j] = (b1 ? w4[2 + j] : w4[j]) + __shfl_xor_sync(kFull, send, 2);
          }
          sm.red[warp][i][lane] = (b0 ? w2[1] : w2[0]) + __shfl_xor_sync(kFull, b0 ? w2[0] : w2[1], 1);
          const float S = row_sum(sGB.x + sGB.y), T = row_sum(sAGw.x + sAGw.y);
          if (qd == q) {  // kept by the lane that prepared the step
            Sq[k & 3] = S;
            Tq[k & 3] = T;
          }
        }
      }
      // The gradients of this lane's own steps, all lanes at once.
      float dus[4], dxs[4];
#pragma unroll
      for (int m = 0; m < 4; m++) {
        const float dx = fmaf(uqv[m], Sq[m], Tq[m]) * sgq[m];
        dus[m] = fmaf(dyq[m], Dd, dlq[m] * Sq[m]);
        dxs[m] = dx;
        dD = fmaf(dyq[m], uqv[m], dD);
        dbias += dx;
      }
      if (row_ok && nq > 0) {
        store4(static_cast<Tin*>(p.du) + grow * L + t0 + 4 * q, nq, p.vec_grad, dus);
        store4(static_cast<Tin*>(p.ddelta) + grow * L + t0 + 4 * q, nq, p.vec_grad, dxs);
      }
    };
    if (len == kBT)
      rerun_and_sweep(std::true_type{});
    else
      rerun_and_sweep(std::false_type{});
    __syncthreads();
    // dB, dC of the chunk: the CTA's warps added up, then one atomic add per (tensor, state, 4 steps).
    {
      // 128 threads: warp = step quad, lane = (tensor, state), so the 32 lanes of a warp read 32 different
      // banks of the warps' sums (lane 8q + r of a warp's sums lies in bank 8q + r).
      const int j = threadIdx.x;
      const int s4 = j >> 5, tensor = (j >> 4) & 1, n = j & 15;
      const int src = (n >> 2) * 8 + tensor * 4 + (n & 3);
      const int steps = quad_len(len, s4);
      if (n < N && steps > 0) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int w = 0; w < kBW; w++)
#pragma unroll
          for (int k = 0; k < 4; k++) acc[k] += sm.red[w][4 * s4 + k][src];
        float* dst = (tensor ? p.dC : p.dB) + (b * N + n) * L + t0 + 4 * s4;
        if (p.vec_dbc && steps == 4) {
          atomicAdd(reinterpret_cast<float4*>(dst), make_float4(acc[0], acc[1], acc[2], acc[3]));
        } else {
#pragma unroll
          for (int k = 0; k < 4; k++)
            if (k < steps) atomicAdd(dst + k, acc[k]);
        }
      }
    }
  }
  dD = row_sum(dD);
  dbias = row_sum(dbias);
  if (!row_ok) return;
#pragma unroll
  for (int k = 0; k < 2; k++) {
    const int n = 4 * q + 2 * k;
    const bool first = kb == 0;  // the block whose start is h0
    if (n < N) {
      if (p.dh0 && first) p.dh0[grow * N + n] = g[k].x;
      atomicAdd(p.dA + dd * N + n, dA[k].x);
    }
    if (n + 1 < N) {
      if (p.dh0 && first) p.dh0[grow * N + n + 1] = g[k].y;
      atomicAdd(p.dA + dd * N + n + 1, dA[k].y);
    }
  }
  if (q == 0) {
    if (p.dD) atomicAdd(p.dD + dd, dD);
    if (p.ddelta_bias) atomicAdd(p.ddelta_bias + dd, dbias);
  }
}

static_assert(kThreads == 2 * kNS * kBT / 4, "one thread per (tensor, state, step quad) of a chunk");

// Summaries of the time blocks (every block computes both; the carries leave the first block's f and
// the last block's e unused).  Over block kb, from a zero start, in one forward sweep:
//   e = the end state (h_t = Ā_t h_{t-1} + Δ_t u_t B_t from h = 0),
//   f = Σ_t (Π_{s ≤ r ≤ t} Ā_r) dy_t C_t, the gradient with respect to the state before the block that
//       the block's dy contributes when the gradient after it is 0 (g ← (g + dy_t C_t) Ā_t undone from
//       the block's end),
//   ΣΔ, whose 2^(A·log2e·ΣΔ) is the product of the block's Ā (it carries h forward and g backward).
template <typename Tin, typename Tg>
__global__ void __launch_bounds__(kThreads) selscan_bwd_summary_kernel(const BwdParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  BwdSmem& sm = *reinterpret_cast<BwdSmem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane & 7, q = lane >> 3;
  const int64_t b = blockIdx.y;
  const int64_t d = static_cast<int64_t>(blockIdx.x) * kRows + warp * 8 + r;
  const bool row_ok = d < p.dim;
  const int64_t dd = row_ok ? d : 0;
  const int64_t grow = b * p.dim + dd;
  const int64_t L = p.seqlen;
  const int N = p.dstate;
  const int nchunks = static_cast<int>((L + kBT - 1) / kBT);
  const int kb = blockIdx.z;
  const int cpb = static_cast<int>(p.tblock / kBT);
  const int cb = kb * cpb, ce = cb + cpb < nchunks ? cb + cpb : nchunks;
  const float bias = p.delta_bias ? p.delta_bias[dd] : 0.f;
  const bool softplus = p.delta_softplus != 0, has_z = p.z != nullptr;
  const Tin* u_row = static_cast<const Tin*>(p.u) + grow * L + 4 * q;
  const Tin* x_row = static_cast<const Tin*>(p.delta) + grow * L + 4 * q;
  const Tin* z_row = has_z ? static_cast<const Tin*>(p.z) + grow * L + 4 * q : nullptr;
  const Tg* go_row = static_cast<const Tg*>(p.dout) + grow * L + 4 * q;
  float2 A2[2], e[2], P[2], f[2];
#pragma unroll
  for (int k = 0; k < 2; k++) {
    const int n = 4 * q + 2 * k;
    A2[k] = f2(n < N ? p.A[dd * N + n] * kLog2e : 0.f, n + 1 < N ? p.A[dd * N + n + 1] * kLog2e : 0.f);
    e[k] = f2(0.f, 0.f);
    P[k] = f2(1.f, 1.f);
    f[k] = f2(0.f, 0.f);
  }
  float sumD = 0.f;  // over this lane's steps
  BCStage<Tin, 2> bs;
  bs.load(p, b, cb);
  Quad<Tin> uq, xq, zq;
  Quad<Tg> gq;
  auto load_inputs = [&](int c) {
    const int n = quad_len(chunk_len(L, c), q);
    const int64_t o = static_cast<int64_t>(c) * kBT;
    uq = load_quad(u_row + o, n, p.vec_in);
    xq = load_quad(x_row + o, n, p.vec_in);
    if (has_z) zq = load_quad(z_row + o, n, p.vec_in);
    gq = load_quad(go_row + o, n, p.vec_dout);
  };
  load_inputs(cb);
  for (int c = cb; c < ce; c++) {
    const int len = chunk_len(L, c);
    const int nq = quad_len(len, q);
    __syncthreads();
    bs.store(sm);
    float dlq[4], duq[4], dyq[4];
#pragma unroll
    for (int m = 0; m < 4; m++) {
      const bool in = m < nq;
      const float x = quad_at(xq, m) + bias;
      const float dl = softplus ? softplus_fast(x) : x;
      const float go = row_ok ? quad_at(gq, m) : 0.f;
      float dy = go;
      if (has_z) {
        const float zz = quad_at(zq, m);
        dy = go * zz * rcp_approx(1.f + ex2_approx(-zz * kLog2e));
      }
      dlq[m] = in ? dl : 0.f;
      duq[m] = in ? dl * quad_at(uq, m) : 0.f;
      dyq[m] = in ? dy : 0.f;
      sumD += dlq[m];
    }
    if (c + 1 < ce) {
      bs.load(p, b, c + 1);
      load_inputs(c + 1);
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kBT; i++) {
      if (i >= len) break;
      const float dl = from_prep(dlq, i, r), du = from_prep(duq, i, r), dy = from_prep(dyq, i, r);
      const float4 Bv = *reinterpret_cast<const float4*>(&sm.bc[0][i][4 * q]);
      const float4 Cv = *reinterpret_cast<const float4*>(&sm.bc[1][i][4 * q]);
      const float2 d2 = f2(dl, dl), du2 = f2(du, du), dy2 = f2(dy, dy);
      const float2 B2[2] = {f2(Bv.x, Bv.y), f2(Bv.z, Bv.w)}, C2[2] = {f2(Cv.x, Cv.y), f2(Cv.z, Cv.w)};
#pragma unroll
      for (int k = 0; k < 2; k++) {
        const float2 x2 = mul2s(d2, A2[k]);
        const float2 a = f2(ex2_approx(x2.x), ex2_approx(x2.y));
        e[k] = fma2s(a, e[k], mul2s(du2, B2[k]));
        P[k] = mul2s(P[k], a);
        f[k] = fma2s(P[k], mul2s(dy2, C2[k]), f[k]);
      }
    }
  }
  sumD = row_sum(sumD);
  if (!row_ok) return;
  const int64_t rows = p.batch * p.dim;
  float* o = p.summ + (static_cast<int64_t>(kb) * rows + grow) * (2 * kNS) + 4 * q;
  *reinterpret_cast<float4*>(o) = make_float4(e[0].x, e[0].y, e[1].x, e[1].y);
  *reinterpret_cast<float4*>(o + kNS) = make_float4(f[0].x, f[0].y, f[1].x, f[1].y);
  if (q == 0) p.sumd[static_cast<int64_t>(kb) * rows + grow] = sumD;
}

// The carries: one thread per (row, state).  Forward: every block's start state from h0 and the
// blocks' end states, h ← 2^(A·log2e·ΣΔ)·h + e.  Backward: every block's end gradient from dh_last,
// g ← 2^(A·log2e·ΣΔ)·g + f, block by block from the last.
__global__ void __launch_bounds__(256) selscan_bwd_carry_kernel(const BwdParams p) {
  const int64_t rows = p.batch * p.dim;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t row = tid / kNS;
  const int n = static_cast<int>(tid % kNS);
  if (row >= rows) return;
  const int N = p.dstate;
  const int nb = p.nblocks;
  const int64_t d = row % p.dim;
  const float a2 = n < N ? p.A[d * N + n] * kLog2e : 0.f;
  float h = (n < N && p.h0) ? p.h0[row * N + n] : 0.f;
  for (int k = 0; k < nb; k++) {
    p.hstart[(static_cast<int64_t>(k) * rows + row) * kNS + n] = h;
    const int64_t s = static_cast<int64_t>(k) * rows + row;
    h = fmaf(ex2_approx(a2 * p.sumd[s]), h, p.summ[s * (2 * kNS) + n]);
  }
  float g = (n < N && p.dh_last) ? p.dh_last[row * N + n] : 0.f;
  for (int k = nb - 1; k >= 0; k--) {
    p.gend[(static_cast<int64_t>(k) * rows + row) * kNS + n] = g;
    const int64_t s = static_cast<int64_t>(k) * rows + row;
    g = fmaf(ex2_approx(a2 * p.sumd[s]), g, p.summ[s * (2 * kNS) + kNS + n]);
  }
}

// Time blocks: enough that the CTAs of all blocks fill the resident slots once (3 CTAs per SM), with
// blocks of at least 256 steps; one block when the rows alone fill the GPU.  SELSCAN_BWD_TBLOCKS forces
// a count.
struct BwdPlan {
  int nblocks;
  int64_t tblock;
};
BwdPlan plan_bwd(int64_t batch, int64_t dim, int64_t L) {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0, v = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    sms = v > 0 ? v : 148;
  }
  const int64_t ctas = ((dim + kRows - 1) / kRows) * batch, slots = static_cast<int64_t>(sms) * kMinBlocks;
  int64_t nb = 1;
  const char* env = getenv("SELSCAN_BWD_TBLOCKS");
  if (env) {
    nb = atoi(env);
  } else if (2 * ctas < slots) {
    nb = slots / (ctas > 0 ? ctas : 1);
    const int64_t by_len = L / 256;
    if (nb > by_len) nb = by_len;
  }
  if (nb < 1) nb = 1;
  int64_t tb = (L + nb - 1) / nb;
  tb = (tb + kBT - 1) / kBT * kBT;
  if (tb < kBT) tb = kBT;
  BwdPlan pl;
  pl.tblock = tb;
  pl.nblocks = static_cast<int>((L + tb - 1) / tb);
  if (pl.nblocks < 1) pl.nblocks = 1;
  return pl;
}

size_t align_floats(size_t n) { return (n + 3) / 4 * 4; }

template <typename Tin, typename Tg>
cudaError_t launch_typed(const BwdParams& p, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>((p.dim + kRows - 1) / kRows), static_cast<unsigned>(p.batch),
                  static_cast<unsigned>(p.nblocks));
  const int smem = static_cast<int>(sizeof(BwdSmem));
  cudaError_t e =
      cudaFuncSetAttribute(selscan_bwd_kernel<Tin, Tg>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (p.nblocks > 1) {
    e = cudaFuncSetAttribute(selscan_bwd_summary_kernel<Tin, Tg>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    selscan_bwd_summary_kernel<Tin, Tg><<<grid, kThreads, smem, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t threads = p.batch * p.dim * kNS;
    selscan_bwd_carry_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launches(2);
  }
  selscan_bwd_kernel<Tin, Tg><<<grid, kThreads, smem, s>>>(p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

size_t bwd_workspace_bytes(int64_t batch, int64_t dim, int64_t seqlen, bool with_ckpt) {
  const size_t rows = static_cast<size_t>(batch) * static_cast<size_t>(dim);
  size_t floats = with_ckpt ? rows * static_cast<size_t>((seqlen + kBT - 1) / kBT) * kNS : 0;  // checkpoints
  const BwdPlan pl = plan_bwd(batch, dim, seqlen);
  if (pl.nblocks > 1) {
    const size_t nb = static_cast<size_t>(pl.nblocks);
    floats += nb * rows * 2 * kNS + align_floats(nb * rows) + 2 * nb * rows * kNS;
  }
  return sizeof(float) * floats;
}

cudaError_t launch_bwd(const BwdParams& p_in, selscan_dtype_t in_dtype, selscan_dtype_t dout_dtype, void* workspace,
                       cudaStream_t s) {
  BwdParams p = p_in;
  const bool own_ckpt = p.ckpt_in == nullptr;
  const size_t ws_bytes = bwd_workspace_bytes(p.batch, p.dim, p.seqlen, own_ckpt);
  void* own = nullptr;
  if (!workspace && ws_bytes > 0) {
    const cudaError_t e = cudaMallocAsync(&own, ws_bytes, s);
    if (e != cudaSuccess) return e;
    workspace = own;
  }
  const BwdPlan pl = plan_bwd(p.batch, p.dim, p.seqlen);
  const size_t rows = static_cast<size_t>(p.batch * p.dim), nb = static_cast<size_t>(pl.nblocks);
  p.nblocks = pl.nblocks;
  p.tblock = pl.tblock;
  float* base = static_cast<float*>(workspace);
  p.ckpt = own_ckpt ? base : nullptr;
  if (pl.nblocks > 1) {
    p.summ = base + (own_ckpt ? rows * static_cast<size_t>((p.seqlen + kBT - 1) / kBT) * kNS : 0);
    p.sumd = p.summ + nb * rows * 2 * kNS;
    p.hstart = p.sumd + align_floats(nb * rows);
    p.gend = p.hstart + nb * rows * kNS;
  }
  cudaError_t e = cudaSuccess;
  if (own_ckpt) {
    // The forward pass by the row-sequential kernel, checkpoints only, where it needs no time blocks: then
    // the backward reruns its chunks from those checkpoints and skips its own phase 1.
    FwdParams f;
    memset(&f, 0, sizeof f);
    const int64_t vin = in_dtype == SELSCAN_F32 ? 4 : 8;  // elements per 16 bytes
    auto a16 = [](const void* q) { return reinterpret_cast<uintptr_t>(q) % 16 == 0; };
    f.batch = p.batch;
    f.dim = p.dim;
    f.seqlen = p.seqlen;
    f.dstate = p.dstate;
    f.u = p.u;
    f.delta = p.delta;
    f.B = p.B;
    f.C = p.C;
    f.A = p.A;
    f.delta_bias = p.delta_bias;
    f.h0 = p.h0;
    f.delta_softplus = p.delta_softplus;
    f.vec_in = a16(p.u) && a16(p.delta) && p.seqlen % vin == 0;
    f.vec_bc = a16(p.B) && a16(p.C) && p.seqlen % vin == 0;
    f.vec_stage = f.vec_in && f.vec_bc;
    f.tblock = p.seqlen;
    f.nblocks = 1;
    f.ckpt = p.ckpt;
    f.ckpt_chunks = (p.seqlen + kBT - 1) / kBT;
    f.ckpt_only = 1;
    bool launched = false;
    if (launch_ckpt_pass(f, in_dtype, s, &launched) == cudaSuccess && launched) {
      p.ckpt_in = p.ckpt;
    } else {
      // The pass could not be set up (nothing of it ran): the backward kernel forms the checkpoints.  An
      // error that outlives the call (a device fault) is reported by the backward kernel's own launch.
      (void)cudaGetLastError();
    }
  }
  if (e == cudaSuccess) {
    if (in_dtype == SELSCAN_F32)
      e = dout_dtype == SELSCAN_F32 ? launch_typed<float, float>(p, s) : launch_typed<float, __nv_bfloat16>(p, s);
    else
      e = dout_dtype == SELSCAN_F32 ? launch_typed<__nv_bfloat16, float>(p, s)
                                    : launch_typed<__nv_bfloat16, __nv_bfloat16>(p, s);
  }
  if (own) {
    const cudaError_t ef = cudaFreeAsync(own, s);
    if (e == cudaSuccess) e = ef;
  }
  return e;
}

}  // namespace selscan

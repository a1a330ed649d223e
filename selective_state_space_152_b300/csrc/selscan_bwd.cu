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
// states [4q, 4q+4) (lane = 8q + r), so the 8 rows of a warp that read one state group read the same
// B, C values (shared-memory broadcast).  The row's lanes add their partial sums (y, Σ G B, Σ A G Ā h)
// with two shuffles.  dB and dC are sums over the channels of a batch entry: per step a warp adds up
// its 8 rows' contributions by recursive halving (7 shuffles leave lane 8q + r holding the sum of value
// r of {dB of states 4q..4q+3, dC of states 4q..4q+3}), the CTA adds its warps in shared memory at the
// end of the chunk, and one 16-byte atomic add per (tensor, state, 4 steps) goes to global memory.  dA,
// dD and dΔ_bias are summed per lane in registers over the sequence and added with one atomic per row.
#include "selscan_internal.cuh"

namespace selscan {
namespace {

constexpr int kBT = 16;         // steps per chunk (checkpoint interval)
constexpr int kBW = 4;          // warps per CTA
constexpr int kRows = kBW * 8;  // channels per CTA
constexpr int kNS = 16;         // states per row held by the 4 lanes (lanes mask states >= N)

struct BwdSmem {
  float bc[2][kBT][kNS];     // B, C of the chunk, [step][state]
  float h[kBW][kBT][32][4];  // per warp: h_{t-1} of every step of the chunk, per lane
  float red[kBW][kBT][32];   // per warp and step: the 8-row sums of dB, dC (lane 8q + r: value r)
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

// softplus(x) and its derivative σ(x) from one exponential: with e = exp(-|x|), softplus = max(x, 0) +
// log(1 + e) (as softplus_fast evaluates it) and σ(x) = 1/(1 + e) for x ≥ 0, e/(1 + e) for x < 0.
__device__ __forceinline__ void softplus_sigmoid(float x, float& sp, float& sg) {
  const float e = ex2_approx(-fabsf(x) * kLog2e);
  const float big = lg2_approx(1.f + e) * kLn2;
  const float small = e * fmaf(e, fmaf(e, fmaf(e, -0.25f, 0.33333334f), -0.5f), 1.f);
  sp = fmaxf(x, 0.f) + (e >= 0.0625f ? big : small);
  sg = (x >= 0.f ? 1.f : e) * rcp_approx(1.f + e);
}

// Up to kBT consecutive values of one row as fp32: 16-byte vector loads when the chunk is whole and the
// row is aligned, else element by element (zeros past len).
template <typename T>
__device__ __forceinline__ void load_chunk(const T* __restrict__ src, int len, bool vec, float (&v)[kBT]) {
  if (vec && len == kBT) {
    if constexpr (sizeof(T) == 2) {
      const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
      for (int j = 0; j < kBT / 8; j++) {
        const uint4 w = __ldg(s + j);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; k++) {
          v[8 * j + 2 * k] = __uint_as_float(ws[k] << 16);
          v[8 * j + 2 * k + 1] = __uint_as_float(ws[k] & 0xffff0000u);
        }
      }
    } else {
      const float4* s = reinterpret_cast<const float4*>(src);
#pragma unroll
      for (int j = 0; j < kBT / 4; j++) {
        const float4 w = __ldg(s + j);
        v[4 * j] = w.x;
        v[4 * j + 1] = w.y;
        v[4 * j + 2] = w.z;
        v[4 * j + 3] = w.w;
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < kBT; i++) v[i] = i < len ? to_f32(src[i]) : 0.f;
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

// B (ntensors = 1) or B and C (2) of steps [t0, t0 + len) of batch entry b as [step][state], zeros past
// N and past len.
template <typename Tin>
__device__ __forceinline__ void stage_bc(BwdSmem& sm, const BwdParams& p, int64_t b, int64_t t0, int len,
                                         int ntensors) {
  const Tin* Bp = static_cast<const Tin*>(p.B);
  const Tin* Cp = static_cast<const Tin*>(p.C);
  for (int i = threadIdx.x; i < ntensors * kBT * kNS; i += kBW * 32) {
    const int tensor = i / (kBT * kNS), rest = i % (kBT * kNS), n = rest / kBT, tt = rest % kBT;
    float v = 0.f;
    if (n < p.dstate && tt < len) v = to_f32((tensor ? Cp : Bp)[(b * p.dstate + n) * p.seqlen + t0 + tt]);
    sm.bc[tensor][tt][n] = v;
  }
}

// Keep `v` (the value of step i of the chunk, equal on the row's 4 lanes) in the slot of the lane q that
// stores steps [4q, 4q + 4).
__device__ __forceinline__ void keep_slot(float (&slot)[4], int i, int q, float v) {
  if ((i >> 2) == q) slot[i & 3] = v;
}

// Values of step quad q of a chunk of len steps that exist (0..4).
__device__ __forceinline__ int quad_len(int len, int q) {
  const int n = len - 4 * q;
  return n < 0 ? 0 : (n > 4 ? 4 : n);
}

template <typename Tin, typename Tg>
__global__ void __launch_bounds__(kBW * 32, 3) selscan_bwd_kernel(const BwdParams p) {
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
  const float bias = p.delta_bias ? p.delta_bias[dd] : 0.f;
  const float Dd = p.D ? p.D[dd] : 0.f;
  const Tin* u_row = static_cast<const Tin*>(p.u) + grow * L;
  const Tin* x_row = static_cast<const Tin*>(p.delta) + grow * L;
  const Tin* z_row = p.z ? static_cast<const Tin*>(p.z) + grow * L : nullptr;
  const Tg* go_row = static_cast<const Tg*>(p.dout) + grow * L;
  float A2[4], Araw[4], h[4];
#pragma unroll
  for (int k = 0; k < 4; k++) {
    const int n = 4 * q + k;
    Araw[k] = n < N ? p.A[dd * N + n] : 0.f;
    A2[k] = Araw[k] * kLog2e;
    h[k] = (n < N && row_ok && p.h0) ? p.h0[grow * N + n] : 0.f;
  }
  float4* ck = reinterpret_cast<float4*>(p.ckpt) + grow * nchunks * (kNS / 4) + q;

  // ---- phase 1: the forward, keeping the state at the start of every chunk --------------------------
  for (int c = 0; c < nchunks; c++) {
    const int64_t t0 = static_cast<int64_t>(c) * kBT;
    const int len = static_cast<int>(L - t0 < kBT ? L - t0 : kBT);
    __syncthreads();  // the previous chunk's B has been read
    stage_bc<Tin>(sm, p, b, t0, len, 1);
    if (row_ok) ck[static_cast<int64_t>(c) * (kNS / 4)] = make_float4(h[0], h[1], h[2], h[3]);
    float uv[kBT], xv[kBT];
    load_chunk(u_row + t0, len, p.vec_in, uv);
    load_chunk(x_row + t0, len, p.vec_in, xv);
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kBT; i++) {
      if (i >= len) break;
      const float x = xv[i] + bias;
      const float dl = p.delta_softplus ? softplus_fast(x) : x;
      const float du = dl * uv[i];
      const float4 Bv = *reinterpret_cast<const float4*>(&sm.bc[0][i][4 * q]);
      const float Bk[4] = {Bv.x, Bv.y, Bv.z, Bv.w};
#pragma unroll
      for (int k = 0; k < 4; k++) h[k] = fmaf(ex2_approx(dl * A2[k]), h[k], du * Bk[k]);
    }
  }

  // ---- phase 2: the chunks from last to first ----------------------------------------------------------
  float g[4], dA[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int k = 0; k < 4; k++) {
    const int n = 4 * q + k;
    g[k] = (n < N && row_ok && p.dh_last) ? p.dh_last[grow * N + n] : 0.f;
  }
  float dD = 0.f, dbias = 0.f;
  const bool has_z = p.z != nullptr;
  for (int c = nchunks - 1; c >= 0; c--) {
    const int64_t t0 = static_cast<int64_t>(c) * kBT;
    const int len = static_cast<int>(L - t0 < kBT ? L - t0 : kBT);
    __syncthreads();  // the previous chunk's B, C and dB/dC sums have been read
    stage_bc<Tin>(sm, p, b, t0, len, 2);
    // (Rows past D have no checkpoints: channel 0's belong to its own row.  Their dout is 0, so every
    // contribution they make is 0 whatever their states are.)
    const float4 c4 = row_ok ? ck[static_cast<int64_t>(c) * (kNS / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
    float hc[4] = {c4.x, c4.y, c4.z, c4.w};
    float uv[kBT], dlv[kBT], dyv[kBT], sgv[kBT];
    {
      float xv[kBT], gov[kBT], zv[kBT];
      load_chunk(u_row + t0, len, p.vec_in, uv);
      load_chunk(x_row + t0, len, p.vec_in, xv);
      load_chunk(go_row + t0, len, p.vec_dout, gov);
      if (has_z) load_chunk(z_row + t0, len, p.vec_in, zv);
      if (!row_ok) {
#pragma unroll
        for (int i = 0; i < kBT; i++) gov[i] = 0.f;
      }
      __syncthreads();
      // Rerun the chunk from its checkpoint: h_{t-1} of every step to shared memory, y, dy and dz.
      float dzs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < kBT; i++) {
        if (i >= len) {
          uv[i] = dlv[i] = dyv[i] = sgv[i] = 0.f;
          continue;
        }
        const float x = xv[i] + bias;
        float dl = x, sg = 1.f;
        if (p.delta_softplus) softplus_sigmoid(x, dl, sg);
        *reinterpret_cast<float4*>(sm.h[warp][i][lane]) = make_float4(hc[0], hc[1], hc[2], hc[3]);
        const float du = dl * uv[i];
        const float4 Bv = *reinterpret_cast<const float4*>(&sm.bc[0][i][4 * q]);
        const float4 Cv = *reinterpret_cast<const float4*>(&sm.bc[1][i][4 * q]);
        const float Bk[4] = {Bv.x, Bv.y, Bv.z, Bv.w}, Ck[4] = {Cv.x, Cv.y, Cv.z, Cv.w};
        float yp = 0.f;
#pragma unroll
        for (int k = 0; k < 4; k++) {
          hc[k] = fmaf(ex2_approx(dl * A2[k]), hc[k], du * Bk[k]);
          yp = fmaf(Ck[k], hc[k], yp);
        }
        float dy = gov[i];
        if (has_z) {
          const float y = fmaf(Dd, uv[i], row_sum(yp));
          const float zz = zv[i];
          const float sz = rcp_approx(1.f + ex2_approx(-zz * kLog2e));
          dy = gov[i] * zz * sz;
          keep_slot(dzs, i, q, gov[i] * y * sz * fmaf(zz, 1.f - sz, 1.f));
        }
        dlv[i] = dl;
        dyv[i] = dy;
        sgv[i] = sg;
      }
      const int nq = quad_len(len, q);
      if (has_z && row_ok && nq > 0) store4(static_cast<Tin*>(p.dz) + grow * L + t0 + 4 * q, nq, p.vec_grad, dzs);
    }
    __syncwarp();
    // The reverse sweep of the chunk; hn holds h_t (the state after the step being undone).
    float hn[4] = {hc[0], hc[1], hc[2], hc[3]};
    float dus[4] = {0.f, 0.f, 0.f, 0.f}, dxs[4] = {0.f, 0.f, 0.f, 0.f};
    const bool b2 = r & 4, b1 = r & 2, b0 = r & 1;
#pragma unroll
    for (int i = kBT - 1; i >= 0; i--) {
      if (i >= len) continue;
      const float4 hp4 = *reinterpret_cast<const float4*>(sm.h[warp][i][lane]);
      const float hp[4] = {hp4.x, hp4.y, hp4.z, hp4.w};
      const float4 Bv = *reinterpret_cast<const float4*>(&sm.bc[0][i][4 * q]);
      const float4 Cv = *reinterpret_cast<const float4*>(&sm.bc[1][i][4 * q]);
      const float Bk[4] = {Bv.x, Bv.y, Bv.z, Bv.w}, Ck[4] = {Cv.x, Cv.y, Cv.z, Cv.w};
      const float dl = dlv[i], uu = uv[i], dy = dyv[i], dlu = dl * uu;
      float sGB = 0.f, sAGw = 0.f, v[8];
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const float ab = ex2_approx(dl * A2[k]);
        const float G = fmaf(dy, Ck[k], g[k]);
        const float t = G * (ab * hp[k]);  // G Ā h_{t-1}
        v[k] = G * dlu;                    // this row's dB
        v[4 + k] = dy * hn[k];             // this row's dC
        sGB = fmaf(G, Bk[k], sGB);
        sAGw = fmaf(Araw[k], t, sAGw);
        dA[k] = fmaf(t, dl, dA[k]);
        g[k] = G * ab;
        hn[k] = hp[k];
      }
      // dB, dC: the sum over the warp's 8 rows by recursive halving; lane 8q + r ends with value r.
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
      const float S = row_sum(sGB), T = row_sum(sAGw);
      const float du = fmaf(dy, Dd, dl * S);
      const float dx = fmaf(uu, S, T) * sgv[i];
      keep_slot(dus, i, q, du);
      keep_slot(dxs, i, q, dx);
      dD = fmaf(dy, uu, dD);
      dbias += dx;
    }
    const int nq = quad_len(len, q);
    if (row_ok && nq > 0) {
      store4(static_cast<Tin*>(p.du) + grow * L + t0 + 4 * q, nq, p.vec_grad, dus);
      store4(static_cast<Tin*>(p.ddelta) + grow * L + t0 + 4 * q, nq, p.vec_grad, dxs);
    }
    __syncthreads();
    // dB, dC of the chunk: the CTA's warps added up, then one atomic add per (tensor, state, 4 steps).
    {
      const int j = threadIdx.x;  // 128 threads: tensor (1 bit), state (4 bits), step quad (2 bits)
      const int tensor = j >> 6, n = (j >> 2) & 15, s4 = j & 3;
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
  if (!row_ok) return;
#pragma unroll
  for (int k = 0; k < 4; k++) {
    const int n = 4 * q + k;
    if (n >= N) continue;
    if (p.dh0) p.dh0[grow * N + n] = g[k];
    atomicAdd(p.dA + dd * N + n, dA[k]);
  }
  if (q == 0) {
    if (p.dD) atomicAdd(p.dD + dd, dD);
    if (p.ddelta_bias) atomicAdd(p.ddelta_bias + dd, dbias);
  }
}

static_assert(kBW * 32 == 2 * kNS * kBT / 4, "one thread per (tensor, state, step quad) of a chunk");

template <typename Tin, typename Tg>
cudaError_t launch_typed(const BwdParams& p, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>((p.dim + kRows - 1) / kRows), static_cast<unsigned>(p.batch));
  const int smem = static_cast<int>(sizeof(BwdSmem));
  cudaError_t e =
      cudaFuncSetAttribute(selscan_bwd_kernel<Tin, Tg>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  selscan_bwd_kernel<Tin, Tg><<<grid, kBW * 32, smem, s>>>(p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

size_t bwd_workspace_bytes(int64_t rows, int64_t seqlen) {
  return sizeof(float) * static_cast<size_t>(rows) * static_cast<size_t>((seqlen + kBT - 1) / kBT) * kNS;
}

cudaError_t launch_bwd(const BwdParams& p_in, selscan_dtype_t in_dtype, selscan_dtype_t dout_dtype, void* workspace,
                       cudaStream_t s) {
  BwdParams p = p_in;
  void* own = nullptr;
  if (!workspace) {
    const cudaError_t e = cudaMallocAsync(&own, bwd_workspace_bytes(p.batch * p.dim, p.seqlen), s);
    if (e != cudaSuccess) return e;
    workspace = own;
  }
  p.ckpt = static_cast<float*>(workspace);
  cudaError_t e;
  if (in_dtype == SELSCAN_F32)
    e = dout_dtype == SELSCAN_F32 ? launch_typed<float, float>(p, s) : launch_typed<float, __nv_bfloat16>(p, s);
  else
    e = dout_dtype == SELSCAN_F32 ? launch_typed<__nv_bfloat16, float>(p, s)
                                  : launch_typed<__nv_bfloat16, __nv_bfloat16>(p, s);
  if (own) {
    const cudaError_t ef = cudaFreeAsync(own, s);
    if (e == cudaSuccess) e = ef;
  }
  return e;
}

}  // namespace selscan

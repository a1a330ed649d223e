// Recurrent decode step: one token per (batch, channel) row, state updated in place.
//
//   Δ = softplus(δ + Δ_bias[d]),  h[n] ← exp(Δ A[d,n]) h[n] + Δ B[b,n] u,
//   y = Σ_n C[b,n] h[n] + D[d] u,  out = y silu(z)
// This is the recurrent (RNN-mode) form of the selective scan with a constant-size state
// ("Mamba架构深度剖析：如何以线性时间重塑序列建模" §3; recurrence from "Mamba状态空间模型深度解析"
// §2.1).  It is a streaming read-modify-write of the fp32 state [B, D, N].  For 16 aligned states and
// D >= 64, four threads per row with B and C staged per CTA (selscan_step_quad_kernel); otherwise
// Q = NS/4 consecutive threads per row, each owning four states (one 16-byte vector), the Q partial
// sums of y meeting with shuffles.  A one-thread-per-row kernel stays selectable for comparison.
#include <cstdlib>

#include "selscan_internal.cuh"

namespace selscan {
namespace {

#ifndef SELSCAN_STEP_ROW_MINB
#define SELSCAN_STEP_ROW_MINB 4
#endif

template <int NS, typename Tin, typename Tout>
__global__ void __launch_bounds__(256) selscan_step_kernel(const StepParams p) {
  constexpr int Q = NS / 4;  // threads per row
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t rows = p.batch * p.dim;
  const int64_t row = gid / Q;
  const int q = static_cast<int>(gid % Q);
  const bool ok = row < rows;  // whole rows are in or out together (Q divides 32)
  const int N = p.dstate;
  const int64_t b = ok ? row / p.dim : 0;
  const int64_t d = ok ? row - b * p.dim : 0;

  float y = 0.f, uu = 0.f;
  if (ok) {
    uu = to_f32(static_cast<const Tin*>(p.u)[row]);
    const float x = to_f32(static_cast<const Tin*>(p.delta)[row]) + (p.delta_bias ? p.delta_bias[d] : 0.f);
    const float dt = p.delta_softplus ? softplus_f(x) : x;
    const float du = dt * uu;
    const Tin* Bb = static_cast<const Tin*>(p.B) + b * N;
    const Tin* Cb = static_cast<const Tin*>(p.C) + b * N;
    float h[4], a[4];
    float* st = p.state + row * N + 4 * q;
    const float* Ar = p.A + d * N + 4 * q;
    const bool vec = p.vec_state && 4 * q + 4 <= N;  // all four of this thread's states exist
    if (vec) {
      const float4 hv = __ldcs(reinterpret_cast<const float4*>(st));
      const float4 av = __ldg(reinterpret_cast<const float4*>(Ar));
      h[0] = hv.x; h[1] = hv.y; h[2] = hv.z; h[3] = hv.w;
      a[0] = av.x; a[1] = av.y; a[2] = av.z; a[3] = av.w;
    } else {
#pragma unroll
      for (int j = 0; j < 4; j++) {
        const bool in = 4 * q + j < N;
        h[j] = in ? st[j] : 0.f;
        a[j] = in ? Ar[j] : 0.f;
      }
    }
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const int n = 4 * q + j;
      if (n < N) {
        h[j] = fmaf(ex2_approx(dt * a[j] * kLog2e), h[j], du * to_f32(Bb[n]));
        y = fmaf(to_f32(Cb[n]), h[j], y);
      }
    }
    if (vec) {
      __stcs(reinterpret_cast<float4*>(st), make_float4(h[0], h[1], h[2], h[3]));
    } else {
#pragma unroll
      for (int j = 0; j < 4; j++)
        if (4 * q + j < N) st[j] = h[j];
    }
  }
  // Sum the Q partial dot products of the row (lanes of a row are adjacent in the warp).
#pragma unroll
  for (int o = 1; o < Q; o <<= 1) y += __shfl_xor_sync(0xffffffffu, y, o);
  if (ok && q == 0) {
    y = fmaf(p.D ? p.D[d] : 0.f, uu, y);
    if (p.z) y *= silu_f(to_f32(static_cast<const Tin*>(p.z)[row]));
    static_cast<Tout*>(p.out)[row] = from_f32<Tout>(y);
  }
}

// One thread per row for 16 states in 16-byte vectors: its four state loads (and A) are all in flight at
// once.  B and C of a batch entry are the same for all of its channels, so each CTA stages them once in
// shared memory (for the one or two batch entries its rows span) and every thread reads them from there
// as broadcast 16-byte loads: 8 shared loads instead of 32 scalar global loads per thread.
template <typename Tin, typename Tout>
__global__ void __launch_bounds__(256, SELSCAN_STEP_ROW_MINB) selscan_step_row16_kernel(const StepParams p) {
  __shared__ __align__(16) float sBC[2][2][16];  // [batch entry of the CTA][B, C][state]
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * blockDim.x;
  const int64_t row = row0 + threadIdx.x;
  const int64_t rows = p.batch * p.dim;
  const int64_t b0 = row0 / p.dim;
  if (threadIdx.x < 64) {
    const int k = threadIdx.x >> 5, tensor = (threadIdx.x >> 4) & 1, n = threadIdx.x & 15;
    const int64_t bb = b0 + k;
    float v = 0.f;
    if (bb < p.batch) v = to_f32(static_cast<const Tin*>(tensor ? p.C : p.B)[bb * 16 + n]);
    sBC[k][tensor][n] = v;
  }
  __syncthreads();
  if (row >= rows) return;
  const int64_t b = row / p.dim, d = row - b * p.dim;
  const float4* st = reinterpret_cast<const float4*>(p.state + row * 16);
  const float4* Ar = reinterpret_cast<const float4*>(p.A + d * 16);
  float4 h[4], a[4];
#pragma unroll
  for (int k = 0; k < 4; k++) h[k] = __ldcs(st + k);
#pragma unroll
  for (int k = 0; k < 4; k++) a[k] = __ldg(Ar + k);
  const float uu = to_f32(static_cast<const Tin*>(p.u)[row]);
  const float x = to_f32(static_cast<const Tin*>(p.delta)[row]) + (p.delta_bias ? p.delta_bias[d] : 0.f);
  const float zz = p.z ? to_f32(static_cast<const Tin*>(p.z)[row]) : 0.f;
  const float Dd = p.D ? p.D[d] : 0.f;
  const float4* Bq = reinterpret_cast<const float4*>(sBC[b - b0][0]);
  const float4* Cq = reinterpret_cast<const float4*>(sBC[b - b0][1]);
  const float dt = p.delta_softplus ? softplus_fast(x) : x;
  const float dtl = dt * kLog2e, du = dt * uu;
  float y = 0.f;
#pragma unroll
  for (int k = 0; k < 4; k++) {
    const float4 bb = Bq[k], cc = Cq[k];
    const float bv[4] = {bb.x, bb.y, bb.z, bb.w}, cv[4] = {cc.x, cc.y, cc.z, cc.w};
    float* hv = reinterpret_cast<float*>(&h[k]);
    const float* av = reinterpret_cast<const float*>(&a[k]);
#pragma unroll
    for (int j = 0; j < 4; j++) {
      hv[j] = fmaf(ex2_approx(dtl * av[j]), hv[j], du * bv[j]);
      y = fmaf(cv[j], hv[j], y);
    }
  }
  float4* sto = reinterpret_cast<float4*>(p.state + row * 16);
#pragma unroll
  for (int k = 0; k < 4; k++) __stcs(sto + k, h[k]);
  y = fmaf(Dd, uu, y);
  if (p.z) y *= silu_fast(zz);
  static_cast<Tout*>(p.out)[row] = from_f32<Tout>(y);
}

// Four threads per row for 16 aligned states, one 16-byte state quad each: a warp reads and writes 512
// contiguous bytes of state per instruction (measured on B300: an 84 MB in-place update in this layout
// reaches 0.79 of the copy bandwidth, one thread per row 0.70).  Each thread reads its four B and C values
// itself (8 or 16 bytes each, shared by every row of the batch entry and so served by L1), and forms Δ and
// the gate itself: no barrier and no value crossing lanes before the y reduction, so every load of a
// thread is in flight at once.
template <typename Tin>
__device__ __forceinline__ float4 load_quad(const Tin* p) {
  if constexpr (sizeof(Tin) == 2) {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(p));
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u), __uint_as_float(w.y << 16),
                       __uint_as_float(w.y & 0xffff0000u));
  } else {
    return __ldg(reinterpret_cast<const float4*>(p));
  }
}

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(256) selscan_step_quad_kernel(const StepParams p) {
  // Grid (channel blocks of 64, batch entries): the row's batch entry and channel come from the grid.
  const int q = threadIdx.x & 3;
  const int64_t b = blockIdx.y;
  const int64_t d = static_cast<int64_t>(blockIdx.x) * 64 + (threadIdx.x >> 2);
  if (d >= p.dim) return;  // whole rows leave together (4 divides the warp)
  const int64_t row = b * p.dim + d;
  float4 h = __ldcs(reinterpret_cast<const float4*>(p.state + row * 16) + q);
  const float4 a = __ldg(reinterpret_cast<const float4*>(p.A + d * 16) + q);
  const float4 bv = load_quad(static_cast<const Tin*>(p.B) + b * 16 + 4 * q);
  const float4 cv = load_quad(static_cast<const Tin*>(p.C) + b * 16 + 4 * q);
  const float uu = to_f32(static_cast<const Tin*>(p.u)[row]);
  const float x = to_f32(static_cast<const Tin*>(p.delta)[row]) + (p.delta_bias ? p.delta_bias[d] : 0.f);
  const float zz = p.z ? to_f32(static_cast<const Tin*>(p.z)[row]) : 0.f;
  const float Dd = p.D ? p.D[d] : 0.f;
  // Each of the row's four threads forms Δ itself: a divergent branch would cost the warp the same
  // issue slots and add a shuffle's latency.
  const float dt = p.delta_softplus ? softplus_fast(x) : x;
  const float dtl = dt * kLog2e, du = dt * uu;
  h.x = fmaf(ex2_approx(dtl * a.x), h.x, du * bv.x);
  h.y = fmaf(ex2_approx(dtl * a.y), h.y, du * bv.y);
  h.z = fmaf(ex2_approx(dtl * a.z), h.z, du * bv.z);
  h.w = fmaf(ex2_approx(dtl * a.w), h.w, du * bv.w);
  __stcs(reinterpret_cast<float4*>(p.state + row * 16) + q, h);
  float y = fmaf(cv.x, h.x, fmaf(cv.y, h.y, fmaf(cv.z, h.z, cv.w * h.w)));
  y += __shfl_xor_sync(kFull, y, 1);
  y += __shfl_xor_sync(kFull, y, 2);
  if (q == 0) {
    y = fmaf(Dd, uu, y);
    if (p.z) y *= silu_fast(zz);
    static_cast<Tout*>(p.out)[row] = from_f32<Tout>(y);
  }
}

template <int NS, typename Tin, typename Tout>
cudaError_t launch_ns(const StepParams& p, cudaStream_t s) {
  // SELSCAN_STEP: "quad", "row" or "generic" (default: the first that applies).
  const char* force = getenv("SELSCAN_STEP");
  const char f = force ? force[0] : 'q';
  if (f == 'q' && NS == 16 && p.dstate == 16 && p.vec_state && p.vec_bc && p.batch <= 65535) {
    const dim3 grid(static_cast<unsigned>((p.dim + 63) / 64), static_cast<unsigned>(p.batch));
    selscan_step_quad_kernel<Tin, Tout><<<grid, 256, 0, s>>>(p);
    count_launches(1);
    return cudaGetLastError();
  }
  // (With at least 256 channels a CTA's 256 rows span at most two batch entries.)
  if (f != 'g' && NS == 16 && p.dstate == 16 && p.vec_state && p.dim >= 256) {
    const int64_t rows = p.batch * p.dim;
    selscan_step_row16_kernel<Tin, Tout><<<static_cast<unsigned>((rows + 255) / 256), 256, 0, s>>>(p);
    count_launches(1);
    return cudaGetLastError();
  }
  constexpr int Q = NS / 4;
  const int64_t threads = p.batch * p.dim * Q;
  const int block = 256;
  const int64_t grid = (threads + block - 1) / block;
  selscan_step_kernel<NS, Tin, Tout><<<static_cast<unsigned>(grid), block, 0, s>>>(p);
  count_launches(1);
  return cudaGetLastError();
}

template <typename Tin, typename Tout>
cudaError_t dispatch_ns(const StepParams& p, cudaStream_t s) {
  if (p.dstate <= 4) return launch_ns<4, Tin, Tout>(p, s);
  if (p.dstate <= 8) return launch_ns<8, Tin, Tout>(p, s);
  return launch_ns<16, Tin, Tout>(p, s);
}

}  // namespace

cudaError_t launch_step(const StepParams& p, selscan_dtype_t in_dtype, selscan_dtype_t out_dtype, cudaStream_t s) {
  if (in_dtype == SELSCAN_F32) {
    return out_dtype == SELSCAN_F32 ? dispatch_ns<float, float>(p, s) : dispatch_ns<float, __nv_bfloat16>(p, s);
  }
  return out_dtype == SELSCAN_F32 ? dispatch_ns<__nv_bfloat16, float>(p, s)
                                  : dispatch_ns<__nv_bfloat16, __nv_bfloat16>(p, s);
}

}  // namespace selscan

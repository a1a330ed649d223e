// Throughput probes of the arithmetic units that bound the selective scan on this GPU: the
// special-function unit (2^x, log2 x, 1/x, tanh x) and the fp32 FMA pipe (scalar and packed fp32x2).
//
// The forward is bound by its N + 4 special-function results per element (N exponentials for
// Ā = exp(ΔA), two for softplus, two for the SiLU gate) and by its fp32 multiply-adds, so its
// roofline needs the rate of each unit per SM and clock.  Each probe runs one CTA per SM (a large
// shared-memory request keeps a second CTA off the SM), every thread applying the unit's operation
// to 8 independent chains for a fixed number of iterations, and each CTA times its own loop with the
// SM cycle counter.  Results per clock per SM = operations of the CTA / its cycles (median over CTAs).
#include <algorithm>
#include <vector>

#include "selscan_internal.cuh"
#include "selscan_probe.h"

namespace selscan {
namespace {

constexpr int kChains = 8;
constexpr int kThreads = 1024;
constexpr int kIters = 4096;
constexpr int kProbeSmem = 160 * 1024;  // more than half of an SM's shared memory: one CTA per SM

template <int UNIT>
__device__ __forceinline__ float unit_op(float x) {
  float r;
  if (UNIT == SELSCAN_PROBE_EX2) {
    asm volatile("{\n .reg .f32 t;\n neg.f32 t, %1;\n ex2.approx.ftz.f32 %0, t;\n}" : "=f"(r) : "f"(x));
  } else if (UNIT == SELSCAN_PROBE_LG2) {
    asm volatile("{\n .reg .f32 t;\n abs.f32 t, %1;\n lg2.approx.ftz.f32 %0, t;\n}" : "=f"(r) : "f"(x));
  } else if (UNIT == SELSCAN_PROBE_RCP) {
    // 1/(x + 1): the added 1 keeps two reciprocals in a row from folding into the identity.
    asm volatile("{\n .reg .f32 t;\n add.f32 t, %1, 0f3F800000;\n rcp.approx.ftz.f32 %0, t;\n}" : "=f"(r) : "f"(x));
  } else if (UNIT == SELSCAN_PROBE_TANH) {
    asm volatile("tanh.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
  } else {
    asm volatile("fma.rn.f32 %0, %1, 0f3F7FBE77, 0f3A83126F;" : "=f"(r) : "f"(x));  // x·0.999 + 0.001
  }
  return r;
}

template <int UNIT>
__global__ void __launch_bounds__(kThreads, 1) probe_kernel(long long* cycles, float* sink) {
  float x[kChains];
#pragma unroll
  for (int c = 0; c < kChains; c++) x[c] = 0.5f + 0.01f * static_cast<float>(c + (threadIdx.x & 7));
  __syncthreads();
  const long long t0 = clock64();
  if (UNIT == SELSCAN_PROBE_FFMA2) {
    float2 v[kChains / 2];
#pragma unroll
    for (int c = 0; c < kChains / 2; c++) v[c] = make_float2(x[2 * c], x[2 * c + 1]);
    const float2 a = make_float2(0.999f, 0.999f), b = make_float2(0.001f, 0.001f);
    for (int i = 0; i < kIters; i++) {
#pragma unroll
      for (int c = 0; c < kChains / 2; c++) v[c] = __ffma2_rn(v[c], a, b);
    }
#pragma unroll
    for (int c = 0; c < kChains / 2; c++) {
      x[2 * c] = v[c].x;
      x[2 * c + 1] = v[c].y;
    }
  } else {
    for (int i = 0; i < kIters; i++) {
#pragma unroll
      for (int c = 0; c < kChains; c++) x[c] = unit_op<UNIT>(x[c]);
    }
  }
  __syncthreads();
  const long long t1 = clock64();
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < kChains; c++) s += x[c];
  sink[blockIdx.x * kThreads + threadIdx.x] = s;
  if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

template <int UNIT>
cudaError_t run_probe(int sms, long long* cycles, float* sink) {
  auto k = probe_kernel<UNIT>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem);
  if (e != cudaSuccess) return e;
  k<<<sms, kThreads, kProbeSmem>>>(cycles, sink);
  return cudaGetLastError();
}

// y[i] = the kernels' own evaluation of function fn at x[i] (x2[i]: A for SELSCAN_FN_ZOH).
__global__ void __launch_bounds__(256) fn_kernel(int fn, const float* __restrict__ x, const float* __restrict__ x2,
                                                 float* __restrict__ y, int64_t n) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float v = x[i];
  float r = 0.f;
  switch (fn) {
    case SELSCAN_FN_EX2: r = ex2_approx(v); break;
    case SELSCAN_FN_SOFTPLUS: r = softplus_fast(v); break;
    case SELSCAN_FN_SILU: r = silu_fast(v); break;
    case SELSCAN_FN_SOFTPLUS_BWD: {
      float sp, sg;
      softplus_sigmoid(v, sp, sg);
      r = sp;
      break;
    }
    case SELSCAN_FN_SIGMOID: {
      float sp, sg;
      softplus_sigmoid(v, sp, sg);
      r = sg;
      break;
    }
    default: {  // SELSCAN_FN_ZOH: the forward's steps for a state with A = x2[i] at Δ = x[i] and u = 1
      const float a2 = x2[i] * kLog2e;   // A·log2 e, as the kernel keeps it
      const float e = v * a2;            // the exponent Δ·A·log2 e
      const float ab = ex2_approx(e);    // Ā
      const float ia = kLog2e / a2;      // 1/A, as the kernel forms it
      r = zoh_factor2(f2(v, v), f2(e, e), f2(ab, ab), f2(ia, ia)).x;
      break;
    }
  }
  y[i] = r;
}

}  // namespace
}  // namespace selscan

// The kernels' own arithmetic of one function on n device values: see include/selscan_probe.h.
extern "C" selscan_status_t selscan_probe_function(int fn, const float* x, const float* x2, float* y, int64_t n,
                                                   void* stream) {
  if (fn < SELSCAN_FN_EX2 || fn > SELSCAN_FN_ZOH) return SELSCAN_ERR_UNSUPPORTED;
  if (n < 0) return SELSCAN_ERR_SHAPE;
  if (n == 0) return SELSCAN_OK;
  if (!x || !y || (fn == SELSCAN_FN_ZOH && !x2)) return SELSCAN_ERR_NULL;
  const int64_t blocks = (n + 255) / 256;
  if (blocks > 0x7fffffff) return SELSCAN_ERR_SHAPE;
  selscan::fn_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(fn, x, x2, y, n);
  return cudaGetLastError() == cudaSuccess ? SELSCAN_OK : SELSCAN_ERR_CUDA;
}

extern "C" selscan_status_t selscan_probe_rate(int unit, double* per_clk_per_sm) {
  using namespace selscan;
  if (!per_clk_per_sm) return SELSCAN_ERR_NULL;
  if (unit < SELSCAN_PROBE_EX2 || unit > SELSCAN_PROBE_FFMA2) return SELSCAN_ERR_UNSUPPORTED;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms <= 0)
    return SELSCAN_ERR_CUDA;
  long long* cycles = nullptr;
  float* sink = nullptr;
  if (cudaMalloc(&cycles, sizeof(long long) * sms) != cudaSuccess) return SELSCAN_ERR_CUDA;
  if (cudaMalloc(&sink, sizeof(float) * sms * kThreads) != cudaSuccess) {
    cudaFree(cycles);
    return SELSCAN_ERR_CUDA;
  }
  cudaError_t e = cudaSuccess;
  switch (unit) {
    case SELSCAN_PROBE_EX2: e = run_probe<SELSCAN_PROBE_EX2>(sms, cycles, sink); break;
    case SELSCAN_PROBE_LG2: e = run_probe<SELSCAN_PROBE_LG2>(sms, cycles, sink); break;
    case SELSCAN_PROBE_RCP: e = run_probe<SELSCAN_PROBE_RCP>(sms, cycles, sink); break;
    case SELSCAN_PROBE_TANH: e = run_probe<SELSCAN_PROBE_TANH>(sms, cycles, sink); break;
    case SELSCAN_PROBE_FFMA: e = run_probe<SELSCAN_PROBE_FFMA>(sms, cycles, sink); break;
    default: e = run_probe<SELSCAN_PROBE_FFMA2>(sms, cycles, sink); break;
  }
  std::vector<long long> host(sms);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(host.data(), cycles, sizeof(long long) * sms, cudaMemcpyDeviceToHost);
  cudaFree(cycles);
  cudaFree(sink);
  if (e != cudaSuccess) return SELSCAN_ERR_CUDA;
  std::sort(host.begin(), host.end());
  const double med = static_cast<double>(host[sms / 2]);
  // Results of one CTA: kChains per thread and iteration (for the packed FMA, kChains / 2 instructions
  // of two results each).
  const double ops = static_cast<double>(kThreads) * kIters * kChains;
  *per_clk_per_sm = med > 0 ? ops / med : 0.0;
  return SELSCAN_OK;
}

// The bounded wait of the forward kernels, made to run out: see include/selscan_probe.h.
extern "C" selscan_status_t selscan_probe_wait_timeout(int64_t polls, int* completed) {
  if (!completed) return SELSCAN_ERR_NULL;
  if (polls < 1 || polls > (int64_t{1} << 20)) return SELSCAN_ERR_SHAPE;
  const cudaError_t e = selscan::probe_wait_timeout(static_cast<long long>(polls), completed);
  return e == cudaSuccess ? SELSCAN_OK : SELSCAN_ERR_CUDA;
}

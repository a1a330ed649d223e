/*
 * libselscan — throughput probes of the arithmetic units that bound the
 * selective-scan forward on this GPU.
 *
 * The forward needs, per element (b, d, t), N exponentials for Ā = exp(Δ·A)
 * ("Mamba架构与SSM模型：高效序列建模技术解析" §2.1), an exponential and a
 * logarithm for Δ = softplus(δ + Δ_bias) (§2.2 of the same page) and an
 * exponential and a reciprocal for the SiLU gate ("Mamba状态空间模型深度解析：
 * 挑战Transformer的下一代序列建模范式" §3.1), plus about 4N + 8 fp32 operations.
 * Its roofline is therefore set by the special-function unit and the FMA pipe;
 * these probes measure their rates so that the roofline rests on numbers taken
 * on the GPU itself rather than on nominal figures.
 *
 * selscan_probe_rate runs one CTA per SM on the current device; every thread
 * applies the unit's operation to 8 independent chains 4096 times and each CTA
 * times its loop with the SM cycle counter.  *per_clk_per_sm receives the fp32
 * results per clock per SM (median over the SMs): for SELSCAN_PROBE_FFMA2 that
 * counts both lanes of each packed instruction.
 *
 * It is synchronous (it waits for the device), allocates two small device
 * buffers with cudaMalloc for the duration of the call, and returns
 * SELSCAN_ERR_NULL (NULL output), SELSCAN_ERR_UNSUPPORTED (unknown unit) or
 * SELSCAN_ERR_CUDA (a CUDA call failed).  It is a measurement utility, not part
 * of the scan.
 */
#ifndef SELSCAN_PROBE_H_
#define SELSCAN_PROBE_H_

#include "selscan.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SELSCAN_PROBE_EX2 = 0,  /* ex2.approx.ftz.f32 (2^x) */
  SELSCAN_PROBE_LG2 = 1,  /* lg2.approx.ftz.f32 (log2 x) */
  SELSCAN_PROBE_RCP = 2,  /* rcp.approx.ftz.f32 (1/x) */
  SELSCAN_PROBE_TANH = 3, /* tanh.approx.f32 */
  SELSCAN_PROBE_FFMA = 4, /* fp32 fused multiply-add */
  SELSCAN_PROBE_FFMA2 = 5 /* packed fp32x2 fused multiply-add */
} selscan_probe_unit_t;

selscan_status_t selscan_probe_rate(int unit, double* per_clk_per_sm);

/*
 * The bounded wait of the forward kernels, made to run out on purpose, so that a caller (or a test) can
 * check on a real GPU that a lost asynchronous copy ends in an error status rather than a hang.  One CTA
 * of 32 threads waits on an mbarrier phase whose one arrival announces 16 bytes that no copy delivers
 * (no copy is issued: nothing is in flight when the waits end).  Each thread polls the phase with the
 * same helper the forward kernels use, at most `polls` times (1 .. 2^20; the kernels themselves use
 * 2^18, about one second at the 3.9 us a poll of an incomplete phase suspends on B300), then gives up: it sets the device status word that selscan_device_status() reads (which then
 * returns 1 until reset) and returns.  *completed receives the number of waits that saw the phase
 * complete (0 when the bound works).  Synchronous; allocates one int with cudaMalloc for the call.
 * Returns SELSCAN_ERR_NULL, SELSCAN_ERR_SHAPE (polls out of range) or SELSCAN_ERR_CUDA.
 */
selscan_status_t selscan_probe_wait_timeout(int64_t polls, int* completed);

/*
 * The kernels' own arithmetic of the functions they approximate, evaluated on n values, so that a test can
 * hold each against a float64 evaluation over its input range:
 *   SELSCAN_FN_EX2          2^x, the special-function unit's ex2.approx.ftz (every Ā = 2^(Δ·A·log2 e));
 *   SELSCAN_FN_SOFTPLUS     softplus(x) as the forward and decode kernels form Δ ("Mamba架构与SSM模型：
 *                           高效序列建模技术解析" §2.2);
 *   SELSCAN_FN_SILU         x·σ(x), the gate ("Mamba状态空间模型深度解析：挑战Transformer的下一代序列建模
 *                           范式" §3.1);
 *   SELSCAN_FN_SOFTPLUS_BWD softplus(x) as the backward forms Δ (together with σ(x) from one exponential);
 *   SELSCAN_FN_SIGMOID      σ(x), the derivative of softplus, as the backward forms it;
 *   SELSCAN_FN_ZOH          the exact zero-order-hold input factor (exp(Δ·A) − 1)/A at Δ = x and A = x2
 *                           (u = 1), through the forward's own steps ("Mamba架构与SSM模型：高效序列建模技术
 *                           解析" §2.1).
 * x, x2 and y are device pointers to n fp32 values (x2 only for SELSCAN_FN_ZOH, else ignored; NULL allowed).
 * Asynchronous on `stream`; allocates nothing.  Returns SELSCAN_ERR_UNSUPPORTED (unknown fn),
 * SELSCAN_ERR_SHAPE (n < 0 or too many blocks), SELSCAN_ERR_NULL or SELSCAN_ERR_CUDA (launch failed).
 */
typedef enum {
  SELSCAN_FN_EX2 = 0,
  SELSCAN_FN_SOFTPLUS = 1,
  SELSCAN_FN_SILU = 2,
  SELSCAN_FN_SOFTPLUS_BWD = 3,
  SELSCAN_FN_SIGMOID = 4,
  SELSCAN_FN_ZOH = 5
} selscan_fn_t;

selscan_status_t selscan_probe_function(int fn, const float* x, const float* x2, float* y, int64_t n, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SELSCAN_PROBE_H_ */

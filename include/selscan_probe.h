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

#ifdef __cplusplus
}
#endif

#endif /* SELSCAN_PROBE_H_ */

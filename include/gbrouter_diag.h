/*
 * gbrouter_diag — measurement and verification aids: the small-M router's
 * latency floor and the error sweep of the FP32 scores. The router pages
 * have no counterpart: these exist to measure how much of a dependent
 * router call is the launch chain itself, and to check the error bound the
 * near-tie guard band rests on.
 *
 * gbr_diag_chain launches n kernels back to back on `stream`, each with the
 * single-cluster router's launch shape (one cluster of 16 CTAs x 512
 * threads) and programmatic dependent launch:
 *   kind 0: release the next kernel, wait for the preceding one, end;
 *   kind 1: as kind 0, then every CTA reads x (x_bytes bytes of a device
 *           buffer, 16-byte aligned, a multiple of 16) with 16-byte loads
 *           and XORs one word per CTA into sink[blockIdx] (sink: device,
 *           16 words, caller-owned).
 * Returns 0, 1 for a bad argument (nothing launched), 3 for a CUDA error.
 * Capturable into a CUDA graph.
 *
 * gbr_diag_act_sweep evaluates the library's FP32 score `act`
 * (GBR_ACT_SQRT_SOFTPLUS or GBR_ACT_SIGMOID: the branch-free forms the
 * kernels use) at every FP32 bit pattern u in [first, first + count) whose
 * value is finite, beside the same score composed of CUDA's expf, log1pf,
 * sqrtf and division, and writes to out (device, 2 floats, caller-owned):
 *   out[0] the largest |a32 - ref| / (2^-23 ref) over inputs with
 *          ref >= 2^-62, rounded up;
 *   out[1] the largest |a32 - ref| over the other inputs.
 * first + count <= 2^32. Returns 0, 1 for a bad argument (nothing
 * launched), 3 for a CUDA error. Asynchronous on `stream`.
 * gbr_diag_act_coef returns the coefficient c of the kernels' error bound
 * |a32 - a| <= c 2^-23 a + 2^-60 for that score (host call, no GPU needed);
 * a sweep maximum plus the reference composition's own bound (2.25 for
 * sqrt-softplus, 3 for the sigmoid) must stay below it.
 *
 * gbr_diag_near_key_cycles times the near-tie key (the double-float score
 * plus bias the selection re-ranks close keys with) for `act`: one warp
 * evaluates it `reps` times per lane in a dependent chain and writes the SM
 * cycles per evaluation to out[0] (device, 2 long longs, caller-owned).
 * Returns 0, 1 for a bad argument, 3 for a CUDA error.
 *
 * The measurement build of the library (build.py variant "stamps",
 * -DGBR_PHASE_STAMPS) also exports router_phase_stamps(), which copies the
 * single-cluster kernel's per-phase %globaltimer stamps to host memory;
 * the product library does not have it.
 */
#ifndef GBROUTER_DIAG_H_
#define GBROUTER_DIAG_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* cudaStream_t;

int gbr_diag_chain(int kind, int n, const void* x, size_t x_bytes, unsigned* sink,
                   cudaStream_t stream);
int gbr_diag_act_sweep(int act, unsigned long long first, unsigned long long count, float* out,
                       cudaStream_t stream);
float gbr_diag_act_coef(int act);
int gbr_diag_near_key_cycles(int act, int reps, long long* out, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GBROUTER_DIAG_H_ */

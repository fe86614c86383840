/*
 * gbrouter_diag — measurement aid for the small-M router's latency floor.
 * The router pages have no counterpart: this exists to measure how much of
 * a dependent router call is the launch chain itself.
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

#ifdef __cplusplus
}
#endif

#endif /* GBROUTER_DIAG_H_ */

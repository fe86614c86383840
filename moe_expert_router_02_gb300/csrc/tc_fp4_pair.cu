// Prefill router kernels for NVFP4 weights, CTA pairs: every list capacity of
// tc_kernel.cuh's kernel for this family, compiled in a translation unit of
// its own so the library's units build in parallel.
#include "tc_kernel.cuh"

namespace gbr {

cudaError_t tc_dispatch_fp4_pair(const CUtensorMap& mx, const CUtensorMap& mw, const TcParams& p,
                                 size_t smem, bool pdl, bool sk, cudaStream_t s, int* q) {
  return dispatch_k<true, true>(mx, mw, p, smem, pdl, sk, s, q);
}

}  // namespace gbr

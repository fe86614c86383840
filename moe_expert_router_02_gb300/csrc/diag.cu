// Floors for the dependent launch chain of the small-M router: chains of
// kernels with the router's launch shape (one cluster of 16 CTAs x 512
// threads, programmatic dependent launch) that do nothing but the parts of
// a router call that cannot overlap the preceding kernel. A router call
// minus such a floor is the time its own work adds.
#include <cuda_runtime.h>

#include "../../include/gbrouter_diag.h"
#include "common.cuh"
#include "dfkey.cuh"

namespace gbr {
namespace {

constexpr int kDiagCtas = 16, kDiagThreads = 512;

// Releases the next kernel, then waits for the preceding one.
__global__ void __launch_bounds__(kDiagThreads) k_diag_wait_only() {
  pdl_launch_dependents();
  pdl_wait();
}

// As above, then reads x [M, H] BF16 the way the single-cluster router does
// (every CTA reads all of it, 16-byte loads spread over its warps), folds it
// to one word per CTA and stores that.
__global__ void __launch_bounds__(kDiagThreads)
    k_diag_read_x(const uint4* __restrict__ x, int n16, unsigned* sink) {
  pdl_launch_dependents();
  pdl_wait();
  unsigned f = 0;
  for (int i = threadIdx.x; i < n16; i += kDiagThreads) {
    const uint4 v = __ldg(x + i);
    f ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  f = __reduce_xor_sync(kFull, f);
  if ((threadIdx.x & 31) == 0) atomicXor(sink + blockIdx.x, f);
}

cudaError_t launch_one(int kind, const void* x, int n16, unsigned* sink, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kDiagCtas);
  cfg.blockDim = dim3(kDiagThreads);
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kDiagCtas;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  if (kind == 0) return cudaLaunchKernelEx(&cfg, k_diag_wait_only);
  return cudaLaunchKernelEx(&cfg, k_diag_read_x, static_cast<const uint4*>(x), n16, sink);
}

// The scores composed of CUDA's own functions, each within its documented
// error bound (expf 2 ulp, log1pf 1 ulp, sqrtf and division correctly
// rounded): the reference the library's branch-free scores are swept
// against.
__device__ float act_libm(int act, float z) {
  if (act == ACT_SIGMOID) return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-z)));
  return sqrtf(fmaxf(z, 0.0f) + log1pf(expf(-fabsf(z))));
}

// out[0]: the largest |act_f32 - act_libm| / (2^-23 act_libm) over inputs
// whose reference is at least 2^-62; out[1]: the largest |act_f32 -
// act_libm| over the others. Both rounded up, as float bit patterns
// (non-negative floats order like their bits).
__global__ void __launch_bounds__(256)
    k_diag_act_sweep(int act, unsigned long long first, unsigned long long count, unsigned* out) {
  unsigned rel = 0u, abs_ = 0u;
  const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
  for (unsigned long long i = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x; i < count;
       i += stride) {
    const float z = __uint_as_float((unsigned)(first + i));
    if (!isfinite(z)) continue;
    const float f = act_f32(act, z), r = act_libm(act, z);
    const float d = __fsub_ru(fmaxf(f, r), fminf(f, r));
    if (r >= 0x1p-62f)
      rel = max(rel, __float_as_uint(__fdiv_ru(d, r * 0x1p-23f)));
    else
      abs_ = max(abs_, __float_as_uint(d));
  }
  rel = __reduce_max_sync(kFull, rel);
  abs_ = __reduce_max_sync(kFull, abs_);
  if ((threadIdx.x & 31) == 0) {
    atomicMax(out, rel);
    atomicMax(out + 1, abs_);
  }
}

// Latency of one near-tie key evaluation: a single warp evaluates it `reps`
// times per lane in a dependent chain; out[0] = SM cycles per evaluation
// (lane 0's clock64 difference / reps).
__global__ void k_diag_near_key_cycles(int act, int reps, long long* out) {
  float z = -3.0f + 0.2f * (float)threadIdx.x;
  float acc = 0.0f;
  const long long t0 = clock64();
  for (int r = 0; r < reps; ++r) {
    const NearKey nk = near_key(act, z, 0.01f);
    acc += nk.lo;
    z += nk.lo * 0x1p-100f;  // a dependence on the previous evaluation, value unchanged
  }
  const long long t1 = clock64();
  if (threadIdx.x == 0) out[0] = (t1 - t0) / (reps > 0 ? reps : 1);
  if (acc == 12345.0f) out[1] = 1;  // keeps the chain live
}

}  // namespace
}  // namespace gbr

extern "C" int gbr_diag_near_key_cycles(int act, int reps, long long* out, cudaStream_t stream) {
  if ((act != gbr::ACT_SQRT_SOFTPLUS && act != gbr::ACT_SIGMOID) || !out || reps < 1) return 1;
  gbr::k_diag_near_key_cycles<<<1, 32, 0, stream>>>(act, reps, out);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

extern "C" float gbr_diag_act_coef(int act) { return gbr::act_err_coef(act); }

extern "C" int gbr_diag_act_sweep(int act, unsigned long long first, unsigned long long count,
                                  float* out, cudaStream_t stream) {
  if ((act != gbr::ACT_SQRT_SOFTPLUS && act != gbr::ACT_SIGMOID) || !out ||
      first > 0x100000000ull || count > 0x100000000ull - first)
    return 1;
  if (cudaMemsetAsync(out, 0, 2 * sizeof(float), stream) != cudaSuccess) return 3;
  if (count == 0) return 0;
  gbr::k_diag_act_sweep<<<152 * 8, 256, 0, stream>>>(act, first, count,
                                                      reinterpret_cast<unsigned*>(out));
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

extern "C" int gbr_diag_chain(int kind, int n, const void* x, size_t x_bytes, unsigned* sink,
                              cudaStream_t stream) {
  if (n < 0 || (kind != 0 && kind != 1) || !sink) return 1;
  if (kind == 1 && (!x || x_bytes % 16 != 0 || (reinterpret_cast<uintptr_t>(x) & 15u) != 0))
    return 1;
  static bool attr_set = false;
  if (!attr_set) {
    // a 16-CTA cluster is a non-portable size
    if (cudaFuncSetAttribute(gbr::k_diag_wait_only, cudaFuncAttributeNonPortableClusterSizeAllowed,
                             1) != cudaSuccess ||
        cudaFuncSetAttribute(gbr::k_diag_read_x, cudaFuncAttributeNonPortableClusterSizeAllowed,
                             1) != cudaSuccess)
      return 3;
    attr_set = true;
  }
  for (int i = 0; i < n; ++i)
    if (gbr::launch_one(kind, x, (int)(x_bytes / 16), sink, stream) != cudaSuccess) return 3;
  return 0;
}

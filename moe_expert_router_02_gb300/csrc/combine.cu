// The unique-route table's consumer: routed gather + shared-expert add.
//
// For each group of T tokens the experts ran once per unique (token, expert)
// route (b70 lab note "MTP1 M=2 gather/shared-add gate", "Real route-direct
// result": "gather retains distinct route weights and may reuse one expert
// output row for duplicate slots"). Token t's output is the weighted sum of
// the rows its k slots map to, accumulated in FP32 in slot order, rounded to
// BF16, plus the shared expert's BF16 output, rounded to BF16 again ("Exact
// arithmetic": FP32 routed accumulation -> BF16 -> add shared BF16 -> BF16).
//
// HBM-bound: each thread owns 8 consecutive elements of one group's rows and
// streams them with 16-byte non-allocating loads; the map and weights of the
// group sit in shared memory.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace gbr {
namespace {

constexpr int kGaThreads = 256;
constexpr int kGaMaxSlots = 128;  // T * k

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// round-to-nearest-even to BF16 bits
__device__ __forceinline__ uint32_t to_bf16_bits(float f) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}

template <bool VEC>
__global__ void __launch_bounds__(kGaThreads)
    k_gather_add(const uint16_t* __restrict__ y, const uint8_t* __restrict__ map,
                 const float* __restrict__ w, const uint16_t* __restrict__ shared, int G, int T,
                 int k, int D, uint16_t* __restrict__ out) {
  __shared__ uint8_t s_map[kGaMaxSlots];
  __shared__ float s_w[kGaMaxSlots];
  const int n = T * k;
  for (int g = blockIdx.y; g < G; g += gridDim.y) {
    __syncthreads();  // the previous group's map and weights are no longer read
    for (int i = threadIdx.x; i < n; i += kGaThreads) {
      s_map[i] = map[(size_t)g * n + i];
      s_w[i] = w[(size_t)g * n + i];
    }
    __syncthreads();
    const int d0 = (blockIdx.x * kGaThreads + threadIdx.x) * (VEC ? 8 : 1);
    if (d0 >= D) continue;
    for (int t = 0; t < T; ++t) {
      float acc[VEC ? 8 : 1];
#pragma unroll
      for (int i = 0; i < (VEC ? 8 : 1); ++i) acc[i] = 0.0f;
      for (int s = 0; s < k; ++s) {
        const int u = s_map[t * k + s];
        if (u >= n) continue;  // not a unique position: contributes nothing
        const float ws = s_w[t * k + s];
        const uint16_t* row = y + (((size_t)g * n + u) * T + t) * D + d0;
        if (VEC) {
          const uint4 v = ld_nc_v4(row);
          const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[2 * i] = __fmaf_rn(ws, bf16_lo(q[i]), acc[2 * i]);
            acc[2 * i + 1] = __fmaf_rn(ws, bf16_hi(q[i]), acc[2 * i + 1]);
          }
        } else {
          acc[0] = __fmaf_rn(ws, __uint_as_float((uint32_t)__ldg(row) << 16), acc[0]);
        }
      }
      const size_t o = ((size_t)g * T + t) * D + d0;
      if (VEC) {
        const uint4 sv = ld_nc_v4(shared + o);
        const uint32_t q[4] = {sv.x, sv.y, sv.z, sv.w};
        uint32_t r[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float lo = __fadd_rn(bf16_lo(to_bf16_bits(acc[2 * i])), bf16_lo(q[i]));
          const float hi = __fadd_rn(bf16_lo(to_bf16_bits(acc[2 * i + 1])), bf16_hi(q[i]));
          r[i] = to_bf16_bits(lo) | (to_bf16_bits(hi) << 16);
        }
        *reinterpret_cast<uint4*>(out + o) = make_uint4(r[0], r[1], r[2], r[3]);
      } else {
        const float sum = __fadd_rn(__uint_as_float(to_bf16_bits(acc[0]) << 16),
                                    __uint_as_float((uint32_t)__ldg(shared + o) << 16));
        out[o] = (uint16_t)to_bf16_bits(sum);
      }
    }
  }
}

}  // namespace

cudaError_t launch_gather_add(const void* y, const uint8_t* map, const float* w,
                              const void* shared, int G, int T, int k, int D, void* out,
                              cudaStream_t stream) {
  const bool vec = D % 8 == 0 &&
                   ((reinterpret_cast<uintptr_t>(y) | reinterpret_cast<uintptr_t>(shared) |
                     reinterpret_cast<uintptr_t>(out)) & 15u) == 0;
  const int per = vec ? 8 * kGaThreads : kGaThreads;
  const dim3 grid((D + per - 1) / per, G < 65535 ? G : 65535);
  const auto* yy = static_cast<const uint16_t*>(y);
  const auto* ss = static_cast<const uint16_t*>(shared);
  auto* oo = static_cast<uint16_t*>(out);
  if (vec)
    k_gather_add<true><<<grid, kGaThreads, 0, stream>>>(yy, map, w, ss, G, T, k, D, oo);
  else
    k_gather_add<false><<<grid, kGaThreads, 0, stream>>>(yy, map, w, ss, G, T, k, D, oo);
  return cudaGetLastError();
}

}  // namespace gbr

// router_select and route_table kernels: the selection stage and the
// unique-route table as standalone launches.
#include "kernels.h"
#include "select.cuh"

namespace gbr {
namespace {

constexpr int kSelWarps = 8;

template <int VPL>
__global__ void __launch_bounds__(kSelWarps * 32)
    k_select(const float* __restrict__ logits, const float* __restrict__ bias, int M, int E, int k,
             int act, int32_t* __restrict__ out_idx, float* __restrict__ out_w) {
  const int row = blockIdx.x * kSelWarps + (threadIdx.x >> 5);
  if (row >= M) return;  // whole warps leave together
  warp_select_row<VPL>(LdPlain{logits + (size_t)row * E}, bias, E, k, act,
                       out_idx + (size_t)row * k, out_w + (size_t)row * k, nullptr);
}

constexpr int kTblWarps = 8;

__global__ void __launch_bounds__(kTblWarps * 32)
    k_route_table(const int32_t* __restrict__ idx, int G, int T, int k,
                  int32_t* __restrict__ unique, uint8_t* __restrict__ mask,
                  uint8_t* __restrict__ map, int32_t* __restrict__ count) {
  __shared__ int32_t s_idx[kTblWarps][128];
  __shared__ int32_t s_rank[kTblWarps][128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x * kTblWarps + warp;
  if (g >= G) return;
  const int n = T * k;
  for (int p = lane; p < n; p += 32) s_idx[warp][p] = idx[(size_t)g * n + p];
  __syncwarp();
  warp_route_table(s_idx[warp], s_rank[warp], T, k, unique + (size_t)g * n, mask + (size_t)g * n,
                   map + (size_t)g * n, count + g);
}

// Groups of n = T*k <= 32 entries: floor(32 / n) groups per warp, one entry
// per lane, so a warp's loads and stores cover consecutive groups'
// contiguous rows; each warp takes kTblChunks such sets of groups and
// issues all of their loads first (enough bytes in flight to stream HBM).
constexpr int kTblChunks = 8;

__global__ void __launch_bounds__(kTblWarps * 32)
    k_route_table32(const int32_t* __restrict__ idx, int G, int T, int k,
                    int32_t* __restrict__ unique, uint8_t* __restrict__ mask,
                    uint8_t* __restrict__ map, int32_t* __restrict__ count) {
  const int lane = threadIdx.x & 31;
  const int n = T * k;
  const int gpw = 32 / n;  // groups per warp and chunk
  const int gl = lane / n, p = lane - gl * n;
  const int gbase = gl * n;
  const uint32_t gmask = gl < gpw ? (n == 32 ? kFull : ((1u << n) - 1u) << gbase) : 0u;
  const long long warp_id = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long g0 = warp_id * kTblChunks * gpw;  // first group of this warp
  int32_t v[kTblChunks];
#pragma unroll
  for (int c = 0; c < kTblChunks; ++c) {
    const long long g = g0 + (long long)c * gpw + gl;
    v[c] = (gl < gpw && g < G) ? __ldg(idx + g * n + p) : 0;
  }
#pragma unroll
  for (int c = 0; c < kTblChunks; ++c) {
    const long long g = g0 + (long long)c * gpw + gl;
    const bool valid = gl < gpw && g < G;
    const TableLane r = table_lanes(v[c], valid, gmask, gbase, T, k);
    if (valid) {
      const long long o = g * n + p;
      unique[o] = r.uniq;
      mask[o] = (uint8_t)r.mask;
      map[o] = (uint8_t)r.map;
      if (p == 0) count[g] = r.count;
    }
  }
}

__global__ void k_near_tie_keys(const float* __restrict__ z, const float* __restrict__ bias, int n,
                                int act, float* __restrict__ hi, float* __restrict__ lo) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const NearKey k = near_key(act, z[i], bias ? bias[i] : 0.0f);
    hi[i] = k.hi;
    lo[i] = k.lo;
  }
}

}  // namespace

cudaError_t launch_near_tie_keys(const float* z, const float* bias, int n, int act, float* hi,
                                 float* lo, cudaStream_t stream) {
  const int blocks = (n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024;
  k_near_tie_keys<<<blocks, 256, 0, stream>>>(z, bias, n, act, hi, lo);
  return cudaGetLastError();
}

cudaError_t launch_select(const float* logits, const float* bias, int M, int E, int k, int act,
                          int32_t* out_idx, float* out_w, cudaStream_t stream) {
  const dim3 grid((M + kSelWarps - 1) / kSelWarps), block(kSelWarps * 32);
  if (E <= 32) k_select<1><<<grid, block, 0, stream>>>(logits, bias, M, E, k, act, out_idx, out_w);
  else if (E <= 64) k_select<2><<<grid, block, 0, stream>>>(logits, bias, M, E, k, act, out_idx, out_w);
  else if (E <= 128) k_select<4><<<grid, block, 0, stream>>>(logits, bias, M, E, k, act, out_idx, out_w);
  else if (E <= 256) k_select<8><<<grid, block, 0, stream>>>(logits, bias, M, E, k, act, out_idx, out_w);
  else k_select<16><<<grid, block, 0, stream>>>(logits, bias, M, E, k, act, out_idx, out_w);
  return cudaGetLastError();
}

cudaError_t launch_route_table(const int32_t* idx, int groups, int T, int k, int32_t* unique,
                               uint8_t* mask, uint8_t* map, int32_t* count, cudaStream_t stream) {
  const dim3 block(kTblWarps * 32);
  if (T * k <= 32) {
    const long long per_warp = (long long)(32 / (T * k)) * kTblChunks;
    const long long warps = (groups + per_warp - 1) / per_warp;
    const dim3 grid((unsigned)((warps + kTblWarps - 1) / kTblWarps));
    k_route_table32<<<grid, block, 0, stream>>>(idx, groups, T, k, unique, mask, map, count);
  } else {
    const dim3 grid((groups + kTblWarps - 1) / kTblWarps);
    k_route_table<<<grid, block, 0, stream>>>(idx, groups, T, k, unique, mask, map, count);
  }
  return cudaGetLastError();
}

}  // namespace gbr

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

// Groups of n = T*k <= 16 entries, one group per lane: a warp stages its 32
// groups' ids in shared memory (coalesced), each lane deduplicates its
// group with compares on register copies (static indices), writes the
// table rows into its own shared-memory row, and the warp stores all rows
// coalesced. Rows are padded to an odd stride (no bank conflicts).
constexpr int kLaneWarps = 8;
constexpr int kLaneMax = 16;
constexpr int kLaneStride = kLaneMax + 1;

__global__ void __launch_bounds__(kLaneWarps * 32)
    k_route_table_lane(const int32_t* __restrict__ idx, int G, int T, int k,
                       int32_t* __restrict__ unique, uint8_t* __restrict__ mask,
                       uint8_t* __restrict__ map, int32_t* __restrict__ count) {
  __shared__ int32_t s_in[kLaneWarps][32 * kLaneStride];
  __shared__ int32_t s_un[kLaneWarps][32 * kLaneStride];
  __shared__ uint8_t s_mk[kLaneWarps][32 * kLaneStride];
  __shared__ uint8_t s_mp[kLaneWarps][32 * kLaneStride];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = T * k;
  const long long g0 = ((long long)blockIdx.x * kLaneWarps + warp) * 32;
  if (g0 >= G) return;  // whole warps leave together
  const int ng = G - g0 < 32 ? (int)(G - g0) : 32;
  const int total = ng * n;
  const uint32_t inv_n = (65536u + (uint32_t)n - 1u) / (uint32_t)n;  // i / n = (i * inv_n) >> 16, i < 512
  int32_t* in = s_in[warp];
  const int32_t* src = idx + g0 * n;
  // every load of the lane in flight at once (total <= 32 * kLaneMax)
  int32_t r[kLaneMax];
#pragma unroll
  for (int u = 0; u < kLaneMax; ++u) {
    const int i = lane + 32 * u;
    r[u] = i < total ? __ldg(src + i) : 0;
  }
#pragma unroll
  for (int u = 0; u < kLaneMax; ++u) {
    const int i = lane + 32 * u;
    if (i < total) {
      const int gl = (int)(((uint32_t)i * inv_n) >> 16);
      in[gl * kLaneStride + (i - gl * n)] = r[u];
    }
  }
  __syncwarp();
  const int row = lane * kLaneStride;
  int32_t v[kLaneMax];
#pragma unroll
  for (int p = 0; p < kLaneMax; ++p) v[p] = p < n ? in[row + p] : 0;
  // first occurrence of each entry's id, and the set of first occurrences
  int fp[kLaneMax];
  uint32_t F = 0u;
#pragma unroll
  for (int p = 0; p < kLaneMax; ++p) {
    int f = p;
#pragma unroll
    for (int q = p - 1; q >= 0; --q) f = (v[q] == v[p]) ? q : f;
    fp[p] = f;
    if (p < n && f == p) F |= 1u << p;
  }
  int32_t* un = s_un[warp] + row;
  uint8_t* mk = s_mk[warp] + row;
  uint8_t* mp = s_mp[warp] + row;
#pragma unroll
  for (int u = 0; u < kLaneMax; ++u) {
    if (u < n) {
      un[u] = -1;
      mk[u] = 0;
    }
  }
  int tok = 0, rem = 0;  // token of entry p = p / k
#pragma unroll
  for (int p = 0; p < kLaneMax; ++p) {
    if (p < n) {
      const int u = __popc(F & ((1u << fp[p]) - 1u));  // unique position of the id
      mp[p] = (uint8_t)u;
      if (fp[p] == p) un[u] = v[p];
      mk[u] = (uint8_t)(mk[u] | (1u << tok));
      if (++rem == k) rem = 0, ++tok;
    }
  }
  __syncwarp();
  const long long o = g0 * n;
  for (int i = lane; i < total; i += 32) {
    const int gl = (int)(((uint32_t)i * inv_n) >> 16);
    const int e = gl * kLaneStride + (i - gl * n);
    unique[o + i] = s_un[warp][e];
    mask[o + i] = s_mk[warp][e];
    map[o + i] = s_mp[warp][e];
  }
  if (lane < ng) count[g0 + lane] = __popc(F);
}

// Groups of N = T*k entries, N a multiple of 4 up to 16, with 16-byte
// aligned ids and 4-byte aligned masks and maps: one lane per group reads
// the group's ids with 16-byte loads straight into registers, finds each
// entry's first occurrence there, and scatters the unique ids and token
// masks into its own shared-memory row (written and read back by the same
// thread, so no barrier), from which it stores its table rows with 16-byte
// (ids) and 4-byte (masks, map) stores.
template <int N>
__global__ void __launch_bounds__(kLaneWarps * 32)
    k_route_table_vec(const int32_t* __restrict__ idx, int G, int k,
                      int32_t* __restrict__ unique, uint8_t* __restrict__ mask,
                      uint8_t* __restrict__ map, int32_t* __restrict__ count) {
  __shared__ __align__(16) int32_t s_un[kLaneWarps * 32][N];
  __shared__ __align__(4) uint8_t s_mk[kLaneWarps * 32][N];
  const long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= G) return;
  int32_t v[N];
  const int4* src = reinterpret_cast<const int4*>(idx + g * N);
#pragma unroll
  for (int c = 0; c < N / 4; ++c) {
    const int4 q = __ldg(src + c);
    v[4 * c] = q.x, v[4 * c + 1] = q.y, v[4 * c + 2] = q.z, v[4 * c + 3] = q.w;
  }
  int32_t* un = s_un[threadIdx.x];
  uint8_t* mk = s_mk[threadIdx.x];
#pragma unroll
  for (int c = 0; c < N / 4; ++c) {
    reinterpret_cast<int4*>(un)[c] = make_int4(-1, -1, -1, -1);
    reinterpret_cast<uint32_t*>(mk)[c] = 0u;
  }
  // first occurrence of each entry's id, and the set of first occurrences
  int fp[N];
  uint32_t F = 0u;
#pragma unroll
  for (int p = 0; p < N; ++p) {
    int f = p;
#pragma unroll
    for (int q = p - 1; q >= 0; --q) f = (v[q] == v[p]) ? q : f;
    fp[p] = f;
    F |= (f == p ? 1u : 0u) << p;
  }
  uint32_t mp[N / 4];
#pragma unroll
  for (int c = 0; c < N / 4; ++c) mp[c] = 0u;
  int tok = 0, rem = 0;  // token of entry p = p / k
#pragma unroll
  for (int p = 0; p < N; ++p) {
    const int u = __popc(F & ((1u << fp[p]) - 1u));  // unique position of the id
    mp[p / 4] |= (uint32_t)u << (8 * (p % 4));
    if (fp[p] == p) un[u] = v[p];
    mk[u] = (uint8_t)(mk[u] | (1u << tok));
    if (++rem == k) rem = 0, ++tok;
  }
  int4* du = reinterpret_cast<int4*>(unique + g * N);
  uint32_t* dk = reinterpret_cast<uint32_t*>(mask + g * N);
  uint32_t* dm = reinterpret_cast<uint32_t*>(map + g * N);
#pragma unroll
  for (int c = 0; c < N / 4; ++c) {
    du[c] = reinterpret_cast<const int4*>(un)[c];
    dk[c] = reinterpret_cast<const uint32_t*>(mk)[c];
    dm[c] = mp[c];
  }
  count[g] = __popc(F);
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
  const int n = T * k;
  const bool vec = n % 4 == 0 && n <= 16 && ((uintptr_t)idx | (uintptr_t)unique) % 16 == 0 &&
                   ((uintptr_t)mask | (uintptr_t)map) % 4 == 0;
  if (vec) {
    const dim3 grid((unsigned)(((long long)groups + kLaneWarps * 32 - 1) / (kLaneWarps * 32)));
    const dim3 lb(kLaneWarps * 32);
    switch (n) {
      case 4: k_route_table_vec<4><<<grid, lb, 0, stream>>>(idx, groups, k, unique, mask, map, count); break;
      case 8: k_route_table_vec<8><<<grid, lb, 0, stream>>>(idx, groups, k, unique, mask, map, count); break;
      case 12: k_route_table_vec<12><<<grid, lb, 0, stream>>>(idx, groups, k, unique, mask, map, count); break;
      default: k_route_table_vec<16><<<grid, lb, 0, stream>>>(idx, groups, k, unique, mask, map, count); break;
    }
  } else if (T * k <= kLaneMax) {
    const long long warps = (groups + 31) / 32;
    const dim3 grid((unsigned)((warps + kLaneWarps - 1) / kLaneWarps));
    k_route_table_lane<<<grid, dim3(kLaneWarps * 32), 0, stream>>>(idx, groups, T, k, unique, mask,
                                                                   map, count);
  } else if (T * k <= 32) {
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

// Selection stage shared by every router kernel: keys, top-k under the
// (key desc, index asc) contract, FP64 guard-band refine, renormalisation,
// and the unique-route table emitter.
//
// Keys (dense_router_decode commit page, "DenseRouterDecodeKernel"):
//   softmax       key = the logit itself. Softmax is strictly increasing, so
//                 ranking logits ranks probabilities, and the full-E
//                 denominator cancels in the renormalisation over the k
//                 chosen experts: w_j = exp(l_j - l_0) / sum_i exp(l_i - l_0).
//   sqrt-softplus a = sqrt(max(z,0) + log1p(exp(-|z|))), key = a + bias;
//                 the weights use the unbiased a: w_j = a_j / sum_i a_i.
// Order (qwisp issue #145, "Bit-exactness"): higher key first, an equal key
// goes to the lower expert index; -0.0 equals +0.0.
//
// Exactness of the sqrt-softplus ranking. FP32 keys carry a bounded error
// (CUDA documents expf <= 2 ulp, log1pf <= 1 ulp, IEEE sqrtf): following
// the three steps gives |key32 - key| <= 2^-23 (2.25 a + 0.5 |key|) plus a
// tiny absolute term for subnormal softplus values. When two neighbouring
// keys among the first k+1 are closer than four times that bound, the
// candidates within the band of the k-th key are re-ranked with keys
// recomputed in FP64, which decides the order the FP64 definition gives.
#pragma once

#include "common.cuh"

namespace gbr {

struct LdPlain {  // generic-address loads (shared memory or read-only global)
  const float* p;
  __device__ __forceinline__ float operator()(int e) const { return p[e]; }
};

struct LdCG {  // global loads that bypass L1 (data written by other CTAs)
  const float* p;
  __device__ __forceinline__ float operator()(int e) const { return __ldcg(p + e); }
};

// Compare-exchange on packed (key, index) pairs: larger packed value first.
__device__ __forceinline__ void cas_desc(uint64_t& a, uint64_t& b) {
  const uint64_t hi = a > b ? a : b, lo = a > b ? b : a;
  a = hi;
  b = lo;
}

// Sorts VPL packed values descending in registers (odd-even transposition;
// fully unrolled, so every index is static).
template <int VPL>
__device__ __forceinline__ void sort_desc(uint64_t (&v)[VPL]) {
#pragma unroll
  for (int pass = 0; pass < VPL; ++pass) {
#pragma unroll
    for (int j = pass & 1; j + 1 < VPL; j += 2) cas_desc(v[j], v[j + 1]);
  }
}

// One warp selects the top-k of one row of E <= 32*VPL logits.
// Lane r < k writes slot r of out_idx / out_w and, if sel_out is not null,
// sel_out[r] (for a route table). All 32 lanes must call.
//
// Each lane packs its entries as (order-preserving key << 32 | ~index) and
// sorts them once; a round takes the warp maximum key (redux.sync), then
// the lowest index among the lanes holding it (redux.sync), and the winning
// lane shifts its sorted list by one. Scores are read back once at the end.
template <int VPL, class Ld>
__device__ __noinline__ void warp_select_row(const Ld ld, const float* __restrict__ bias, int E,
                                             int k, int act, int32_t* __restrict__ out_idx,
                                             float* __restrict__ out_w, int32_t* sel_out) {
  const int lane = threadIdx.x & 31;
  uint64_t pk[VPL];  // (key << 32) | (0xffffffff - expert); 0 = empty
  float amax = 0.0f, kabs = 0.0f;
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = lane + 32 * j;
    pk[j] = 0ull;
    if (e < E) {
      const float z = ld(e);
      float key = z;
      if (act != ACT_SOFTMAX) {
        const float a = sqrt_softplus_f32(z);
        key = bias ? a + __ldg(bias + e) : a;
        amax = fmaxf(amax, a);
        kabs = fmaxf(kabs, fabsf(key));
      }
      pk[j] = ((uint64_t)ord_of(key) << 32) | (uint64_t)(0xffffffffu - (uint32_t)e);
    }
  }
  sort_desc<VPL>(pk);

  // k+1 rounds: the (k+1)-th key is kept for the gap test.
  const int kk = min(k + 1, E);
  int sel_idx = -1;
  float sel_key = 0.0f;
  for (int r = 0; r < kk; ++r) {
    const uint32_t bo = (uint32_t)(pk[0] >> 32);
    const uint32_t wbest = __reduce_max_sync(kFull, bo);
    const uint32_t cand = (bo == wbest) ? 0xffffffffu - (uint32_t)pk[0] : 0xffffffffu;
    const uint32_t widx = __reduce_min_sync(kFull, cand);  // lowest index among equal keys
    if (lane == r) {
      sel_idx = (int)widx;
      sel_key = float_of_ord(wbest);
    }
    if ((int)(widx & 31u) == lane) {
#pragma unroll
      for (int j = 0; j + 1 < VPL; ++j) pk[j] = pk[j + 1];
      pk[VPL - 1] = 0ull;
    }
  }

  if (act == ACT_SQRT_SOFTPLUS) {
    // FP32 key error bound; non-negative floats order like their bit patterns
    const float amax_w = __uint_as_float(__reduce_max_sync(kFull, __float_as_uint(amax)));
    const float kabs_w = __uint_as_float(__reduce_max_sync(kFull, __float_as_uint(kabs)));
    const double err = 0x1p-23 * (2.25 * (double)amax_w + 0.5 * (double)kabs_w) + 0x1p-60;
    const double band = 4.0 * err;
    const float next_key = __shfl_down_sync(kFull, sel_key, 1);
    const bool close = (lane < kk - 1) && ((double)sel_key - (double)next_key <= band);
    if (__any_sync(kFull, close)) {
      // re-rank every expert whose FP32 key lies within the band of the k-th
      const double thr = (double)__shfl_sync(kFull, sel_key, k - 1) - band;
      double k64[VPL];
      uint32_t cmask = 0;
#pragma unroll
      for (int j = 0; j < VPL; ++j) {
        k64[j] = 0.0;
        const int e = lane + 32 * j;
        if (e < E) {
          const float z = ld(e);
          const float a = sqrt_softplus_f32(z);
          const float kv = bias ? a + __ldg(bias + e) : a;
          if ((double)kv >= thr) {
            cmask |= 1u << j;
            k64[j] = sqrt_softplus_f64((double)z) + (bias ? (double)__ldg(bias + e) : 0.0);
          }
        }
      }
      for (int r = 0; r < k; ++r) {
        double bv = -INFINITY;
        int bidx = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
          if (((cmask >> j) & 1u) && (bidx == 0x7fffffff || k64[j] > bv)) {
            bv = k64[j];
            bidx = lane + 32 * j;
          }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          const double ov = __shfl_xor_sync(kFull, bv, off);
          const int oi = __shfl_xor_sync(kFull, bidx, off);
          if (ov > bv || (ov == bv && oi < bidx)) {
            bv = ov;
            bidx = oi;
          }
        }
        if ((bidx & 31) == lane) cmask &= ~(1u << (bidx >> 5));
        if (lane == r) sel_idx = bidx;
      }
    }
  }

  // weights over the chosen k, summed in slot order
  float s = 0.0f;
  if (act == ACT_SOFTMAX) {
    // the key is the logit (-0.0 read back as +0.0, which exp treats alike)
    const float z0 = __shfl_sync(kFull, sel_key, 0);
    if (lane < k) s = expf(sel_key - z0);
  } else if (lane < k) {
    s = sqrt_softplus_f32(ld(sel_idx));
  }
  float sum = 0.0f;
#pragma unroll
  for (int r = 0; r < kMaxK; ++r) {
    const float v = __shfl_sync(kFull, s, r);
    if (r < k) sum += v;
  }
  if (lane < k) {
    out_idx[lane] = sel_idx;
    out_w[lane] = (sum > 0.0f) ? s / sum : 1.0f / (float)k;
    if (sel_out) sel_out[lane] = sel_idx;
  }
}

// One warp emits the unique-route table of one group of T tokens x k slots
// from ids in shared memory s_idx[T*k] (T*k <= 128); s_rank[T*k] is shared
// scratch. Equivalent to the serial walk over (token, slot): the first
// occurrence of an id defines its unique position, ranked by a prefix count.
// (b70 lab note, "Unique-route router screen": stable dedup, prefix ranking,
// token masks, slot mapping.)
static __device__ __noinline__ void warp_route_table(const int32_t* s_idx, int32_t* s_rank, int T, int k,
                                              int32_t* __restrict__ unique,
                                              uint8_t* __restrict__ mask,
                                              uint8_t* __restrict__ map,
                                              int32_t* __restrict__ count) {
  const int lane = threadIdx.x & 31;
  const int n = T * k;
  int first[4];
  int base = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int p = lane + 32 * i;
    int f = -1;
    if (p < n) {
      const int32_t v = s_idx[p];
      f = p;
      for (int q = 0; q < p; ++q) {
        if (s_idx[q] == v) {
          f = q;
          break;
        }
      }
    }
    first[i] = f;
    const bool is_first = (p < n) && (f == p);
    const unsigned b = __ballot_sync(kFull, is_first);
    if (is_first) s_rank[p] = base + __popc(b & ((1u << lane) - 1u));
    base += __popc(b);
  }
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int p = lane + 32 * i;
    if (p < n) {
      const int32_t v = s_idx[p];
      const int u = s_rank[first[i]];
      map[p] = (uint8_t)u;
      if (first[i] == p) {
        uint32_t bits = 0;
        for (int q = p; q < n; ++q)
          if (s_idx[q] == v) bits |= 1u << (q / k);
        unique[u] = v;
        mask[u] = (uint8_t)bits;
      }
    }
  }
  for (int u = base + lane; u < n; u += 32) {
    unique[u] = -1;
    mask[u] = 0;
  }
  if (lane == 0) *count = base;
  __syncwarp();
}

}  // namespace gbr

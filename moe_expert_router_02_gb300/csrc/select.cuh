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
//   sigmoid       a = 1 / (1 + exp(-z)), key = a + bias, weights as above
//                 (the biased sigmoid score of the same page's routing).
//   softmax+bias  p = exp(z - max) / sum_e exp(z_e - max) over all E,
//                 key = p + bias, weights the unbiased p renormalised (the
//                 bias variant of the softmax route, qwisp issue #145,
//                 "Gates"); near ties are re-ranked with FP64 keys.
// Order (qwisp issue #145, "Bit-exactness"): higher key first, an equal key
// goes to the lower expert index; -0.0 equals +0.0.
//
// Exactness of the biased rankings. FP32 keys carry a bounded error: the
// branch-free scores of common.cuh are within c 2^-23 a + 2^-60 of the exact
// score (c = act_err_coef, checked at every FP32 input against CUDA's
// documented expf/log1pf/sqrtf composition), so |key32 - key| <=
// 2^-23 (c a + 0.5 |key|) + 2^-59 (key_err_bound). Two keys whose exact
// order differs from their FP32 order are then within twice that bound,
// and so is every exact top-k member of the k-th FP32 key. When two
// neighbouring keys among the first k+1 are that close, the candidates
// within that band of the k-th key are re-ranked with
// double-float keys (relative error near 2^-42, FP32 arithmetic only); a
// pair of those still too close to call, from different inputs, is ranked
// with FP64 keys, which decide the order the FP64 definition gives.
#pragma once

#include "common.cuh"
#include "dfkey.cuh"

namespace gbr {

#ifdef GBR_PHASE_STAMPS
// Measurement build only: lane 0 of a selecting warp of CTA b < 16 stamps
// %globaltimer at the selection's sub-phases (0 keys loaded and packed,
// 1 sorted, 2 k+1 rounds done, 3 weights computed, 4 stored); the last
// selection of each CTA rank wins.
namespace {
__device__ unsigned long long g_sel_stamps[16][5];
// rows whose selection took the near-tie re-rank, of those the rows that
// went on to FP64 keys, and rows whose 32-bit rounds met equal truncated
// keys and ran again on (key, index) pairs (warp selections of this
// translation unit)
__device__ unsigned long long g_sel_refines[3];
}
#define SEL_STAMP(i)                                                           \
  do {                                                                         \
    if ((threadIdx.x & 31) == 0 && blockIdx.x < 16) {                          \
      unsigned long long t_;                                                   \
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_)::"memory");         \
      g_sel_stamps[blockIdx.x][i] = t_;                                        \
    }                                                                          \
  } while (0)
#else
#define SEL_STAMP(i) \
  do {               \
  } while (0)
#endif

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

// Sorts VPL packed values descending in registers, fully unrolled so that
// every index is static: 4 and 8 values by the minimal comparator networks
// (5 comparators in 3 layers; 19 in 6 layers, Knuth TAOCP vol. 3,
// sec. 5.3.4), any other count by odd-even transposition.
template <int VPL>
__device__ __forceinline__ void sort_desc(uint64_t (&v)[VPL]) {
  if constexpr (VPL == 8) {
    cas_desc(v[0], v[2]), cas_desc(v[1], v[3]), cas_desc(v[4], v[6]), cas_desc(v[5], v[7]);
    cas_desc(v[0], v[4]), cas_desc(v[1], v[5]), cas_desc(v[2], v[6]), cas_desc(v[3], v[7]);
    cas_desc(v[0], v[1]), cas_desc(v[2], v[3]), cas_desc(v[4], v[5]), cas_desc(v[6], v[7]);
    cas_desc(v[2], v[4]), cas_desc(v[3], v[5]);
    cas_desc(v[1], v[4]), cas_desc(v[3], v[6]);
    cas_desc(v[1], v[2]), cas_desc(v[3], v[4]), cas_desc(v[5], v[6]);
  } else if constexpr (VPL == 4) {
    cas_desc(v[0], v[1]), cas_desc(v[2], v[3]);
    cas_desc(v[0], v[2]), cas_desc(v[1], v[3]);
    cas_desc(v[1], v[2]);
  } else {
#pragma unroll
    for (int pass = 0; pass < VPL; ++pass) {
#pragma unroll
      for (int j = pass & 1; j + 1 < VPL; j += 2) cas_desc(v[j], v[j + 1]);
    }
  }
}

// The same networks on 32-bit values (one max and one min per comparator).
__device__ __forceinline__ void cas_desc32(uint32_t& a, uint32_t& b) {
  const uint32_t hi = max(a, b), lo = min(a, b);
  a = hi;
  b = lo;
}

template <int VPL>
__device__ __forceinline__ void sort_desc32(uint32_t (&v)[VPL]) {
  if constexpr (VPL == 8) {
    cas_desc32(v[0], v[2]), cas_desc32(v[1], v[3]), cas_desc32(v[4], v[6]), cas_desc32(v[5], v[7]);
    cas_desc32(v[0], v[4]), cas_desc32(v[1], v[5]), cas_desc32(v[2], v[6]), cas_desc32(v[3], v[7]);
    cas_desc32(v[0], v[1]), cas_desc32(v[2], v[3]), cas_desc32(v[4], v[5]), cas_desc32(v[6], v[7]);
    cas_desc32(v[2], v[4]), cas_desc32(v[3], v[5]);
    cas_desc32(v[1], v[4]), cas_desc32(v[3], v[6]);
    cas_desc32(v[1], v[2]), cas_desc32(v[3], v[4]), cas_desc32(v[5], v[6]);
  } else if constexpr (VPL == 4) {
    cas_desc32(v[0], v[1]), cas_desc32(v[2], v[3]);
    cas_desc32(v[0], v[2]), cas_desc32(v[1], v[3]);
    cas_desc32(v[1], v[2]);
  } else {
#pragma unroll
    for (int pass = 0; pass < VPL; ++pass) {
#pragma unroll
      for (int j = pass & 1; j + 1 < VPL; j += 2) cas_desc32(v[j], v[j + 1]);
    }
  }
}

// k rounds of (key desc, index asc) over the FP64 keys of the candidates in
// cmask (lane + 32 j holds k64[j]); returns this lane's pick (lane < k).
template <int VPL>
__device__ __forceinline__ int fp64_rounds(const double (&k64)[VPL], uint32_t cmask, int k) {
  const int lane = threadIdx.x & 31;
  int pick = -1;
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
    if (lane == r) pick = bidx;
  }
  return pick;
}

// The FP64 re-ranking of the candidates in cmask (k rounds of
// (key desc, index asc)); returns this lane's pick (lane < k). Out of line:
// FP64 is slow on this part and must not be issued on the common path.
template <int VPL, class Ld>
__device__ __noinline__ int select_fp64(const Ld ld, const float* __restrict__ bias, int act, int k,
                                        uint32_t cmask) {
  const int lane = threadIdx.x & 31;
  double k64[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = lane + 32 * j;
    k64[j] = 0.0;
    if ((cmask >> j) & 1u)
      k64[j] = act_f64(act, (double)ld(e)) + (bias ? (double)bias[e] : 0.0);
  }
  return fp64_rounds<VPL>(k64, cmask, k);
}

// Softmax probability + bias in FP64 for the candidates in cmask: the row's
// FP64 denominator over all E experts (relative to the row maximum zmax),
// then the rounds. Every lane ends the butterfly with the same sum.
template <int VPL, class Ld>
__device__ __noinline__ int select_softmax_bias_fp64(const Ld ld, const float* __restrict__ bias,
                                                     int E, int k, float zmax, uint32_t cmask) {
  const int lane = threadIdx.x & 31;
  double ex[VPL];
  double part = 0.0;
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = lane + 32 * j;
    ex[j] = 0.0;
    if (e < E) {
      ex[j] = exp((double)ld(e) - (double)zmax);
      part += ex[j];
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(kFull, part, off);
  double k64[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = lane + 32 * j;
    k64[j] = ((cmask >> j) & 1u) ? ex[j] / part + (double)bias[e] : 0.0;
  }
  return fp64_rounds<VPL>(k64, cmask, k);
}

// FP32 softmax-probability + bias key of one expert, given the row maximum
// and the FP32 denominator (the main pass and the near-tie candidate mask
// compute it the same way).
__device__ __forceinline__ float softmax_bias_key32(float z, float zmax, float zsum, float b) {
  return __fadd_rn(__fdiv_rn(expf(__fsub_rn(z, zmax)), zsum), b);
}

// Bound on |key32 - key| for the softmax-probability + bias key, u = 2^-24:
// z - max rounds to d (1 + u), expf adds at most 2 ulp (4u), the FP32
// denominator sums each term through at most VPL - 1 + 5 roundings, the
// division and the bias add one rounding each. With pmax the row's largest
// FP32 probability, s1z = sum_e e^d |d| / Z (the exp argument's error
// carried into the denominator) and p |d| <= 1 / (e Z):
//   |key32 - key| <= u ((VPL + 14 + 1.01 s1z) pmax + 0.37 / Z + |key|max).
__device__ __forceinline__ float softmax_bias_err_bound(int vpl, float pmax, float s1z, float zsum,
                                                        float kabs) {
  const float c = __fadd_ru((float)(vpl + 14), __fmul_ru(1.01f, s1z));
  const float t = __fadd_ru(__fmaf_ru(c, pmax, __fdiv_ru(0.37f, zsum)), kabs);
  return __fadd_ru(__fmul_ru(t, 0x1p-24f), 0x1p-60f);
}

// The near-tie re-ranking of one row (all lanes call): every expert whose
// FP32 key lies within `band` of the k-th is re-keyed; returns this lane's
// pick (lane < k). Out of line: it runs rarely, and the common path's
// instructions stay contiguous.
template <int VPL, class Ld>
__device__ __noinline__ int refine_near_ties(const Ld ld, const float* __restrict__ bias, int act, int E,
                                             int k, int kk, float sel_key, int sel_idx,
                                             float band) {
  const int lane = threadIdx.x & 31;
  // re-rank every expert whose FP32 key lies within the band of the k-th
  const float thr = __fsub_rd(__shfl_sync(kFull, sel_key, k - 1), band);
  uint32_t cmask = 0;
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = lane + 32 * j;
    if (e < E) {
      const float a = act_f32(act, ld(e));
      const float kv = bias ? a + bias[e] : a;
      if (kv >= thr) cmask |= 1u << j;
    }
  }
  // double-float keys, one candidate per lane per round
  float khi[VPL], klo[VPL], ksc[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) khi[j] = klo[j] = ksc[j] = 0.0f;
  uint32_t todo = cmask;
  while (__any_sync(kFull, todo != 0u)) {
    const bool has = todo != 0u;
    const int j = has ? __ffs(todo) - 1 : 0;
    const int e = lane + 32 * j;
    const float z = has ? ld(e) : 0.0f;
    const float b = (has && bias) ? bias[e] : 0.0f;
    const NearKey nk = near_key_ool(act, z, b);
#pragma unroll
    for (int jj = 0; jj < VPL; ++jj) {
      if (has && jj == j) {
        khi[jj] = nk.hi;
        klo[jj] = nk.lo;
        ksc[jj] = nk.scale;
      }
    }
    todo &= todo - 1u;
  }
  // k+1 rounds of (key desc, index asc) over the candidates; a pair of
  // consecutive picks too close for the double-float keys, from
  // different inputs, sends the row to FP64
  bool amb = false;
  float ph = 0.0f, pl = 0.0f, psc = 0.0f, pz = 0.0f, pb = 0.0f;
  int pick = -1;
  uint32_t left = cmask;
  for (int r = 0; r < kk; ++r) {
    float bh = -INFINITY, bl = 0.0f, bsc = 0.0f;
    int bidx = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      if (((left >> j) & 1u) && (bidx == 0x7fffffff || df_gt(khi[j], klo[j], bh, bl))) {
        bh = khi[j];
        bl = klo[j];
        bsc = ksc[j];
        bidx = lane + 32 * j;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float oh = __shfl_xor_sync(kFull, bh, off);
      const float ol = __shfl_xor_sync(kFull, bl, off);
      const float os = __shfl_xor_sync(kFull, bsc, off);
      const int oi = __shfl_xor_sync(kFull, bidx, off);
      const bool take = oi != 0x7fffffff &&
                        (bidx == 0x7fffffff || df_gt(oh, ol, bh, bl) ||
                         (oh == bh && ol == bl && oi < bidx));
      if (take) {
        bh = oh;
        bl = ol;
        bsc = os;
        bidx = oi;
      }
    }
    if (bidx == 0x7fffffff) break;  // fewer candidates than rounds
    if ((bidx & 31) == lane) left &= ~(1u << (bidx >> 5));
    const float wz = ld(bidx);
    const float wb = bias ? bias[bidx] : 0.0f;
    if (r > 0 && !near_distinct(ph, pl, psc, bh, bl, bsc) && !(pz == wz && pb == wb))
      amb = true;
    ph = bh, pl = bl, psc = bsc, pz = wz, pb = wb;
    if (lane == r) pick = bidx;
  }
  if (!amb) {
    if (lane < k) sel_idx = pick;
  } else {
#ifdef GBR_PHASE_STAMPS
    if (lane == 0) atomicAdd(&g_sel_refines[1], 1ull);
#endif
    const int pick64 = select_fp64<VPL>(ld, bias, act, k, cmask);
    if (lane < k) sel_idx = pick64;
  }
  return sel_idx;
}

// The sum of the first k of v[0..KC) in the tree order of the warp
// selection's butterfly (j + j^8, then ^4, ^2, ^1 over 16 slots), for
// kernels that hold a row's chosen scores in one thread.
template <int KC>
__device__ __forceinline__ float slot_tree_sum(const float (&v)[KC], int k) {
  float t[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) t[j] = (j < KC && j < k) ? v[j < KC ? j : 0] : 0.0f;
#pragma unroll
  for (int w = 8; w > 0; w >>= 1) {
#pragma unroll
    for (int j = 0; j < w; ++j) t[j] = t[j] + t[j + w];
  }
  return t[0];
}

// One warp selects the top-k of one row of E <= 32*VPL logits.
// Lane r < k writes slot r of out_idx / out_w and, if sel_out is not null,
// sel_out[r] (for a route table). All 32 lanes must call.
//
// Each lane packs its entries as (order-preserving key << 32 | ~index) and
// sorts them once; a round takes the warp maximum key (redux.sync), then
// the lowest index among the lanes holding it (redux.sync), and the winning
// lane shifts its sorted list by one. Scores are read back once at the end.
// One copy per activation: the kernels run it once per row and call, so the
// instruction fetches of code for the other activation would be paid cold.
template <int VPL, int act, class Ld>
__device__ __noinline__ void warp_select_row_act(const Ld ld, const float* __restrict__ bias,
                                                 int E, int k, int32_t* __restrict__ out_idx,
                                                 float* __restrict__ out_w, int32_t* sel_out) {
  const int lane = threadIdx.x & 31;
  uint64_t pk[VPL];  // (key << 32) | (0xffffffff - expert); 0 = empty
  float av[VPL];     // sqrt-softplus / sigmoid: the scores, for the weights
  float amax = 0.0f, kabs = 0.0f;
  // softmax + bias: the row maximum, the FP32 denominator and the bound term
  float zmax = 0.0f, zsum = 1.0f, s1z = 0.0f;
  if (act == ACT_SOFTMAX_BIAS) {
    float zv[VPL], ev[VPL];
    uint32_t mo = 0u;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int e = lane + 32 * j;
      zv[j] = e < E ? ld(e) : 0.0f;
      if (e < E) mo = max(mo, ord_of(zv[j]));
    }
    zmax = float_of_ord(__reduce_max_sync(kFull, mo));
    float zs = 0.0f, s1 = 0.0f;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int e = lane + 32 * j;
      ev[j] = 0.0f;
      if (e < E) {
        const float d = __fsub_rn(zv[j], zmax);
        ev[j] = expf(d);
        zs = __fadd_rn(zs, ev[j]);
        s1 = __fmaf_rn(ev[j], -d, s1);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      zs = __fadd_rn(zs, __shfl_xor_sync(kFull, zs, off));
      s1 = __fadd_rn(s1, __shfl_xor_sync(kFull, s1, off));
    }
    zsum = zs;  // >= 1: the maximum's term is exp(0)
    s1z = __fdiv_ru(s1, zs);
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int e = lane + 32 * j;
      pk[j] = 0ull;
      if (e < E) {
        const float p = __fdiv_rn(ev[j], zsum);
        const float key = __fadd_rn(p, bias[e]);  // as softmax_bias_key32
        amax = fmaxf(amax, p);
        kabs = fmaxf(kabs, fabsf(key));
        pk[j] = ((uint64_t)ord_of(key) << 32) | (uint64_t)(0xffffffffu - (uint32_t)e);
      }
    }
  } else {
    // every load first, at an index clamped into the row (no branch per
    // value), then the scores: the chains of the VPL values interleave
    float zv[VPL], bv[VPL];
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int ec = min(lane + 32 * j, E - 1);
      zv[j] = ld(ec);
      bv[j] = (act != ACT_SOFTMAX && bias) ? bias[ec] : 0.0f;
    }
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int e = lane + 32 * j;
      const bool in = e < E;
      float key = zv[j];
      if (act != ACT_SOFTMAX) {
        const float a = act_f32(act, zv[j]);
        key = a + bv[j];  // a >= +0: adding +0 (no bias) leaves it unchanged
        av[j] = a;
        amax = in ? fmaxf(amax, a) : amax;
        kabs = in ? fmaxf(kabs, fabsf(key)) : kabs;
      }
      pk[j] = in ? (((uint64_t)ord_of(key) << 32) | (uint64_t)(0xffffffffu - (uint32_t)e)) : 0ull;
    }
  }
  SEL_STAMP(0);
  // k+1 rounds for the biased scores: the (k+1)-th key is kept for the gap
  // test; softmax has none and stops at k.
  const int kk = act == ACT_SOFTMAX ? k : min(k + 1, E);
  int sel_idx = -1;
  float sel_key = 0.0f;
  bool exact = true;
  if constexpr (VPL <= 8 && act == ACT_SOFTMAX) {
    // Softmax, E <= 256: rounds over one 32-bit word per entry, the key's
    // top 24 bits and 255 - index in the low 8 (a larger word: a larger
    // truncated key, or the same one and a lower index), so a round is one
    // warp maximum. (The biased scores measured slower this way.)
    // Truncation keeps order (t(a) > t(b) implies a > b), so when the kk
    // words picked and the best word left have strictly decreasing
    // truncated keys, the kk picked are the top kk of the exact keys in
    // exact order; otherwise the rounds below on (key, index) pairs decide.
    uint32_t c[VPL];
#pragma unroll
    for (int j = 0; j < VPL; ++j)
      c[j] = pk[j] ? (((uint32_t)(pk[j] >> 32) & 0xffffff00u) | (255u - (uint32_t)(lane + 32 * j)))
                   : 0u;
    sort_desc32<VPL>(c);
    SEL_STAMP(1);
    uint32_t mine = 0u;  // lane r <= kk: the word of round r
    for (int r = 0; r <= kk; ++r) {
      const uint32_t wbest = __reduce_max_sync(kFull, c[0]);
      mine = lane == r ? wbest : mine;
      const bool win = (int)(wbest & 31u) == (31 - lane);  // (255 - e) & 31 = 31 - e % 32
#pragma unroll
      for (int j = 0; j + 1 < VPL; ++j) c[j] = win ? c[j + 1] : c[j];
      c[VPL - 1] = win ? 0u : c[VPL - 1];
    }
    const uint32_t after = __shfl_down_sync(kFull, mine, 1);
    const bool tie = lane < kk && after != 0u && (mine >> 8) == (after >> 8);
    exact = __any_sync(kFull, tie);
#ifdef GBR_PHASE_STAMPS
    if (exact && lane == 0) atomicAdd(&g_sel_refines[2], 1ull);
#endif
    if (!exact) {
      // lane r < kk: its expert, and the exact key from the lane holding it
      const int e = 255 - (int)(mine & 0xffu);
      const int src = e & 31, js = lane < kk ? e >> 5 : -1;
      uint32_t ko = 0u;
#pragma unroll
      for (int j = 0; j < VPL; ++j) {
        const uint32_t v = __shfl_sync(kFull, (uint32_t)(pk[j] >> 32), src);
        ko = j == js ? v : ko;
      }
      if (lane < kk) {
        sel_idx = e;
        sel_key = float_of_ord(ko);
      }
    }
  }
  if (exact) {
    sort_desc<VPL>(pk);
    SEL_STAMP(1);
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
  }

  SEL_STAMP(2);
  if (act != ACT_SOFTMAX) {
    // FP32 key error bound; non-negative floats order like their bit patterns
    const float amax_w = __uint_as_float(__reduce_max_sync(kFull, __float_as_uint(amax)));
    const float kabs_w = __uint_as_float(__reduce_max_sync(kFull, __float_as_uint(kabs)));
    // two FP32 keys in the wrong exact order lie within 2 err of each
    // other, and every exact top-k member within 2 err of the k-th FP32 key;
    // the softmax + bias bound keeps a factor of 2 on top
    const float band = act == ACT_SOFTMAX_BIAS
                           ? 4.0f * softmax_bias_err_bound(VPL, amax_w, s1z, zsum, kabs_w)
                           : 2.0f * key_err_bound(amax_w, kabs_w, act_err_coef(act));
    const float next_key = __shfl_down_sync(kFull, sel_key, 1);
    // the difference rounded down: a gap of at most band is never missed
    const bool close = (lane < kk - 1) && __fsub_rd(sel_key, next_key) <= band;
    if (__any_sync(kFull, close)) {
#ifdef GBR_PHASE_STAMPS
      if (lane == 0) atomicAdd(&g_sel_refines[0], 1ull);
#endif
      if (act == ACT_SOFTMAX_BIAS) {
        // FP64 keys for every expert within the band of the k-th key
        const float thr = __fsub_rd(__shfl_sync(kFull, sel_key, k - 1), band);
        uint32_t cmask = 0u;
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
          const int e = lane + 32 * j;
          if (e < E && softmax_bias_key32(ld(e), zmax, zsum, bias[e]) >= thr)
            cmask |= 1u << j;
        }
        const int pick = select_softmax_bias_fp64<VPL>(ld, bias, E, k, zmax, cmask);
        if (lane < k) sel_idx = pick;
      } else {
        sel_idx = refine_near_ties<VPL>(ld, bias, act, E, k, kk, sel_key, sel_idx, band);
      }
    }
  }

  // weights over the chosen k, summed in slot order
  float s = 0.0f;
  if (act == ACT_SOFTMAX) {
    // the key is the logit (-0.0 read back as +0.0, which exp treats alike)
    const float z0 = __shfl_sync(kFull, sel_key, 0);
    if (lane < k) s = expf(sel_key - z0);
  } else if (act == ACT_SOFTMAX_BIAS) {
    // the unbiased probabilities renormalised: exp(z_j - zc) / sum, zc the
    // largest chosen logit (the bias may rank a smaller logit first)
    const float zj = lane < k ? ld(sel_idx) : -INFINITY;
    const float zc = float_of_ord(__reduce_max_sync(kFull, lane < k ? ord_of(zj) : 0u));
    if (lane < k) s = expf(zj - zc);
  } else {
    // the chosen scores come from the lanes that hold them (no reload)
    const int src = sel_idx & 31, js = sel_idx >> 5;  // lanes >= k: js = -1, no match
    float sv = 0.0f;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const float v = __shfl_sync(kFull, av[j], src);
      sv = j == js ? v : sv;
    }
    if (lane < k) s = sv;
    const float smax = __uint_as_float(__reduce_max_sync(kFull, __float_as_uint(s)));
    if (!(smax >= 0x1p-50f)) {
      // every chosen activation is tiny (FP32 keeps few or no bits of it):
      // the ratios come from the log domain
      const float la = lane < k ? log_act(act, ld(sel_idx)) : -INFINITY;
      float lm = la;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) lm = fmaxf(lm, __shfl_xor_sync(kFull, lm, off));
      s = (lane < k && lm > -INFINITY) ? expf(la - lm) : 0.0f;
    }
  }
  // summed over the slots by a fixed tree (slot j + slot j^8, then ^4, ^2,
  // ^1; slots >= k add 0): every lane gets the same sum, in the order
  // slot_tree_sum follows
  float sum = lane < k ? s : 0.0f;
  sum += __shfl_xor_sync(kFull, sum, 8);
  sum += __shfl_xor_sync(kFull, sum, 4);
  sum += __shfl_xor_sync(kFull, sum, 2);
  sum += __shfl_xor_sync(kFull, sum, 1);
  SEL_STAMP(3);
  if (lane < k) {
    out_idx[lane] = sel_idx;
    out_w[lane] = (sum > 0.0f) ? s / sum : 1.0f / (float)k;
    if (sel_out) sel_out[lane] = sel_idx;
  }
  SEL_STAMP(4);
}

template <int VPL, class Ld>
__device__ __forceinline__ void warp_select_row(const Ld ld, const float* __restrict__ bias, int E,
                                                int k, int act, int32_t* __restrict__ out_idx,
                                                float* __restrict__ out_w, int32_t* sel_out) {
  if (act == ACT_SOFTMAX)
    warp_select_row_act<VPL, ACT_SOFTMAX>(ld, bias, E, k, out_idx, out_w, sel_out);
  else if (act == ACT_SOFTMAX_BIAS)
    warp_select_row_act<VPL, ACT_SOFTMAX_BIAS>(ld, bias, E, k, out_idx, out_w, sel_out);
  else if (act == ACT_SIGMOID)
    warp_select_row_act<VPL, ACT_SIGMOID>(ld, bias, E, k, out_idx, out_w, sel_out);
  else
    warp_select_row_act<VPL, ACT_SQRT_SOFTPLUS>(ld, bias, E, k, out_idx, out_w, sel_out);
}

// The unique-route table of groups of n = T*k <= 32 (token, slot) entries
// laid over a warp's lanes in row-major order: the lanes gbase .. gbase+n-1
// (gmask) hold one group, lane gbase + p its entry p with id v (b70 lab
// note, "Unique-route router screen": stable dedup, prefix ranking, token
// masks, slot mapping, done with warp match and ballot). The lowest lane
// holding an id is its first occurrence; its unique position is the number
// of first occurrences below it. Returns, for this lane: map (the entry's
// unique position), the unique id and token mask of unique position
// p = lane - gbase (-1 and 0 past the count), and the count. All lanes call.
struct TableLane {
  int32_t uniq;
  uint32_t mask;
  uint32_t map;
  int count;
};

__device__ __forceinline__ TableLane table_lanes(int32_t v, bool valid, uint32_t gmask, int gbase,
                                                 int T, int k) {
  const int lane = threadIdx.x & 31;
  const uint32_t eq = __match_any_sync(kFull, v) & gmask;  // lanes of this group holding v
  const int first = eq ? __ffs(eq) - 1 : lane;  // eq == 0: a lane outside every group
  const uint32_t fb = __ballot_sync(kFull, valid && first == lane) & gmask;
  TableLane r;
  r.map = (uint32_t)__popc(fb & ((1u << first) - 1u));
  r.count = __popc(fb);
  // bit t when token t (lanes gbase + t k .. gbase + t k + k - 1) holds v
  const uint32_t slots = (k == 32 ? kFull : (1u << k) - 1u);
  uint32_t tm = 0u;
  for (int t = 0; t < T; ++t) tm |= ((eq >> (gbase + t * k)) & slots) ? (1u << t) : 0u;
  // lane gbase + u takes the id and mask of the u-th first occurrence
  const int u = lane - gbase;
  const bool has = valid && u < r.count;
  uint32_t src = (uint32_t)lane;
  if (has) asm("fns.b32 %0, %1, 0, %2;" : "=r"(src) : "r"(fb), "r"(u + 1));
  const int32_t uv = __shfl_sync(kFull, v, (int)src);
  const uint32_t um = __shfl_sync(kFull, tm, (int)src);
  r.uniq = has ? uv : -1;
  r.mask = has ? um : 0u;
  return r;
}

// One group of T x k <= 32 entries from ids in shared memory s_idx[T*k]
// (one warp; lanes >= T*k idle).
__device__ __forceinline__ void warp_route_table_small(const int32_t* s_idx, int T, int k,
                                                       int32_t* __restrict__ unique,
                                                       uint8_t* __restrict__ mask,
                                                       uint8_t* __restrict__ map,
                                                       int32_t* __restrict__ count) {
  const int lane = threadIdx.x & 31;
  const int n = T * k;
  const bool valid = lane < n;
  const int32_t v = valid ? s_idx[lane] : 0;
  const TableLane r = table_lanes(v, valid, n == 32 ? kFull : (1u << n) - 1u, 0, T, k);
  if (valid) {
    unique[lane] = r.uniq;
    mask[lane] = (uint8_t)r.mask;
    map[lane] = (uint8_t)r.map;
    if (lane == 0) *count = r.count;
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

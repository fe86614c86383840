// Near-tie keys in double-float ("float-float") arithmetic.
//
// The selection re-ranks experts whose FP32 keys sqrt(softplus(z)) + b lie
// within the FP32 error band of the k-th (the FP64 guard band). FP64
// transcendentals run at a small fraction of the FP32 rate on this part
// (one FP64 sqrt(softplus) costs a warp some 24,000 cycles), so the key is
// evaluated as an unevaluated sum hi + lo of two floats with a relative
// error near 2^-42, from FP32 operations only. A pair of keys closer than
// the bound kDfRel allows (and not computed from identical inputs) still
// goes to FP64 (key64 in the callers): the double-float keys only decide
// the orders that FP64 would decide the same way.
//
// Methods: error-free sum and product (Knuth's TwoSum, Dekker's Fast2Sum,
// the FMA product residual) and Dekker's double-length multiplication;
// exp by Cody and Waite's argument reduction with ln 2 split in three
// parts, the Taylor series of expm1 on x / 4 (double-float terms through
// y^5/120, the rest in FP32) and two doublings expm1(2y) = expm1(y)
// (expm1(y) + 2); log1p(u) as 2 atanh(u / (2 + u)) by its power series
// (double-float terms through w^5/11 in w = s^2 <= 1/9, the rest in FP32);
// sqrt by one Newton (Heron) step. The constants are ln 2, 1/k! and
// 1/(2k+1) rounded to float, or split into two floats where a term needs
// more: C1 is ln 2 to 15 significant bits (n * C1 is exact for n < 2^8), C2
// and C3 the next float-rounded parts (C1 + C2 + C3 - ln 2 = -1.3e-21).
#pragma once

#include <cstdint>

#include "common.cuh"

namespace gbr {

struct df32 {
  float hi, lo;
};

__device__ __forceinline__ df32 two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, e};
}

// |a| >= |b| (or a == 0)
__device__ __forceinline__ df32 fast_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

__device__ __forceinline__ df32 two_prod(float a, float b) {
  const float p = __fmul_rn(a, b);
  return {p, __fmaf_rn(a, b, -p)};
}

__device__ __forceinline__ df32 df_add(df32 x, df32 y) {
  df32 s = two_sum(x.hi, y.hi);
  const df32 t = two_sum(x.lo, y.lo);
  s.lo = __fadd_rn(s.lo, t.hi);
  s = fast_two_sum(s.hi, s.lo);
  s.lo = __fadd_rn(s.lo, t.lo);
  return fast_two_sum(s.hi, s.lo);
}

__device__ __forceinline__ df32 df_add_f(df32 x, float b) {
  df32 s = two_sum(x.hi, b);
  s.lo = __fadd_rn(s.lo, x.lo);
  return fast_two_sum(s.hi, s.lo);
}

// x + y for |x.hi| >= |y.hi| (Fast2Sum on the leading parts): the Horner
// steps below, whose coefficient dominates the running product.
__device__ __forceinline__ df32 df_add_big(df32 x, df32 y) {
  df32 s = fast_two_sum(x.hi, y.hi);
  s.lo = __fadd_rn(s.lo, __fadd_rn(x.lo, y.lo));
  return fast_two_sum(s.hi, s.lo);
}

__device__ __forceinline__ df32 df_mul(df32 x, df32 y) {
  df32 p = two_prod(x.hi, y.hi);
  p.lo = __fmaf_rn(x.hi, y.lo, p.lo);
  p.lo = __fmaf_rn(x.lo, y.hi, p.lo);
  return fast_two_sum(p.hi, p.lo);
}

__device__ __forceinline__ df32 df_scale(df32 x, float pow2) {  // exact for powers of two
  return {__fmul_rn(x.hi, pow2), __fmul_rn(x.lo, pow2)};
}

// expm1(x) for |x| <= 0.75, relative error below 2^-44: y = x / 4 (|y| <=
// 0.1875), the Taylor series y (1 + y/2 + y^2/6 + y^3/24 + y^4/120 + y^5 t)
// by Horner's rule in double-float, with t = 1/720 + ... + y^4/3628800 in
// FP32 (its terms are below 2^-21 of the result, and the first one dropped
// below 2^-47), then two doublings. This path only runs for near ties, so
// its code is cold whenever it runs: the function stays out of line, which
// keeps the instruction fetches few.
static __device__ __noinline__ df32 expm1_df(df32 x) {
  const df32 y = df_scale(x, 0x1p-2f);
  float t = __fmaf_rn(y.hi, 0x1.27e4fcp-22f, 0x1.71de3ap-19f);  // 1/10!, 1/9!
  t = __fmaf_rn(t, y.hi, 0x1.a01a02p-16f);                      // 1/8!
  t = __fmaf_rn(t, y.hi, 0x1.a01a02p-13f);                      // 1/7!
  t = __fmaf_rn(t, y.hi, 0x1.6c16c2p-10f);                      // 1/6!
  df32 p = fast_two_sum(0x1.111112p-7f, __fmaf_rn(y.hi, t, -0x1.dddddep-32f));  // 1/120 + y t
  p = df_add_big(df32{0x1.555556p-5f, -0x1.555556p-30f}, df_mul(y, p));       // 1/24 + y p
  p = df_add_big(df32{0x1.555556p-3f, -0x1.555556p-28f}, df_mul(y, p));       // 1/6 + y p
  p = df_add_big(df32{0.5f, 0.0f}, df_mul(y, p));                              // 1/2 + y p
  p = df_add_big(df32{1.0f, 0.0f}, df_mul(y, p));                              // 1 + y p
  df32 e = df_mul(y, p);
  e = df_mul(e, df_add_f(e, 2.0f));  // expm1(2v) from expm1(v)
  return df_mul(e, df_add_f(e, 2.0f));
}

// Largest |z| the double-float path takes; beyond it the callers use FP64.
constexpr float kDfMaxAbsZ = 30.0f;
// Bound used to call two double-float keys distinct: |key_a - key_b| must
// exceed kDfRel * (s_a + |key_a| + s_b + |key_b|). The evaluation error is
// near 2^-42 relative; the margin is 64x.
constexpr float kDfRel = 0x1p-36f;

// sqrt(softplus(z)) with softplus(z) = max(z, 0) + log1p(exp(-|z|)), for
// |z| <= kDfMaxAbsZ.
__device__ __forceinline__ df32 sqrt_softplus_df(float z) {
  const float a = fabsf(z);
  const float n = rintf(__fmul_rn(a, 0x1.715476p+0f));  // 0 .. 44
  // r = a - n ln 2 (Cody and Waite): a - n*C1 is exact, n*C2 is exact as a
  // product pair, n*C3 is below 2^-38
  const float r0 = __fmaf_rn(-n, 0x1.62e4p-1f, a);
  const df32 nc2 = two_prod(n, 0x1.7f7d1cp-20f);
  df32 r = df_add(df32{r0, 0.0f}, df32{-nc2.hi, -nc2.lo});
  r = df_add_f(r, -__fmul_rn(n, 0x1.ef357ap-45f));
  // u = exp(-a) = 2^-n (1 + expm1(-r))
  const df32 em = expm1_df(df32{-r.hi, -r.lo});
  df32 u = df_add_f(em, 1.0f);
  u = df_scale(u, __int_as_float((127 - (int)n) << 23));  // 2^-n, n in 0..44
  // log1p(u) = 2 atanh(s), s = u / (2 + u) in (0, 1/3]: s to FP32, then
  // the remainder u - s (2 + u), whose leading part cancels exactly
  const df32 dd = df_add_f(u, 2.0f);
  const float q0 = __fdividef(u.hi, dd.hi);
  const df32 qd = two_prod(q0, dd.hi);
  const float rem = __fadd_rn(__fsub_rn(__fsub_rn(u.hi, qd.hi), qd.lo),
                              __fsub_rn(u.lo, __fmul_rn(q0, dd.lo)));
  const df32 sv = fast_two_sum(q0, __fdividef(rem, dd.hi));
  df32 w = two_prod(sv.hi, sv.hi);  // w = s^2 <= 1/9
  w = fast_two_sum(w.hi, __fmaf_rn(2.0f * sv.hi, sv.lo, w.lo));
  // 1 + w/3 + w^2/5 + ...: terms from w^6/13 on in FP32 (below 2^-22 of the
  // sum; the first one dropped, w^14/29, below 2^-48)
  float t = __fmaf_rn(w.hi, 0x1.2f684cp-5f, 0x1.47ae14p-5f);  // 1/27, 1/25
  t = __fmaf_rn(t, w.hi, 0x1.642c86p-5f);                     // 1/23
  t = __fmaf_rn(t, w.hi, 0x1.861862p-5f);                     // 1/21
  t = __fmaf_rn(t, w.hi, 0x1.af286cp-5f);                     // 1/19
  t = __fmaf_rn(t, w.hi, 0x1.e1e1e2p-5f);                     // 1/17
  t = __fmaf_rn(t, w.hi, 0x1.111112p-4f);                     // 1/15
  t = __fmaf_rn(t, w.hi, 0x1.3b13b2p-4f);                     // 1/13
  df32 P = fast_two_sum(0x1.745d18p-4f, __fmaf_rn(w.hi, t, -0x1.745d18p-29f));  // 1/11 + w t
  P = df_add_big(df32{0x1.c71c72p-4f, -0x1.c71c72p-31f}, df_mul(w, P));  // 1/9 + w P
  P = df_add_big(df32{0x1.24924ap-3f, -0x1.b6db6ep-28f}, df_mul(w, P));  // 1/7 + w P
  P = df_add_big(df32{0x1.99999ap-3f, -0x1.99999ap-29f}, df_mul(w, P));  // 1/5 + w P
  P = df_add_big(df32{0x1.555556p-2f, -0x1.555556p-27f}, df_mul(w, P));  // 1/3 + w P
  P = df_add_big(df32{1.0f, 0.0f}, df_mul(w, P));                        // 1 + w P
  df32 sp = df_scale(df_mul(sv, P), 2.0f);
  if (z > 0.0f) sp = df_add_f(sp, z);
  // sqrt: s0 = RN(sqrt(sp.hi)); s = s0 + (sp - s0^2) / (2 s0), s0^2 exact as a product pair
  const float s0 = __fsqrt_rn(sp.hi);
  const df32 sq = two_prod(s0, s0);
  const float res = __fadd_rn(__fsub_rn(__fsub_rn(sp.hi, sq.hi), sq.lo), sp.lo);
  return fast_two_sum(s0, __fdiv_rn(res, __fmul_rn(2.0f, s0)));
}

// sigmoid(z) = 1 / (1 + exp(-z)) for |z| <= kDfMaxAbsZ: u = exp(-|z|) as
// above, 1 / (1 + u) by one Newton step on the FP32 reciprocal, times u
// when z < 0 (sigmoid(z) = u / (1 + u) there).
__device__ __forceinline__ df32 sigmoid_df(float z) {
  const float a = fabsf(z);
  const float n = rintf(__fmul_rn(a, 0x1.715476p+0f));
  const float r0 = __fmaf_rn(-n, 0x1.62e4p-1f, a);
  const df32 nc2 = two_prod(n, 0x1.7f7d1cp-20f);
  df32 r = df_add(df32{r0, 0.0f}, df32{-nc2.hi, -nc2.lo});
  r = df_add_f(r, -__fmul_rn(n, 0x1.ef357ap-45f));
  df32 u = df_add_f(expm1_df(df32{-r.hi, -r.lo}), 1.0f);
  u = df_scale(u, __int_as_float((127 - (int)n) << 23));
  const df32 s = df_add_f(u, 1.0f);  // 1 + u in [1, 2]
  const float q0 = __fdiv_rn(1.0f, s.hi);
  const df32 sq = two_prod(s.hi, q0);
  const float res = __fsub_rn(__fsub_rn(__fsub_rn(1.0f, sq.hi), sq.lo), __fmul_rn(s.lo, q0));
  const df32 inv = fast_two_sum(q0, __fmul_rn(q0, res));
  return z >= 0.0f ? inv : df_mul(u, inv);
}

// Upper bound on |key32 - key| for FP32 keys whose largest activation is
// amax and largest |key| is kabs: 2^-23 (c amax + 0.5 kabs) + 2^-59 with c
// the activation's coefficient (act_err_coef; the absolute term covers the
// score's 2^-60 and the rounding of tiny keys), every step rounded up.
__device__ __forceinline__ float key_err_bound(float amax, float kabs, float coef) {
  return __fadd_ru(__fmul_ru(__fmaf_ru(coef, amax, __fmul_ru(0.5f, kabs)), 0x1p-23f), 0x1p-59f);
}

// A near-tie key: a(z) + b as a double-float (a = sqrt-softplus or sigmoid),
// with the scale a + |key| its distinctness test uses. Beyond the
// double-float range of z the activation comes from FP64.
struct NearKey {
  float hi, lo, scale;
};

// FP64 activation split into two floats; out of line, so that no FP64
// instruction is issued (not even predicated off) unless |z| is large.
static __device__ __noinline__ df32 act_split64(int act, float z) {
  const double v = act_f64(act, (double)z);
  df32 s;
  s.hi = (float)v;
  s.lo = isfinite(s.hi) ? (float)(v - (double)s.hi) : 0.0f;
  return s;
}

__device__ __forceinline__ NearKey near_key(int act, float z, float b) {
  const df32 s = fabsf(z) <= kDfMaxAbsZ
                     ? (act == ACT_SIGMOID ? sigmoid_df(z) : sqrt_softplus_df(z))
                     : act_split64(act, z);
  const df32 key = df_add_f(s, b);
  return {key.hi, isfinite(key.hi) ? key.lo : 0.0f, __fadd_ru(fabsf(s.hi), fabsf(key.hi))};
}

// near_key out of line: its callers run on cold paths, where one shared
// copy of the code costs fewer instruction fetches.
static __device__ __noinline__ NearKey near_key_ool(int act, float z, float b) {
  return near_key(act, z, b);
}

// True when two near-tie keys are far enough apart that their double-float
// order is the order FP64 gives.
__device__ __forceinline__ bool near_distinct(float ah, float al, float asc, float bh, float bl,
                                              float bsc) {
  const float d = fabsf(__fadd_rn(__fsub_rn(ah, bh), __fsub_rn(al, bl)));
  return d > kDfRel * __fadd_ru(asc, bsc);
}

// (hi, lo) ordering of normalised double-float keys.
__device__ __forceinline__ bool df_gt(float ah, float al, float bh, float bl) {
  return ah > bh || (ah == bh && al > bl);
}

// Row-local top list of double-float keys, sorted by (key desc, index asc),
// with FP32 comparisons only.
template <int KC>
struct TopListDF {
  float h[KC], l[KC];
  int i[KC];
  float z[KC];
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int j = 0; j < KC; ++j) {
      h[j] = -INFINITY;
      l[j] = 0.0f;
      i[j] = 0x7fffffff;
      z[j] = 0.0f;
    }
  }
  __device__ __forceinline__ static bool ahead(float kh, float kl, int idx, float vh, float vl,
                                               int vi) {
    return df_gt(kh, kl, vh, vl) || (kh == vh && kl == vl && idx < vi);
  }
  __device__ __forceinline__ void push(float kh, float kl, int idx, float zz) {
#pragma unroll
    for (int j = KC - 1; j > 0; --j) {
      if (ahead(kh, kl, idx, h[j], l[j], i[j])) {
        const bool up = ahead(kh, kl, idx, h[j - 1], l[j - 1], i[j - 1]);
        h[j] = up ? h[j - 1] : kh;
        l[j] = up ? l[j - 1] : kl;
        i[j] = up ? i[j - 1] : idx;
        z[j] = up ? z[j - 1] : zz;
      }
    }
    if (ahead(kh, kl, idx, h[0], l[0], i[0])) {
      h[0] = kh;
      l[0] = kl;
      i[0] = idx;
      z[0] = zz;
    }
  }
};

}  // namespace gbr

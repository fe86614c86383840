// Large-M (prefill) fused router on the 5th-generation tensor cores: the
// kernel and its launch templates. tc.cu holds the host side; the
// tc_*.cu files instantiate the kernel families, one per translation unit.
//
// A CTA owns 128 token rows and all E <= 256 experts, so a row's logits
// never leave the SM: TMA streams x [128 x 64] and W_gate [E x 64] BF16
// tiles (128-byte swizzle) into a shared-memory ring; one thread issues
// tcgen05.mma (kind::f16, K=16) into an FP32 accumulator in tensor memory;
// after the last k-step eight epilogue warps read the rows back with
// tcgen05.ld (thread = row, two warps per TMEM lane quadrant, each half of
// the columns) and run the activation, top-k and renormalisation. This is
// the warp-specialised layout the dense_router_decode commit page sketches
// ("Warp 5 (TMA) ... Warp 4 (MMA) ... Warps 0-3 (EPI)", "the heap
// accumulates across subtiles, then merge+renorm+store once per row"),
// written directly in PTX for sm_103a.
//
// By default two CTAs form a pair for 256 rows (M = 256 MMAs issued by the
// even CTA, each CTA staging half of every W tile). When there are fewer
// tiles than resident pairs the launch is stream-K: the tiles x k-steps
// units are split evenly over one pair per two SMs, a pair publishes the
// partial accumulator of the tile it starts in the workspace and finishes
// the tile it ends in after adding the partials of the pairs before it.
//
// NVFP4 weights (the same page's "NVFP4 blockscaled GEMM"): x stays BF16,
// and tcgen05 has no BF16 x FP4 kind, so the CTAs decode W once per launch,
// exactly, into a BF16 copy in the workspace that the producers load like
// BF16 weights: e2m1 * e4m3 has at most 6 significant bits and fits BF16's
// exponent range, so the copy equals W / g bit for bit; the FP32 global
// scale g multiplies the accumulator in the epilogue.
//
// Every wait (mbarriers, flags in global memory) gives up after about a
// second of %globaltimer, records GBR_ETIMEOUT in a device status word and
// lets the CTA unwind (free tensor memory, return) instead of hanging.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/gbrouter.h"
#include "kernels.h"
#include "dfkey.cuh"
#include "select.cuh"

namespace gbr {

// Host helpers the launch templates use (tc.cu): the stream-K group count
// for U = tiles x nk units over at most G groups, and the groups of this
// kernel that are resident at once.
int tc_sk_groups_for(int tiles, int nk, int G);
int tc_sk_resident_groups(const void* kern, size_t smem, int cl);

namespace {


constexpr int BM = 128;   // token rows per CTA (= MMA M, = TMEM lanes)
constexpr int BK = 64;    // BF16 elements per k-step (one 128-byte swizzle atom)
constexpr int kEpiWarps = 8;  // two per TMEM lane quadrant, each half of the columns
constexpr uint64_t kWaitNs = 1000000000ull;

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

#ifdef GBR_PHASE_STAMPS
#define TC_STAMP(i)                                                                      \
  do {                                                                                   \
    if (threadIdx.x == 0 && p.stamps) p.stamps[blockIdx.x * kTcStamps + (i)] = globaltimer(); \
  } while (0)
#else
#define TC_STAMP(i) \
  do {              \
  } while (0)
#endif

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for a whole warp: lane 0 polls with a growing sleep so the
// waiting warp leaves the issue slots to the TMA and MMA threads, then the
// warp synchronises. All lanes get the result.
__device__ __forceinline__ bool mbar_wait_warp(unsigned* st, uint32_t bar, uint32_t parity) {
  uint32_t ok = 1;
  if ((threadIdx.x & 31) == 0 && !mbar_try(bar, parity)) {
    const uint64_t t0 = globaltimer();
    uint32_t ns = 32;
    while (!mbar_try(bar, parity)) {
      __nanosleep(ns);
      if (ns < 512) ns <<= 1;
      if (globaltimer() - t0 > kWaitNs) {
        if (st) atomicOr(st, 1u);
        ok = 0;
        break;
      }
    }
  }
  ok = __shfl_sync(kFull, ok, 0);
  __syncwarp();  // orders lane 0's observation of the phase before the other lanes' accesses
  return ok != 0;
}

// Bounded wait; false (and the status word set) when it gave up.
__device__ __forceinline__ bool mbar_wait(unsigned* st, uint32_t bar, uint32_t parity) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (!mbar_try(bar, parity)) {
    if (globaltimer() - t0 > kWaitNs) {
      if (st) atomicOr(st, 1u);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
      : "memory");
}

// The CTA-pair form: the completion goes to the mbarrier at `bar`, a
// shared::cluster address that may lie in the other CTA of the pair (both
// CTAs load their own operand halves and signal the even CTA's barrier).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int c0,
                                                 int c1, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".cta_group::2.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
      : "memory");
}

// L2 eviction policies: x streams through once (first to go), W_gate is
// read by every CTA (last to go). Keeping the stream from flushing the
// rest of L2 also keeps the kernel's own code there: the epilogue's rarely
// run paths are otherwise fetched from DRAM.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded wait for a flag in global memory to take the value want.
__device__ __forceinline__ bool wait_flag(unsigned* st, const unsigned* f, unsigned want) {
  if (ld_acquire_u32(f) == want) return true;
  const uint64_t t0 = globaltimer();
  uint32_t ns = 32;
  while (ld_acquire_u32(f) != want) {
    __nanosleep(ns);
    if (ns < 256) ns <<= 1;
    if (globaltimer() - t0 > kWaitNs) {
      if (st) atomicOr(st, 1u);
      return false;
    }
  }
  return true;
}

// Bounded wait until flags f[0..n) (n <= 8) all hold `want`: the relaxed
// loads of a round go out together, and one acq_rel fence after the round
// that sees them all set orders what follows after the flags' release
// stores (an acquire pattern), so a batch costs one round trip.
__device__ __forceinline__ bool wait_flags8(unsigned* st, const unsigned* f, int n, unsigned want) {
  const uint64_t t0 = globaltimer();
  uint32_t ns = 32;
  for (;;) {
    unsigned v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[j] = want;
      if (j < n) asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v[j]) : "l"(f + j) : "memory");
    }
    bool all = true;
#pragma unroll
    for (int j = 0; j < 8; ++j) all = all && v[j] == want;
    if (all) break;
    __nanosleep(ns);
    if (ns < 256) ns <<= 1;
    if (globaltimer() - t0 > kWaitNs) {
      if (st) atomicOr(st, 1u);
      return false;
    }
  }
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
  return true;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// AND of a predicate over the kEpiWarps epilogue warps (named barrier 2,
// used for nothing else).
__device__ __forceinline__ bool epi_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 2, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(v ? 1u : 0u), "r"(kEpiWarps * 32)
      : "memory");
  return r != 0u;
}

__device__ __forceinline__ void cluster_sync_tc() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle,
// 8-row core-matrix groups 1024 bytes apart, descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;               // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;     // stride byte offset
  d |= (uint64_t)1 << 46;               // version
  d |= (uint64_t)2 << 61;               // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: FP32 accumulator, BF16 A and B, both
// K-major, N = E, M = 128.
__host__ __device__ constexpr uint32_t idesc_bf16(int N, int M = BM) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// A CTA pair's MMA (M = 256: each CTA's 128 rows of A, each CTA's half of
// the N rows of B, D in each CTA's tensor memory), issued by the even CTA.
__device__ __forceinline__ void mma_bf16_pair(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on the mbarrier at this offset in both CTAs of the pair once the
// pair MMAs issued so far have completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"((uint16_t)3)
      : "memory");
}

__device__ __forceinline__ uint32_t mapa_u32(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive FP32 accumulator columns of this thread's TMEM lane,
// without waiting (tmem_wait_ld makes the registers valid).
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 consecutive FP32 accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from global to this CTA's shared memory, completing on the mbarrier.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void st_cg_v4(float* p, float a, float b, float c, float d) {
  asm volatile("st.global.cg.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}

// Writes 32 consecutive FP32 columns of this thread's TMEM lane (the
// caller waits with tcgen05.wait::st before the columns are read again).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

// Sorts N (a power of two) floats descending in registers: a bitonic
// network, fully unrolled (every index static).
template <int N>
__device__ __forceinline__ void sort_desc_bitonic(float (&v)[N]) {
#pragma unroll
  for (int size = 2; size <= N; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
      for (int i = 0; i < N; ++i) {
        const int j = i ^ stride;
        if (j > i) {
          const bool desc = (i & size) == 0;  // the direction of i's block
          const float a = v[i], b = v[j];
          v[i] = desc ? fmaxf(a, b) : fminf(a, b);
          v[j] = desc ? fminf(a, b) : fmaxf(a, b);
        }
      }
    }
  }
}

// Row-local top list of capacity KC (>= k+1), kept sorted by (key desc,
// index asc). Columns arrive in increasing expert order, so a strict
// comparison keeps the lower index ahead on equal keys.
template <int KC>
struct TopList {
  uint32_t o[KC];  // order-preserving key
  int i[KC];
  float z[KC];     // the score the weights use (logit for softmax, activation otherwise)
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int j = 0; j < KC; ++j) {
      o[j] = 0u;
      i[j] = 0x7fffffff;
      z[j] = 0.0f;
    }
  }
  // Branch-free insertion (selects only): the lanes of a warp insert at
  // different positions, and per-slot branches would diverge.
  __device__ __forceinline__ void push(uint32_t ok, int idx, float zz) {
    if (ok <= o[KC - 1]) return;
#pragma unroll
    for (int j = KC - 1; j > 0; --j) {
      const bool c = ok > o[j];
      const bool u = ok > o[j - 1];
      const uint32_t no = u ? o[j - 1] : ok;
      const int ni = u ? i[j - 1] : idx;
      const float nz = u ? z[j - 1] : zz;
      o[j] = c ? no : o[j];
      i[j] = c ? ni : i[j];
      z[j] = c ? nz : z[j];
    }
    const bool c0 = ok > o[0];
    o[0] = c0 ? ok : o[0];
    i[0] = c0 ? idx : i[0];
    z[0] = c0 ? zz : z[0];
  }
};

template <int KC>
struct TopList64 {
  double v[KC];
  int i[KC];
  float z[KC];
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int j = 0; j < KC; ++j) {
      v[j] = -INFINITY;
      i[j] = 0x7fffffff;
      z[j] = 0.0f;
    }
  }
  // (kv, idx) ahead of (v[j], i[j]): larger key, or equal key and lower index
  __device__ __forceinline__ static bool ahead(double kv, int idx, double vj, int ij) {
    return kv > vj || (kv == vj && idx < ij);
  }
  __device__ __forceinline__ void push(double kv, int idx, float zz) {
    if (!ahead(kv, idx, v[KC - 1], i[KC - 1])) return;
#pragma unroll
    for (int j = KC - 1; j > 0; --j) {
      if (ahead(kv, idx, v[j], i[j])) {
        const bool up = ahead(kv, idx, v[j - 1], i[j - 1]);
        v[j] = up ? v[j - 1] : kv;
        i[j] = up ? i[j - 1] : idx;
        z[j] = up ? z[j - 1] : zz;
      }
    }
    if (ahead(kv, idx, v[0], i[0])) {
      v[0] = kv;
      i[0] = idx;
      z[0] = zz;
    }
  }
};

// FP64 key of one expert; out of line so that the FP64 work runs only for
// the entries that need it.
__device__ __noinline__ double key64(int act, float z, float b) {
  return act_f64(act, (double)z) + (double)b;
}

// FP64 re-ranking of one row (see select.cuh): every lane of the warp calls
// it (the TMEM loads are warp-collective); lanes with close == false only
// take part in the loads. Kept out of line so the common path's top list
// stays in registers.
template <int KC, bool FP4>
__device__ __noinline__ void refine_row(uint32_t trow, int E, float g, const float* bias, int act,
                                        float thr, bool close, int* out_i, float* out_z) {
  // out_i / out_z: KC entries, BM apart (shared memory)
  TopList64<KC> t64;
  t64.init();
  for (int c0 = 0; c0 < E; c0 += 32) {
    float v[32];
    tmem_ld32(trow + c0, v);
    if (close) {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int e = c0 + j;
        if (e < E) {
          const float z = FP4 ? v[j] * g : v[j];
          const float av = act_f32(act, z);
          const float key = bias ? av + __ldg(bias + e) : av;
          if (key >= thr)
            t64.push(act_f64(act, (double)z) + (bias ? (double)__ldg(bias + e) : 0.0), e, av);
        }
      }
    }
  }
  if (close) {
#pragma unroll
    for (int j = 0; j < KC; ++j) {
      out_i[j * BM] = t64.i[j];
      out_z[j * BM] = t64.z[j];
    }
  }
}

// The FP64 stage of refine_in_list (all lanes call): FP64 keys for every
// pooled entry; rows with amb set re-rank their list (still as stored) with
// them. Out of line: FP64 is slow on this part and must not be issued on
// the common path.
template <int KC>
__device__ __noinline__ void refine_fp64(int act, const uint32_t* l_o, int32_t* l_i, float* l_z,
                                         uint32_t need, bool amb, int qoff, int qtotal,
                                         const float* zq, const float* sb, const uint32_t* wl) {
  const int lane = threadIdx.x & 31;
  double kd[KC];
#pragma unroll
  for (int j = 0; j < KC; ++j) kd[j] = (double)float_of_ord(l_o[j * BM]);
  for (int base = 0; base < qtotal; base += 32) {
    double key = 0.0;
    if (base + lane < qtotal) {
      const uint32_t item = wl[base + lane];
      const int e = (int)(item >> 16);
      key = key64(act, zq[e * BM + (int)((item >> 5) & 31u)], sb ? sb[e] : 0.0f);
    }
#pragma unroll
    for (int j = 0; j < KC; ++j) {
      const int qj = qoff + __popc(need & ((1u << j) - 1u));
      const bool mine = ((need >> j) & 1u) && qj >= base && qj < base + 32;
      const double kv = __shfl_sync(kFull, key, mine ? qj - base : lane);
      if (mine) kd[j] = kv;
    }
  }
  if (amb) {
    TopList64<KC> t64;
    t64.init();
#pragma unroll
    for (int j = 0; j < KC; ++j)
      if (l_o[j * BM] != 0u) t64.push(kd[j], l_i[j * BM], l_z[j * BM]);
#pragma unroll
    for (int j = 0; j < KC; ++j) {
      l_i[j * BM] = t64.i[j];
      l_z[j * BM] = t64.z[j];
    }
  }
}

// Near ties inside the merged list of one row (all 32 lanes call; lanes
// with close == false take part in the pooled evaluations only). The list
// (KC entries, BM apart in shared memory: order keys, experts, scores) is
// re-ranked in place. When every key at or above the band below the k-th
// is in the list, only entries next to a gap of at most `band` need a
// better key; the others keep their FP32 key, which orders them correctly
// against everything more than `band` away. Those keys are double-float
// (dfkey.cuh); a pair still too close to call, from different inputs,
// takes FP64 keys. The warp pools the entries its rows need and evaluates
// them one per lane (zq: the warp's logit copy, [E][BM] from its first
// row; sb: the bias in shared memory or null). Returns true when the near
// ties reach past the list (the caller then re-ranks every column).
// This runs for about one row in four thousand, so its code is cold in the
// instruction cache whenever it runs and every distinct instruction costs a
// fetch: the loops stay rolled and work in shared memory (the row's list,
// and the warp's spent candidate list wl for the pooled items).
template <int KC>
__device__ __noinline__ bool refine_in_list(int act, const uint32_t* l_o, int32_t* l_i, float* l_z,
                                            bool close, float band, float thr, const float* zq,
                                            const float* sb, uint32_t* wl) {
  const int lane = threadIdx.x & 31;
  bool in_list = false;
  uint32_t need = 0u;
  if (close) {
    // the whole list at once (one shared-memory round trip), then the
    // entries next to a gap of at most `band`; empty entries (0) sort last
    uint32_t o[KC];
#pragma unroll
    for (int j = 0; j < KC; ++j) o[j] = l_o[j * BM];
    const float lo = __fsub_rd(thr, band);
    in_list = o[KC - 1] == 0u || float_of_ord(o[KC - 1]) < lo;
    if (in_list) {
#pragma unroll
      for (int j = 0; j < KC; ++j) {
        const float kj = float_of_ord(o[j]);
        const bool up = j > 0 && __fsub_rd(float_of_ord(o[j > 0 ? j - 1 : 0]), kj) <= band;
        const bool dn = j + 1 < KC && o[j + 1 < KC ? j + 1 : j] != 0u &&
                        __fsub_rd(kj, float_of_ord(o[j + 1 < KC ? j + 1 : j])) <= band;
        if (o[j] != 0u && kj >= lo && (up || dn)) need |= 1u << j;
      }
    }
  }
  // pool (expert, owner lane, slot) items of the needed entries
  const int nneed = __popc(need);
  int qoff = nneed;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int t = __shfl_up_sync(kFull, qoff, d);
    if (lane >= d) qoff += t;
  }
  const int qtotal = __shfl_sync(kFull, qoff, 31);
  qoff -= nneed;
  if (qtotal == 0) return close && !in_list;
  // items in wl[0, 256), their double-float keys (hi, lo) and scales after
  // them; more than 256 items (a warp full of near ties) go to FP64
  const bool fits = qtotal <= 256;
  uint32_t* it_e = wl;
  float* it_h = reinterpret_cast<float*>(wl + 256);
  float* it_l = reinterpret_cast<float*>(wl + 512);
  float* it_s = reinterpret_cast<float*>(wl + 768);
  {
    int q = qoff;
#pragma unroll
    for (int j = 0; j < KC; ++j)
      if ((need >> j) & 1u)
        it_e[q++] = ((uint32_t)l_i[j * BM] << 16) | ((uint32_t)lane << 5) | (uint32_t)j;
  }
  __syncwarp();
  bool amb = !fits;
  if (fits) {
    // double-float keys, one item per lane
#pragma unroll 1
    for (int q = lane; q < qtotal; q += 32) {
      const uint32_t item = it_e[q];
      const int e = (int)(item >> 16);
      const NearKey nk = near_key_ool(act, zq[e * BM + (int)((item >> 5) & 31u)], sb ? sb[e] : 0.0f);
      it_h[q] = nk.hi;
      it_l[q] = nk.lo;
      it_s[q] = nk.scale;
    }
    __syncwarp();
    // Re-rank this row's items. Runs of consecutive needed entries lie more
    // than `band` apart, beyond what the keys' errors can cross, so sorting
    // all of the row's items by (key desc, expert asc) keeps every item in
    // its run; they then refill the needed slots in order.
#pragma unroll 1
    for (int q = qoff + 1; q < qoff + nneed; ++q) {
      const uint32_t ie = it_e[q];
      const float h = it_h[q], l = it_l[q], c = it_s[q];
      int p = q;
#pragma unroll 1
      while (p > qoff) {
        const float ph = it_h[p - 1], pl = it_l[p - 1];
        const bool ahead = df_gt(h, l, ph, pl) ||
                           (h == ph && l == pl && (ie >> 16) < (it_e[p - 1] >> 16));
        if (!ahead) break;
        it_e[p] = it_e[p - 1], it_h[p] = ph, it_l[p] = pl, it_s[p] = it_s[p - 1];
        --p;
      }
      it_e[p] = ie, it_h[p] = h, it_l[p] = l, it_s[p] = c;
    }
    // consecutive items must be distinct or come from identical inputs (a
    // misordered pair always leaves such a consecutive pair)
#pragma unroll 1
    for (int q = qoff; q + 1 < qoff + nneed; ++q) {
      if (!near_distinct(it_h[q], it_l[q], it_s[q], it_h[q + 1], it_l[q + 1], it_s[q + 1])) {
        const int e0 = (int)(it_e[q] >> 16), e1 = (int)(it_e[q + 1] >> 16);
        const bool same = zq[e0 * BM + lane] == zq[e1 * BM + lane] && (sb ? sb[e0] == sb[e1] : true);
        if (!same) amb = true;
      }
    }
  }
  // rare: FP64 keys decide the rows the double-float keys could not (it
  // reads the list as still stored and pools its own items)
  if (__any_sync(kFull, amb)) {
    __syncwarp();
    if (amb) {  // back to slot order (the other rows keep their sorted items)
      int q = qoff;
#pragma unroll 1
      for (int j = 0; j < KC; ++j)
        if ((need >> j) & 1u)
          wl[q++] = ((uint32_t)l_i[j * BM] << 16) | ((uint32_t)lane << 5) | (uint32_t)j;
    }
    __syncwarp();
    refine_fp64<KC>(act, l_o, l_i, l_z, need, amb, qoff, qtotal, zq, sb, wl);
  }
  if (need != 0u && !amb) {
    // the sorted items and their scores (from their original slots), all
    // read before the needed slots are refilled in order
    uint32_t ev[KC];
    float sv[KC];
#pragma unroll
    for (int j = 0; j < KC; ++j) {
      ev[j] = 0u;
      sv[j] = 0.0f;
      if ((need >> j) & 1u) {
        ev[j] = it_e[qoff + __popc(need & ((1u << j) - 1u))];
        sv[j] = l_z[(int)(ev[j] & 31u) * BM];
      }
    }
#pragma unroll
    for (int j = 0; j < KC; ++j) {
      if ((need >> j) & 1u) {
        l_i[j * BM] = (int)(ev[j] >> 16);
        l_z[j * BM] = sv[j];
      }
    }
  }
  return close && !in_list;
}

constexpr size_t kCandOffset = 32768;  // the logits copy starts after the exchange area
constexpr int kListCap = 1024;         // words of each warp's candidate list area (4 KB)
constexpr int kPool = 336;             // pooled candidates per warp: items, keys, scores

}  // namespace

struct TcParams {
  RouterArgs a;
  int stages;
  uint32_t stage_bytes, a_bytes, b_bytes;
  int tmem_cols;
  int pair;  // CTA pairs run M = 256 MMAs, each CTA holding half of every W tile
  // NVFP4 only, both in the workspace: W decoded to a BF16 [E, H] copy,
  // and [0] claim counter, [1] epoch, [2 + kb] flag of column block kb
  uint8_t* wdec;
  unsigned* wsync;
  // Stream-K (sk = 1): the tiles x k-steps units are split evenly over
  // `groups` work groups (one CTA, or one CTA pair, per group), so every SM
  // runs the main loop even when there are fewer tiles than SMs. A group's
  // range covers at most the tail of one tile (which it finishes) and the
  // head of the next (whose partial accumulator it publishes); the second
  // accumulator sits `acc2` columns into tensor memory.
  int sk, groups, tiles, acc2;
  float* sk_part;     // [grid CTAs][E/4][BM][4] partial accumulators
  unsigned* sk_flag;  // [grid CTAs] this launch's epoch + 1 once the partial is out
  // measurement build only (-DGBR_PHASE_STAMPS): [CTA][kTcStamps] phase
  // stamps of the launch (null: none)
  unsigned long long* stamps;
};

// Phase stamps of the prefill kernel (measurement build): %globaltimer ns
// that thread 0 of each CTA takes at 0 entry, 1 set-up done, 2 epilogue
// set-up done, 3 accumulator complete, 4 partials added, 5 pass A and the
// bound merged, 6 passes B and C done, 7 halves merged (and near ties
// re-ranked), 8 rows stored, 9 CTA end; slot 10 holds 1 when a warp of the
// CTA re-ranked near ties, slot 11 the time the first MMA was issued (even
// CTAs), 12 threshold computed, 13 pass B masks built, 14 pooled
// activations done, 15 insertion done; slots 16 and 17 hold thread 0's
// candidate count and its warp's pooled total, 18 the SM the CTA ran on,
// 19 its plan (2 x segments + 1 if it finishes a tile), 20 its partial
// accumulator complete, 21 that partial published, 22 the early partials
// of its tile streamed in, 23 its last MMA issued (even CTAs); of the
// partials added after the main loop, the first one's flag seen (24),
// copy landed (25) and sum stored (26), and the same for the last (27-29);
// per first-half warp q (0..3) that re-ranked near ties, slots 30 + 4q..:
// re-rank start, list re-ranked, every-column pass done (0: none), and
// whether that pass ran.
constexpr int kTcStamps = 46;

namespace {


// One group's work: up to two segments of k-steps, the partial one first
// (other groups wait for it), then the one that finishes its tile. Scalar
// fields with select accessors keep the plan in registers.
struct TcPlan {
  int nseg;
  int t0, a0, b0, t1, a1, b1;  // segment s: tile t_s, k-steps [a_s, b_s)
  bool f0, f1;                 // segment s finishes its tile
  int p0;  // first group holding a partial of the finished tile (== group: none)
  __device__ __forceinline__ int t(int s) const { return s ? t1 : t0; }
  __device__ __forceinline__ int kb0(int s) const { return s ? a1 : a0; }
  __device__ __forceinline__ int kb1(int s) const { return s ? b1 : b0; }
  __device__ __forceinline__ bool fin(int s) const { return s ? f1 : f0; }
};

__device__ __forceinline__ TcPlan tc_plan(const TcParams& p, int grp, int nk) {
  TcPlan s;
  s.nseg = 1;
  s.t0 = grp, s.a0 = 0, s.b0 = nk, s.f0 = true;
  s.t1 = 0, s.a1 = 0, s.b1 = 0, s.f1 = false;
  s.p0 = grp;
  if (!p.sk) return s;
  const long long U = (long long)p.tiles * nk, G = p.groups;
  const long long u0 = U * grp / G, u1 = U * (grp + 1) / G;
  const int t0 = (int)(u0 / nk);
  const long long te = (long long)(t0 + 1) * nk;
  const int a0 = (int)(u0 - (long long)t0 * nk);
  // the group owning unit u is ceil((u + 1) G / U) - 1
  s.p0 = (int)((((long long)t0 * nk + 1) * G + U - 1) / U - 1);
  if (u1 > te) {
    // the tail of tile t0 runs to its end; the head of t0 + 1 is shorter
    // than a tile (a range spans at most nk units)
    s.nseg = 2;
    s.t0 = t0 + 1, s.a0 = 0, s.b0 = (int)(u1 - te), s.f0 = false;
    s.t1 = t0, s.a1 = a0, s.b1 = nk, s.f1 = true;
  } else {
    s.t0 = t0, s.a0 = a0, s.b0 = (int)(u1 - (long long)t0 * nk);
    s.f0 = s.b0 == nk;
  }
  return s;
}

// Serial unique-route table for one pair of rows (the thread owning the
// even row of the pair builds it from ids in shared memory). The running
// table lives in the output arrays themselves, which only this thread
// touches, so no per-thread array is needed.
__device__ void pair_table(const int32_t* r0, const int32_t* r1, int k, int32_t* unique,
                           uint8_t* mask, uint8_t* map, int32_t* count) {
  int n = 0;
  for (int p = 0; p < 2 * k; ++p) {
    const int t = p >= k ? 1 : 0;
    const int32_t v = t ? r1[p - k] : r0[p];
    int f = p;
    for (int q = 0; q < p; ++q) {
      if ((q >= k ? r1[q - k] : r0[q]) == v) {
        f = q;
        break;
      }
    }
    if (f == p) {
      unique[n] = v;
      mask[n] = (uint8_t)(1u << t);
      map[p] = (uint8_t)n;
      ++n;
    } else {
      const int u = map[f];
      map[p] = (uint8_t)u;
      mask[u] = (uint8_t)(mask[u] | (1u << t));
    }
  }
  for (int u = n; u < 2 * k; ++u) {
    unique[u] = -1;
    mask[u] = 0;
  }
  *count = n;
}

template <int KC, bool FP4, bool PAIR>
__global__ void __launch_bounds__((kEpiWarps + 2) * 32, 1)
    k_tc_router(const __grid_constant__ CUtensorMap tmap_x,
                const __grid_constant__ CUtensorMap tmap_w, const TcParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint32_t s_lut[256];  // NVFP4: byte of two E2M1 codes -> two BF16 values
  __shared__ __align__(8) uint64_t s_wready;  // NVFP4: s_epoch is set
  __shared__ unsigned s_epoch, s_claim;
  __shared__ float s_bias[256];    // the selection bias (sqrt-softplus)
  __shared__ float s_gbmin[2][32];  // least bias per column group (sqrt-softplus)
  __shared__ __align__(8) uint64_t s_pbar;  // stream-K: a partial has landed
  __shared__ int s_go;                      // stream-K: prefetch the next partial
  const RouterArgs& a = p.a;
  unsigned* const wstat = a.status;  // set when a bounded wait gives up
  TC_STAMP(0);
#ifdef GBR_PHASE_STAMPS
  __shared__ int s_refined;
  if (threadIdx.x == 0) s_refined = 0;
#endif
  const int S = p.stages;
  // 1024-byte aligned tile ring, then barriers
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  uint8_t* tiles = base;
  uint64_t* full = reinterpret_cast<uint64_t*>(tiles + (size_t)S * p.stage_bytes);
  uint64_t* empty = full + S;
  uint64_t* accf = empty + S;  // the finishing accumulator is complete
  uint64_t* accp = accf + 1;   // the partial accumulator is complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accp + 1);
  int32_t* s_sel = reinterpret_cast<int32_t*>(tmem_slot + 4);  // [BM][kMaxK] for tables

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int producer_warp = kEpiWarps, mma_warp = kEpiWarps + 1;
  const int crank = PAIR ? (int)cluster_rank() : 0;
  const int nk = a.H / BK;
  const int E = a.E;
  const int grp = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const TcPlan plan = tc_plan(p, grp, nk);
  const int tile_rows = PAIR ? 2 * BM : BM;
  const bool has_fin = plan.f0 || plan.f1;
  const bool has_part = !plan.f0;  // a partial segment always comes first
  // first row of this CTA's 128 rows of the finished tile
  const int m0 = (plan.f0 ? plan.t0 : plan.t1) * tile_rows + (PAIR ? crank * BM : 0);
#ifdef GBR_PHASE_STAMPS
  if (threadIdx.x == 0 && p.stamps) {
    unsigned sm;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
    p.stamps[blockIdx.x * kTcStamps + 18] = sm;
    p.stamps[blockIdx.x * kTcStamps + 19] = (unsigned)(2 * plan.nseg + (has_fin ? 1 : 0));
  }
#endif

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(accf), 1);
    mbar_init(smem_u32(accp), 1);
    mbar_init(smem_u32(&s_pbar), 1);
    if (FP4) mbar_init(smem_u32(&s_wready), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == mma_warp) {
    if (PAIR) {
      // both CTAs of the pair allocate; the MMAs use the even CTA's address
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(tmem_slot)),
                   "r"(p.tmem_cols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(tmem_slot)),
                   "r"(p.tmem_cols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  // the pair's barriers are initialised and its allocations made before
  // either CTA signals the other
  if (PAIR) cluster_sync_tc();
  tc_fence_after();
  const uint32_t tmem_own = *tmem_slot;
  uint32_t tmem = tmem_own;
  if (PAIR) {
    asm volatile("ld.shared::cluster.u32 %0, [%1];"
                 : "=r"(tmem)
                 : "r"(mapa_u32(smem_u32(tmem_slot), 0u))
                 : "memory");
  }

  pdl_launch_dependents();
  TC_STAMP(1);

  if (warp == producer_warp) {
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_x)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_w)) : "memory");
      pdl_wait();
      const uint64_t pol_x = policy_evict_first(), pol_w = policy_evict_last();
      int issued = 0;
      unsigned want = 0u;  // NVFP4: the flag value of a tile decoded by this launch
      bool go = true;
      if (FP4) {
        go = mbar_wait(wstat, smem_u32(&s_wready), 0);
        want = *reinterpret_cast<volatile unsigned*>(&s_epoch) + 1u;
      }
      for (int sg = 0; sg < plan.nseg && go; ++sg) {
        const int mrow = plan.t(sg) * tile_rows + (PAIR ? crank * BM : 0);
        int decoded_to = plan.kb0(sg);  // NVFP4: column blocks seen decoded, exclusive end
        for (int kb = plan.kb0(sg); kb < plan.kb1(sg); ++kb) {
          const int s = issued % S;  // ring position: k-steps issued so far
          const uint32_t ph = (uint32_t)(issued / S) & 1u;
          if (!mbar_wait(wstat, smem_u32(&empty[s]), ph ^ 1u)) {
            go = false;
            break;
          }
          uint8_t* st = tiles + (size_t)s * p.stage_bytes;
          const uint32_t fb = smem_u32(&full[s]);
          if (PAIR) {
            // both CTAs' halves land on the even CTA's barrier
            const uint32_t fb0 = mapa_u32(fb, 0u);
            if (crank == 0) mbar_expect_tx(fb, 2u * (p.a_bytes + p.b_bytes));
            tma_load_2d_pair(smem_u32(st), &tmap_x, kb * BK, mrow, fb0, pol_x);
            ++issued;
            if (FP4 && kb >= decoded_to) {  // the decoded copy: the next blocks, in batches
              const int nb = min(kb == plan.kb0(sg) ? 1 : 8, plan.kb1(sg) - kb);  // first block alone
              if (!wait_flags8(wstat, p.wsync + 2 + kb, nb, want)) {
                go = false;
                break;
              }
              asm volatile("fence.proxy.async.global;" ::: "memory");
              decoded_to = kb + nb;
            }
            tma_load_2d_pair(smem_u32(st + p.a_bytes), &tmap_w, kb * BK, crank * (E / 2), fb0,
                             pol_w);
            continue;
          }
          mbar_expect_tx(fb, p.a_bytes + p.b_bytes);
          tma_load_2d(smem_u32(st), &tmap_x, kb * BK, mrow, fb, pol_x);
          ++issued;
          if (FP4 && kb >= decoded_to) {  // the decoded copy: the next blocks, in batches
            const int nb = min(kb == plan.kb0(sg) ? 1 : 8, plan.kb1(sg) - kb);  // first block alone
            if (!wait_flags8(wstat, p.wsync + 2 + kb, nb, want)) {
              go = false;
              break;
            }
            asm volatile("fence.proxy.async.global;" ::: "memory");
            decoded_to = kb + nb;
          }
          tma_load_2d(smem_u32(st + p.a_bytes), &tmap_w, kb * BK, 0, fb, pol_w);
        }
      }
      // let copies still in flight land before the CTA can exit (a pair's
      // odd CTA cannot see them: its exit waits for the pair's last MMA)
      if (!PAIR || crank == 0)
        for (int i = (issued > S ? issued - S : 0); i < issued; ++i)
          mbar_wait(wstat, smem_u32(&full[i % S]), (uint32_t)(i / S) & 1u);
    }
  } else if (warp == mma_warp) {
    if (lane == 0 && (!PAIR || crank == 0)) {
      // the even CTA of a pair issues M = 256 MMAs for both
      const uint32_t idesc = PAIR ? idesc_bf16(E, 2 * BM) : idesc_bf16(E);
      int it = 0;  // ring position
      bool go = true;
      for (int sg = 0; sg < plan.nseg && go; ++sg) {
        const uint32_t acc = plan.fin(sg) ? tmem : tmem + (uint32_t)p.acc2;
        for (int kb = plan.kb0(sg); kb < plan.kb1(sg); ++kb, ++it) {
          const int s = it % S;
          const uint32_t ph = (uint32_t)(it / S) & 1u;
          if (!mbar_wait(wstat, smem_u32(&full[s]), ph)) {
            go = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(tiles + (size_t)s * p.stage_bytes);
          const uint32_t sb = sa + p.a_bytes;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint32_t accum = (kb > plan.kb0(sg) || kk > 0) ? 1u : 0u;
#ifdef GBR_PHASE_STAMPS
            if (it == 0 && kk == 0 && p.stamps) p.stamps[blockIdx.x * kTcStamps + 11] = globaltimer();
#endif
            if (PAIR)
              mma_bf16_pair(acc, smem_desc_sw128(sa + kk * 32), smem_desc_sw128(sb + kk * 32),
                            idesc, accum);
            else
              mma_bf16(acc, smem_desc_sw128(sa + kk * 32), smem_desc_sw128(sb + kk * 32), idesc,
                       accum);
          }
          if (PAIR) mma_commit_pair(smem_u32(&empty[s]));
          else mma_commit(smem_u32(&empty[s]));
        }
        // after a give-up the accumulator is incomplete: no commit, so the
        // epilogue's wait for it gives up too instead of reading it
        if (!go) break;
        const uint32_t done = smem_u32(plan.fin(sg) ? accf : accp);
        if (PAIR) mma_commit_pair(done);
        else mma_commit(done);
      }
#ifdef GBR_PHASE_STAMPS
      if (p.stamps) p.stamps[blockIdx.x * kTcStamps + 23] = globaltimer();
#endif
    }
  } else if (warp < kEpiWarps) {
    // epilogue: warp w reads TMEM lanes 32(w%4).. of columns half w/4
    const int quad = warp & 3, half = warp >> 2;
    const int row = quad * 32 + lane;
    const int m = m0 + row;
    const int E2 = ((E / 2 + 31) / 32) * 32;
    const int c_lo = half * E2, c_hi = half ? E : min(E, E2);
    const float g = FP4 ? a.w_global : 1.0f;
    const int k = a.k;
    // sp: a biased activation (sqrt-softplus or sigmoid) rather than softmax
    const int act = a.act;
    const bool sp = act != ACT_SOFTMAX;
    const bool sig = act == ACT_SIGMOID;
    const bool has_bias = sp && a.bias != nullptr;
    // range of the selection-only bias (read before the accumulator is ready)
    float bmin = 0.0f, bmax = 0.0f;
    if (has_bias) {
      bmin = INFINITY;
      bmax = -INFINITY;
      for (int e = lane; e < E; e += 32) {
        const float b = __ldg(a.bias + e);
        bmin = fminf(bmin, b);
        bmax = fmaxf(bmax, b);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        bmin = fminf(bmin, __shfl_xor_sync(kFull, bmin, off));
        bmax = fmaxf(bmax, __shfl_xor_sync(kFull, bmax, off));
      }
    }
    if (has_bias && warp == 0)
      for (int e = lane; e < E; e += 32) s_bias[e] = __ldg(a.bias + e);
    if (sp && warp == 1) {
      // least bias of each interleaved column group of each half (the
      // groups of pass A: column c_lo + q + G t is in group q)
      constexpr int G = KC <= 4 ? 4 : (KC <= 6 ? 8 : (KC <= 10 ? 16 : 32));
      for (int hq = lane; hq < 2 * G; hq += 32) {
        const int h = hq / G, q = hq % G;
        const int lo = h * E2, hi = h ? E : min(E, E2);
        float m = INFINITY;
        for (int c = lo + q; c < hi; c += G) m = fminf(m, has_bias ? __ldg(a.bias + c) : 0.0f);
        s_gbmin[h][q] = m;
      }
    }
    if (!FP4 && p.sk && threadIdx.x == 0) {
      // this launch's epoch (the flags it sets are epoch + 1): read after the
      // previous launch has finished, then one arrival per CTA; the last
      // arrival resets the counter and advances the epoch for the next launch
      pdl_wait();
      s_epoch = ld_acquire_u32(p.wsync + 1);
      const unsigned t = atomicAdd(p.wsync, 1u);
      if (t == gridDim.x - 1u) {
        asm volatile("st.relaxed.gpu.global.u32 [%0], 0;" ::"l"(p.wsync) : "memory");
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p.wsync + 1) : "memory");
      }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
    if (FP4) {
      // NVFP4: W is decoded once per launch, not once per CTA. The CTAs claim
      // k-step column blocks from a counter in the workspace; the 256 threads
      // of a claim decode the E x 64 block (thread r owns row r) into a BF16
      // [E, H] copy and flag it with this launch's epoch; producers load
      // flagged blocks with the same TMA tiles as BF16 weights.
      // Claims never wait, so no CTA needs another to be resident. Each CTA
      // makes one failing claim; the last of them (ticket nk + grid - 1)
      // resets the counter and advances the epoch for the next launch.
      const int r = threadIdx.x;  // 0..255
      for (int b = r; b < 256; b += kEpiWarps * 32) {
        const uint32_t lo = __float_as_uint(e2m1_to_f32(b & 15u)) >> 16;
        const uint32_t hi = __float_as_uint(e2m1_to_f32((uint32_t)b >> 4)) >> 16;
        s_lut[b] = lo | (hi << 16);
      }
      pdl_wait();  // the decoded copy is read by the preceding launch until here
      if (r == 0) {
        s_epoch = ld_acquire_u32(p.wsync + 1);
        mbar_arrive(smem_u32(&s_wready));
      }
      const uint8_t* qp = static_cast<const uint8_t*>(a.w);
      const int Hb = a.H / 2, Hs = a.H / 16;
      const unsigned nclaim = (unsigned)nk + gridDim.x;
      for (;;) {
        if (r == 0) {
          const unsigned t = atomicAdd(p.wsync, 1u);
          if (t == nclaim - 1u) {  // every claim of this launch is in
            asm volatile("st.relaxed.gpu.global.u32 [%0], 0;" ::"l"(p.wsync) : "memory");
            asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p.wsync + 1) : "memory");
          }
          s_claim = t;
        }
        asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
        const unsigned t = *reinterpret_cast<volatile unsigned*>(&s_claim);
        const unsigned want = *reinterpret_cast<volatile unsigned*>(&s_epoch) + 1u;
        asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
        if (t >= (unsigned)nk) break;
        if (r < E) {
          const uint4* src = reinterpret_cast<const uint4*>(qp + (size_t)r * Hb + t * (BK / 2));
          const uint4 q0 = __ldg(src), q1 = __ldg(src + 1);
          const uint32_t sc =
              __ldg(reinterpret_cast<const uint32_t*>(a.w_scales + (size_t)r * Hs + t * (BK / 16)));
          const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
          // row r, elements 64t..64t+63 of the decoded [E, H] BF16 copy
          uint8_t* dst = p.wdec + ((size_t)r * a.H + (size_t)t * BK) * 2;
#pragma unroll
          for (int c = 0; c < 8; ++c) {  // 16-byte chunk c = elements 8c..8c+7
            // the block scale in BF16 (exact: at most 4 significant bits), twice
            const uint32_t sb16 = __float_as_uint(e4m3_to_f32((sc >> (8 * (c >> 1))) & 0xffu)) >> 16;
            const __nv_bfloat162 scale2 = __halves2bfloat162(
                __ushort_as_bfloat16((unsigned short)sb16), __ushort_as_bfloat16((unsigned short)sb16));
            uint32_t outw[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              const uint32_t pair = s_lut[(qw[c] >> (8 * jj)) & 0xffu];
              __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&pair);
              v = __hmul2(v, scale2);  // exact: the product has at most 6 significant bits
              outw[jj] = *reinterpret_cast<const uint32_t*>(&v);
            }
            *reinterpret_cast<uint4*>(dst + c * 16) = make_uint4(outw[0], outw[1], outw[2], outw[3]);
          }
        }
        // the producers read the tile through the async proxy
        asm volatile("fence.proxy.async.global;" ::: "memory");
        asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
        if (r == 0)
          asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p.wsync + 2 + t), "r"(want)
                       : "memory");
      }
    }
    TC_STAMP(2);
    const unsigned sk_want = *reinterpret_cast<volatile unsigned*>(&s_epoch) + 1u;
    const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
    if (has_part) {
      // publish the partial accumulator: this CTA's slot of the workspace,
      // [E/4][BM][4] (a warp stores 512 contiguous bytes per 4 columns), then
      // the flag; finishers fetch it with one bulk copy
      const bool okp = mbar_wait_warp(wstat, smem_u32(accp), 0);
      TC_STAMP(20);
      tc_fence_after();
      if (okp) {
        // two 32-column loads in flight per round
        float* part = p.sk_part + (size_t)blockIdx.x * E * BM + row * 4;
        for (int c0 = c_lo; c0 < c_hi; c0 += 64) {
          const bool two = c0 + 32 < c_hi;
          uint32_t r[2][32];
          tmem_ld32_issue(trow + (uint32_t)p.acc2 + c0, r[0]);
          if (two) tmem_ld32_issue(trow + (uint32_t)p.acc2 + c0 + 32, r[1]);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (h == 0 || two) {
#pragma unroll
              for (int i = 0; i < 8; ++i)  // E % 16 == 0: a group of 4 is all in or all out
                if (c0 + 32 * h + 4 * i < c_hi)
                  st_cg_v4(part + (size_t)((c0 + 32 * h) / 4 + i) * BM * 4,
                           __uint_as_float(r[h][4 * i]), __uint_as_float(r[h][4 * i + 1]),
                           __uint_as_float(r[h][4 * i + 2]), __uint_as_float(r[h][4 * i + 3]));
            }
          }
        }
      }
      asm volatile("fence.proxy.async.global;" ::: "memory");  // read by bulk copies
      asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
      if (threadIdx.x == 0) {
        __threadfence();
        asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p.sk_flag + blockIdx.x),
                     "r"(sk_want)
                     : "memory");
      }
      TC_STAMP(21);
    }
    // The finished tile's other partials P_q (groups p0 .. grp-1) are summed
    // in group order into S in the spare accumulator columns, and the tile's
    // logits are fin + S: the same additions in the same order whichever
    // way each partial arrives. While the main loop still runs, partials
    // whose flags are already set stream in through registers; the rest land
    // in the idle tile ring by bulk copies once the accumulator is complete.
    const int nparts = has_fin ? grp - plan.p0 : 0;
    const uint32_t tS = trow + (uint32_t)p.acc2;
    int pre = 0;
    for (int q = plan.p0; q < plan.p0 + nparts; ++q) {
      const int slot = q * (PAIR ? 2 : 1) + crank;
      if (threadIdx.x == 0) {
        // whichever comes first: the partial (prefetch it) or the end of the
        // main loop (the bulk copies below are then faster)
        int go = 0;
        const uint64_t t0 = globaltimer();
        uint32_t ns = 64;
        for (;;) {
          // once the main loop is done the bulk copies win, even for a
          // partial that is already out
          if (mbar_try(smem_u32(accf), 0)) break;
          if (ld_acquire_u32(p.sk_flag + slot) == sk_want) {
            go = 1;
            break;
          }
          if (globaltimer() - t0 > kWaitNs) break;
          __nanosleep(ns);
          if (ns < 512) ns <<= 1;
        }
        s_go = go;
      }
      asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
      const bool go = *reinterpret_cast<volatile int*>(&s_go) != 0;
      asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
      if (!go) break;
      wait_flag(wstat, p.sk_flag + slot, sk_want);  // set: this thread's own acquire
      const float* part = p.sk_part + (size_t)slot * E * BM + row * 4;
      for (int c0 = c_lo; c0 < c_hi; c0 += 64) {
        // two 32-column groups of loads in flight per round
        float v[2][32];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            // E % 16 == 0: a group of 4 columns is all in or all out
            const int g4 = min((c0 + 32 * h) / 4 + i, E / 4 - 1);
            const float4 u = __ldcg(reinterpret_cast<const float4*>(part + (size_t)g4 * BM * 4));
            v[h][4 * i] = u.x, v[h][4 * i + 1] = u.y, v[h][4 * i + 2] = u.z, v[h][4 * i + 3] = u.w;
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (c0 + 32 * h < c_hi) {
            if (pre > 0) {
              float w[32];
              tmem_ld32(tS + c0 + 32 * h, w);
#pragma unroll
              for (int j = 0; j < 32; ++j) v[h][j] = w[j] + v[h][j];
            }
            tmem_st32(tS + c0 + 32 * h, v[h]);
          }
        }
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      ++pre;
    }
    TC_STAMP(22);
    // a CTA whose range ends inside a tile has no rows to finish
    const bool ok = has_fin && mbar_wait_warp(wstat, smem_u32(accf), 0);
    TC_STAMP(3);
    tc_fence_after();
    // one answer for all epilogue warps (the blocks it guards hold named
    // barriers): a warp whose bounded wait gave up just before the
    // accumulator landed must not leave its peers waiting at them
    const bool all_ok = epi_all(ok);
    if (all_ok && nparts > 0) {
      const uint32_t pbytes = (uint32_t)E * BM * 4;
      for (int q = plan.p0 + pre; q <= grp; ++q) {
        // q < grp: P_q lands in the ring (S += P_q, and on the last one the
        // logits fin + S); q == grp: every partial came early, fin + S only
        const bool last = q >= grp - 1;
        const bool have = q < grp;
        bool okq = true;
#ifdef GBR_PHASE_STAMPS
        const int sfirst = q == plan.p0 + pre ? 24 : -1, slast = last ? 27 : -1;
#endif
        if (have) {
          const int slot = q * (PAIR ? 2 : 1) + crank;
          wait_flag(wstat, p.sk_flag + slot, sk_want);
#ifdef GBR_PHASE_STAMPS
          if (sfirst >= 0) TC_STAMP(24);
          if (slast >= 0) TC_STAMP(27);
#endif
          if (threadIdx.x == 0) {
            asm volatile("fence.proxy.async.global;" ::: "memory");
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_expect_tx(smem_u32(&s_pbar), pbytes);
            // eight copies in flight rather than one (pbytes / 8 = 64 E bytes)
            const uint8_t* src = reinterpret_cast<const uint8_t*>(p.sk_part + (size_t)slot * E * BM);
#pragma unroll
            for (int c = 0; c < 8; ++c)
              bulk_g2s(smem_u32(tiles) + c * (pbytes / 8), src + c * (pbytes / 8), pbytes / 8,
                       smem_u32(&s_pbar));
          }
          okq = mbar_wait_warp(wstat, smem_u32(&s_pbar), (uint32_t)(q - plan.p0 - pre) & 1u);
#ifdef GBR_PHASE_STAMPS
          if (sfirst >= 0) TC_STAMP(25);
          if (slast >= 0) TC_STAMP(28);
#endif
        }
        if (okq) {
          const bool hasS = q > plan.p0;  // S holds P_p0 .. P_(q-1)
          const float4* sp4 = reinterpret_cast<const float4*>(tiles) + row;
          for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
            // the tensor-memory loads (S, and the accumulator on the last
            // round) are in flight together while the staged partial is read
            uint32_t ws[32], fs[32];
            if (hasS) tmem_ld32_issue(tS + c0, ws);
            if (last) tmem_ld32_issue(trow + c0, fs);
            float v[32];
            if (have) {
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float4 u = sp4[(size_t)min(c0 / 4 + i, E / 4 - 1) * BM];
                v[4 * i] = u.x, v[4 * i + 1] = u.y, v[4 * i + 2] = u.z, v[4 * i + 3] = u.w;
              }
            }
            if (hasS || last) tmem_wait_ld();
            if (hasS) {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                v[j] = have ? __uint_as_float(ws[j]) + v[j] : __uint_as_float(ws[j]);
            }
            if (last) {
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(fs[j]) + v[j];
              tmem_st32(trow + c0, v);
            } else {
              tmem_st32(tS + c0, v);
            }
          }
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        }
        // every warp is done with the staged partial before the next lands
        // (or, after the last, before pass A writes over the ring)
        asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
#ifdef GBR_PHASE_STAMPS
        if (sfirst >= 0 && have) TC_STAMP(26);
        if (slast >= 0 && have) TC_STAMP(29);
#endif
        if (last) break;
      }
    }
    TC_STAMP(4);
    // the idle tile ring: exchange area, then per-(half, row) candidate lists
    uint32_t* xo = reinterpret_cast<uint32_t*>(tiles);       // [KC][BM]
    int32_t* xi = reinterpret_cast<int32_t*>(xo + KC * BM);  // [KC][BM]
    float* xz = reinterpret_cast<float*>(xi + KC * BM);      // [KC][BM]
    float* xm = xz + KC * BM;                                 // [3][BM]
    float* zbuf = reinterpret_cast<float*>(tiles + kCandOffset);  // [E][BM] logits, column-major
    TopList<KC> top;
    top.init();
    float amax = 0.0f, kabs = 0.0f;
    if (all_ok) {
      // Pass A: a lower bound L on the row's k-th largest key, branch-free.
      // Each half splits its columns into G interleaved groups and takes each
      // group's largest logit z_q; that expert's key a(z_q) + b is at least
      // LB_q = sqrt(max(z_q, 0)) + (least bias in the group), since
      // a(z) >= sqrt(max(z, 0)) (rounded down: LB_q never exceeds it). The
      // groups of both halves are 2G distinct experts, so the k-th largest
      // LB_q over the row is at most the k-th largest key. An expert can
      // then reach the top k (or the FP32 band below it) only if
      // a(z) + b_max >= L - margin, i.e. z >= a^-1(L - margin - b_max).
      // For softmax the key is the logit and LB_q = z_q, so z >= L.
      constexpr int G = KC <= 4 ? 4 : (KC <= 6 ? 8 : (KC <= 10 ? 16 : 32));  // >= 2 (KC - 2) >= 2k
      float gmax[G];
#pragma unroll
      for (int q = 0; q < G; ++q) gmax[q] = -INFINITY;
      for (int c0 = c_lo; c0 < c_hi; c0 += (KC <= 10 ? 64 : 32)) {
        // two 32-column loads in flight, one wait (the condition is warp-uniform)
        uint32_t r0[32], r1[32];
        const bool two = KC <= 10 && c0 + 32 < c_hi;  // long lists: one load at a time
        tmem_ld32_issue(trow + c0, r0);
        if (two) tmem_ld32_issue(trow + c0 + 32, r1);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (c0 + j < c_hi) {
            const float z = FP4 ? __uint_as_float(r0[j]) * g : __uint_as_float(r0[j]);
            gmax[j % G] = fmaxf(gmax[j % G], z);
            zbuf[(c0 + j) * BM + row] = z;  // lanes store consecutive words
          }
        }
        if (two) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (c0 + 32 + j < c_hi) {
              const float z = FP4 ? __uint_as_float(r1[j]) * g : __uint_as_float(r1[j]);
              gmax[j % G] = fmaxf(gmax[j % G], z);
              zbuf[(c0 + 32 + j) * BM + row] = z;
            }
          }
        }
      }
      // this half's LB_q, sorted descending by a bitonic network (G is a
      // power of two); its KC - 1 >= k largest go to the other half
      float lbv[G];
#pragma unroll
      for (int q = 0; q < G; ++q) {
        float xq = gmax[q];
        if (sp && xq > -INFINITY) {
          // a lower bound of a(z_q): sqrt(max(z, 0)) as z * rsqrt(z) (rsqrtf
          // is within 2 ulp) lowered by 2^-20, or the FP32 sigmoid lowered
          // by 2^-20 (its error is at most 3 * 2^-23)
          const float zz = fmaxf(xq, 0.0f);
          const float lb = sig ? sigmoid_f32(xq) * (1.0f - 0x1p-20f)
                               : (zz > 0.0f ? zz * rsqrtf(zz) * (1.0f - 0x1p-20f) : 0.0f);
          xq = __fadd_rd(lb, s_gbmin[half][q]);
        }
        lbv[q] = xq;
      }
      sort_desc_bitonic<G>(lbv);
      // the other half's list comes through the idle tile ring: past the
      // list exchange area when it fits below the logits copy (nothing else
      // writes there), else over it, with a second barrier so it is not
      // reused before both halves have read
      constexpr int kLbxOff = (3 * KC + 3) * BM * 4;
      constexpr bool kSepLbx = kLbxOff + 2 * (KC - 1) * BM * 4 <= (int)kCandOffset;
      float* lbx = reinterpret_cast<float*>(tiles + (kSepLbx ? kLbxOff : 0));  // [2][KC - 1][BM]
#pragma unroll
      for (int j = 0; j < KC - 1; ++j) lbx[(half * (KC - 1) + j) * BM + row] = lbv[j];
      asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
      // L: the k-th largest of the union of the two sorted lists, the
      // largest over i of min(i-th of mine, (k-i)-th of the other's); and
      // the largest LB of the row
      const float* other = lbx + (1 - half) * (KC - 1) * BM + row;
      float lz = -INFINITY;
#pragma unroll
      for (int i = 0; i < KC - 1; ++i) {
        if (i <= k) {
          const float ai = i == 0 ? INFINITY : lbv[i > 0 ? i - 1 : 0];
          const float bj = i == k ? INFINITY : other[(k - i - 1) * BM];
          lz = fmaxf(lz, fminf(ai, bj));
        }
      }
      const float lb_top = fmaxf(lbv[0], other[0]);
      if (!kSepLbx) asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
      TC_STAMP(5);
      // The threshold. Margins: the FP32 keys are within
      // err = 2^-23 (c a + 0.5 |key|) + 2^-59 of the exact ones (c =
      // act_err_coef <= 6); the band is 2 err and the list must hold keys
      // down to two bands below the k-th FP32 key, so the exact keys to
      // keep reach L - 6 err (the margin below allows 10); with a <= A = (largest LB) -
      // b_min + 0.84 (a(z) <= sqrt(max(z, 0)) + sqrt(ln 2)) the margin
      // 2^-16 (4 A + |b|max + 1) covers that many times over. a^-1(y) =
      // log(expm1(y^2)) is then taken on y shrunk by 2^-18 and the result
      // lowered by 2^-16 (1 + |t|), far beyond the FP32 errors of expm1f and
      // logf; above y^2 = 80, log(expm1(u)) = u - O(e^-80).
      float tz;
      if (!(lz > -INFINITY)) {
        tz = -INFINITY;  // fewer than k experts bounded: keep them all
      } else if (!sp) {
        tz = lz;  // softmax: the key is the logit, exactly
      } else {
        const float A = sig ? 1.0f : lb_top - bmin + 0.84f;
        const float babs = fmaxf(fabsf(bmin), fabsf(bmax));
        const float margin = 0x1p-16f * (4.0f * fabsf(A) + babs + 1.0f);
        const float y = (lz - margin - bmax) * (1.0f - 0x1p-18f);
        if (!(y > 0.0f)) {
          tz = -INFINITY;
        } else {
          const float u = y * y;
          // a^-1(y): sqrt-softplus log(expm1(y^2)), sigmoid log(y / (1 - y));
          // L never exceeds the k-th key, so y < 1 for the sigmoid
          const float t = sig ? logf(y / (1.0f - y)) : (u > 80.0f ? u : logf(expm1f(u)));
          tz = t - 0x1p-16f * (1.0f + fabsf(t));
        }
      }
      TC_STAMP(12);
      // Pass B: a bit per candidate column, branch-free (at most 4 chunks of 32)
      uint32_t cm[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        const int c0 = c_lo + 32 * ch;
        if (c0 < c_hi) {
          float v[32];
          tmem_ld32(trow + c0, v);
          uint32_t mbits = 0u;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            mbits |= ((c0 + j < c_hi) && (FP4 ? v[j] * g : v[j]) >= tz ? 1u : 0u) << j;
          cm[ch] = mbits;
        }
      }
      TC_STAMP(13);
      // Pass C. The warp pools its 32 rows' candidates into one list (lane,
      // expert) in expert order per row, then computes each item's score
      // (the logit, or its activation) and key (score + bias) spread evenly
      // over the lanes, four independent items per lane at a time; every
      // row then inserts its own items from the list, loaded one step
      // ahead, into its sorted top list (lanes in lockstep). A warp with
      // more than kPool candidates falls back to per-row evaluation.
      const int ncand = __popc(cm[0]) + __popc(cm[1]) + __popc(cm[2]) + __popc(cm[3]);
      int off = ncand;  // inclusive warp scan of the counts
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int t = __shfl_up_sync(kFull, off, d);
        if (lane >= d) off += t;
      }
      const int total = __shfl_sync(kFull, off, 31);
      off -= ncand;
      uint32_t* wl = reinterpret_cast<uint32_t*>(tiles + kCandOffset + (size_t)E * BM * 4) +
                     warp * kListCap;         // items: lane << 8 | expert
      float* wk = reinterpret_cast<float*>(wl + kPool);      // keys
      float* ws = reinterpret_cast<float*>(wl + 2 * kPool);  // scores
      const bool pooled = total <= kPool;
      if (pooled) {
        uint32_t mm[4] = {cm[0], cm[1], cm[2], cm[3]};
        int o = off;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          while (mm[ch]) {
            const int col = 32 * ch + __ffs(mm[ch]) - 1;
            mm[ch] &= mm[ch] - 1u;
            wl[o++] = ((uint32_t)lane << 8) | (uint32_t)(c_lo + col);
          }
        }
        __syncwarp();
        constexpr int AU = KC <= 10 ? 4 : 1;  // items per lane in flight (long lists: 1)
        for (int t0 = lane; t0 < total; t0 += 32 * AU) {
          float z[AU];
          int ex[AU];
#pragma unroll
          for (int u = 0; u < AU; ++u) {
            const int t = t0 + 32 * u;
            ex[u] = 0;
            z[u] = 0.0f;
            if (t < total) {
              const uint32_t item = wl[t];
              ex[u] = (int)(item & 255u);
              z[u] = zbuf[ex[u] * BM + quad * 32 + (int)(item >> 8)];
            }
          }
#pragma unroll
          for (int u = 0; u < AU; ++u) {
            const int t = t0 + 32 * u;
            if (t < total) {
              const float sc = sp ? act_f32(act, z[u]) : z[u];
              ws[t] = sc;
              wk[t] = has_bias ? sc + s_bias[ex[u]] : sc;
            }
          }
        }
        __syncwarp();
      }
      TC_STAMP(14);
#ifdef GBR_PHASE_STAMPS
      if (threadIdx.x == 0 && p.stamps) {
        p.stamps[blockIdx.x * kTcStamps + 16] = (unsigned)ncand;
        p.stamps[blockIdx.x * kTcStamps + 17] = (unsigned)total;
      }
#endif
      const int nmax = (int)__reduce_max_sync(kFull, (uint32_t)ncand);
      if (pooled) {
        uint32_t it_n = 0u;
        float k_n = 0.0f, s_n = 0.0f;
        if (ncand > 0) it_n = wl[off], k_n = wk[off], s_n = ws[off];
        for (int i = 0; i < nmax; ++i) {
          const uint32_t it = it_n;
          const float key = k_n, sc = s_n;
          if (i + 1 < ncand) it_n = wl[off + i + 1], k_n = wk[off + i + 1], s_n = ws[off + i + 1];
          if (i < ncand) {
            if (sp) {
              amax = fmaxf(amax, sc);
              kabs = fmaxf(kabs, fabsf(key));
            }
            top.push(ord_of(key), (int)(it & 255u), sc);
          }
        }
      } else {
        for (int i = 0; i < nmax; ++i) {
          if (i < ncand) {
            // next candidate column, branch-free: the lowest set bit of the
            // first non-empty chunk mask
            const bool n0 = cm[0] != 0u, n1 = cm[1] != 0u, n2 = cm[2] != 0u;
            const uint32_t mw = n0 ? cm[0] : (n1 ? cm[1] : (n2 ? cm[2] : cm[3]));
            const int base = n0 ? 0 : (n1 ? 32 : (n2 ? 64 : 96));
            const uint32_t rest = mw & (mw - 1u);
            cm[0] = n0 ? rest : cm[0];
            cm[1] = (!n0 && n1) ? rest : cm[1];
            cm[2] = (!n0 && !n1 && n2) ? rest : cm[2];
            cm[3] = (!n0 && !n1 && !n2) ? rest : cm[3];
            const int e = c_lo + base + __ffs(mw) - 1;
            float sc = zbuf[e * BM + row];  // the score: the logit, or its activation
            if (sp) sc = act_f32(act, sc);
            float key = sc;
            if (sp) {
              key = has_bias ? sc + s_bias[e] : sc;
              amax = fmaxf(amax, sc);
              kabs = fmaxf(kabs, fabsf(key));
            }
            top.push(ord_of(key), e, sc);
          }
        }
      }
      TC_STAMP(15);
    }
    TC_STAMP(6);
    // hand the second half's list to the first half
    if (half == 1) {
#pragma unroll
      for (int j = 0; j < KC; ++j) {
        xo[j * BM + row] = top.o[j];
        xi[j * BM + row] = top.i[j];
        xz[j * BM + row] = top.z[j];
      }
      xm[row] = amax;
      xm[BM + row] = kabs;
    }
    // (stream-K: the first half reads columns the second half wrote back)
    tc_fence_before();
    asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
    tc_fence_after();
    if (half == 0 && all_ok) {
#pragma unroll
      for (int j = 0; j < KC; ++j) top.push(xo[j * BM + row], xi[j * BM + row], xz[j * BM + row]);
      amax = fmaxf(amax, xm[row]);
      kabs = fmaxf(kabs, xm[BM + row]);
      // guard-band refine (see select.cuh); FP32 bounds, rounded outwards
      bool close = false;
      float band = 0.0f;
      if (sp) {
        band = 2.0f * key_err_bound(amax, kabs, act_err_coef(act));  // as in select.cuh
        const int kk = min(k + 1, E);
#pragma unroll
        for (int j = 0; j + 1 < KC; ++j)
          if (j + 1 < kk &&
              __fsub_rd(float_of_ord(top.o[j]), float_of_ord(top.o[j + 1])) <= band)
            close = true;
      }
      // the k-th key is the smallest of the first k (the list is sorted);
      // a min avoids an index by k, which would push the list to local memory
      uint32_t kth = 0xffffffffu;
#pragma unroll
      for (int j = 0; j < KC; ++j)
        if (j < k) kth = min(kth, top.o[j]);
      const float thr = __fsub_rd(float_of_ord(kth), band);
      bool slow = false;
#ifdef GBR_PHASE_STAMPS
      if (__any_sync(kFull, close) && lane == 0) s_refined = 1;
#endif
      if (__any_sync(kFull, close)) {
        // the list goes through the exchange area (free after the merge), so
        // the rare refine runs out of line without holding it in registers
#pragma unroll
        for (int j = 0; j < KC; ++j) {
          xo[j * BM + row] = top.o[j];
          xi[j * BM + row] = top.i[j];
          xz[j * BM + row] = top.z[j];
        }
        uint32_t* wl = reinterpret_cast<uint32_t*>(tiles + kCandOffset + (size_t)E * BM * 4) +
                       warp * kListCap;  // this warp's candidate list is spent
#ifdef GBR_PHASE_STAMPS
        if (lane == 0 && p.stamps) p.stamps[blockIdx.x * kTcStamps + 30 + 4 * quad] = globaltimer();
#endif
        slow = refine_in_list<KC>(act, xo + row, xi + row, xz + row, close, band, thr,
                                  zbuf + quad * 32, has_bias ? s_bias : nullptr, wl);
#ifdef GBR_PHASE_STAMPS
        if (lane == 0 && p.stamps) p.stamps[blockIdx.x * kTcStamps + 31 + 4 * quad] = globaltimer();
#endif
        if (close) {
#pragma unroll
          for (int j = 0; j < KC; ++j) {
            top.i[j] = xi[j * BM + row];
            top.z[j] = xz[j * BM + row];
          }
        }
      }
      if (__any_sync(kFull, slow)) {  // near ties reaching past the list: every column
        refine_row<KC, FP4>(trow, E, g, a.bias, act, thr, slow, xi + row, xz + row);
#ifdef GBR_PHASE_STAMPS
        if (lane == 0 && p.stamps) {
          p.stamps[blockIdx.x * kTcStamps + 32 + 4 * quad] = globaltimer();
          p.stamps[blockIdx.x * kTcStamps + 33 + 4 * quad] = 1;
        }
#endif
        if (slow) {
#pragma unroll
          for (int j = 0; j < KC; ++j) {
            top.i[j] = xi[j * BM + row];
            top.z[j] = xz[j * BM + row];
          }
        }
      }
      TC_STAMP(7);
      if (m < a.M) {
        float sv[KC];
#pragma unroll
        for (int j = 0; j < KC; ++j)
          sv[j] = sp ? top.z[j] : expf(top.z[j] - top.z[0]);  // the list keeps scores
        float sum = slot_tree_sum<KC>(sv, k);  // the warp selection's summation order
        if (sp) {
          float smax = 0.0f;
#pragma unroll
          for (int j = 0; j < KC; ++j)
            if (j < k) smax = fmaxf(smax, sv[j]);
          if (!(smax >= 0x1p-50f)) {
            // every chosen activation is tiny (FP32 keeps few or no bits of
            // it): the ratios come from the log domain
            float la[KC], lm = -INFINITY;
#pragma unroll
            for (int j = 0; j < KC; ++j) {
              la[j] = j < k ? log_act(act, zbuf[top.i[j] * BM + row]) : -INFINITY;
              lm = fmaxf(lm, la[j]);
            }
#pragma unroll
            for (int j = 0; j < KC; ++j) sv[j] = lm > -INFINITY ? expf(la[j] - lm) : 0.0f;
            sum = slot_tree_sum<KC>(sv, k);
          }
        }
        const float inv = 1.0f / (float)k;
#pragma unroll
        for (int j = 0; j < KC; ++j) sv[j] = sum > 0.0f ? sv[j] / sum : inv;
        int32_t* oi = a.out_idx + (size_t)m * k;
        float* ow = a.out_w + (size_t)m * k;
        if ((k & 3) == 0 && ((reinterpret_cast<uintptr_t>(oi) | reinterpret_cast<uintptr_t>(ow)) & 15u) == 0) {
#pragma unroll
          for (int j = 0; j + 3 < KC; j += 4) {  // 16-byte stores
            if (j < k) {
              *reinterpret_cast<int4*>(oi + j) = make_int4(top.i[j], top.i[j + 1], top.i[j + 2], top.i[j + 3]);
              *reinterpret_cast<float4*>(ow + j) = make_float4(sv[j], sv[j + 1], sv[j + 2], sv[j + 3]);
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < KC; ++j) {
            if (j < k) {
              oi[j] = top.i[j];
              ow[j] = sv[j];
            }
          }
        }
        if (a.tbl_unique) {
#pragma unroll
          for (int j = 0; j < KC; ++j)
            if (j < k) s_sel[row * kMaxK + j] = top.i[j];
        }
      }
      if (a.logits) {  // telemetry tap; the loads are warp-collective, the stores per row
        for (int c0 = 0; c0 < E; c0 += 32) {
          float v[32];
          tmem_ld32(trow + c0, v);
          if (m < a.M) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (c0 + j < E) a.logits[(size_t)m * E + c0 + j] = FP4 ? v[j] * g : v[j];
          }
        }
      }
      if (a.tbl_unique) {
        __syncwarp();
        if ((lane & 1) == 0 && m + 1 < a.M) {
          const size_t gi = (size_t)(m >> 1);
          pair_table(s_sel + row * kMaxK, s_sel + (row + 1) * kMaxK, k,
                     a.tbl_unique + gi * 2 * k, a.tbl_mask + gi * 2 * k, a.tbl_map + gi * 2 * k,
                     a.tbl_count + gi);
        }
      }
    }
  }
  TC_STAMP(8);
  tc_fence_before();
  __syncthreads();
  TC_STAMP(9);
#ifdef GBR_PHASE_STAMPS
  if (threadIdx.x == 0 && p.stamps) p.stamps[blockIdx.x * kTcStamps + 10] = (unsigned)s_refined;
#endif
  // the peer may still signal this CTA's barriers (or read its tensor
  // memory) until it is done as well
  if (PAIR) cluster_sync_tc();
  if (warp == mma_warp) {
    tc_fence_after();
    if (PAIR)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_own),
                   "r"(p.tmem_cols)
                   : "memory");
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_own),
                   "r"(p.tmem_cols)
                   : "memory");
  }
}

template <int KC, bool FP4, bool PAIR>
cudaError_t launch_kc(const CUtensorMap& mx, const CUtensorMap& mw, const TcParams& p0,
                      size_t smem, bool pdl, bool want_sk, cudaStream_t stream, int* query) {
  auto kern = k_tc_router<KC, FP4, PAIR>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  TcParams p = p0;
  const int cl = PAIR ? 2 : 1;
  int grid = ((p.a.M + BM - 1) / BM + cl - 1) / cl * cl;
  if (want_sk) {
    // stream-K when there are fewer tiles than resident groups: the
    // tiles x k-steps units split evenly over as many of them as keep every
    // tile within four groups
    const int tiles = (p.a.M + cl * BM - 1) / (cl * BM);
    const int nk = p.a.H / BK;
    const int Gr = tc_sk_resident_groups(reinterpret_cast<const void*>(kern), smem, cl);
    const int G = Gr > tiles ? tc_sk_groups_for(tiles, nk, Gr) : 0;
    if (G > 0 && 2 * p.tmem_cols <= 512) {
      p.sk = 1;
      p.groups = G;
      p.tiles = tiles;
      p.acc2 = p.tmem_cols;
      p.tmem_cols *= 2;
      grid = G * cl;
    }
  }
  if (query) {  // report the choice without launching
    *query = p.sk ? p.groups : 0;
    return cudaSuccess;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3((kEpiWarps + 2) * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (cl > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = cl;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, mx, mw, p);
}

template <bool FP4, bool PAIR>
cudaError_t dispatch_k(const CUtensorMap& mx, const CUtensorMap& mw, const TcParams& p,
                       size_t smem, bool pdl, bool sk, cudaStream_t s, int* q) {
  // KC >= k + 2: the list keeps one key past the (k+1)-th, so a near tie at
  // the k / k+1 boundary can be settled inside the list
  const int k = p.a.k;
  if (k <= 2) return launch_kc<4, FP4, PAIR>(mx, mw, p, smem, pdl, sk, s, q);
  if (k <= 4) return launch_kc<6, FP4, PAIR>(mx, mw, p, smem, pdl, sk, s, q);
  if (k <= 6) return launch_kc<8, FP4, PAIR>(mx, mw, p, smem, pdl, sk, s, q);
  if (k <= 8) return launch_kc<10, FP4, PAIR>(mx, mw, p, smem, pdl, sk, s, q);
  return launch_kc<18, FP4, PAIR>(mx, mw, p, smem, pdl, sk, s, q);
}

}  // namespace

// One kernel family (all list capacities) per translation unit.
cudaError_t tc_dispatch_bf16_pair(const CUtensorMap& mx, const CUtensorMap& mw, const TcParams& p,
                                  size_t smem, bool pdl, bool sk, cudaStream_t s, int* q);
cudaError_t tc_dispatch_bf16_cta(const CUtensorMap& mx, const CUtensorMap& mw, const TcParams& p,
                                 size_t smem, bool pdl, bool sk, cudaStream_t s, int* q);
cudaError_t tc_dispatch_fp4_pair(const CUtensorMap& mx, const CUtensorMap& mw, const TcParams& p,
                                 size_t smem, bool pdl, bool sk, cudaStream_t s, int* q);
cudaError_t tc_dispatch_fp4_cta(const CUtensorMap& mx, const CUtensorMap& mw, const TcParams& p,
                                size_t smem, bool pdl, bool sk, cudaStream_t s, int* q);

}  // namespace gbr

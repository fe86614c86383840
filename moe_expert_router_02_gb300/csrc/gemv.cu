// Small-M (decode / verify widths) fused routers and the generic router.
//
// At M <= 64 the router reads W_gate (E x H BF16, 1-4 MiB) once and little
// else, so it is bound by HBM and by latency. W rows are bulk-copied into
// shared memory before each kernel waits on the preceding one (programmatic
// dependent launch), so back-to-back calls overlap their W streams with the
// previous call's tail. The contraction runs on the tensor cores with
// mma.sync m16n8k16 (experts as the 16-row operand, 8 tokens per n-tile).
// The logits are combined on chip in a fixed order (deterministic): inside
// one cluster of E/16 CTAs that holds all of W (single-cluster kernel), or
// over clusters that each hold a slice of H, through distributed shared
// memory and an L2-resident buffer with an arrival ticket (split-cluster
// kernel). Both are the "threadgroup-level reduction" option that qwisp
// issue #145 ("Change") leaves to measurement, with the E logits kept on
// chip or in L2 instead of a separate launch.
#include <cuda_bf16.h>

#include <map>
#include <mutex>
#include <tuple>

#include "kernels.h"
#include "select.cuh"

namespace gbr {
namespace {


__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

__device__ __forceinline__ float dsmem_ld_f32(const float* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(r));
  return v;
}

__device__ __forceinline__ void dsmem_st_u32(uint32_t* p, uint32_t rank, uint32_t v) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(r), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}

__device__ __forceinline__ void atom_exch_relaxed_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.exch.relaxed.gpu.global.b32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
}

// ---------------------------------------------------------------------------
// Single-cluster small-M router (M <= 64, E <= 256; one cluster per group
// of 4, 8 or 16 rows, each routing its rows on its own). One cluster of E/16
// CTAs holds all of W_gate in shared memory: CTA r owns experts
// [16r, 16r+16) over the whole H, so there are no partial sums to combine
// and no logits leave the cluster. Each CTA starts bulk copies of its 16 W
// rows (L2 evict-first: the weight stream must not push x or the kernel's
// code out of L2) before it waits on the preceding kernel (programmatic
// dependent launch); NVFP4 rows are decoded to BF16 in shared memory there
// too, when the copy fits. After the wait it reads x, runs the mma.sync
// contraction from shared memory and sums its warps' partials. Row m is
// selected by one CTA of the cluster (rows spread over the CTAs, a table's
// row pairs kept together): every CTA sends its 16 logits of row m to that
// CTA with st.async stores that complete on the receiver's mbarrier, whose
// expected byte count the receiver set at start. No global scratch, no
// atomics, no second cluster barrier.

#ifdef GBR_PHASE_STAMPS
// Measurement build only: %globaltimer stamps (ns) that thread 0 of each
// CTA of the single-cluster kernel's first row group takes at phase
// boundaries, kept for the last kStampCalls launches (slot = launch count of
// that CTA rank):
//   0 entry, 1 W copies issued and dependents released, 2 wait on the
//   preceding kernel returned, 3 W in shared memory, 4 warps' partials
//   stored, 5 logits sent, 6 (selecting CTAs) this CTA's rows landed,
//   7 row selected and stored.
constexpr int kStampCalls = 256, kStampPhases = 8;
__device__ unsigned long long g_stamps[kStampCalls][16][kStampPhases];
__device__ unsigned g_stamp_seq[16];
// The split-cluster kernel's stamps: [call slot][CTA = group * CL + rank]
// [phase], phases 0 entry, 1 W copy issued, 2 wait returned, 3 W in shared
// memory, 4 warps' partials stored, 5 slices ready (cluster barrier), 6 the
// cluster's logits stored, 7 cluster barrier, 8 ticket known to the
// cluster, 9 (last cluster) rows selected.
constexpr int kSplitStampCalls = 64, kSplitStampCtas = 128, kSplitStampPhases = 10;
__device__ unsigned long long g_split_stamps[kSplitStampCalls][kSplitStampCtas][kSplitStampPhases];
__device__ unsigned g_split_seq[kSplitStampCtas];
#define GBR_SPLIT_STAMP(slot, cta, i)                                       \
  do {                                                                      \
    if (threadIdx.x == 0 && (cta) < kSplitStampCtas) {                      \
      unsigned long long t_;                                                \
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_)::"memory");      \
      g_split_stamps[slot][cta][i] = t_;                                    \
    }                                                                       \
  } while (0)
#define GBR_STAMP(slot, i)                                                  \
  do {                                                                      \
    if (threadIdx.x == 0 && blockIdx.y == 0) {                              \
      unsigned long long t_;                                                \
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_)::"memory");      \
      g_stamps[slot][blockIdx.x][i] = t_;                                   \
    }                                                                       \
  } while (0)
#else
#define GBR_STAMP(slot, i) \
  do {                     \
  } while (0)
#define GBR_SPLIT_STAMP(slot, cta, i) \
  do {                                \
  } while (0)
#endif

constexpr int k1cWarps = 16;
constexpr int k1cBatch = 8;  // 32-element chunks of x held in registers per warp

constexpr int kMaxE1c = 256;
constexpr int kPartPitch = 20;  // floats per (warp, token) row of partials: 16 experts + pad

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 16 bytes into shared memory of a CTA of the cluster (shared::cluster
// address), completing 16 bytes of that CTA's mbarrier transaction count.
__device__ __forceinline__ void st_async_v4(uint32_t dst, float a, float b, float c, float d,
                                            uint32_t bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::
          "r"(dst),
      "f"(a), "f"(b), "f"(c), "f"(d), "r"(bar)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_parity(uint32_t bar, uint32_t parity) {
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

// Bounded wait (about one second of %globaltimer); false when it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, unsigned* status) {
  if (mbar_try_parity(bar, parity)) return true;
  uint64_t t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  while (!mbar_try_parity(bar, parity)) {
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 > 1000000000ull) {
      if (status) atomicOr(status, 1u);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ bool mbar_try_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait with cluster-scope acquire (about one second of %globaltimer).
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, unsigned* status) {
  if (mbar_try_cluster(bar, parity)) return true;
  uint64_t t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  while (!mbar_try_cluster(bar, parity)) {
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 > 1000000000ull) {
      if (status) atomicOr(status, 1u);
      return false;
    }
  }
  return true;
}

// Eight NVFP4 values (4 packed bytes, element 2j in the low nibble of byte j)
// times their E4M3 block scale, as four BF16 pairs in memory order. Exact:
// e2m1 * e4m3 has at most 6 significant bits and fits BF16's exponent range.
__device__ __forceinline__ uint4 fp4_frag(uint32_t packed, uint8_t scale_code, const uint32_t* lut) {
  const uint32_t sb = __float_as_uint(e4m3_to_f32(scale_code)) >> 16;
  const __nv_bfloat162 s2 = __halves2bfloat162(__ushort_as_bfloat16((unsigned short)sb),
                                               __ushort_as_bfloat16((unsigned short)sb));
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t pair = lut[(packed >> (8 * j)) & 0xffu];
    __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&pair);
    v = __hmul2(v, s2);
    o[j] = *reinterpret_cast<const uint32_t*>(&v);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Which CTA of the cluster selects row m, and in which of its row slots.
// Without a table row m goes to CTA m % CL; with one, the pair (2g, 2g+1)
// goes to CTA g % CL (the emitter needs both rows of a pair in one CTA).
struct RowOwner {
  int CL;
  bool table;
  uint32_t inv;  // (65536 + CL - 1) / CL: i / CL = (i * inv) >> 16 exactly for i < 512
  __device__ __forceinline__ int div(int i) const { return (int)(((uint32_t)i * inv) >> 16); }
  __device__ __forceinline__ int cta(int m) const {
    const int i = table ? m >> 1 : m;
    return i - CL * div(i);
  }
  __device__ __forceinline__ int slot(int m) const {
    return table ? 2 * div(m >> 1) + (m & 1) : div(m);
  }
  __device__ __forceinline__ int row(int c, int s) const {
    return table ? 2 * (c + CL * (s >> 1)) + (s & 1) : c + CL * s;
  }
  __device__ __forceinline__ int count(int c, int M) const {
    if (table) {
      const int pairs = M >> 1;
      return c < pairs ? 2 * ((pairs - c + CL - 1) / CL) : 0;
    }
    return c < M ? (M - c + CL - 1) / CL : 0;
  }
};

// Row groups: the single-cluster kernel runs one cluster per group of rows
// (blockIdx.y), each a complete router for its rows that stages all of W
// itself; this is the sub-problem of group rg (rows a multiple of 2, so a
// table's row pairs stay in one group).
constexpr int k1cMaxM = 64;
__device__ __forceinline__ RouterArgs row_group(RouterArgs a, int rg, int rows) {
  if (rg == 0 && a.M <= rows) return a;
  const int m0 = rows * rg;
  a.M = min(rows, a.M - m0);
  a.x = static_cast<const uint16_t*>(a.x) + (size_t)m0 * a.H;
  a.out_idx += (size_t)m0 * a.k;
  a.out_w += (size_t)m0 * a.k;
  if (a.logits) a.logits += (size_t)m0 * a.E;
  if (a.tbl_unique) {  // row pairs: m0 is even
    const size_t g0 = (size_t)(m0 / 2);
    a.tbl_unique += g0 * 2 * a.k;
    a.tbl_mask += g0 * 2 * a.k;
    a.tbl_map += g0 * 2 * a.k;
    a.tbl_count += g0;
  }
  return a;
}

// NVFP4 weights: the CTA stages its 16 packed rows (fpitch bytes apart) and
// their E4M3 block scales. With PREDEC the rows are decoded to BF16 in
// shared memory before the wait on the preceding kernel, so the contraction
// after it is the BF16 one; otherwise each 16-byte A fragment (8 BF16
// values) is decoded from 4 packed bytes as it is used. Either way the MMA
// sees W / g exactly (a byte -> two-BF16 table, one exact BF16 multiply by
// the block scale) and g multiplies the FP32 sums.
template <int NT, int VPL, bool FP4, bool PREDEC>
__device__ __forceinline__ void gemv1c_body(const RouterArgs& a, int pitch, int fpitch) {
  constexpr int NTOK = 8 * NT;
  constexpr bool kFrag4 = FP4 && !PREDEC;  // NVFP4 fragments decoded in the MMA loop
  // BF16 rows [16][pitch] (BF16 weights, or NVFP4 decoded there); NVFP4:
  // packed rows [16][fpitch] at fbase, then the block scales [16][H/16]
  extern __shared__ __align__(128) uint8_t s_w[];
  __shared__ uint32_t s_lut[FP4 ? 256 : 1];
  __shared__ __align__(16) float s_part[k1cWarps][NTOK][kPartPitch];
  __shared__ __align__(16) float s_all[16][kMaxE1c];  // logits of the rows this CTA selects
  __shared__ int32_t s_sel[k1cWarps * kMaxK];
  __shared__ __align__(8) uint64_t s_bar;   // this CTA's W rows have landed
  __shared__ __align__(8) uint64_t s_join;  // every logit of this CTA's rows has landed
  __shared__ float s_bias[kMaxE];           // the selection bias (CTAs that select)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int rank = blockIdx.x;  // one cluster spans the grid
  const int CL = gridDim.x;
  const int e0 = rank * 16;
  const int H = a.H, M = a.M, E = a.E;
  const bool table = a.tbl_unique != nullptr;
  const RowOwner own{CL, table, (65536u + (uint32_t)CL - 1u) / (uint32_t)CL};
  const int nown = own.count(rank, M);
  const uint32_t bar = smem_u32(&s_bar), join = smem_u32(&s_join);
  const uint32_t wsm = smem_u32(s_w);
#ifdef GBR_PHASE_STAMPS
  const int stamp = threadIdx.x == 0 && blockIdx.y == 0
                        ? (int)(atomicAdd(&g_stamp_seq[blockIdx.x], 1u) % kStampCalls)
                        : 0;
#endif
  GBR_STAMP(stamp, 0);

  const int row_bytes = FP4 ? H / 2 : H * 2;
  const int scale_bytes = FP4 ? 16 * (H / 16) : 0;
  const int fbase = PREDEC ? 16 * pitch : 0;  // packed NVFP4 rows
  const int spitch = FP4 ? fpitch : pitch;    // pitch of the staged rows
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(join) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"((uint32_t)(16 * row_bytes + scale_bytes))
                 : "memory");
    if (nown > 0)  // the other CTAs' stores complete this many bytes on it
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(join),
                   "r"((uint32_t)(nown * E * 4))
                   : "memory");
  }
  if (FP4) {
    for (int b = tid; b < 256; b += k1cWarps * 32) {
      const uint32_t lo = __float_as_uint(e2m1_to_f32(b & 15u)) >> 16;
      const uint32_t hi = __float_as_uint(e2m1_to_f32((uint32_t)b >> 4)) >> 16;
      s_lut[b] = lo | (hi << 16);
    }
  }
  __syncthreads();
  // publish the barriers' initialisation (the matching wait follows the W
  // copies' issue, before the wait on the preceding kernel)
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  if (tid < 17) {
    const uint64_t pol = policy_evict_first();
    if (tid < 16) {  // this CTA's 16 W rows, one bulk copy per row into the padded pitch
      const uint8_t* w = static_cast<const uint8_t*>(a.w) + (size_t)(e0 + tid) * row_bytes;
      bulk_g2s(wsm + fbase + tid * spitch, w, row_bytes, bar, pol);
    } else if (FP4) {  // the 16 rows of block scales are contiguous
      bulk_g2s(wsm + fbase + 16 * spitch, a.w_scales + (size_t)e0 * (H / 16), scale_bytes, bar,
               pol);
    }
  }
  // the bias is a weight: staged before the wait (read after a later
  // __syncthreads), so the selection does not wait on L2 for it
  if (a.bias && nown > 0)
    for (int e = tid; e < E; e += k1cWarps * 32) s_bias[e] = a.bias[e];
  pdl_launch_dependents();
  // every CTA of the cluster has initialised its barriers (they all arrived
  // above): the remote stores below may target them. Waiting here keeps the
  // cluster barrier off the chain that starts at the preceding kernel's end.
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  GBR_STAMP(stamp, 1);
  bool w_ok = true;
  if (PREDEC) {
    // W does not depend on the preceding kernel: decode it before the wait
    w_ok = mbar_wait_bounded(bar, 0, a.status);
    const int n8 = H / 8;  // 8-element chunks per row
    const uint8_t* sc = s_w + fbase + 16 * fpitch;
    for (int i = tid; i < 16 * n8; i += k1cWarps * 32) {
      const int r = i / n8, c8 = i - r * n8;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (w_ok)
        v = fp4_frag(*reinterpret_cast<const uint32_t*>(s_w + fbase + r * fpitch + c8 * 4),
                     sc[r * (H / 16) + (c8 >> 1)], s_lut);
      *reinterpret_cast<uint4*>(s_w + r * pitch + c8 * 16) = v;
    }
    __syncthreads();
  }
  pdl_wait();  // x and the outputs belong to the preceding kernel until here
  GBR_STAMP(stamp, 2);

  const uint16_t* __restrict__ x = static_cast<const uint16_t*>(a.x);
  const int nchunk = H / 32;
  const int cpw = warp < nchunk ? (nchunk - warp + k1cWarps - 1) / k1cWarps : 0;
  float acc[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.0f;
  const uint8_t* w0 = s_w + g * (kFrag4 ? fpitch : pitch) + (kFrag4 ? 4 : 16) * t;
  const uint8_t* w1 = w0 + 8 * (kFrag4 ? fpitch : pitch);
  const uint8_t* sc0 = s_w + 16 * fpitch + g * (H / 16) + (t >> 1);  // kFrag4 block scales
  const uint8_t* sc1 = sc0 + 8 * (H / 16);
  for (int jb = 0; jb < cpw; jb += k1cBatch) {
    uint4 xv[k1cBatch][NT];
#pragma unroll
    for (int i = 0; i < k1cBatch; ++i) {
      const int hoff = (warp + k1cWarps * (jb + i)) * 32 + 8 * t;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const int tok = n * 8 + g;
        xv[i][n] = make_uint4(0u, 0u, 0u, 0u);
        if (jb + i < cpw && tok < M)
          xv[i][n] = __ldg(reinterpret_cast<const uint4*>(x + (size_t)tok * H + hoff));
      }
    }
    if (!PREDEC && jb == 0) {
      w_ok = mbar_wait_bounded(bar, 0, a.status);  // x loads in flight
      GBR_STAMP(stamp, 3);
    }
#pragma unroll
    for (int i = 0; i < k1cBatch; ++i) {
      if (jb + i < cpw && w_ok) {
        const int c = warp + k1cWarps * (jb + i);
        uint4 wa, wb;
        if (kFrag4) {
          wa = fp4_frag(*reinterpret_cast<const uint32_t*>(w0 + c * 16), sc0[2 * c], s_lut);
          wb = fp4_frag(*reinterpret_cast<const uint32_t*>(w1 + c * 16), sc1[2 * c], s_lut);
        } else {
          wa = *reinterpret_cast<const uint4*>(w0 + c * 64);
          wb = *reinterpret_cast<const uint4*>(w1 + c * 64);
        }
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          mma_bf16_16816(acc[n], wa.x, wb.x, wa.y, wb.y, xv[i][n].x, xv[i][n].y);
          mma_bf16_16816(acc[n], wa.z, wb.z, wa.w, wb.w, xv[i][n].z, xv[i][n].w);
        }
      }
    }
  }
  if (!PREDEC && cpw == 0) mbar_wait_bounded(bar, 0, a.status);  // never leave with copies in flight
  // accumulator layout: c0,c1 -> expert g, tokens 2t, 2t+1; c2,c3 -> expert g+8
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    s_part[warp][n * 8 + 2 * t][g] = acc[n][0];
    s_part[warp][n * 8 + 2 * t + 1][g] = acc[n][1];
    s_part[warp][n * 8 + 2 * t][g + 8] = acc[n][2];
    s_part[warp][n * 8 + 2 * t + 1][g + 8] = acc[n][3];
  }
  __syncthreads();
  GBR_STAMP(stamp, 4);
  // sum the warps' partials in a fixed order; four experts of a row per
  // thread go to the CTA that selects the row
  for (int i = tid; i < 4 * M; i += k1cWarps * 32) {
    const int m = i >> 2, q = i & 3;
    float4 u[k1cWarps];
#pragma unroll
    for (int w = 0; w < k1cWarps; ++w) u[w] = *reinterpret_cast<const float4*>(&s_part[w][m][4 * q]);
#pragma unroll
    for (int h = k1cWarps / 2; h > 0; h >>= 1) {  // a fixed tree: warp w + warp w + h
#pragma unroll
      for (int w = 0; w < h; ++w) {
        u[w].x += u[w + h].x, u[w].y += u[w + h].y;
        u[w].z += u[w + h].z, u[w].w += u[w + h].w;
      }
    }
    float4 v = u[0];
    if (FP4) {
      v.x *= a.w_global, v.y *= a.w_global, v.z *= a.w_global, v.w *= a.w_global;
    }
    if (a.logits) {
      float* lg = a.logits + (size_t)m * E + e0 + 4 * q;
      lg[0] = v.x, lg[1] = v.y, lg[2] = v.z, lg[3] = v.w;
    }
    const uint32_t dst_cta = (uint32_t)own.cta(m);
    uint32_t dst, dbar;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(dst)
                 : "r"(smem_u32(&s_all[own.slot(m)][e0 + 4 * q])), "r"(dst_cta));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(dbar) : "r"(join), "r"(dst_cta));
    st_async_v4(dst, v.x, v.y, v.z, v.w, dbar);
  }
  GBR_STAMP(stamp, 5);
  if (nown == 0) return;  // no row to select; no CTA reads this one's shared memory
  if (!mbar_wait_cluster(join, 0, a.status)) return;
  GBR_STAMP(stamp, 6);

  // warp s selects the CTA's row slot s; rows 2g and 2g+1 of a table's pair
  // sit in slots 2p and 2p + 1
  const int k = a.k;
  const int row = own.row(rank, warp);
  if (warp < nown)
    warp_select_row<VPL>(LdPlain{&s_all[warp][0]}, a.bias ? s_bias : nullptr, E, k, a.act,
                         a.out_idx + (size_t)row * k, a.out_w + (size_t)row * k,
                         s_sel + warp * k);
  GBR_STAMP(stamp, 7);
  if (table) {
    __syncthreads();
    if ((warp & 1) == 0 && warp + 1 < nown) {
      const size_t gi = (size_t)(row >> 1);
      warp_route_table_small(s_sel + warp * k, 2, k, a.tbl_unique + gi * 2 * k,
                             a.tbl_mask + gi * 2 * k, a.tbl_map + gi * 2 * k, a.tbl_count + gi);
    }
  }
}

// One cluster (one row group): the body reads the launch parameters in place.
template <int NT, int VPL, bool FP4, bool PREDEC>
__global__ void __launch_bounds__(k1cWarps * 32)
    k_gemv1c_router(const RouterArgs a, int pitch, int fpitch) {
  gemv1c_body<NT, VPL, FP4, PREDEC>(a, pitch, fpitch);
}

// A cluster per group of `rows` rows: each cluster takes its row group's
// sub-problem (a copy of the parameters with its rows' pointers).
template <int NT, int VPL, bool FP4, bool PREDEC>
__global__ void __launch_bounds__(k1cWarps * 32)
    k_gemv1c_router_rows(const RouterArgs a, int pitch, int fpitch, int rows) {
  const RouterArgs g = row_group(a, (int)blockIdx.y, rows);
  gemv1c_body<NT, VPL, FP4, PREDEC>(g, pitch, fpitch);
}


// ---------------------------------------------------------------------------
// Split-cluster small-M router (M <= 64; used where the single-cluster
// kernel is not, and for the logits-only half of the unfused A/B pair).
// CTA (r, eg) owns expert group eg (16 experts) and the r-th of CL slices
// of H; the CL CTAs of an expert group form a cluster. Each CTA bulk-copies
// its 16 x H/CL slice of W into shared memory (L2 evict-first) before it
// waits on the preceding kernel. Its 8 warps split the work by token tile
// and chunk group: warp w takes the 8-token tile w % NT over every
// (8/NT)-th 32-element chunk of the slice, so each warp issues all of its
// x loads at once. The cluster sums its H slices over distributed shared
// memory in a fixed order and writes the 16 x M logits to an L2-resident
// buffer [M, E] (or the caller's logits tap); the cluster that arrives last
// on a ticket selects, one warp per row across its CTAs, and resets the
// ticket. The K permutation inside a 32-element chunk is the one of the
// single-cluster kernel: thread t of a quad owns elements [8t, 8t+8), and
// for MMA j its logical k slots {2t, 2t+1, 2t+8, 2t+9} are the physical
// elements 8t + 4j + {0,1,2,3}, the same for W (A) and x (B).
constexpr int kSplitWarps = 8;  // two CTAs fit an SM: the next call's CTAs can start early

template <int NT, int VPL, bool SELECT>
__global__ void __launch_bounds__(kSplitWarps * 32)
    k_gemv_router(const RouterArgs a, int CL, int pitch) {
  constexpr int NTOK = 8 * NT;
  constexpr int NG = kSplitWarps / NT;  // chunk groups: warps per token tile
  constexpr int kSplitXB = NG == 1 ? 16 : 8;  // x chunks per warp held in registers at once
  extern __shared__ __align__(128) uint8_t s_w[];  // [16][pitch]: this CTA's W slice
  __shared__ float s_part[NG][16][NTOK];
  __shared__ float s_cta[16][NTOK];
  __shared__ int32_t s_sel[kSplitWarps * kMaxK];
  __shared__ float s_bias[SELECT ? kMaxE : 1];  // the selection bias
  __shared__ uint32_t s_flag;
  __shared__ __align__(8) uint64_t s_bar;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int rank = blockIdx.x;  // the grid's x extent equals the cluster size
  const int e0 = blockIdx.y * 16;
  const int H = a.H, M = a.M, E = a.E;
  const int Hc = H / CL, nchunk = Hc / 32, h_begin = rank * Hc;
  const int tile = warp % NT, cg = warp / NT;
  const uint32_t bar = smem_u32(&s_bar);
#ifdef GBR_PHASE_STAMPS
  const int scta = blockIdx.y * CL + rank;
  const int sslot = (threadIdx.x == 0 && scta < kSplitStampCtas)
                        ? (int)(atomicAdd(&g_split_seq[scta], 1u) % kSplitStampCalls)
                        : 0;
#endif
  GBR_SPLIT_STAMP(sslot, scta, 0);

  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"((uint32_t)(16 * Hc * 2))
                 : "memory");
  }
  __syncthreads();
  if (tid < 16) {  // row tid of the slice: H/CL contiguous BF16 values
    const uint16_t* src = static_cast<const uint16_t*>(a.w) + (size_t)(e0 + tid) * H + h_begin;
    bulk_g2s(smem_u32(s_w) + tid * pitch, src, (uint32_t)(Hc * 2), bar, policy_evict_first());
  }
  // any cluster may arrive last: each stages the bias (a weight) before the
  // wait; a later __syncthreads orders it before the selection
  if (SELECT && a.bias)
    for (int e = tid; e < E; e += kSplitWarps * 32) s_bias[e] = a.bias[e];
  pdl_launch_dependents();
  GBR_SPLIT_STAMP(sslot, scta, 1);
  pdl_wait();  // x, the scratch and the ticket belong to the preceding call until here
  GBR_SPLIT_STAMP(sslot, scta, 2);

  const uint16_t* __restrict__ x = static_cast<const uint16_t*>(a.x);
  const int tok = tile * 8 + g;
  const uint8_t* w0 = s_w + g * pitch + 16 * t;
  const uint8_t* w1 = w0 + 8 * pitch;
  // two accumulators (even and odd chunks of a batch) halve the chain of
  // dependent MMAs; they are added once at the end
  float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f}, acc2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  bool w_ok = true, waited = false;
  for (int cb = cg; cb < nchunk; cb += NG * kSplitXB) {
    uint4 xv[kSplitXB];
#pragma unroll
    for (int i = 0; i < kSplitXB; ++i) {
      const int c = cb + NG * i;
      xv[i] = make_uint4(0u, 0u, 0u, 0u);
      if (c < nchunk && tok < M)
        xv[i] = __ldg(reinterpret_cast<const uint4*>(x + (size_t)tok * H + h_begin + c * 32 + 8 * t));
    }
    if (!waited) {  // the x loads are in flight meanwhile
      w_ok = mbar_wait_bounded(bar, 0, a.status);
      waited = true;
      GBR_SPLIT_STAMP(sslot, scta, 3);
    }
#pragma unroll
    for (int i = 0; i < kSplitXB; ++i) {
      const int c = cb + NG * i;
      if (c < nchunk && w_ok) {
        const uint4 wa = *reinterpret_cast<const uint4*>(w0 + c * 64);
        const uint4 wb = *reinterpret_cast<const uint4*>(w1 + c * 64);
        float (&ac)[4] = (i & 1) ? acc2 : acc;
        mma_bf16_16816(ac, wa.x, wb.x, wa.y, wb.y, xv[i].x, xv[i].y);
        mma_bf16_16816(ac, wa.z, wb.z, wa.w, wb.w, xv[i].z, xv[i].w);
      }
    }
  }
  if (!waited) mbar_wait_bounded(bar, 0, a.status);  // never leave with the copy in flight
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j] += acc2[j];

  // accumulator layout: c0,c1 -> expert g, tokens 2t, 2t+1; c2,c3 -> expert g+8
  s_part[cg][g][tile * 8 + 2 * t] = acc[0];
  s_part[cg][g][tile * 8 + 2 * t + 1] = acc[1];
  s_part[cg][g + 8][tile * 8 + 2 * t] = acc[2];
  s_part[cg][g + 8][tile * 8 + 2 * t + 1] = acc[3];
  __syncthreads();
  GBR_SPLIT_STAMP(sslot, scta, 4);
  for (int i = tid; i < 16 * NTOK; i += kSplitWarps * 32) {
    const int el = i / NTOK, m = i % NTOK;
    float v = s_part[0][el][m];
#pragma unroll
    for (int q = 1; q < NG; ++q) v += s_part[q][el][m];
    s_cta[el][m] = v;
  }
  cluster_sync_all();
  GBR_SPLIT_STAMP(sslot, scta, 5);

  // cluster reduction over the CL slices of H; item i = m * 16 + el
  for (int i = rank + CL * tid; i < 16 * M; i += CL * kSplitWarps * 32) {
    const int m = i >> 4, el = i & 15;
    float part[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) part[q] = q < CL ? dsmem_ld_f32(&s_cta[el][m], (uint32_t)q) : 0.0f;
    float v = part[0];
#pragma unroll
    for (int q = 1; q < 8; ++q) v += part[q];  // fixed order; absent slices add +0
    a.logits[(size_t)m * E + e0 + el] = v;
  }
  if (!SELECT) {
    cluster_sync_all();  // keep shared memory alive until every peer has read it
    return;
  }
  GBR_SPLIT_STAMP(sslot, scta, 6);
  // The cluster barrier (release/acquire) orders every peer's logits stores
  // before rank 0's acq_rel arrival on the ticket; the arrivals form one
  // release sequence, so the cluster that arrives last observes all logits
  // and hands them to its peers through the next cluster barrier.
  cluster_sync_all();
  GBR_SPLIT_STAMP(sslot, scta, 7);
  if (rank == 0 && tid == 0) {
    const uint32_t old = atom_add_acq_rel_gpu(a.ticket, 1u);
    const uint32_t last = (old == gridDim.y - 1) ? 1u : 0u;
    if (last) atom_exch_relaxed_gpu(a.ticket, 0u);
    for (int q = 0; q < CL; ++q) dsmem_st_u32(&s_flag, (uint32_t)q, last);
  }
  cluster_sync_all();
  GBR_SPLIT_STAMP(sslot, scta, 8);
  if (!s_flag) return;

  // the last cluster selects: warp w of CTA r takes rows r*8 + w, then
  // every CL*8 rows further; rows 2p and 2p+1 share a CTA
  const bool table = a.tbl_unique != nullptr;
  const int k = a.k;
  for (int base = rank * kSplitWarps; base < M; base += CL * kSplitWarps) {
    const int row = base + warp;
    if (row < M)
      warp_select_row<VPL>(LdCG{a.logits + (size_t)row * E}, a.bias ? s_bias : nullptr, E, k,
                           a.act,
                           a.out_idx + (size_t)row * k, a.out_w + (size_t)row * k,
                           s_sel + warp * k);
    if (table) {
      __syncthreads();
      if ((warp & 1) == 0 && row + 1 < M) {
        const size_t gi = (size_t)(row >> 1);
        warp_route_table_small(s_sel + warp * k, 2, k, a.tbl_unique + gi * 2 * k,
                               a.tbl_mask + gi * 2 * k, a.tbl_map + gi * 2 * k, a.tbl_count + gi);
      }
      __syncthreads();
    }
  }
  GBR_SPLIT_STAMP(sslot, scta, 9);
}

// Generic router: one CTA per row (two rows when a table is fused), any
// dtype, any H. W is decoded element by element (NVFP4: e2m1 * e4m3, the
// global scale applied to the FP32 sum). Each expert's dot product is a
// fixed per-lane FMA order followed by a fixed butterfly.
constexpr int kGenWarps = 8;

__device__ __forceinline__ float x_at(const RouterArgs& a, size_t i) {
  return a.x_dtype == DT_F32 ? static_cast<const float*>(a.x)[i]
                             : bf16_bits_to_f32(static_cast<const uint16_t*>(a.x)[i]);
}

__device__ __forceinline__ float w_at(const RouterArgs& a, int e, int h) {
  if (a.w_dtype == DT_F32) return static_cast<const float*>(a.w)[(size_t)e * a.H + h];
  if (a.w_dtype == DT_BF16)
    return bf16_bits_to_f32(static_cast<const uint16_t*>(a.w)[(size_t)e * a.H + h]);
  const uint32_t byte = static_cast<const uint8_t*>(a.w)[(size_t)e * (a.H / 2) + h / 2];
  const uint32_t code = (h & 1) ? (byte >> 4) : (byte & 15u);
  return e2m1_to_f32(code) * e4m3_to_f32(a.w_scales[(size_t)e * (a.H / 16) + h / 16]);
}

template <int VPL>
__global__ void __launch_bounds__(kGenWarps * 32) k_generic_router(const RouterArgs a, int rows) {
  __shared__ float s_log[2][kMaxE];
  __shared__ int32_t s_sel[2 * kMaxK];
  pdl_launch_dependents();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = blockIdx.x * rows;
  const int M = a.M, H = a.H, E = a.E, k = a.k;
  for (int r = 0; r < rows; ++r) {
    const int m = row0 + r;
    if (m >= M) break;
    for (int e = warp; e < E; e += kGenWarps) {
      float acc = 0.0f;
      for (int h = lane; h < H; h += 32) acc = fmaf(x_at(a, (size_t)m * H + h), w_at(a, e, h), acc);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(kFull, acc, off);
      if (lane == 0) {
        const float l = (a.w_dtype == DT_NVFP4) ? acc * a.w_global : acc;
        s_log[r][e] = l;
        if (a.logits) a.logits[(size_t)m * E + e] = l;
      }
    }
  }
  __syncthreads();
  if (warp < rows && row0 + warp < M) {
    const size_t m = (size_t)(row0 + warp);
    warp_select_row<VPL>(LdPlain{s_log[warp]}, a.bias, E, k, a.act, a.out_idx + m * k,
                         a.out_w + m * k, s_sel + warp * k);
  }
  __syncthreads();
  if (a.tbl_unique && rows == 2 && warp == 0 && row0 + 1 < M) {
    const size_t gi = (size_t)(row0 >> 1);
    warp_route_table_small(s_sel, 2, k, a.tbl_unique + gi * 2 * k, a.tbl_mask + gi * 2 * k,
                           a.tbl_map + gi * 2 * k, a.tbl_count + gi);
  }
}

template <class Kern>
cudaError_t launch_ex(Kern kern, dim3 grid, dim3 block, int cluster, bool pdl, cudaStream_t stream,
                      const RouterArgs& a, int extra) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int n = 0;
  if (cluster > 1) {
    attrs[n].id = cudaLaunchAttributeClusterDimension;
    attrs[n].val.clusterDim.x = cluster;
    attrs[n].val.clusterDim.y = 1;
    attrs[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl) {
    attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, a, extra);
}

// Row pitch of a CTA's W slice (H/CL BF16 values per row), padded to 64
// (mod 128) bytes like the single-cluster kernel's rows.
int split_pitch(int Hc) { return 2 * Hc + ((2 * Hc) % 128 == 0 ? 64 : 0); }

template <class Kern>
cudaError_t launch_split(Kern kern, const RouterArgs& a, int CL, bool pdl, cudaStream_t stream) {
  const int pitch = split_pitch(a.H / CL);
  const size_t dsmem = (size_t)16 * pitch;
  if (dsmem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)dsmem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL, a.E / 16);
  cfg.blockDim = dim3(kSplitWarps * 32);
  cfg.dynamicSmemBytes = dsmem;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int n = 0;
  attrs[n].id = cudaLaunchAttributeClusterDimension;
  attrs[n].val.clusterDim.x = CL;
  attrs[n].val.clusterDim.y = 1;
  attrs[n].val.clusterDim.z = 1;
  ++n;
  if (pdl) {
    attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, a, CL, pitch);
}

template <int NT, bool SELECT>
cudaError_t gemv_dispatch_vpl(const RouterArgs& a, int CL, bool pdl, cudaStream_t s) {
  if (a.E <= 128) return launch_split(k_gemv_router<NT, 4, SELECT>, a, CL, pdl, s);
  if (a.E <= 256) return launch_split(k_gemv_router<NT, 8, SELECT>, a, CL, pdl, s);
  return launch_split(k_gemv_router<NT, 16, SELECT>, a, CL, pdl, s);
}

template <bool SELECT>
cudaError_t gemv_dispatch(const RouterArgs& a, int CL, bool pdl, cudaStream_t s) {
  if (a.M <= 8) return gemv_dispatch_vpl<1, SELECT>(a, CL, pdl, s);
  if (a.M <= 16) return gemv_dispatch_vpl<2, SELECT>(a, CL, pdl, s);
  if (a.M <= 32) return gemv_dispatch_vpl<4, SELECT>(a, CL, pdl, s);
  return gemv_dispatch_vpl<8, SELECT>(a, CL, pdl, s);
}

// Row pitch of the staged W rows: BF16 rows padded to 64 (mod 128) bytes and
// NVFP4 rows to 16 (mod 32) bytes, which keeps the fragment loads free of
// bank conflicts.
int gemv1c_pitch(int H) { return 2 * H + ((2 * H) % 128 == 0 ? 64 : 0); }
int gemv1c_fpitch(int H) { return H / 2 + ((H / 2) % 32 == 16 ? 0 : 16); }

// Dynamic shared memory of the single-cluster kernel: BF16 rows, NVFP4 packed
// rows and scales, or both when NVFP4 rows are decoded before the wait.
size_t gemv1c_smem(int H, bool fp4, bool predec) {
  const size_t bf = (size_t)16 * gemv1c_pitch(H);
  const size_t f4 = (size_t)16 * gemv1c_fpitch(H) + (size_t)16 * (H / 16);
  return fp4 ? (predec ? bf + f4 : f4) : bf;
}

constexpr size_t k1cMaxDynSmem = 180 * 1024;  // leaves room for the static arrays (about 40 KB)

// NVFP4 rows are decoded before the wait whenever both copies fit.
bool gemv1c_predec(int H) { return gemv1c_smem(H, true, true) <= k1cMaxDynSmem; }

// Launches (or, with probe, only sizes) the single-cluster kernel.
template <int NT, int VPL, bool FP4, bool PREDEC>
cudaError_t launch_1c_inst(const RouterArgs& a, int rows, bool pdl, cudaStream_t stream,
                           bool probe, bool* fits) {
  const bool grouped = a.M > rows;
  const int CL = a.E / 16;
  const size_t dsmem = gemv1c_smem(a.H, FP4, PREDEC);
  const void* kern = grouped ? (const void*)k_gemv1c_router_rows<NT, VPL, FP4, PREDEC>
                             : (const void*)k_gemv1c_router<NT, VPL, FP4, PREDEC>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)dsmem);
  if (e != cudaSuccess) return e;
  if (CL > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL, (a.M + rows - 1) / rows);  // a cluster per row group
  cfg.blockDim = dim3(k1cWarps * 32);
  cfg.dynamicSmemBytes = dsmem;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = CL;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = pdl ? 2 : 1;
  if (probe) {
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    *fits = (e == cudaSuccess && n > 0);
    return cudaSuccess;
  }
  const int pitch = gemv1c_pitch(a.H), fpitch = gemv1c_fpitch(a.H);
  if (grouped)
    return cudaLaunchKernelEx(&cfg, k_gemv1c_router_rows<NT, VPL, FP4, PREDEC>, a, pitch, fpitch,
                              rows);
  return cudaLaunchKernelEx(&cfg, k_gemv1c_router<NT, VPL, FP4, PREDEC>, a, pitch, fpitch);
}

template <int NT, bool FP4, bool PREDEC>
cudaError_t launch_1c_vpl(const RouterArgs& a, int rows, bool pdl, cudaStream_t s, bool probe,
                          bool* fits) {
  if (a.E <= 128) return launch_1c_inst<NT, 4, FP4, PREDEC>(a, rows, pdl, s, probe, fits);
  return launch_1c_inst<NT, 8, FP4, PREDEC>(a, rows, pdl, s, probe, fits);
}

template <int NT>
cudaError_t launch_1c_nt(const RouterArgs& a, int rows, bool pdl, cudaStream_t s, bool probe,
                         bool* fits) {
  if (a.w_dtype != DT_NVFP4) return launch_1c_vpl<NT, false, false>(a, rows, pdl, s, probe, fits);
  if (gemv1c_predec(a.H)) return launch_1c_vpl<NT, true, true>(a, rows, pdl, s, probe, fits);
  return launch_1c_vpl<NT, true, false>(a, rows, pdl, s, probe, fits);
}

// Rows per cluster. Every CTA of a cluster reads all of its rows' x from L2
// (about 0.1 TB/s per SM), so fewer rows per cluster shorten the dependent
// chain, but a call of eight clusters (128 CTAs) took about twice as long as
// one of four: BF16 takes four rows up to six clusters, then eight rows up
// to four clusters, then sixteen. NVFP4 W, whose rows are decoded before
// the wait, lost from four clusters on (the fewer calls fit the GPU at
// once, the less time a call has to stage and decode W before its
// predecessor ends): four rows up to two clusters, eight up to three, then
// sixteen (all measured on GB300 at M = 1..64). Four and eight rows take one
// token tile (NT = 1), sixteen two.
int rows_per_cluster(int M, bool fp4) {
  if (fp4) return M <= 8 ? 4 : M <= 24 ? 8 : 16;
  return M <= 24 ? 4 : M <= 32 ? 8 : 16;
}

cudaError_t launch_1c(const RouterArgs& a, bool pdl, cudaStream_t s, bool probe, bool* fits) {
  const int rows = rows_per_cluster(a.M, a.w_dtype == DT_NVFP4);
  return rows <= 8 ? launch_1c_nt<1>(a, rows, pdl, s, probe, fits)
                   : launch_1c_nt<2>(a, rows, pdl, s, probe, fits);
}

}  // namespace

bool gemv1c_eligible(int M, int H, int E, bool fp4) {
  if (M < 1 || M > k1cMaxM || E % 16 != 0 || E < 16 || E > 256 || H % (fp4 ? 256 : 32) != 0)
    return false;
  if (gemv1c_smem(H, fp4, fp4 && gemv1c_predec(H)) > k1cMaxDynSmem) return false;
  // the cluster must be schedulable with this much shared memory per CTA
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int>, bool> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const auto key = std::make_tuple(dev, 2 * rows_per_cluster(M, fp4) + (fp4 ? 1 : 0), E, H);  // one cluster's fit
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  RouterArgs probe_args{};
  probe_args.M = M, probe_args.H = H, probe_args.E = E;
  probe_args.w_dtype = fp4 ? DT_NVFP4 : DT_BF16;
  bool fits = false;
  if (launch_1c(probe_args, true, 0, true, &fits) != cudaSuccess) fits = false;
  (void)cudaGetLastError();
  cache[key] = fits;
  return fits;
}

#ifdef GBR_PHASE_STAMPS
// The split-cluster kernel's stamps [kSplitStampCalls][kSplitStampCtas]
// [kSplitStampPhases], copied to host memory; the launch counters cleared.
extern "C" int router_split_phase_stamps(unsigned long long* host, int* calls, int* ctas,
                                         int* phases) {
  *calls = kSplitStampCalls, *ctas = kSplitStampCtas, *phases = kSplitStampPhases;
  if (!host) return 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return 3;
  if (cudaMemcpyFromSymbol(host, g_split_stamps, sizeof(g_split_stamps)) != cudaSuccess) return 3;
  static const unsigned zero[kSplitStampCtas] = {};
  return cudaMemcpyToSymbol(g_split_seq, zero, sizeof(zero)) == cudaSuccess ? 0 : 3;
}

// Copies the stamps [kStampCalls][16][kStampPhases] to host memory and
// clears the launch counters (measurement build only).
extern "C" int router_phase_stamps(unsigned long long* host, int* calls, int* ctas, int* phases) {
  *calls = kStampCalls, *ctas = 16, *phases = kStampPhases;
  if (!host) return 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return 3;
  if (cudaMemcpyFromSymbol(host, g_stamps, sizeof(g_stamps)) != cudaSuccess) return 3;
  // the last selection's sub-phase stamps of each CTA rank follow
  if (cudaMemcpyFromSymbol(host + kStampCalls * 16 * kStampPhases, g_sel_stamps,
                           sizeof(g_sel_stamps)) != cudaSuccess)
    return 3;
  // then the re-rank counts since the last call (rows re-ranked, rows
  // taken to FP64, rows whose 32-bit rounds ran again on (key, index)
  // pairs), which restart from zero
  if (cudaMemcpyFromSymbol(host + kStampCalls * 16 * kStampPhases + 16 * 5, g_sel_refines,
                           sizeof(g_sel_refines)) != cudaSuccess)
    return 3;
  static const unsigned long long zr[3] = {};
  if (cudaMemcpyToSymbol(g_sel_refines, zr, sizeof(zr)) != cudaSuccess) return 3;
  static const unsigned zero[16] = {};
  return cudaMemcpyToSymbol(g_stamp_seq, zero, sizeof(zero)) == cudaSuccess ? 0 : 3;
}
#endif

cudaError_t launch_gemv1c(const RouterArgs& a, bool pdl, cudaStream_t stream) {
  bool unused = false;
  return launch_1c(a, pdl, stream, false, &unused);
}

int gemv_cluster_size(int H) {
  for (int cl = 8; cl > 1; cl >>= 1)
    if (H % (32 * cl) == 0) return cl;
  return 1;
}

cudaError_t launch_gemv(const RouterArgs& a, bool select, bool pdl, cudaStream_t stream) {
  const int CL = gemv_cluster_size(a.H);
  return select ? gemv_dispatch<true>(a, CL, pdl, stream) : gemv_dispatch<false>(a, CL, pdl, stream);
}

cudaError_t launch_generic(const RouterArgs& a, bool pdl, cudaStream_t stream) {
  const int rows = a.tbl_unique ? 2 : 1;
  const dim3 grid((a.M + rows - 1) / rows), block(kGenWarps * 32);
  if (a.E <= 32) return launch_ex(k_generic_router<1>, grid, block, 1, pdl, stream, a, rows);
  if (a.E <= 64) return launch_ex(k_generic_router<2>, grid, block, 1, pdl, stream, a, rows);
  if (a.E <= 128) return launch_ex(k_generic_router<4>, grid, block, 1, pdl, stream, a, rows);
  if (a.E <= 256) return launch_ex(k_generic_router<8>, grid, block, 1, pdl, stream, a, rows);
  return launch_ex(k_generic_router<16>, grid, block, 1, pdl, stream, a, rows);
}

}  // namespace gbr

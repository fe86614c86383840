// Large-M (prefill) fused router: host side. Tensor maps, the stream-K
// plan, the workspace layout, the launch (the kernel itself is in
// tc_kernel.cuh, instantiated by the tc_*.cu files) and the device status
// word every bounded wait reports to.
#include <cuda.h>
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <tuple>

#include "tc_kernel.cuh"

namespace gbr {

// bit 0 set when a bounded wait of a prefill kernel gave up (the kernels
// receive its address in RouterArgs::status)
static __device__ unsigned g_tc_status = 0;

#ifdef GBR_PHASE_STAMPS
// measurement build: the last prefill launch's phase stamps per CTA
constexpr int kTcStampCtas = 160;
static __device__ unsigned long long g_tc_stamps[kTcStampCtas * kTcStamps];

unsigned long long* tc_stamp_buffer() {
  void* p = nullptr;
  return cudaGetSymbolAddress(&p, g_tc_stamps) == cudaSuccess
             ? static_cast<unsigned long long*>(p)
             : nullptr;
}
#endif

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &p, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D BF16 tensor [rows, cols] row-major, box [box_rows, 64], 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* ptr, int rows, int cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kSkMaxCtas = 160;    // stream-K flag and partial slots in the workspace
constexpr int kSkMinRows = 256;    // smaller M gets no partial slots
constexpr int kSkMaxParts = 3;     // partials a finishing group may add

// Largest number of other groups holding units of one tile when U = tiles *
// nk units are split evenly over G groups (the group owning unit u is
// ceil((u + 1) G / U) - 1).
int sk_max_parts(int tiles, int nk, int G) {
  const long long U = (long long)tiles * nk;
  auto owner = [&](long long u) { return (int)(((u + 1) * G + U - 1) / U - 1); };
  int mx = 0;
  for (int t = 0; t < tiles; ++t) {
    const int n = owner((long long)(t + 1) * nk - 1) - owner((long long)t * nk);
    mx = n > mx ? n : mx;
  }
  return mx;
}

// The most groups, up to G, that split U = tiles * nk units with no tile
// over more than kSkMaxParts + 1 groups and every range non-empty (0: none,
// more groups than tiles being the point). Cached: a launch only looks it up.
}  // namespace

int tc_sk_groups_for(int tiles, int nk, int G) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int>, int> cache;
  std::lock_guard<std::mutex> lk(mu);
  const auto key = std::make_tuple(tiles, nk, G);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int g = G;
  if ((long long)tiles * nk < g) g = (int)((long long)tiles * nk);
  while (g > tiles && sk_max_parts(tiles, nk, g) > kSkMaxParts) --g;
  const int r = g > tiles ? g : 0;
  cache[key] = r;
  return r;
}

// Work groups that are resident at once, one CTA (or pair) per SM at most;
// the stream-K finishers wait for other groups' partials, so the whole grid
// has to fit. Cached per kernel, shared-memory size and device.
int tc_sk_resident_groups(const void* kern, size_t smem, int cl) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, size_t, int>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lk(mu);
  const auto key = std::make_tuple(kern, smem, dev);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int sms = 0, n = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) sms = 0;
  if (cl > 1) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cl);
    cfg.blockDim = dim3((kEpiWarps + 2) * 32);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeClusterDimension;
    at.val.clusterDim.x = cl;
    at.val.clusterDim.y = 1;
    at.val.clusterDim.z = 1;
    cfg.attrs = &at;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  } else {
    int per = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kern, (kEpiWarps + 2) * 32, smem) !=
        cudaSuccess)
      per = 0;
    n = per * sms;
  }
  (void)cudaGetLastError();  // a failed query leaves no sticky error
  if (n > sms / cl) n = sms / cl;
  if (n > kSkMaxCtas / cl) n = kSkMaxCtas / cl;
  cache[key] = n;
  return n;
}


bool tc_eligible(int M, int H, int E, int k, int x_dtype, int w_dtype) {
  return M >= 1 && x_dtype == DT_BF16 && (w_dtype == DT_BF16 || w_dtype == DT_NVFP4) &&
         E % 16 == 0 && E >= 16 && E <= 256 && H % BK == 0 && k <= kMaxK;
}

// Workspace. The small-M kernels' ticket and logits may share it (one
// library workspace per stream), so the prefill kernel's part starts past
// their largest extent: words [0] claim / arrival counter, [1] epoch,
// [2, 2 + H/64) NVFP4 column-block flags, then the stream-K flags; from the
// next 256-byte boundary the stream-K partial accumulators (M >=
// kSkMinRows), then the decoded NVFP4 W. Every flag holds the epoch + 1 of
// the launch that set it, and the epoch only grows, so no stale flag
// matches a later launch.
static size_t tc_flag_bytes(int H) {
  return ((size_t)(2 + H / BK + kSkMaxCtas) * 4 + 255) / 256 * 256;
}

static bool tc_sk_sized(int M) { return M >= kSkMinRows; }

static size_t tc_part_bytes(int E) { return (size_t)kSkMaxCtas * E * BM * 4; }

size_t tc_workspace(int M, int H, int E, int w_dtype) {
  const bool fp4 = w_dtype == DT_NVFP4, sk = tc_sk_sized(M);
  if (!fp4 && !sk) return 0;
  return kSmallMScratchBytes + tc_flag_bytes(H) + (sk ? tc_part_bytes(E) : 0) +
         (fp4 ? (size_t)E * H * 2 : 0);
}

cudaError_t launch_tc(const RouterArgs& a, bool pdl, cudaStream_t stream, int* query) {
  const bool fp4 = a.w_dtype == DT_NVFP4;
  TcParams p{};
  p.a = a;
  if (fp4 && !a.ticket) return cudaErrorInvalidValue;
  const bool sk_ws = a.ticket && tc_sk_sized(a.M);
  if (a.ticket && !query) {  // a query only needs to know a workspace is there
    uint8_t* ws = reinterpret_cast<uint8_t*>(a.ticket) + kSmallMScratchBytes;
    p.wsync = reinterpret_cast<unsigned*>(ws);
    p.sk_flag = p.wsync + 2 + a.H / BK;
    p.sk_part = sk_ws ? reinterpret_cast<float*>(ws + tc_flag_bytes(a.H)) : nullptr;
    if (fp4) p.wdec = ws + tc_flag_bytes(a.H) + (sk_ws ? tc_part_bytes(a.E) : 0);
  }
  // stream-K where it applies, unless the caller turns it off
  const bool want_sk = !(a.flags & GBR_FLAG_TC_NO_STREAMK) && sk_ws;
  // CTA pairs unless the caller asks for single CTAs: each CTA stages its
  // 128 rows of x and half of the W tile, and the even CTA issues M = 256
  // MMAs for both, so each SM's shared memory carries a third less traffic
  // per k-step
  p.pair = !(a.flags & GBR_FLAG_TC_SINGLE_CTA) && a.E % 32 == 0;
  p.a_bytes = BM * BK * 2;
  p.b_bytes = (uint32_t)(p.pair ? a.E / 2 : a.E) * BK * 2;
  p.stage_bytes = p.a_bytes + p.b_bytes;
  const size_t extra = 1024 /*align*/ + 2 * 8 * 8 + 16 + 16 + BM * kMaxK * 4;
  const size_t budget = 227 * 1024 - 4096;  // the rest holds the static shared arrays
  int S = (int)((budget - extra) / p.stage_bytes);
  if (S > 6) S = 6;
  if (S < 2) return cudaErrorInvalidValue;
  p.stages = S;
  int cols = 32;
  while (cols < a.E) cols <<= 1;
  p.tmem_cols = cols;
  // after the main loop the tile ring holds the exchange area and a copy
  // of the logits [E][BM]
  if ((size_t)S * p.stage_bytes < kCandOffset + (size_t)a.E * BM * 4 + (size_t)kEpiWarps * kListCap * 4)
    return cudaErrorInvalidValue;
  const size_t smem = (size_t)S * p.stage_bytes + extra;
#ifdef GBR_PHASE_STAMPS
  if (!query) p.stamps = tc_stamp_buffer();
#endif

  CUtensorMap mx{}, mw{};
  if (!query) {
    if (!make_map(&mx, a.x, a.M, a.H, BM)) return cudaErrorInvalidValue;
    // NVFP4: the kernel decodes W into the workspace as a BF16 [E, H] copy
    if (!make_map(&mw, fp4 ? static_cast<const void*>(p.wdec) : a.w, a.E, a.H,
                  p.pair ? a.E / 2 : a.E))
      return cudaErrorInvalidValue;
  }
  if (p.pair)
    return fp4 ? tc_dispatch_fp4_pair(mx, mw, p, smem, pdl, want_sk, stream, query)
               : tc_dispatch_bf16_pair(mx, mw, p, smem, pdl, want_sk, stream, query);
  return fp4 ? tc_dispatch_fp4_cta(mx, mw, p, smem, pdl, want_sk, stream, query)
             : tc_dispatch_bf16_cta(mx, mw, p, smem, pdl, want_sk, stream, query);
}

unsigned* status_word() {
  static std::mutex mu;
  static unsigned* ptr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_tc_status) == cudaSuccess) ptr[dev] = static_cast<unsigned*>(p);
  }
  return ptr[dev];
}

int tc_read_status(int clear) {
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_tc_status, sizeof v) != cudaSuccess) return -1;
  if (clear) {
    const unsigned z = 0;
    if (cudaMemcpyToSymbol(g_tc_status, &z, sizeof z) != cudaSuccess) return -1;
  }
  return v ? 1 : 0;
}

#ifdef GBR_PHASE_STAMPS
// Measurement build only: the stamps [160][kTcStamps] of the prefill
// launches since the previous read (zeros where nothing stamped), copied to
// host memory; the buffer is then cleared.
extern "C" int router_tc_phase_stamps(unsigned long long* host, int* ctas, int* phases) {
  *ctas = kTcStampCtas, *phases = kTcStamps;
  if (!host) return 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return 3;
  if (cudaMemcpyFromSymbol(host, g_tc_stamps, sizeof(g_tc_stamps)) != cudaSuccess) return 3;
  void* d = nullptr;
  if (cudaGetSymbolAddress(&d, g_tc_stamps) != cudaSuccess) return 3;
  if (cudaMemset(d, 0, sizeof(g_tc_stamps)) != cudaSuccess) return 3;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : 3;
}
#endif

}  // namespace gbr

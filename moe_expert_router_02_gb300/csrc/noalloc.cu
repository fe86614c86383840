// router_forward_noalloc: the small-M fused router for callers that cannot
// allocate device memory.
//
// Some callers may not call cudaMalloc at all: runtimes whose device memory
// is planned ahead by a static memory planner, plugin interfaces that get a
// stream but no allocator, and code on a path where an allocation could
// block or fail at the wrong time. router_forward needs a scratch buffer
// (an arrival ticket and the FP32 logits [M, E]) and allocates one per
// stream on first use; this entry point instead uses one file-scope device
// array that the library holds from the moment it is loaded until the
// process exits, on every GPU that loads it.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/gbrouter.h"
#include "kernels.h"

namespace {

constexpr int kNoAllocMaxM = 64;
constexpr int kNoAllocMaxE = 512;
// every E the library accepts must fit the array (larger E is rejected
// before this entry point looks at its scratch)
static_assert(kNoAllocMaxE >= gbr::kMaxE, "static scratch smaller than the largest E");
constexpr size_t kTicketRegion = 256;  // the arrival ticket, alone in the first 256 bytes
constexpr size_t kNoAllocBytes = kTicketRegion + (size_t)kNoAllocMaxM * kNoAllocMaxE * 4;

// 131,328 bytes per device. Host code must not use this name as an address:
// it only names a host-side stand-in; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device with that device current.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GBR_ECUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return GBR_ECUDA;
    g_ptr[dev] = p;
  }
  *out = g_ptr[dev];
  return GBR_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int router_forward_noalloc(const void* x, const void* W_gate, const float* bias, int M,
                                      int H, int E, int k, int act, int32_t* out_idx,
                                      float* out_w, cudaStream_t stream) {
  if (M < 0 || H < 1 || E < 1 || k < 1 || k > E) return GBR_EINVAL;
  if (act != GBR_ACT_SOFTMAX && act != GBR_ACT_SQRT_SOFTPLUS && act != GBR_ACT_SIGMOID)
    return GBR_EINVAL;
  if (E > gbr::kMaxE || k > gbr::kMaxK) return GBR_EUNSUPPORTED;
  if (M > kNoAllocMaxM) return GBR_EWORKSPACE;  // beyond the static scratch
  if (M == 0) return GBR_OK;
  if (!x || !W_gate || !out_idx || !out_w) return GBR_EINVAL;
  if (E % 16 != 0 || H % 32 != 0 || !aligned16(x) || !aligned16(W_gate)) return GBR_EUNSUPPORTED;

  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != GBR_OK) return rc;
  // The array keeps the previous call's contents; the ticket must start at zero.
  if (cudaMemsetAsync(scratch, 0, sizeof(uint32_t), stream) != cudaSuccess) return GBR_ECUDA;

  gbr::RouterArgs a{};
  a.x = x;
  a.w = W_gate;
  a.w_global = 1.0f;
  a.bias = bias;
  a.M = M, a.H = H, a.E = E, a.k = k, a.act = gbr::internal_act(act, bias);
  a.x_dtype = gbr::DT_BF16, a.w_dtype = gbr::DT_BF16;
  a.out_idx = out_idx;
  a.out_w = out_w;
  a.ticket = static_cast<uint32_t*>(scratch);
  a.logits = reinterpret_cast<float*>(static_cast<unsigned char*>(scratch) + kTicketRegion);
  return gbr::launch_gemv(a, true, true, stream) == cudaSuccess ? GBR_OK : GBR_ECUDA;
}

// C-ABI entry points: argument checks, workspace, regime choice, launch.
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <utility>

#include "../../include/gbrouter.h"
#include "kernels.h"

namespace {

using gbr::RouterArgs;

constexpr size_t kTicketBytes = 256;  // the arrival ticket sits alone in the first 256 bytes

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Shape {
  int M, H, E, k, act, x_dtype, w_dtype, flags;
  bool table, has_bias, has_scales;
};

// Argument checks that need no pointer values beyond null-ness.
int check_shape(const Shape& s) {
  if (s.M < 0 || s.H < 1 || s.E < 1 || s.k < 1 || s.k > s.E) return GBR_EINVAL;
  if (s.act != GBR_ACT_SOFTMAX && s.act != GBR_ACT_SQRT_SOFTPLUS && s.act != GBR_ACT_SIGMOID)
    return GBR_EINVAL;
  if (s.x_dtype != GBR_F32 && s.x_dtype != GBR_BF16) return GBR_EINVAL;
  if (s.w_dtype != GBR_F32 && s.w_dtype != GBR_BF16 && s.w_dtype != GBR_NVFP4) return GBR_EINVAL;
  if (s.w_dtype == GBR_NVFP4 && (s.H % 16 != 0 || !s.has_scales)) return GBR_EINVAL;
  if (s.table && (s.M % 2 != 0)) return GBR_EINVAL;
  if (s.E > gbr::kMaxE || s.k > gbr::kMaxK) return GBR_EUNSUPPORTED;
  return GBR_OK;
}

bool gemv_eligible(const Shape& s) {
  return s.x_dtype == GBR_BF16 && s.w_dtype == GBR_BF16 && s.M >= 1 && s.M <= 64 &&
         s.E % 16 == 0 && s.H % 32 == 0;
}

int regime_of(const Shape& s) {
  const int f = s.flags;
  if (f & GBR_FLAG_FORCE_GENERIC) return GBR_REGIME_GENERIC;
  // softmax with a selection bias: not in the prefill kernel's epilogue (the
  // generic kernel serves those shapes)
  const bool tc = gbr::tc_eligible(s.M, s.H, s.E, s.k, s.x_dtype, s.w_dtype) &&
                  !(s.act == GBR_ACT_SOFTMAX && s.has_bias);
  const bool gv = gemv_eligible(s);
  if (f & GBR_FLAG_UNFUSED) return gv ? GBR_REGIME_UNFUSED : GBR_REGIME_GENERIC;
  if ((f & GBR_FLAG_FORCE_TC) && tc) return GBR_REGIME_TC;
  const bool one_cluster = gv && !(f & GBR_FLAG_NO_SINGLE_CLUSTER) &&
                           gbr::gemv1c_eligible(s.M, s.H, s.E, false);
  // NVFP4 weights at small M: only the single-cluster kernel decodes them
  if (s.x_dtype == GBR_BF16 && s.w_dtype == GBR_NVFP4 && !(f & GBR_FLAG_NO_SINGLE_CLUSTER) &&
      !(f & GBR_FLAG_FORCE_TC) && gbr::gemv1c_eligible(s.M, s.H, s.E, true))
    return GBR_REGIME_GEMV1C;
  if ((f & GBR_FLAG_FORCE_GEMV) && gv) return one_cluster ? GBR_REGIME_GEMV1C : GBR_REGIME_GEMV;
  if (gv) return one_cluster ? GBR_REGIME_GEMV1C : GBR_REGIME_GEMV;
  if (tc && s.M > 64) return GBR_REGIME_TC;
  return GBR_REGIME_GENERIC;
}

size_t workspace_for(const Shape& s, int regime) {
  // ticket in the first 256 bytes, FP32 logits [M, E] after it. The
  // single-cluster kernel needs none, but reports the same size so that a
  // workspace sized on one device also fits a device where it is not chosen.
  if (regime == GBR_REGIME_GEMV || regime == GBR_REGIME_GEMV1C || regime == GBR_REGIME_UNFUSED)
    return kTicketBytes + round_up((size_t)s.M * s.E * 4, 256);
  // the prefill kernel keeps stream-K partial sums and the NVFP4 W it
  // decodes once per launch in the workspace
  if (regime == GBR_REGIME_TC) return gbr::tc_workspace(s.M, s.H, s.E, s.w_dtype);
  return 0;
}

Shape make_shape(int M, int H, int E, int k, int act, const float* bias, const gbr_opts* o) {
  Shape s{};
  s.M = M, s.H = H, s.E = E, s.k = k, s.act = act;
  s.x_dtype = o ? o->x_dtype : GBR_BF16;
  s.w_dtype = o ? o->w_dtype : GBR_BF16;
  s.flags = o ? o->flags : 0;
  s.table = o && o->tbl_unique;
  s.has_bias = bias != nullptr;
  s.has_scales = o && o->w_scales;
  return s;
}

// Library-owned workspaces, one per (device, stream), grown on demand and
// zero-filled when (re)allocated.
struct Ws {
  void* ptr = nullptr;
  size_t bytes = 0;
};
std::mutex g_ws_mu;
std::map<std::pair<int, cudaStream_t>, Ws> g_ws;

int library_workspace(cudaStream_t stream, size_t need, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GBR_ECUDA;
  std::lock_guard<std::mutex> lk(g_ws_mu);
  Ws& w = g_ws[{dev, stream}];
  if (w.bytes < need) {
    if (w.ptr) {
      if (cudaStreamSynchronize(stream) != cudaSuccess) return GBR_ECUDA;
      cudaFree(w.ptr);
      w.ptr = nullptr;
      w.bytes = 0;
    }
    const size_t bytes = round_up(need < (1u << 20) ? (1u << 20) : need, 1u << 20);
    if (cudaMalloc(&w.ptr, bytes) != cudaSuccess) return GBR_ECUDA;
    if (cudaMemsetAsync(w.ptr, 0, bytes, stream) != cudaSuccess) return GBR_ECUDA;
    w.bytes = bytes;
  }
  *out = w.ptr;
  return GBR_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

const char* router_strerror(int status) {
  switch (status) {
    case GBR_OK: return "ok";
    case GBR_EINVAL: return "invalid argument";
    case GBR_EUNSUPPORTED: return "unsupported shape (E > 512 or k > 16)";
    case GBR_ECUDA: return "CUDA runtime error";
    case GBR_EWORKSPACE: return "workspace too small";
    case GBR_ETIMEOUT: return "a bounded device-side wait expired";
    default: return "unknown status";
  }
}

size_t router_workspace_size(int M, int H, int E, int k, const gbr_opts* opt) {
  const Shape s = make_shape(M, H, E, k, GBR_ACT_SOFTMAX, nullptr, opt);
  if (check_shape(s) != GBR_OK) return 0;
  return workspace_for(s, regime_of(s));
}

int router_regime(int M, int H, int E, int k, const gbr_opts* opt) {
  const Shape s = make_shape(M, H, E, k, GBR_ACT_SOFTMAX, nullptr, opt);
  if (check_shape(s) != GBR_OK) return -1;
  return regime_of(s);
}

int router_tc_groups(int M, int H, int E, int k, const gbr_opts* opt) {
  const Shape s = make_shape(M, H, E, k, GBR_ACT_SOFTMAX, nullptr, opt);
  if (check_shape(s) != GBR_OK) return -1;
  if (regime_of(s) != GBR_REGIME_TC) return 0;
  gbr::RouterArgs a{};
  a.M = M, a.H = H, a.E = E, a.k = k, a.act = GBR_ACT_SOFTMAX;
  a.x_dtype = s.x_dtype, a.w_dtype = s.w_dtype;
  a.flags = s.flags;
  // the launch gets a workspace whenever workspace_for asks for one (a
  // query only tests the pointer for null)
  static uint32_t present;
  a.ticket = workspace_for(s, GBR_REGIME_TC) ? &present : nullptr;
  int groups = 0;
  if (gbr::launch_tc(a, false, nullptr, &groups) != cudaSuccess) {
    (void)cudaGetLastError();
    return -1;
  }
  return groups;
}

int router_forward_ex(const void* x, const void* W_gate, const float* bias, int M, int H, int E,
                      int k, int act, int32_t* out_idx, float* out_w, const gbr_opts* opt,
                      cudaStream_t stream) {
  const Shape s = make_shape(M, H, E, k, act, bias, opt);
  int rc = check_shape(s);
  if (rc != GBR_OK) return rc;
  if (opt) {
    const int n_tbl = (opt->tbl_unique != nullptr) + (opt->tbl_mask != nullptr) +
                      (opt->tbl_map != nullptr) + (opt->tbl_count != nullptr);
    if (n_tbl != 0 && n_tbl != 4) return GBR_EINVAL;
  }
  if (M == 0) return GBR_OK;
  if (!x || !W_gate || !out_idx || !out_w) return GBR_EINVAL;

  int regime = regime_of(s);
  if ((regime == GBR_REGIME_GEMV || regime == GBR_REGIME_GEMV1C || regime == GBR_REGIME_UNFUSED ||
       regime == GBR_REGIME_TC) &&
      (!aligned16(x) || !aligned16(W_gate) || H % 8 != 0 ||
       (s.w_dtype == GBR_NVFP4 && !aligned16(opt->w_scales))))
    regime = GBR_REGIME_GENERIC;

  RouterArgs a{};
  a.x = x;
  a.w = W_gate;
  a.w_scales = opt ? opt->w_scales : nullptr;
  a.w_global = opt ? opt->w_global_scale : 1.0f;
  a.bias = bias;
  a.M = M, a.H = H, a.E = E, a.k = k, a.act = gbr::internal_act(act, bias);
  a.x_dtype = s.x_dtype, a.w_dtype = s.w_dtype;
  a.flags = s.flags;
  a.out_idx = out_idx;
  a.out_w = out_w;
  a.logits = opt ? opt->out_logits : nullptr;
  if (s.table) {
    a.tbl_unique = opt->tbl_unique;
    a.tbl_mask = opt->tbl_mask;
    a.tbl_map = opt->tbl_map;
    a.tbl_count = opt->tbl_count;
  }
  const bool pdl = !(s.flags & GBR_FLAG_NO_PDL);
  a.status = gbr::status_word();

  const size_t need = workspace_for(s, regime);
  void* ws = nullptr;
  if (need) {
    if (opt && opt->workspace) {
      if (opt->workspace_bytes < need) return GBR_EWORKSPACE;
      ws = opt->workspace;
    } else {
      rc = library_workspace(stream, need, &ws);
      if (rc != GBR_OK) return rc;
    }
  }

  cudaError_t err = cudaSuccess;
  switch (regime) {
    case GBR_REGIME_GEMV:
      a.ticket = static_cast<uint32_t*>(ws);
      if (!a.logits) a.logits = reinterpret_cast<float*>(static_cast<char*>(ws) + kTicketBytes);
      err = gbr::launch_gemv(a, true, pdl, stream);
      break;
    case GBR_REGIME_GEMV1C:
      err = gbr::launch_gemv1c(a, pdl, stream);
      break;
    case GBR_REGIME_UNFUSED: {
      if (!a.logits) a.logits = reinterpret_cast<float*>(static_cast<char*>(ws) + kTicketBytes);
      err = gbr::launch_gemv(a, false, pdl, stream);
      if (err == cudaSuccess)
        err = gbr::launch_select(a.logits, bias, M, E, k, a.act, out_idx, out_w, stream);
      if (err == cudaSuccess && s.table)
        err = gbr::launch_route_table(out_idx, M / 2, 2, k, a.tbl_unique, a.tbl_mask, a.tbl_map,
                                      a.tbl_count, stream);
      break;
    }
    case GBR_REGIME_TC:
      a.ticket = static_cast<uint32_t*>(ws);
      err = gbr::launch_tc(a, pdl, stream);
      break;
    default:
      err = gbr::launch_generic(a, pdl, stream);
      break;
  }
  return err == cudaSuccess ? GBR_OK : GBR_ECUDA;
}

int router_forward(const void* x, const void* W_gate, const float* bias, int M, int H, int E, int k,
                   int act, int32_t* out_idx, float* out_w, cudaStream_t stream) {
  return router_forward_ex(x, W_gate, bias, M, H, E, k, act, out_idx, out_w, nullptr, stream);
}

int router_select(const float* logits, const float* bias, int M, int E, int k, int act,
                  int32_t* out_idx, float* out_w, cudaStream_t stream) {
  if (M < 0 || E < 1 || k < 1 || k > E) return GBR_EINVAL;
  if (act != GBR_ACT_SOFTMAX && act != GBR_ACT_SQRT_SOFTPLUS && act != GBR_ACT_SIGMOID)
    return GBR_EINVAL;
  if (E > gbr::kMaxE || k > gbr::kMaxK) return GBR_EUNSUPPORTED;
  if (M == 0) return GBR_OK;
  if (!logits || !out_idx || !out_w) return GBR_EINVAL;
  return gbr::launch_select(logits, bias, M, E, k, gbr::internal_act(act, bias), out_idx, out_w,
                            stream) == cudaSuccess
             ? GBR_OK
             : GBR_ECUDA;
}

int router_near_tie_keys(const float* z, const float* bias, int n, int act, float* key_hi,
                         float* key_lo, cudaStream_t stream) {
  if (n < 0 || (act != GBR_ACT_SQRT_SOFTPLUS && act != GBR_ACT_SIGMOID)) return GBR_EINVAL;
  if (n == 0) return GBR_OK;
  if (!z || !key_hi || !key_lo) return GBR_EINVAL;
  return gbr::launch_near_tie_keys(z, bias, n, act, key_hi, key_lo, stream) == cudaSuccess
             ? GBR_OK
             : GBR_ECUDA;
}

int route_gather_add(const void* y, const uint8_t* map, const float* w, const void* shared,
                     int groups, int tokens_per_group, int k, int D, void* out,
                     cudaStream_t stream) {
  if (groups < 0 || tokens_per_group < 1 || tokens_per_group > 8 || k < 1 || k > gbr::kMaxK ||
      D < 1)
    return GBR_EINVAL;
  if (groups == 0) return GBR_OK;
  if (!y || !map || !w || !shared || !out) return GBR_EINVAL;
  return gbr::launch_gather_add(y, map, w, shared, groups, tokens_per_group, k, D, out, stream) ==
                 cudaSuccess
             ? GBR_OK
             : GBR_ECUDA;
}

int route_table(const int32_t* idx, int groups, int tokens_per_group, int k, int32_t* out_unique,
                uint8_t* out_mask, uint8_t* out_map, int32_t* out_count, cudaStream_t stream) {
  if (groups < 0 || tokens_per_group < 1 || tokens_per_group > 8 || k < 1 || k > gbr::kMaxK)
    return GBR_EINVAL;
  if (groups == 0) return GBR_OK;
  if (!idx || !out_unique || !out_mask || !out_map || !out_count) return GBR_EINVAL;
  return gbr::launch_route_table(idx, groups, tokens_per_group, k, out_unique, out_mask, out_map,
                                 out_count, stream) == cudaSuccess
             ? GBR_OK
             : GBR_ECUDA;
}

int router_device_status(int clear) {
  if (cudaDeviceSynchronize() != cudaSuccess) return GBR_ECUDA;
  const int st = gbr::tc_read_status(clear);
  if (st < 0) return GBR_ECUDA;
  return st ? GBR_ETIMEOUT : GBR_OK;
}

}  // extern "C"

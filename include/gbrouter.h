/*
 * gbrouter — fused MoE router for one NVIDIA GB300 (sm_103a). C ABI.
 *
 * One call computes, for M token rows x[m, :]:
 *   1. the gate projection  logits[m, e] = sum_h x[m, h] * W_gate[e, h]
 *      with FP32 accumulation, kept on chip
 *      (qwisp issue #145, "Observation" and "Change": postNorm[H] ->
 *      gateLogits[E], "one kernel producing inds/scores directly from
 *      postNorm", logits held on chip instead of round-tripping);
 *   2. the score: softmax over E, or a = sqrt(softplus(logit)) with the
 *      stable softplus max(z,0) + log1p(exp(-|z|)), or a = sigmoid(logit) =
 *      1 / (1 + exp(-logit)); a per-expert bias, when given, is added to the
 *      score for selection only (softmax: to the full-E probability; without
 *      a bias the softmax key is the logit, which orders alike)
 *      (dense_router_decode commit page, "DenseRouterDecodeKernel: BF16 GEMM
 *      + sqrt(softplus) + bias + top-k", "Numerically stable softplus", heap
 *      of "(score, index, unbiased act)"; qwisp issue #145, "Gates": the bias
 *      variant of the softmax route; the sigmoid score and the softmax bias
 *      are this library's widening of the same biased-score contract);
 *   3. top-k under the fixed comparison: higher key first, an equal key goes
 *      to the lower expert index; slots are returned in that order
 *      (qwisp issue #145, "Bit-exactness": the tie-break order is part of
 *      the contract);
 *   4. renormalisation of the chosen weights, w_j = s_j / sum_{i<k} s_i,
 *      where s is the softmax probability or the unbiased activation
 *      (commit page, "top-k + renorm");
 *   5. optionally the M=2 unique-route table: encounter-ordered unique
 *      experts, per-unique-expert token masks, slot-to-unique map and count
 *      (b70 lab note "MTP1 M=2 gather/shared-add gate", section
 *      "Unique-route router screen").
 *
 * Conventions shared by every entry point
 *   - Every data pointer is a caller-owned DEVICE pointer; the library never
 *     frees or retains it. Arrays are dense row-major.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream). The
 *     return value reports argument errors and launch errors only.
 *   - Argument errors return before any CUDA call: nothing is launched and
 *     nothing is written.
 *   - M == 0 (or groups == 0) returns GBR_OK without a launch.
 *   - Inputs must be finite. -0.0 and +0.0 compare equal (lower index wins).
 *   - If every chosen score of a row is zero, its weights are 1/k.
 *   - W_gate, bias and NVFP4 scales may be read before the kernel waits on
 *     the preceding kernel of the stream (programmatic dependent launch).
 *     If the immediately preceding kernel writes them, set GBR_FLAG_NO_PDL.
 */
#ifndef GBROUTER_H_
#define GBROUTER_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* cudaStream_t;

/* status codes */
enum {
  GBR_OK = 0,
  GBR_EINVAL = 1,       /* bad argument: null pointer, k < 1, k > E, bad enum, ... */
  GBR_EUNSUPPORTED = 2, /* valid but beyond the library's limits: E > 512, k > 16 */
  GBR_ECUDA = 3,        /* a CUDA runtime call or launch failed */
  GBR_EWORKSPACE = 4,   /* caller workspace smaller than router_workspace_size() */
  GBR_ETIMEOUT = 5      /* a bounded device-side wait expired (see router_device_status) */
};

/* score activation */
enum { GBR_ACT_SOFTMAX = 0, GBR_ACT_SQRT_SOFTPLUS = 1, GBR_ACT_SIGMOID = 2 };

/* element types. NVFP4 is for W_gate only: packed E2M1 codes [E, H/2]
 * (element 2j in the low nibble of byte j, 2j+1 in the high nibble), one
 * E4M3 scale per 16 elements along H in w_scales [E, H/16], and an FP32
 * global scale: W[e,h] = e2m1 * e4m3 * w_global_scale
 * (dense_router_decode commit page, "NVFP4 blockscaled GEMM"). */
enum { GBR_F32 = 0, GBR_BF16 = 1, GBR_NVFP4 = 2 };

/* option flags */
enum {
  GBR_FLAG_NO_PDL = 1,        /* launch without programmatic dependent launch */
  GBR_FLAG_FORCE_GENERIC = 2, /* use the generic row-per-CTA kernel (A/B and tests) */
  GBR_FLAG_FORCE_GEMV = 4,    /* use the small-M tensor-core GEMV kernel when eligible */
  GBR_FLAG_FORCE_TC = 8,      /* use the tcgen05 prefill kernel when eligible */
  GBR_FLAG_UNFUSED = 16,      /* two launches: gate logits, then router_select (A/B only) */
  GBR_FLAG_NO_SINGLE_CLUSTER = 32, /* small M: skip the single-cluster kernel (A/B only) */
  GBR_FLAG_TC_NO_STREAMK = 64,    /* prefill: one CTA pair (or CTA) per tile, no stream-K */
  GBR_FLAG_TC_SINGLE_CTA = 128    /* prefill: single CTAs (M = 128 MMAs) instead of CTA pairs */
};

/* kernel families reported by router_regime() */
enum {
  GBR_REGIME_GENERIC = 0, /* one CTA per row, any dtype and shape */
  GBR_REGIME_GEMV = 1,    /* M <= 64: clusters split H, last cluster selects */
  GBR_REGIME_TC = 2,      /* M > 64: tcgen05 GEMM with the selection in its epilogue */
  GBR_REGIME_UNFUSED = 3, /* logits kernel + router_select (A/B baseline) */
  GBR_REGIME_GEMV1C = 4   /* M <= 64, E <= 256: a cluster per 4, 8 or 16 rows holds W_gate in shared memory */
};

typedef struct {
  int x_dtype;                /* GBR_F32 or GBR_BF16 (default for router_forward: BF16) */
  int w_dtype;                /* GBR_F32, GBR_BF16 or GBR_NVFP4 */
  const uint8_t* w_scales;    /* NVFP4 only: E4M3 codes [E, H/16] */
  float w_global_scale;       /* NVFP4 only */
  void* workspace;            /* nullable: library-owned per (device, stream) if NULL.
                                 Must be 256-byte aligned and zero-filled before its
                                 first use; every call leaves it ready for the next. */
  size_t workspace_bytes;
  /* optional M=2 unique-route table; all four or none; M must be even and
     group g covers rows 2g and 2g+1 (layouts as in route_table, T = 2) */
  int32_t* tbl_unique;        /* [M/2, 2k] */
  uint8_t* tbl_mask;          /* [M/2, 2k] */
  uint8_t* tbl_map;           /* [M/2, 2, k] */
  int32_t* tbl_count;         /* [M/2] */
  float* out_logits;          /* nullable FP32 [M, E]: the raw gate logits the
                                 selection used (telemetry tap) */
  int flags;                  /* GBR_FLAG_* */
} gbr_opts;

/*
 * router_forward — steps 1-4 in one launch, BF16 x [M, H] and BF16
 * W_gate [E, H], FP32 bias [E] (nullable; selection only, every
 * activation). Softmax with a bias at M > 64 runs the generic kernel (the
 * prefill kernel's epilogue does not take the probability key).
 * Outputs: out_idx int32 [M, k] (expert ids in slot order), out_w FP32
 * [M, k]. Uses a library-owned workspace for (current device, stream),
 * allocated and zero-filled on first use (call once before capturing the
 * stream into a CUDA graph). Thread-safe.
 * Errors: GBR_EINVAL for null required pointers, M < 0, H < 1, E < 1,
 * k < 1, k > E, act outside the enum; GBR_EUNSUPPORTED for E > 512 or
 * k > 16; GBR_ECUDA if allocation or launch fails.
 */
int router_forward(const void* x, const void* W_gate, const float* bias, int M, int H, int E,
                   int k, int act, int32_t* out_idx, float* out_w, cudaStream_t stream);

/*
 * router_forward_ex — as router_forward with dtypes, NVFP4 weights, an
 * explicit workspace, the fused M=2 route table and the logits tap.
 * opt may be NULL (BF16 x and W, library workspace). Extra errors:
 * GBR_EINVAL for a partial table pointer set, a table with odd M, NVFP4
 * without scales or with H % 16 != 0, dtypes outside the enums;
 * GBR_EWORKSPACE when workspace_bytes < router_workspace_size(...).
 * Concurrent calls that share one workspace race; give each stream its own.
 */
int router_forward_ex(const void* x, const void* W_gate, const float* bias, int M, int H, int E,
                      int k, int act, int32_t* out_idx, float* out_w, const gbr_opts* opt,
                      cudaStream_t stream);

/* Bytes of workspace router_forward_ex needs for this shape (0 if none). */
size_t router_workspace_size(int M, int H, int E, int k, const gbr_opts* opt);

/* Which kernel family router_forward_ex would launch (GBR_REGIME_*) for a
 * call without a bias or with a non-softmax activation, or -1 for arguments
 * it would reject. */
int router_regime(int M, int H, int E, int k, const gbr_opts* opt);

/* Stream-K work groups the prefill kernel (GBR_REGIME_TC) would split this
 * shape over on the current device: the tiles x k-steps units divided
 * evenly over up to one CTA pair (or CTA) per two SMs (per SM), as many as
 * keep every tile within four groups; each group finishes at most one tile
 * after adding the other groups' partial accumulators from the workspace.
 * 0 when every tile gets its own CTA pair (fewer than 256 rows, at least as
 * many tiles as groups, GBR_FLAG_TC_NO_STREAMK in opt->flags) or the shape
 * takes another kernel family; -1 for arguments router_forward_ex would
 * reject or a failed device query. Launches nothing. */
int router_tc_groups(int M, int H, int E, int k, const gbr_opts* opt);

/*
 * router_select — steps 2-4 alone, on caller FP32 logits [M, E]; bias
 * nullable FP32 [E] (every activation). The same selection code the fused
 * kernels run; it exists so the selection stage can be checked on identical
 * FP32 logits (qwisp issue #145, "Gates", G-A: synthetic logits with exact
 * and near ties at the top-k boundary). Errors as router_forward.
 */
int router_select(const float* logits, const float* bias, int M, int E, int k, int act,
                  int32_t* out_idx, float* out_w, cudaStream_t stream);

/*
 * router_near_tie_keys — the key the selection re-ranks near ties with
 * (the biased activations): key[i] = a(z[i]) + bias[i], a = sqrt-softplus
 * (act = GBR_ACT_SQRT_SOFTPLUS) or sigmoid (GBR_ACT_SIGMOID), bias nullable
 * (0), returned as an unevaluated sum key_hi[i] + key_lo[i] of two floats
 * with |lo| <= ulp(hi)/2, from FP32 arithmetic only (double-float
 * evaluation, relative error near 2^-42; |z| > 30 goes through FP64).
 * Step 2 of the router as the guard-band refine evaluates it; exposed so
 * that its error can be measured against an FP64 definition. z, bias,
 * key_hi, key_lo: device FP32 [n]. Errors: GBR_EINVAL for n < 0, another
 * act, or null z / key pointers (n == 0: no launch).
 */
int router_near_tie_keys(const float* z, const float* bias, int n, int act, float* key_hi,
                         float* key_lo, cudaStream_t stream);

/*
 * route_table — step 5 alone for `groups` groups of T = tokens_per_group
 * rows (1 <= T <= 8), k slots each (1 <= k <= 16):
 *   idx        int32 [groups, T, k]  expert ids (expected >= 0)
 *   out_unique int32 [groups, T*k]   unique experts in encounter order
 *                                    (token-major, slot order), -1 past count
 *   out_mask   uint8 [groups, T*k]   bit t set when token t routes to
 *                                    out_unique[u]; 0 past count
 *   out_map    uint8 [groups, T, k]  u such that out_unique[u] == idx[t][s]
 *   out_count  int32 [groups]        number of unique experts
 * Duplicates within a row map to the same u. Weights and ids are untouched
 * (the b70 note requires them preserved bit-for-bit).
 * Errors: GBR_EINVAL for null pointers, groups < 0, T or k out of range.
 */
int route_table(const int32_t* idx, int groups, int tokens_per_group, int k, int32_t* out_unique,
                uint8_t* out_mask, uint8_t* out_map, int32_t* out_count, cudaStream_t stream);

/*
 * router_forward_noalloc — router_forward for callers that must not
 * allocate device memory (no counterpart on the router pages; it exists for
 * this library's users). Runtimes that plan all device memory ahead of time,
 * plugin interfaces that receive a stream but no allocator, and paths where
 * an allocation may block or fail cannot let router_forward create its
 * per-stream workspace. This entry point allocates nothing: its scratch (an
 * arrival ticket and FP32 logits [M, E]) is one file-scope device array of
 * 131,328 bytes that every GPU loading the library holds until the process
 * exits. Limits: M <= 64 (beyond it: GBR_EWORKSPACE); E <= 512 as for every
 * entry point (beyond it: GBR_EUNSUPPORTED); BF16 x and W_gate with
 * E % 16 == 0, H % 32 == 0 and 16-byte aligned x and W_gate (otherwise
 * GBR_EUNSUPPORTED). Other arguments and errors as router_forward.
 * The first call on a device looks up the array's device address, so make
 * that first call before any stream capture. Every call on a device shares
 * the one array: calls that overlap on the GPU (other streams, other host
 * threads) race and must be serialised by the caller. Each call clears the
 * ticket with a 4-byte cudaMemsetAsync on `stream` before its launch.
 */
int router_forward_noalloc(const void* x, const void* W_gate, const float* bias, int M, int H,
                           int E, int k, int act, int32_t* out_idx, float* out_w,
                           cudaStream_t stream);

/*
 * route_gather_add — the table's consumer (b70 lab note "MTP1 M=2
 * gather/shared-add gate": "Exact arithmetic", "Real route-direct result").
 * The experts ran once per unique (token, expert) route of each group; this
 * combines their rows. For group g, token t < T = tokens_per_group and
 * element d < D:
 *   acc = 0; for s = 0..k-1: acc = fma(w[g][t][s], y[g][map[g][t][s]][t][d], acc)
 *   out[g][t][d] = bf16(float(bf16(acc)) + float(shared[g][t][d]))
 * FP32 fma accumulation in slot order, FP32 add, round-to-nearest-even to
 * BF16 at both steps. Layouts (dense, row-major, device):
 *   y      BF16 [groups, T*k, T, D]  row (u, t): unique expert u's output
 *                                     for token t (rows no slot maps to are
 *                                     not read)
 *   map    uint8 [groups, T, k]      as route_table's out_map
 *   w      FP32 [groups, T, k]       the router's weights
 *   shared BF16 [groups, T, D]       the shared expert's output
 *   out    BF16 [groups, T, D]
 * A map entry >= T*k contributes nothing. 16-byte aligned y, shared and out
 * with D % 8 == 0 take the vector path. Errors: GBR_EINVAL for groups < 0,
 * T outside 1..8, k outside 1..16, D < 1, null pointers (groups == 0: no
 * launch).
 */
int route_gather_add(const void* y, const uint8_t* map, const float* w, const void* shared,
                     int groups, int tokens_per_group, int k, int D, void* out,
                     cudaStream_t stream);

/* Static text for a status code. */
const char* router_strerror(int status);

/*
 * router_device_status — synchronises the current device and reports
 * GBR_ETIMEOUT if any kernel of this library gave up a bounded wait since
 * the last clear (its outputs for that call are then undefined), else
 * GBR_OK; GBR_ECUDA if the device cannot be queried. clear != 0 resets it.
 */
int router_device_status(int clear);

#ifdef __cplusplus
}
#endif

#endif /* GBROUTER_H_ */

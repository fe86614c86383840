// Host-side launchers of the router kernels (internal to the library).
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace gbr {

cudaError_t launch_select(const float* logits, const float* bias, int M, int E, int k, int act,
                          int32_t* out_idx, float* out_w, cudaStream_t stream);

// Near-tie keys (double-float activation + bias) for n logits.
cudaError_t launch_near_tie_keys(const float* z, const float* bias, int n, int act, float* hi,
                                 float* lo, cudaStream_t stream);

// The table's consumer: routed gather + shared-expert add (BF16 rows).
cudaError_t launch_gather_add(const void* y, const uint8_t* map, const float* w,
                              const void* shared, int G, int T, int k, int D, void* out,
                              cudaStream_t stream);

cudaError_t launch_route_table(const int32_t* idx, int groups, int T, int k, int32_t* unique,
                               uint8_t* mask, uint8_t* map, int32_t* count, cudaStream_t stream);

// Small-M tensor-core GEMV router. select == false writes the logits only
// (first half of the unfused A/B pair).
int gemv_cluster_size(int H);
cudaError_t launch_gemv(const RouterArgs& a, bool select, bool pdl, cudaStream_t stream);

// Small-M single-cluster router (E <= 256, W_gate in shared memory): one
// cluster per group of 4, 8 or 16 rows (at most four clusters), M <= 64.
bool gemv1c_eligible(int M, int H, int E, bool fp4);
cudaError_t launch_gemv1c(const RouterArgs& a, bool pdl, cudaStream_t stream);

// Row-per-CTA router for any dtype and shape.
cudaError_t launch_generic(const RouterArgs& a, bool pdl, cudaStream_t stream);

// tcgen05 prefill router.
bool tc_eligible(int M, int H, int E, int k, int x_dtype, int w_dtype);
// With query set nothing launches: *query receives the stream-K group count
// the launch would use (0: one CTA or CTA pair per tile).
cudaError_t launch_tc(const RouterArgs& a, bool pdl, cudaStream_t stream, int* query = nullptr);
// The M <= 64 kernels' part of a workspace: the arrival ticket (256 bytes)
// and FP32 logits [M, E] for M <= 64, E <= 512.
constexpr size_t kSmallMScratchBytes = 256 + 64 * 512 * 4;
// Workspace the prefill router needs (flags, stream-K partial accumulators
// for M >= 256, NVFP4 W decoded); launch_tc takes it as RouterArgs::ticket.
size_t tc_workspace(int M, int H, int E, int w_dtype);
int tc_read_status(int clear);  // 0 ok, 1 a bounded wait expired, -1 query failed
unsigned* status_word();        // device address of that status word (current device)

}  // namespace gbr

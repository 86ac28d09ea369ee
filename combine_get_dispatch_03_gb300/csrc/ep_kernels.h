// ep_kernels.h -- host-side launchers of the EP kernels (internal to the library).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ep.h"

namespace ep {

// Launch shapes, chosen once per device when a handle is created.
struct LaunchPlan {
    int num_sms = 0;        // SMs the data kernels may fill: the device's, or ep_config.max_sms if fewer
    bool sm_limited = false;  // num_sms was capped by max_sms: one resident wave covers all tokens
    int dispatch_blocks[3] = {0, 0, 0};  // per payload mode
    int combine_blocks[4] = {0, 0, 0, 0};  // bf16 out, fp32 out; then the same with the all-ranks batch
    int ll_dispatch_blocks[2] = {0, 0};  // bf16, fp8
    int ll_combine_blocks = 0;
    int ll_combine_blocks_small_k = 0;  // the variant with every top-k slot in one batch
    int bulk_stages[3] = {0, 0, 0};      // bulk-copy dispatch: stages per CTA (0 = not usable)
    unsigned bulk_smem[3] = {0, 0, 0};   // its dynamic shared memory
    int bulk_resident[3] = {1, 1, 1};    // its CTAs resident on the GPU at once
};

constexpr int kLayoutThreads = 1024;
constexpr int kNotifyThreads = 1024;
constexpr int kDispatchThreads = 512;
constexpr int kCombineThreads = 256;
constexpr int kLLCountThreads = 512;
constexpr int kLLDispatchThreads = 512;
constexpr int kLLCombineThreads = 256;

enum DispatchMode { kModeBf16 = 0, kModeCastFp8 = 1, kModeFp8In = 2 };

cudaError_t plan_launches(LaunchPlan* plan, int device, int num_experts);

// rank_mask: int32 [R] (nonzero = masked) or NULL; slots that start or end on a masked rank are left out.
cudaError_t launch_get_dispatch_layout(const int64_t* topk_idx, const int32_t* rank_mask, int R, int T, int K,
                                       int E, int32_t* tpr, int32_t* tprdma, int32_t* tpe, uint8_t* itr,
                                       int32_t* status, cudaStream_t stream);

cudaError_t launch_dispatch_notify(int R, int T, int E, int C, int A, int64_t cap, const int32_t* tpr,
                                   const uint8_t* itr, const int32_t* tpe, int32_t* rank_prefix,
                                   int32_t* channel_prefix, int32_t* recv_channel_prefix, int32_t* num_recv,
                                   int32_t* send_head, int32_t* recv_src_idx, int32_t* num_recv_per_expert,
                                   int32_t* rdma_channel_prefix, int32_t* recv_rdma_rank_prefix, int32_t* status,
                                   cudaStream_t stream);

// Layout and the dispatch record in one pass (a decoupled look-back scan over token tiles of 512),
// for T >= 1; with rdma_channel_prefix and recv_rdma_rank_prefix (whole nodes of 8, R > 8) the
// node-level record as well.  scratch: layout_scan_scratch_words(R, E, maxT) words of device
// memory, zero before the first launch; launches sharing it must be ordered.
size_t layout_scan_scratch_words(int R, int E, int max_tokens);
cudaError_t launch_layout_scan(const int64_t* topk_idx, const int32_t* rank_mask, int R, int T, int K, int E, int C,
                               int A, int64_t cap, int32_t* tpr, int32_t* tprdma, int32_t* tpe, uint8_t* itr,
                               int32_t* rank_prefix, int32_t* channel_prefix, int32_t* recv_channel_prefix,
                               int32_t* num_recv, int32_t* send_head, int32_t* recv_src_idx,
                               int32_t* num_recv_per_expert, int32_t* rdma_channel_prefix,
                               int32_t* recv_rdma_rank_prefix, uint32_t* scratch, int32_t* status,
                               cudaStream_t stream);

cudaError_t launch_dispatch(const LaunchPlan& plan, int mode, int R, int T, int H, int K, int EL, int64_t cap,
                            const void* x, const float* x_scales, const int64_t* topk_idx,
                            const float* topk_weights, const int32_t* send_head, void* recv_x,
                            float* recv_x_scales, int64_t* recv_topk_idx, float* recv_topk_weights,
                            int32_t* status, cudaStream_t stream);

// work: two words of device memory, zero before the first launch, through which the combine's
// warps claim tokens; each launch leaves them zero again.  Launches sharing them must be ordered.
cudaError_t launch_combine(const LaunchPlan& plan, bool out_fp32, int R, int T, int H, int K, int64_t cap,
                           const int32_t* send_head, const void* y, const float* recv_topk_weights,
                           const void* bias0, const void* bias1, void* out, float* combined_topk_weights,
                           uint32_t* work, cudaStream_t stream);

cudaError_t launch_ll_dispatch(const LaunchPlan& plan, int R, int T, int maxT, int H, int K, int E,
                               const void* x, const int64_t* topk_idx, bool use_fp8, bool round_scale,
                               bool use_ue8m0, const int32_t* rank_mask, int32_t* slot, int32_t* cnt,
                               void* recv_msgs, int32_t* packed_recv_count, int64_t* layout_range,
                               int32_t* stats, int32_t* status, cudaStream_t stream);

cudaError_t launch_bounded_wait_selftest(uint32_t max_iterations, int rank, int32_t* rank_mask, int32_t* status,
                                         cudaStream_t stream);

cudaError_t launch_ll_combine(const LaunchPlan& plan, int R, int T, int maxT, int H, int K, int E,
                              const void* y, int64_t y_row_bytes, const int64_t* topk_idx, const float* topk_weights,
                              const int32_t* slot, void* out, cudaStream_t stream);

}  // namespace ep

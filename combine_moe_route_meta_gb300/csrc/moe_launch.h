// moe_launch.h -- host-side launch interface between the C-ABI entry points and the kernels.
// Arguments arrive here already validated by moe_abi.cu.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace moe {

// Launch-time facts about the current device, queried once per entry-point call.
struct LaunchCtx {
    cudaStream_t stream;
    int num_sms;
};

// Route metadata: pairs are cut into chunks of 1024*R consecutive pairs, one per
// thread block. One block handles everything when n_pairs <= kRouteSingleMax.
constexpr int kRouteThreads = 1024;
constexpr int kRouteRMax = 16;
constexpr int64_t kRouteSingleMax = 8192;
constexpr int kRouteTargetBlocks = 128;

struct RoutePlan {
    bool single;
    int rounds;        // R: rounds of 32 pairs per warp
    int blocks;        // B
    size_t ws_bytes;   // scratch: ticket + per-block count table [B][E]
};
RoutePlan plan_route_meta(int64_t n_pairs, int num_experts);

cudaError_t launch_route_meta(const LaunchCtx& ctx, const RoutePlan& plan, const int32_t* topk_ids,
                              int64_t n_pairs, int K, int E, int P, int M, int64_t* seg_indptr,
                              int32_t* src2dst, int32_t* reorder_topk_ids, int32_t* masked_m,
                              int32_t* partition_counts, void* workspace, int32_t* dev_status);

cudaError_t launch_dispatch(const LaunchCtx& ctx, int mode, int quant, const uint16_t* x, int64_t T,
                            int H, const int32_t* topk_ids, int K, int E, int M,
                            const int32_t* src2dst, const int64_t* seg_indptr, float global_scale,
                            void* out_q, void* out_scales, int32_t* dev_status);

cudaError_t launch_convert_probe(const LaunchCtx& ctx, const float* in, int64_t n, uint8_t* e4m3,
                                 uint8_t* e2m1, float* e4m3_value);

cudaError_t launch_combine(const LaunchCtx& ctx, int mode, const uint16_t* expert_out, int64_t T,
                           int H, int K, int E, int M, const int32_t* topk_ids,
                           const int32_t* src2dst, const int64_t* seg_indptr,
                           const float* topk_weights, uint16_t* out, int32_t* dev_status);

}  // namespace moe

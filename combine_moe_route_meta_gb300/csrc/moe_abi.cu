// moe_abi.cu -- the extern "C" entry points declared in include/moe_dispatch.h (the hot path)
// and include/moe_diag.h (test hooks).
//
// Each entry point validates its arguments on the host (returning a status and launching
// nothing on failure), reads the SM count of the current device, and hands the launch to
// the kernel files. The library allocates no memory and keeps no state between calls.
#include <climits>
#include <cstdint>
#include <cuda_runtime.h>

#include "moe_diag.h"
#include "moe_dispatch.h"
#include "moe_launch.h"

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

moe_status_t make_ctx(moe_stream_t stream, moe::LaunchCtx* ctx) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MOE_ERR_CUDA;
    ctx->stream = reinterpret_cast<cudaStream_t>(stream);
    ctx->num_sms = sms > 0 ? sms : 1;
    ctx->device = dev;
    return MOE_OK;
}

moe_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// shared checks of (T, K, E)
moe_status_t check_shape(int64_t T, int K, int E) {
    if (T < 0) return MOE_ERR_INVALID_ARG;
    if (K < 1 || E < 1) return MOE_ERR_INVALID_ARG;
    if (K > MOE_MAX_TOPK || E > MOE_MAX_EXPERTS) return MOE_ERR_UNSUPPORTED;
    if (T > 0 && T > int64_t(INT32_MAX) / K) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

}  // namespace

extern "C" {

int moe_abi_version(void) { return MOE_ABI_VERSION; }

const char* moe_status_string(moe_status_t s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: invalid argument (size, null or misaligned pointer)";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: size beyond the library's limits";
        case MOE_ERR_CAPACITY: return "MOE_ERR_CAPACITY: an expert received more than max_tokens_per_expert pairs";
        case MOE_ERR_BAD_EXPERT_ID: return "MOE_ERR_BAD_EXPERT_ID: an expert id outside [-1, num_experts) was skipped";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT: a bounded device wait gave up";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA runtime call or launch failed";
        default: return "MOE_ERR_UNKNOWN";
    }
}

size_t moe_route_meta_workspace_size(int64_t num_tokens, int topk, int num_experts) {
    if (check_shape(num_tokens, topk, num_experts) != MOE_OK) return 0;
    return moe::plan_route_meta(num_tokens * topk, num_experts).ws_bytes;
}

static moe_status_t route_meta_impl(const void* topk_ids, int ids_bytes, int64_t num_tokens, int topk,
                                    int num_experts, int num_partitions, int max_tokens_per_expert,
                                    int expert_alignment, int64_t* seg_indptr, int32_t* src2dst,
                                    int32_t* reorder_topk_ids, int32_t* masked_m, int32_t* partition_counts,
                                    int32_t* ids_out, int32_t* expected_m_host, void* workspace,
                                    size_t workspace_bytes, int32_t* dev_status, moe_stream_t stream) {
    if (ids_bytes != 4 && ids_bytes != 8) return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_shape(num_tokens, topk, num_experts);
    if (st != MOE_OK) return st;
    if (num_partitions < 1 || num_experts % num_partitions != 0) return MOE_ERR_INVALID_ARG;
    if (max_tokens_per_expert < 0) return MOE_ERR_INVALID_ARG;
    if (expert_alignment < 1) return MOE_ERR_INVALID_ARG;
    if (expert_alignment > 1024) return MOE_ERR_UNSUPPORTED;
    const int64_t n_pairs = num_tokens * topk;
    if (n_pairs + int64_t(num_experts) * (expert_alignment - 1) > int64_t(INT32_MAX)) return MOE_ERR_UNSUPPORTED;
    if (!seg_indptr || !masked_m || !dev_status) return MOE_ERR_INVALID_ARG;
    if ((n_pairs > 0 || expert_alignment > 1) && !reorder_topk_ids) return MOE_ERR_INVALID_ARG;
    if (n_pairs > 0 && (!topk_ids || !src2dst)) return MOE_ERR_INVALID_ARG;
    if (!aligned(seg_indptr, 8) || !aligned(topk_ids, uintptr_t(ids_bytes)) || !aligned(src2dst, 4) ||
        !aligned(reorder_topk_ids, 4) || !aligned(masked_m, 4) || !aligned(partition_counts, 4) ||
        !aligned(ids_out, 4) || !aligned(dev_status, 4))
        return MOE_ERR_INVALID_ARG;
    const moe::RoutePlan plan = moe::plan_route_meta(n_pairs, num_experts);
    if (plan.ws_bytes > 0 && (!workspace || workspace_bytes < plan.ws_bytes || !aligned(workspace, 256)))
        return MOE_ERR_INVALID_ARG;
    moe::LaunchCtx ctx;
    st = make_ctx(stream, &ctx);
    if (st != MOE_OK) return st;
    if (expected_m_host) *expected_m_host = int32_t((n_pairs + num_experts) / num_experts);
    const bool i64 = ids_bytes == 8;
    return from_cuda(moe::launch_route_meta(
        ctx, plan, i64 ? nullptr : static_cast<const int32_t*>(topk_ids), n_pairs, topk, num_experts,
        num_partitions, max_tokens_per_expert, seg_indptr, src2dst, reorder_topk_ids, masked_m, partition_counts,
        workspace, dev_status, expert_alignment, i64 ? static_cast<const int64_t*>(topk_ids) : nullptr, ids_out));
}

moe_status_t moe_route_meta(const int32_t* topk_ids, int64_t num_tokens, int topk, int num_experts,
                            int num_partitions, int max_tokens_per_expert, int64_t* seg_indptr,
                            int32_t* src2dst, int32_t* reorder_topk_ids, int32_t* masked_m,
                            int32_t* partition_counts, int32_t* expected_m_host, void* workspace,
                            size_t workspace_bytes, int32_t* dev_status, moe_stream_t stream) {
    return route_meta_impl(topk_ids, 4, num_tokens, topk, num_experts, num_partitions, max_tokens_per_expert, 1,
                           seg_indptr, src2dst, reorder_topk_ids, masked_m, partition_counts, nullptr,
                           expected_m_host, workspace, workspace_bytes, dev_status, stream);
}

moe_status_t moe_route_meta_ex(const void* topk_ids, int topk_ids_bytes, int64_t num_tokens, int topk,
                               int num_experts, int num_partitions, int max_tokens_per_expert,
                               int expert_alignment, int64_t* seg_indptr, int32_t* src2dst,
                               int32_t* reorder_topk_ids, int32_t* masked_m, int32_t* partition_counts,
                               int32_t* topk_ids_i32_out, int32_t* expected_m_host, void* workspace,
                               size_t workspace_bytes, int32_t* dev_status, moe_stream_t stream) {
    return route_meta_impl(topk_ids, topk_ids_bytes, num_tokens, topk, num_experts, num_partitions,
                           max_tokens_per_expert, expert_alignment, seg_indptr, src2dst, reorder_topk_ids,
                           masked_m, partition_counts, topk_ids_i32_out, expected_m_host, workspace,
                           workspace_bytes, dev_status, stream);
}

static bool valid_quant(moe_quant_t q) {
    return q == MOE_QUANT_NONE || q == MOE_QUANT_FP8_G128 || q == MOE_QUANT_NVFP4_B16 ||
           q == MOE_QUANT_FP8_G128_UE8M0 || q == MOE_QUANT_FP8_PASSTHROUGH;
}

// A pass-through row of H one-byte codes moves exactly like a bf16 row of H/2 elements.
static void passthrough_as_copy(moe_quant_t* q, int* hidden) {
    if (*q == MOE_QUANT_FP8_PASSTHROUGH) {
        *q = MOE_QUANT_NONE;
        *hidden /= 2;
    }
}

static bool is_fp8(moe_quant_t q) { return q == MOE_QUANT_FP8_G128 || q == MOE_QUANT_FP8_G128_UE8M0; }

static moe_status_t dispatch_impl(moe_mode_t mode, moe_quant_t quant, moe_scale_layout_t layout,
                                  const uint16_t* hidden_states, int64_t num_tokens, int hidden,
                                  const int32_t* topk_ids, int topk, int num_experts, int max_tokens_per_expert,
                                  int64_t out_rows, const int32_t* src2dst, const int64_t* seg_indptr,
                                  float input_global_scale, void* out_q, void* out_scales, int32_t* dev_status,
                                  moe_stream_t stream) {
    if (mode != MOE_MODE_NORMAL && mode != MOE_MODE_MASKED) return MOE_ERR_INVALID_ARG;
    if (!valid_quant(quant)) return MOE_ERR_INVALID_ARG;
    if (layout != MOE_SCALES_ROW_MAJOR && layout != MOE_SCALES_COL_MAJOR && layout != MOE_SCALES_SWIZZLED_128X4)
        return MOE_ERR_INVALID_ARG;
    if (layout == MOE_SCALES_COL_MAJOR && !is_fp8(quant)) return MOE_ERR_INVALID_ARG;
    if (layout == MOE_SCALES_SWIZZLED_128X4 && (quant != MOE_QUANT_NVFP4_B16 || hidden % 64 != 0))
        return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_shape(num_tokens, topk, num_experts);
    if (st != MOE_OK) return st;
    if (hidden <= 0 || hidden % 16 != 0) return MOE_ERR_INVALID_ARG;
    if (is_fp8(quant) && hidden % 128 != 0) return MOE_ERR_INVALID_ARG;
    if (quant == MOE_QUANT_FP8_PASSTHROUGH && hidden % 32 != 0) return MOE_ERR_INVALID_ARG;
    passthrough_as_copy(&quant, &hidden);
    const bool masked = mode == MOE_MODE_MASKED;
    if (masked && max_tokens_per_expert < 1) return MOE_ERR_INVALID_ARG;
    if (!masked && out_rows != 0 && out_rows < num_tokens * topk) return MOE_ERR_INVALID_ARG;
    if (!dev_status) return MOE_ERR_INVALID_ARG;
    if (num_tokens == 0) return MOE_OK;
    if (!hidden_states || !src2dst || !out_q) return MOE_ERR_INVALID_ARG;
    if (masked && (!topk_ids || !seg_indptr)) return MOE_ERR_INVALID_ARG;
    if (quant != MOE_QUANT_NONE && !out_scales) return MOE_ERR_INVALID_ARG;
    if (!aligned(hidden_states, 16) || !aligned(out_q, 16) || !aligned(src2dst, 4) ||
        !aligned(topk_ids, 4) || !aligned(seg_indptr, 8) || !aligned(dev_status, 4))
        return MOE_ERR_INVALID_ARG;
    if ((quant == MOE_QUANT_FP8_G128 || layout == MOE_SCALES_SWIZZLED_128X4) && !aligned(out_scales, 4))
        return MOE_ERR_INVALID_ARG;
    moe::LaunchCtx ctx;
    st = make_ctx(stream, &ctx);
    if (st != MOE_OK) return st;
    return from_cuda(moe::launch_dispatch(ctx, int(mode), int(quant), hidden_states, num_tokens,
                                          hidden, topk_ids, topk, num_experts,
                                          masked ? max_tokens_per_expert : 0, src2dst, seg_indptr,
                                          input_global_scale, out_q, out_scales, dev_status, int(layout),
                                          masked ? 0 : out_rows));
}

moe_status_t moe_dispatch(moe_mode_t mode, moe_quant_t quant, const uint16_t* hidden_states,
                          int64_t num_tokens, int hidden, const int32_t* topk_ids, int topk,
                          int num_experts, int max_tokens_per_expert, const int32_t* src2dst,
                          const int64_t* seg_indptr, float input_global_scale, void* out_q,
                          void* out_scales, int32_t* dev_status, moe_stream_t stream) {
    return dispatch_impl(mode, quant, MOE_SCALES_ROW_MAJOR, hidden_states, num_tokens, hidden, topk_ids, topk,
                         num_experts, max_tokens_per_expert, 0, src2dst, seg_indptr, input_global_scale, out_q,
                         out_scales, dev_status, stream);
}

moe_status_t moe_dispatch_ex(moe_mode_t mode, moe_quant_t quant, moe_scale_layout_t scale_layout,
                             const uint16_t* hidden_states, int64_t num_tokens, int hidden,
                             const int32_t* topk_ids, int topk, int num_experts, int max_tokens_per_expert,
                             int64_t out_rows, const int32_t* src2dst, const int64_t* seg_indptr,
                             float input_global_scale, void* out_q, void* out_scales, int32_t* dev_status,
                             moe_stream_t stream) {
    return dispatch_impl(mode, quant, scale_layout, hidden_states, num_tokens, hidden, topk_ids, topk, num_experts,
                         max_tokens_per_expert, out_rows, src2dst, seg_indptr, input_global_scale, out_q,
                         out_scales, dev_status, stream);
}

moe_status_t moe_route_dispatch(moe_mode_t mode, moe_quant_t quant, const uint16_t* hidden_states,
                                int64_t num_tokens, int hidden, const int32_t* topk_ids, int topk,
                                int num_experts, int num_partitions, int max_tokens_per_expert,
                                float input_global_scale, int64_t* seg_indptr, int32_t* src2dst,
                                int32_t* reorder_topk_ids, int32_t* masked_m, int32_t* partition_counts,
                                int32_t* expected_m_host, void* workspace, size_t workspace_bytes,
                                void* out_q, void* out_scales, int32_t* dev_status, moe_stream_t stream) {
    if (mode != MOE_MODE_NORMAL && mode != MOE_MODE_MASKED) return MOE_ERR_INVALID_ARG;
    if (!valid_quant(quant)) return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_shape(num_tokens, topk, num_experts);
    if (st != MOE_OK) return st;
    if (num_partitions < 1 || num_experts % num_partitions != 0) return MOE_ERR_INVALID_ARG;
    if (hidden <= 0 || hidden % 16 != 0) return MOE_ERR_INVALID_ARG;
    if (is_fp8(quant) && hidden % 128 != 0) return MOE_ERR_INVALID_ARG;
    if (quant == MOE_QUANT_FP8_PASSTHROUGH && hidden % 32 != 0) return MOE_ERR_INVALID_ARG;
    passthrough_as_copy(&quant, &hidden);
    const bool masked = mode == MOE_MODE_MASKED;
    if (masked ? max_tokens_per_expert < 1 : max_tokens_per_expert < 0) return MOE_ERR_INVALID_ARG;
    if (!seg_indptr || !masked_m || !dev_status) return MOE_ERR_INVALID_ARG;
    const int64_t n_pairs = num_tokens * topk;
    if (n_pairs > 0 && (!topk_ids || !src2dst || !reorder_topk_ids || !hidden_states || !out_q))
        return MOE_ERR_INVALID_ARG;
    if (n_pairs > 0 && quant != MOE_QUANT_NONE && !out_scales) return MOE_ERR_INVALID_ARG;
    if (!aligned(seg_indptr, 8) || !aligned(topk_ids, 4) || !aligned(src2dst, 4) ||
        !aligned(reorder_topk_ids, 4) || !aligned(masked_m, 4) || !aligned(partition_counts, 4) ||
        !aligned(dev_status, 4) || !aligned(hidden_states, 16) || !aligned(out_q, 16))
        return MOE_ERR_INVALID_ARG;
    if (quant == MOE_QUANT_FP8_G128 && !aligned(out_scales, 4)) return MOE_ERR_INVALID_ARG;
    const int M = masked ? max_tokens_per_expert : 0;
    const bool fused = moe::route_dispatch_fusable(num_tokens, topk);
    const moe::RoutePlan plan = moe::plan_route_meta(n_pairs, num_experts);
    if (!fused && plan.ws_bytes > 0 &&
        (!workspace || workspace_bytes < plan.ws_bytes || !aligned(workspace, 256)))
        return MOE_ERR_INVALID_ARG;
    moe::LaunchCtx ctx;
    st = make_ctx(stream, &ctx);
    if (st != MOE_OK) return st;
    if (expected_m_host) *expected_m_host = int32_t((n_pairs + num_experts) / num_experts);
    if (fused)
        return from_cuda(moe::launch_route_dispatch_small(
            ctx, int(mode), int(quant), hidden_states, num_tokens, hidden, topk_ids, topk, num_experts,
            num_partitions, M, input_global_scale, seg_indptr, src2dst, reorder_topk_ids, masked_m,
            partition_counts, out_q, out_scales, dev_status));
    st = from_cuda(moe::launch_route_meta(ctx, plan, topk_ids, n_pairs, topk, num_experts, num_partitions,
                                          M, seg_indptr, src2dst, reorder_topk_ids, masked_m,
                                          partition_counts, workspace, dev_status));
    if (st != MOE_OK || num_tokens == 0) return st;
    return from_cuda(moe::launch_dispatch(ctx, int(mode), int(quant), hidden_states, num_tokens, hidden,
                                          topk_ids, topk, num_experts, M, src2dst, seg_indptr,
                                          input_global_scale, out_q, out_scales, dev_status));
}

static moe_status_t combine_impl(moe_mode_t mode, const uint16_t* expert_out, int64_t num_tokens, int hidden,
                                 int topk, int num_experts, int max_tokens_per_expert, int64_t expert_out_rows,
                                 const int32_t* topk_ids, const int32_t* src2dst, const int64_t* seg_indptr,
                                 const float* topk_weights, uint16_t* out, int32_t* dev_status,
                                 moe_stream_t stream) {
    if (mode != MOE_MODE_NORMAL && mode != MOE_MODE_MASKED) return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_shape(num_tokens, topk, num_experts);
    if (st != MOE_OK) return st;
    if (hidden <= 0 || hidden % 16 != 0) return MOE_ERR_INVALID_ARG;
    const bool masked = mode == MOE_MODE_MASKED;
    if (masked && max_tokens_per_expert < 1) return MOE_ERR_INVALID_ARG;
    if (!masked && expert_out_rows != 0 && expert_out_rows < num_tokens * topk) return MOE_ERR_INVALID_ARG;
    if (!dev_status) return MOE_ERR_INVALID_ARG;
    if (num_tokens == 0) return MOE_OK;
    if (!expert_out || !src2dst || !topk_weights || !out) return MOE_ERR_INVALID_ARG;
    if (masked && (!topk_ids || !seg_indptr)) return MOE_ERR_INVALID_ARG;
    if (!aligned(expert_out, 16) || !aligned(out, 16) || !aligned(src2dst, 4) ||
        !aligned(topk_ids, 4) || !aligned(seg_indptr, 8) || !aligned(topk_weights, 4) ||
        !aligned(dev_status, 4))
        return MOE_ERR_INVALID_ARG;
    moe::LaunchCtx ctx;
    st = make_ctx(stream, &ctx);
    if (st != MOE_OK) return st;
    return from_cuda(moe::launch_combine(ctx, int(mode), expert_out, num_tokens, hidden, topk,
                                         num_experts, masked ? max_tokens_per_expert : 0, topk_ids,
                                         src2dst, seg_indptr, topk_weights, out, dev_status,
                                         masked ? 0 : expert_out_rows));
}

moe_status_t moe_combine(moe_mode_t mode, const uint16_t* expert_out, int64_t num_tokens, int hidden,
                         int topk, int num_experts, int max_tokens_per_expert,
                         const int32_t* topk_ids, const int32_t* src2dst, const int64_t* seg_indptr,
                         const float* topk_weights, uint16_t* out, int32_t* dev_status,
                         moe_stream_t stream) {
    return combine_impl(mode, expert_out, num_tokens, hidden, topk, num_experts, max_tokens_per_expert, 0,
                        topk_ids, src2dst, seg_indptr, topk_weights, out, dev_status, stream);
}

moe_status_t moe_combine_ex(moe_mode_t mode, const uint16_t* expert_out, int64_t num_tokens, int hidden,
                            int topk, int num_experts, int max_tokens_per_expert, int64_t expert_out_rows,
                            const int32_t* topk_ids, const int32_t* src2dst, const int64_t* seg_indptr,
                            const float* topk_weights, uint16_t* out, int32_t* dev_status, moe_stream_t stream) {
    return combine_impl(mode, expert_out, num_tokens, hidden, topk, num_experts, max_tokens_per_expert,
                        expert_out_rows, topk_ids, src2dst, seg_indptr, topk_weights, out, dev_status, stream);
}

moe_status_t moe_dispatch_layout(const int32_t* topk_ids, int64_t num_tokens, int topk, int num_experts,
                                 int num_partitions, int32_t* num_tokens_per_rank, uint8_t* is_token_in_rank,
                                 int32_t* num_tokens_per_expert, int32_t* dev_status, moe_stream_t stream) {
    moe_status_t st = check_shape(num_tokens, topk, num_experts);
    if (st != MOE_OK) return st;
    if (num_partitions < 1 || num_experts % num_partitions != 0) return MOE_ERR_INVALID_ARG;
    if (!num_tokens_per_rank || !dev_status) return MOE_ERR_INVALID_ARG;
    if (num_tokens > 0 && (!topk_ids || !is_token_in_rank)) return MOE_ERR_INVALID_ARG;
    if (!aligned(topk_ids, 4) || !aligned(num_tokens_per_rank, 4) || !aligned(num_tokens_per_expert, 4) ||
        !aligned(dev_status, 4))
        return MOE_ERR_INVALID_ARG;
    moe::LaunchCtx ctx;
    st = make_ctx(stream, &ctx);
    if (st != MOE_OK) return st;
    return from_cuda(moe::launch_dispatch_layout(ctx, topk_ids, num_tokens, topk, num_experts, num_partitions,
                                                 num_tokens_per_rank, is_token_in_rank, num_tokens_per_expert,
                                                 dev_status));
}

static moe_status_t check_partitioned(int64_t T, int64_t S, int H, int K, int E, int P) {
    moe_status_t st = check_shape(T, K, E);
    if (st != MOE_OK) return st;
    if (P < 1 || E % P != 0 || S < T) return MOE_ERR_INVALID_ARG;
    if (P > moe::kMaxPartitionsA2A) return MOE_ERR_UNSUPPORTED;
    if (S > 0 && S * P > int64_t(INT32_MAX) / (K > 0 ? K : 1)) return MOE_ERR_UNSUPPORTED;
    if (H <= 0 || H % 16 != 0) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

static moe_status_t dispatch_partitioned_impl(moe_quant_t quant, moe_scale_layout_t layout,
                                              const uint16_t* hidden_states, int64_t num_tokens,
                                              int64_t num_slots, int hidden, const int32_t* topk_ids,
                                              const float* topk_weights, int topk, int num_experts,
                                              int num_partitions, int32_t invalid_expert_id,
                                              float input_global_scale, void* recv_x, uint8_t* recv_scales,
                                              int32_t* recv_topk_ids, float* recv_topk_weights,
                                              int32_t* dev_status, moe_stream_t stream) {
    if (quant != MOE_QUANT_NONE && quant != MOE_QUANT_NVFP4_B16) return MOE_ERR_INVALID_ARG;
    if (layout != MOE_SCALES_ROW_MAJOR && layout != MOE_SCALES_SWIZZLED_128X4) return MOE_ERR_INVALID_ARG;
    if (layout == MOE_SCALES_SWIZZLED_128X4 &&
        (quant != MOE_QUANT_NVFP4_B16 || hidden % 64 != 0 || !aligned(recv_scales, 4)))
        return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_partitioned(num_tokens, num_slots, hidden, topk, num_experts, num_partitions);
    if (st != MOE_OK) return st;
    if (!dev_status) return MOE_ERR_INVALID_ARG;
    if (num_slots == 0) return MOE_OK;
    if (!recv_topk_ids || !recv_topk_weights || !recv_x) return MOE_ERR_INVALID_ARG;
    if (num_tokens > 0 && (!hidden_states || !topk_ids || !topk_weights)) return MOE_ERR_INVALID_ARG;
    if (quant == MOE_QUANT_NVFP4_B16 && !recv_scales) return MOE_ERR_INVALID_ARG;
    if (!aligned(hidden_states, 16) || !aligned(recv_x, 16) || !aligned(topk_ids, 4) || !aligned(topk_weights, 4) ||
        !aligned(recv_topk_ids, 4) || !aligned(recv_topk_weights, 4) || !aligned(dev_status, 4))
        return MOE_ERR_INVALID_ARG;
    moe::LaunchCtx ctx;
    st = make_ctx(stream, &ctx);
    if (st != MOE_OK) return st;
    return from_cuda(moe::launch_dispatch_partitioned(ctx, int(quant), hidden_states, num_tokens, num_slots, hidden,
                                                      topk_ids, topk_weights, topk, num_experts, num_partitions,
                                                      invalid_expert_id, input_global_scale, recv_x, recv_scales,
                                                      recv_topk_ids, recv_topk_weights, dev_status, int(layout)));
}

moe_status_t moe_dispatch_partitioned(moe_quant_t quant, const uint16_t* hidden_states, int64_t num_tokens,
                                      int64_t num_slots, int hidden, const int32_t* topk_ids,
                                      const float* topk_weights, int topk, int num_experts, int num_partitions,
                                      int32_t invalid_expert_id, float input_global_scale, void* recv_x,
                                      uint8_t* recv_scales, int32_t* recv_topk_ids, float* recv_topk_weights,
                                      int32_t* dev_status, moe_stream_t stream) {
    return dispatch_partitioned_impl(quant, MOE_SCALES_ROW_MAJOR, hidden_states, num_tokens, num_slots, hidden,
                                     topk_ids, topk_weights, topk, num_experts, num_partitions, invalid_expert_id,
                                     input_global_scale, recv_x, recv_scales, recv_topk_ids, recv_topk_weights,
                                     dev_status, stream);
}

moe_status_t moe_dispatch_partitioned_ex(moe_quant_t quant, moe_scale_layout_t scale_layout,
                                         const uint16_t* hidden_states, int64_t num_tokens, int64_t num_slots,
                                         int hidden, const int32_t* topk_ids, const float* topk_weights, int topk,
                                         int num_experts, int num_partitions, int32_t invalid_expert_id,
                                         float input_global_scale, void* recv_x, uint8_t* recv_scales,
                                         int32_t* recv_topk_ids, float* recv_topk_weights, int32_t* dev_status,
                                         moe_stream_t stream) {
    return dispatch_partitioned_impl(quant, scale_layout, hidden_states, num_tokens, num_slots, hidden, topk_ids,
                                     topk_weights, topk, num_experts, num_partitions, invalid_expert_id,
                                     input_global_scale, recv_x, recv_scales, recv_topk_ids, recv_topk_weights,
                                     dev_status, stream);
}

moe_status_t moe_combine_partitioned(const uint16_t* partial, int64_t num_tokens, int64_t num_slots, int hidden,
                                     const int32_t* topk_ids, int topk, int num_experts, int num_partitions,
                                     uint16_t* out, int32_t* dev_status, moe_stream_t stream) {
    moe_status_t st = check_partitioned(num_tokens, num_slots, hidden, topk, num_experts, num_partitions);
    if (st != MOE_OK) return st;
    if (!dev_status) return MOE_ERR_INVALID_ARG;
    if (num_tokens == 0) return MOE_OK;
    if (!partial || !topk_ids || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned(partial, 16) || !aligned(out, 16) || !aligned(topk_ids, 4) || !aligned(dev_status, 4))
        return MOE_ERR_INVALID_ARG;
    moe::LaunchCtx ctx;
    st = make_ctx(stream, &ctx);
    if (st != MOE_OK) return st;
    return from_cuda(moe::launch_combine_partitioned(ctx, partial, num_tokens, num_slots, hidden, topk_ids, topk,
                                                     num_experts, num_partitions, out, dev_status));
}

moe_status_t moe_fp8_division_check(unsigned long long* result, moe_stream_t stream) {
    if (!result || !aligned(result, 8)) return MOE_ERR_INVALID_ARG;
    moe::LaunchCtx ctx;
    moe_status_t st = make_ctx(stream, &ctx);
    if (st != MOE_OK) return st;
    return from_cuda(moe::launch_fp8_division_check(ctx, result));
}

moe_status_t moe_wait_timeout_check(int32_t* dev_status, int64_t limit_ns, int complete, moe_stream_t stream) {
    if (!dev_status || !aligned(dev_status, 4)) return MOE_ERR_INVALID_ARG;
    if (limit_ns <= 0 || limit_ns > 10000000000ll || (complete != 0 && complete != 1)) return MOE_ERR_INVALID_ARG;
    moe::LaunchCtx ctx;
    moe_status_t st = make_ctx(stream, &ctx);
    if (st != MOE_OK) return st;
    return from_cuda(moe::launch_wait_timeout_check(ctx, dev_status, uint64_t(limit_ns), complete));
}

moe_status_t moe_convert_probe(const float* in, int64_t n, uint8_t* e4m3, uint8_t* e2m1,
                               float* e4m3_value, moe_stream_t stream) {
    if (n < 0 || n % 2 != 0) return MOE_ERR_INVALID_ARG;
    if (n == 0) return MOE_OK;
    if (!in || !aligned(in, 8) || !aligned(e4m3_value, 4)) return MOE_ERR_INVALID_ARG;
    moe::LaunchCtx ctx;
    moe_status_t st = make_ctx(stream, &ctx);
    if (st != MOE_OK) return st;
    return from_cuda(moe::launch_convert_probe(ctx, in, n, e4m3, e2m1, e4m3_value));
}

}  // extern "C"

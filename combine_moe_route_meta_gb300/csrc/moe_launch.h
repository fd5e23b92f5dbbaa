// moe_launch.h -- host-side launch interface between the C-ABI entry points and the kernels.
// Arguments arrive here already validated by moe_abi.cu.
#pragma once

#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

namespace moe {

// Launch-time facts about the current device, queried once per entry-point call.
struct LaunchCtx {
    cudaStream_t stream;
    int num_sms;
    int device;
};

// Launch `kern` as a programmatic dependent of the previous kernel in the stream: its
// launch may overlap that kernel's execution, and every kernel of this library executes
// griddepcontrol.wait before its first global-memory access, so it still sees all of the
// previous kernel's writes.
template <typename Kernel, typename... Args>
cudaError_t launch_pdl(const LaunchCtx& ctx, Kernel kern, dim3 grid, dim3 block, size_t smem, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = ctx.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Resident blocks per SM of `kern` at (threads, smem), cached per device and kernel: the
// answer depends only on the compiled kernel and the device, so it is queried once.
// Kernels that cannot be resident at all report 0.
template <typename Kernel>
cudaError_t blocks_per_sm(const LaunchCtx& ctx, Kernel kern, int threads, size_t smem, int* out) {
    constexpr int kDevices = 64, kSlots = 16;
    struct Entry {
        const void* fn;
        int threads;
        size_t smem;
        int value;  // -1: not cached
    };
    static std::mutex mu;
    static Entry cache[kDevices][kSlots];
    static bool init = false;
    const void* fn = reinterpret_cast<const void*>(kern);
    const int dev = ctx.device >= 0 && ctx.device < kDevices ? ctx.device : -1;
    if (dev >= 0) {
        std::lock_guard<std::mutex> lock(mu);
        if (!init) {
            for (auto& row : cache)
                for (Entry& e : row) e = Entry{nullptr, 0, 0, -1};
            init = true;
        }
        for (const Entry& e : cache[dev])
            if (e.value >= 0 && e.fn == fn && e.threads == threads && e.smem == smem) {
                *out = e.value;
                return cudaSuccess;
            }
    }
    int v = 0;
    cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, threads, smem);
    if (err != cudaSuccess) return err;
    if (dev >= 0) {
        std::lock_guard<std::mutex> lock(mu);
        for (Entry& e : cache[dev])
            if (e.value < 0) {
                e = Entry{fn, threads, smem, v};
                break;
            }
    }
    *out = v;
    return cudaSuccess;
}

// Route metadata: pairs are cut into chunks of 1024*R consecutive pairs, one per
// thread block. One block handles everything when n_pairs <= kRouteSingleMax.
constexpr int kRouteThreads = 1024;
constexpr int kRouteRMax = 16;
// one block up to 2048 pairs (2 rounds per warp). Measured after an L2 flush: one block
// 8.5 / 10.2 / 11.3 / 14.3 / 18.4 us at 256 / 1024 / 2048 / 4096 / 8192 pairs, the count +
// place kernels 11.3 / 12.8 / 12.8 / 12.9 / 13.3 us.
constexpr int64_t kRouteSingleMax = 2048;
constexpr int kRouteTargetBlocks = 128;

struct RoutePlan {
    bool single;
    int rounds;        // R: rounds of 32 pairs per warp
    int blocks;        // B
    size_t ws_bytes;   // scratch: the per-block count table [B][E] (int32)
};
RoutePlan plan_route_meta(int64_t n_pairs, int num_experts);

cudaError_t launch_route_meta(const LaunchCtx& ctx, const RoutePlan& plan, const int32_t* topk_ids,
                              int64_t n_pairs, int K, int E, int P, int M, int64_t* seg_indptr,
                              int32_t* src2dst, int32_t* reorder_topk_ids, int32_t* masked_m,
                              int32_t* partition_counts, void* workspace, int32_t* dev_status, int A = 1,
                              const int64_t* topk_ids64 = nullptr, int32_t* ids_out = nullptr);

cudaError_t launch_dispatch(const LaunchCtx& ctx, int mode, int quant, const uint16_t* x, int64_t T,
                            int H, const int32_t* topk_ids, int K, int E, int M,
                            const int32_t* src2dst, const int64_t* seg_indptr, float global_scale,
                            void* out_q, void* out_scales, int32_t* dev_status, int scale_layout = 0,
                            int64_t out_rows = 0);

// The FlashInfer one-row-per-partition layout through the bulk (TMA) dispatch kernels, for
// batches of at least kBulkMinTokens tokens whose rows fit the bulk geometry (bf16 or NVFP4).
// Sets *launched = false, launching nothing, when the bulk path does not apply.
cudaError_t launch_dispatch_partitioned_bulk(const LaunchCtx& ctx, int quant, const uint16_t* x, int64_t T,
                                             int64_t S, int H, const int32_t* ids, const float* w, int K, int E,
                                             int P, int32_t invalid_id, float g, void* recv_x, uint8_t* recv_sf,
                                             int32_t* recv_ids, float* recv_w, int32_t* dev_status,
                                             int scale_layout, bool* launched, bool keep_scales_in_l2 = false);

// moe_dispatch_layout runs as one block (ids staged in shared memory, no memsets, no global
// atomics) up to this many (token, k) pairs. Measured after an L2 flush: one block 10.2 us
// against 13.0 us for memsets + several blocks at 128 x 8 pairs, but 43.0 against 14.6 us at
// 4096 x 8 (one block's time grows by about 1 us per 1000 pairs).
constexpr int64_t kLayoutSingleMaxPairs = 4096;

// Fused route + dispatch for small batches (one kernel, one block per token).
// every block of the fused kernel counts all T*K ids, so its cost grows with T: measured
// against route metadata + dispatch after an L2 flush, fused 8.2 / 11.2 / 20.5 us against
// 13.6 / 16.9 / 21.5 us at 128 / 256 / 512 tokens x 8, but 26.6 against 25.6 us at 1024 x 4
constexpr int64_t kFusedMaxPairs = 4096;
constexpr int64_t kFusedMaxTokens = 512;
bool route_dispatch_fusable(int64_t T, int K);
cudaError_t launch_route_dispatch_small(const LaunchCtx& ctx, int mode, int quant, const uint16_t* x,
                                        int64_t T, int H, const int32_t* topk_ids, int K, int E, int P,
                                        int M, float global_scale, int64_t* seg_indptr, int32_t* src2dst,
                                        int32_t* reorder_topk_ids, int32_t* masked_m,
                                        int32_t* partition_counts, void* out_q, void* out_scales,
                                        int32_t* dev_status);

// The 128 x 4 swizzled NVFP4 scale layout by whole tiles (sf_swizzle.cu): the touched 128-row
// blocks of the [R, C] scale matrix (sf 4-byte aligned, C % 4 == 0) are cleared, the dispatch
// writes its scale rows row-major into the same buffer, and the blocks are then interleaved
// in place.
constexpr int kSfTilesAll = 0;          // contiguous layout: every block of [0, roundup(R, 128))
constexpr int kSfTilesMasked = 1;       // blocks overlapping e*M + [0, min(M, seg[e+1] - seg[e]))
constexpr int kSfTilesPartitioned = 2;  // blocks overlapping p*S + [0, T)
struct SfTiles {
    uint8_t* sf;
    int64_t R;          // rows of the scale matrix
    int C;              // columns (bytes per row), C % 4 == 0
    int kind;
    const int64_t* seg; // masked: seg_indptr [E+1]
    int E, M;           // masked
    int P;              // partitioned
    int64_t S, T;       // partitioned: slots per partition, tokens
    int64_t n_blocks;   // roundup(R, 128) / 128
    int64_t q_per_group;  // CTAs per expert / partition (sf_tiles_q_per_group)
    int32_t* status;      // MOE_ERR_TIMEOUT if a bounded wait of the interleave gives up
    const int32_t* ids;   // partitioned: topk_ids [T, K] (which slots a partition receives)
    int K, ep;            // partitioned: top-k, experts per partition
};
// CTAs per group for groups of about `rows_per_group_guess` touched rows.
int64_t sf_tiles_q_per_group(int64_t rows_per_group_guess, int64_t groups);
// Whether the blocks can be interleaved in place (sf 16-byte aligned, a 128-row block fits in
// shared memory); otherwise the dispatch stores each scale word at its tile position.
bool sf_tiles_interleavable(const SfTiles& a);
// Whether the interleave itself zeroes the rows of a touched block that the dispatch does not
// write (masked and partitioned layouts), so that no clear has to run before the dispatch.
bool sf_tiles_interleave_zeroes(const SfTiles& a);
cudaError_t launch_sf_tiles_clear(const LaunchCtx& ctx, const SfTiles& a);
cudaError_t launch_sf_tiles_interleave(const LaunchCtx& ctx, const SfTiles& a);

// Per-partition layout and the FlashInfer all-to-all layout (partitioned.cu).
constexpr int kMaxPartitionsA2A = 32;
cudaError_t launch_dispatch_layout(const LaunchCtx& ctx, const int32_t* ids, int64_t T, int K, int E, int P,
                                   int32_t* num_tokens_per_rank, uint8_t* is_token_in_rank,
                                   int32_t* num_tokens_per_expert, int32_t* dev_status);
cudaError_t launch_dispatch_partitioned(const LaunchCtx& ctx, int quant, const uint16_t* x, int64_t T, int64_t S,
                                        int H, const int32_t* ids, const float* w, int K, int E, int P,
                                        int32_t invalid_id, float g, void* recv_x, uint8_t* recv_sf,
                                        int32_t* recv_ids, float* recv_w, int32_t* dev_status,
                                        int scale_layout = 0);
cudaError_t launch_combine_partitioned(const LaunchCtx& ctx, const uint16_t* partial, int64_t T, int64_t S, int H,
                                       const int32_t* ids, int K, int E, int P, uint16_t* out, int32_t* dev_status);

cudaError_t launch_wait_timeout_check(const LaunchCtx& ctx, int32_t* status, uint64_t limit_ns, int complete);
cudaError_t launch_fp8_division_check(const LaunchCtx& ctx, unsigned long long* result);
cudaError_t launch_convert_probe(const LaunchCtx& ctx, const float* in, int64_t n, uint8_t* e4m3,
                                 uint8_t* e2m1, float* e4m3_value);

cudaError_t launch_combine(const LaunchCtx& ctx, int mode, const uint16_t* expert_out, int64_t T,
                           int H, int K, int E, int M, const int32_t* topk_ids,
                           const int32_t* src2dst, const int64_t* seg_indptr,
                           const float* topk_weights, uint16_t* out, int32_t* dev_status,
                           int64_t expert_out_rows = 0);

}  // namespace moe

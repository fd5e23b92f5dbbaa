// route_meta.cu -- routing metadata: expert histogram, exclusive scan, stable per-pair rank.
//
// Computes, for the flattened (token, k) pairs i = t*K + k of topk_ids
// (deepep_run_moe_deep_preprocess as consumed by _DeepEPDispatcherImplNormal._deepep_permute,
// "sglang 0.4.4.post2 -> 0.4.4.post4, ep_moe/token_dispatcher.py" diff):
//   seg_indptr[e+1] = seg_indptr[e] + count[e]
//   src2dst[i]      = seg_indptr[id_i] + #{j < i valid : id_j = id_i}   (stable counting sort)
//   reorder_topk_ids[src2dst[i]] = id_i
// plus masked_m / per-partition counts of the low-latency path (deepep.py page).
//
// Design (sm_103a, 1024-thread blocks):
//  * Each block owns a contiguous chunk of 1024*R pairs; each warp a contiguous
//    sub-chunk of 32*R pairs, walked in R rounds of 32 lanes. Within a round,
//    __match_any_sync groups the lanes holding the same expert; the group's lowest
//    lane adds the group size to the warp's shared-memory counter, and each lane's
//    rank inside its warp is that counter plus the number of lower lanes in its group.
//    Walking rounds in order keeps the rank stable (flattened order).
//  * A per-expert exclusive scan over the 32 warp counters turns warp ranks into
//    block ranks and gives the block's histogram.
//  * One block (n_pairs <= 8192): block-wide scan of the histogram -> seg_indptr, and
//    the final positions are written in the same kernel.
//  * Several blocks: each block publishes its histogram row to a [B][E] table and
//    writes block ranks into src2dst. The last block to finish (atomic ticket,
//    threadfence pattern -- no block ever waits for another) scans the table column
//    by column into per-block expert offsets and scans the totals into seg_indptr.
//    A second kernel adds seg_indptr[e] + offset[b][e] to every rank and scatters
//    reorder_topk_ids. Nothing spins, so no wait needs a bound.
#include <cstdint>

#include "moe_device.cuh"
#include "moe_launch.h"

namespace moe {
namespace {

constexpr int kWarps = kRouteThreads / 32;

// workspace layout: [0] ticket (uint32), table at byte offset 256: int32 [B][E]
constexpr size_t kTableOffset = 256;

// Block-wide exclusive scan of one int per thread (blockDim == 1024).
// `warp_sums` is 32 ints of shared memory. Returns the exclusive prefix; *total gets the sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(kFullMask, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[w] = x;
    __syncthreads();
    if (w == 0) {
        int s = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(kFullMask, s, o);
            if (lane >= o) s += y;
        }
        warp_sums[lane] = s;
    }
    __syncthreads();
    const int excl = x - v + (w > 0 ? warp_sums[w - 1] : 0);
    *total = warp_sums[31];
    __syncthreads();
    return excl;
}

// Final per-expert outputs from the histogram held in shared memory.
// hist[e] (e < E) -> seg (shared, E+1 ints), seg_indptr, masked_m, partition_counts.
__device__ void finish_histogram(const int* hist, int* seg, int* warp_sums, int E, int P, int M,
                                 int64_t* seg_indptr, int32_t* masked_m, int32_t* partition_counts,
                                 int32_t* status) {
    const int e = threadIdx.x;  // E <= 1024 == blockDim
    const int c = e < E ? hist[e] : 0;
    int total;
    const int excl = block_exclusive_scan(c, warp_sums, &total);
    if (e < E) {
        seg[e] = excl;
        seg_indptr[e] = excl;
        int mm = c;
        if (M > 0 && c > M) {
            mm = M;
            set_status(status, MOE_ERR_CAPACITY);
        }
        masked_m[e] = mm;
    }
    if (e == 0) {
        seg[E] = total;
        seg_indptr[E] = total;
    }
    __syncthreads();
    if (partition_counts != nullptr && e < P) {
        const int ep = E / P;
        partition_counts[e] = seg[(e + 1) * ep] - seg[e * ep];
    }
}

// Phase 1 of every block: per-warp stable ranks and per-warp counters.
// cnt: shared [32][E]. Fills e_r / rank_r for the R rounds of this thread.
template <int RMAX>
__device__ __forceinline__ void warp_ranks(const int32_t* __restrict__ ids, int64_t n_pairs, int E,
                                           int R, int64_t warp_base, int* cnt, int (&e_r)[RMAX],
                                           int (&rank_r)[RMAX], int32_t* status) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const unsigned lt = (1u << lane) - 1u;
    int* my = cnt + w * E;
    bool bad = false;
#pragma unroll
    for (int r = 0; r < RMAX; r++) {
        e_r[r] = -1;
        rank_r[r] = 0;
        if (r < R) {
            const int64_t i = warp_base + r * 32 + lane;
            int e = -1;
            if (i < n_pairs) {
                e = __ldg(ids + i);
                if (e < -1 || e >= E) {
                    bad = true;
                    e = -1;
                }
                if (e < 0) e = -1;
            }
            const unsigned peers = __match_any_sync(kFullMask, e);
            int base = 0;
            if (e >= 0) base = my[e];
            __syncwarp();
            if (e >= 0 && lane == __ffs(peers) - 1) my[e] = base + __popc(peers);
            __syncwarp();
            e_r[r] = e;
            rank_r[r] = base + __popc(peers & lt);
        }
    }
    if (__any_sync(kFullMask, bad) && lane == 0) set_status(status, MOE_ERR_BAD_EXPERT_ID);
}

// Exclusive scan of cnt[w][e] over the 32 warps, per expert; returns block totals in hist.
__device__ __forceinline__ void scan_warps(int* cnt, int* hist, int E) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = 0;
#pragma unroll 8
        for (int w = 0; w < kWarps; w++) {
            const int c = cnt[w * E + e];
            cnt[w * E + e] = run;
            run += c;
        }
        hist[e] = run;
    }
}

struct RouteArgs {
    const int32_t* ids;
    int64_t n_pairs;
    int E, P, M, R;
    int64_t* seg_indptr;
    int32_t* src2dst;
    int32_t* reorder;
    int32_t* masked_m;
    int32_t* partition_counts;
    unsigned* ticket;
    int32_t* table;  // [B][E]
    int32_t* status;
};

// shared memory: cnt[32][E] | hist[E] | seg[E+1] | warp_sums[32] | flag
__host__ __device__ constexpr size_t route_smem_bytes(int E) {
    return sizeof(int) * (size_t(kWarps) * E + E + (E + 1) + 32 + 1);
}

// One block for all pairs.
template <int RMAX>
__global__ void __launch_bounds__(kRouteThreads, 1) route_meta_single_kernel(RouteArgs a) {
    extern __shared__ int smem[];
    const int E = a.E;
    int* cnt = smem;
    int* hist = cnt + kWarps * E;
    int* seg = hist + E;
    int* warp_sums = seg + E + 1;
    for (int j = threadIdx.x; j < kWarps * E; j += blockDim.x) cnt[j] = 0;
    __syncthreads();
    pdl_launch_dependents();

    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t warp_base = int64_t(w) * 32 * a.R;
    int e_r[RMAX], rank_r[RMAX];
    warp_ranks<RMAX>(a.ids, a.n_pairs, E, a.R, warp_base, cnt, e_r, rank_r, a.status);
    __syncthreads();
    scan_warps(cnt, hist, E);
    __syncthreads();
    finish_histogram(hist, seg, warp_sums, E, a.P, a.M, a.seg_indptr, a.masked_m,
                     a.partition_counts, a.status);
    // finish_histogram ends with __syncthreads: seg[] and the warp offsets in cnt are final
#pragma unroll
    for (int r = 0; r < RMAX; r++) {
        if (r < a.R) {
            const int64_t i = warp_base + r * 32 + lane;
            if (i < a.n_pairs) {
                const int e = e_r[r];
                if (e >= 0) {
                    const int d = seg[e] + cnt[w * E + e] + rank_r[r];
                    a.src2dst[i] = d;
                    a.reorder[d] = e;
                } else {
                    a.src2dst[i] = -1;
                }
            }
        }
    }
}

// Several blocks, kernel 1: block ranks + histogram rows; the last block scans.
template <int RMAX>
__global__ void __launch_bounds__(kRouteThreads, 1) route_meta_count_kernel(RouteArgs a) {
    extern __shared__ int smem[];
    const int E = a.E;
    int* cnt = smem;
    int* hist = cnt + kWarps * E;
    int* seg = hist + E;
    int* warp_sums = seg + E + 1;
    int* flag = warp_sums + 32;
    for (int j = threadIdx.x; j < kWarps * E; j += blockDim.x) cnt[j] = 0;
    __syncthreads();

    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int B = gridDim.x;
    const int64_t block_base = int64_t(blockIdx.x) * kRouteThreads * a.R;
    const int64_t warp_base = block_base + int64_t(w) * 32 * a.R;
    int e_r[RMAX], rank_r[RMAX];
    warp_ranks<RMAX>(a.ids, a.n_pairs, E, a.R, warp_base, cnt, e_r, rank_r, a.status);
    __syncthreads();
    scan_warps(cnt, hist, E);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) a.table[size_t(blockIdx.x) * E + e] = hist[e];
#pragma unroll
    for (int r = 0; r < RMAX; r++) {
        if (r < a.R) {
            const int64_t i = warp_base + r * 32 + lane;
            if (i < a.n_pairs) a.src2dst[i] = e_r[r] >= 0 ? cnt[w * E + e_r[r]] + rank_r[r] : -1;
        }
    }

    // ---- last block: column scan of the [B][E] table, then seg_indptr ----
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) *flag = (atomicInc(a.ticket, unsigned(B - 1)) == unsigned(B - 1));
    __syncthreads();
    if (!*flag) return;
    __threadfence();

    // G threads per expert column, each owning a contiguous run of rows; G <= 32 keeps
    // the partial sums [G][E] inside the cnt[32][E] region they reuse.
    const int G = min(kRouteThreads / E, kWarps);  // >= 1
    const int rows_per = (B + G - 1) / G;
    int* part = cnt;  // reuse: [G][E]
    const int tid = threadIdx.x;
    const int col = tid % E, g = tid / E;
    const bool active = tid < G * E;
    const int b0 = g * rows_per, b1 = min(B, b0 + rows_per);
    int psum = 0;
    if (active) {
        for (int b = b0; b < b1; b++) psum += __ldcg(a.table + size_t(b) * E + col);
        part[g * E + col] = psum;
    }
    __syncthreads();
    if (active) {
        int off = 0;
        for (int g2 = 0; g2 < g; g2++) off += part[g2 * E + col];
        for (int b = b0; b < b1; b++) {
            int32_t* p = a.table + size_t(b) * E + col;
            const int v = __ldcg(p);
            __stcg(p, off);
            off += v;
        }
        if (g == G - 1) hist[col] = off;  // column total
    }
    __syncthreads();
    finish_histogram(hist, seg, warp_sums, E, a.P, a.M, a.seg_indptr, a.masked_m,
                     a.partition_counts, a.status);
}

// Several blocks, kernel 2: final positions.
__global__ void __launch_bounds__(kRouteThreads) route_meta_place_kernel(RouteArgs a) {
    extern __shared__ int base[];  // [E]
    pdl_wait();
    const int E = a.E;
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        base[e] = int(a.seg_indptr[e]) + __ldcg(a.table + size_t(blockIdx.x) * E + e);
    if (blockIdx.x == 0 && threadIdx.x == 0) *a.ticket = 0u;
    __syncthreads();
    const int64_t b0 = int64_t(blockIdx.x) * kRouteThreads * a.R;
    const int64_t b1 = min(a.n_pairs, b0 + int64_t(kRouteThreads) * a.R);
    for (int64_t i = b0 + threadIdx.x; i < b1; i += blockDim.x) {
        const int d = a.src2dst[i];
        if (d >= 0) {
            const int e = __ldg(a.ids + i);
            const int dst = base[e] + d;
            a.src2dst[i] = dst;
            a.reorder[dst] = e;
        }
    }
}

template <int RMAX>
cudaError_t launch_rmax(const LaunchCtx& ctx, const RoutePlan& plan, const RouteArgs& a, int E) {
    const size_t smem = route_smem_bytes(E);
    if (plan.single) {
        auto k = route_meta_single_kernel<RMAX>;
        if (smem > 48 * 1024) {
            cudaError_t err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
            if (err != cudaSuccess) return err;
        }
        k<<<1, kRouteThreads, smem, ctx.stream>>>(a);
        return cudaGetLastError();
    }
    auto k1 = route_meta_count_kernel<RMAX>;
    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (err != cudaSuccess) return err;
    }
    k1<<<plan.blocks, kRouteThreads, smem, ctx.stream>>>(a);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;

    // kernel 2 as a programmatic dependent: its launch overlaps kernel 1's tail and
    // griddepcontrol.wait orders every read after kernel 1's writes.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.blocks);
    cfg.blockDim = dim3(kRouteThreads);
    cfg.dynamicSmemBytes = sizeof(int) * size_t(E);
    cfg.stream = ctx.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, route_meta_place_kernel, a);
}

}  // namespace

RoutePlan plan_route_meta(int64_t n_pairs, int num_experts) {
    RoutePlan p{};
    if (n_pairs <= kRouteSingleMax) {
        p.single = true;
        p.rounds = int(n_pairs > 0 ? (n_pairs + kRouteThreads - 1) / kRouteThreads : 1);
        p.blocks = 1;
        p.ws_bytes = 0;
        return p;
    }
    const int64_t per_round = int64_t(kRouteThreads) * kRouteTargetBlocks;
    int64_t R = (n_pairs + per_round - 1) / per_round;
    if (R < 1) R = 1;
    if (R > kRouteRMax) R = kRouteRMax;
    const int64_t chunk = int64_t(kRouteThreads) * R;
    p.single = false;
    p.rounds = int(R);
    p.blocks = int((n_pairs + chunk - 1) / chunk);
    p.ws_bytes = kTableOffset + sizeof(int32_t) * size_t(p.blocks) * size_t(num_experts);
    return p;
}

cudaError_t launch_route_meta(const LaunchCtx& ctx, const RoutePlan& plan, const int32_t* topk_ids,
                              int64_t n_pairs, int K, int E, int P, int M, int64_t* seg_indptr,
                              int32_t* src2dst, int32_t* reorder_topk_ids, int32_t* masked_m,
                              int32_t* partition_counts, void* workspace, int32_t* dev_status) {
    (void)K;
    RouteArgs a{};
    a.ids = topk_ids;
    a.n_pairs = n_pairs;
    a.E = E;
    a.P = P;
    a.M = M;
    a.R = plan.rounds;
    a.seg_indptr = seg_indptr;
    a.src2dst = src2dst;
    a.reorder = reorder_topk_ids;
    a.masked_m = masked_m;
    a.partition_counts = partition_counts;
    a.status = dev_status;
    if (!plan.single) {
        a.ticket = static_cast<unsigned*>(workspace);
        a.table = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + kTableOffset);
    }
    if (plan.rounds <= 1) return launch_rmax<1>(ctx, plan, a, E);
    if (plan.rounds <= 2) return launch_rmax<2>(ctx, plan, a, E);
    if (plan.rounds <= 4) return launch_rmax<4>(ctx, plan, a, E);
    if (plan.rounds <= 8) return launch_rmax<8>(ctx, plan, a, E);
    return launch_rmax<16>(ctx, plan, a, E);
}

}  // namespace moe

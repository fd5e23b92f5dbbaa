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
//  * One block (n_pairs <= 2048): block-wide scan of the histogram -> seg_indptr, and
//    the final positions are written in the same kernel.
//  * Several blocks: each block publishes its histogram row to a [B][E] table and writes
//    block ranks into src2dst. A second kernel (launched as a programmatic dependent)
//    gives every block the whole table in one batch of L2 loads: the column sums over
//    the rows before its own are its per-expert offsets, the full column sums scanned
//    over the experts are seg_indptr (block 0 writes the per-expert outputs); it then
//    finalises its own pairs. No block ever waits for another, so nothing spins.
#include <algorithm>
#include <climits>
#include <cstdint>

#include "moe_device.cuh"
#include "moe_launch.h"

namespace moe {
namespace {

constexpr int kWarps = kRouteThreads / 32;

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
// Segments are padded to a multiple of A rows (expert_alignment; A = 1: no padding).
// With `write` false only the shared seg[] is produced; with `write` the per-expert outputs
// go to memory (the padding rows of reorder_topk_ids: write_padding).
__device__ void finish_histogram(const int* hist, int* seg, int* warp_sums, int E, int P, int M, int A,
                                 int64_t* seg_indptr, int32_t* masked_m, int32_t* partition_counts,
                                 int32_t* status, bool write = true) {
    const int e = threadIdx.x;  // E <= 1024 == blockDim
    const int c = e < E ? hist[e] : 0;
    const int padded = (c + A - 1) / A * A;
    int total;
    const int excl = block_exclusive_scan(padded, warp_sums, &total);
    if (e < E) {
        seg[e] = excl;
        if (write) {
            seg_indptr[e] = excl;
            int mm = c;
            if (M > 0 && c > M) {
                mm = M;
                set_status(status, MOE_ERR_CAPACITY);
            }
            masked_m[e] = mm;
        }
    }
    if (e == 0) {
        seg[E] = total;
        if (write) seg_indptr[E] = total;
    }
    __syncthreads();
    if (write && partition_counts != nullptr) {
        // warp w sums the histogram over partition w's experts (lane-strided, then reduced)
        const int ep = E / P, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
        for (int p = w; p < P; p += int(blockDim.x >> 5)) {
            int n = 0;
            for (int x = p * ep + lane; x < (p + 1) * ep; x += 32) n += hist[x];
            n = __reduce_add_sync(kFullMask, n);
            if (lane == 0) partition_counts[p] = n;
        }
    }
}

// -1 in reorder_topk_ids on the padding rows [seg[e] + hist[e], seg[e] + roundup(hist[e], A)) of
// every expert's segment (A > 1 only). One warp per expert, its lanes on consecutive rows;
// the experts are dealt out over `parts` blocks, this block taking share `part`. Needs the
// final seg[] (shared, as left by finish_histogram).
__device__ void write_padding(const int* hist, const int* seg, int E, int A, int32_t* reorder, int part, int parts) {
    if (A == 1) return;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = int(blockDim.x >> 5);
    for (int e = part * nw + w; e < E; e += parts * nw) {
        const int c = hist[e];
        const int padded = (c + A - 1) / A * A;
        for (int r = c + lane; r < padded; r += 32) reorder[seg[e] + r] = -1;
    }
}

// Row stride of the per-warp counter table cnt[32][S]: odd, so the 32 lanes of a warp
// reading one expert's column (lane l -> row l) hit 32 different banks.
__host__ __device__ constexpr int cnt_stride(int E) { return E | 1; }

// A pair's expert and in-warp rank packed in one register: rank (< 32*16) above bit 11,
// expert + 1 (0 = no valid expert, E <= 1024) in the low 11 bits.
__device__ __forceinline__ int pack_er(int e, int rank) { return (rank << 11) | (e + 1); }
__device__ __forceinline__ int er_expert(int p) { return (p & 0x7ff) - 1; }
__device__ __forceinline__ int er_rank(int p) { return p >> 11; }

// Phase 1 of every block: per-warp stable ranks and per-warp counters.
// cnt: shared [32][S]. Fills er[r] (packed expert, rank) for the R rounds of this thread.
// Expert id of pair i as int32. int64 ids outside the int32 range map to INT32_MIN / INT32_MAX,
// which are outside [-1, E) and so count as bad ids; ids_out (if set) receives the value.
__device__ __forceinline__ int read_id(const int32_t* __restrict__ ids, const int64_t* __restrict__ ids64,
                                       int64_t i) {
    if (ids64 == nullptr) return __ldg(ids + i);
    const long long v = __ldg(reinterpret_cast<const long long*>(ids64) + i);
    return v < INT32_MIN ? INT32_MIN : (v > INT32_MAX ? INT32_MAX : int(v));
}

template <int RMAX>
__device__ __forceinline__ void warp_ranks(const int32_t* __restrict__ ids, const int64_t* __restrict__ ids64,
                                           int32_t* ids_out, int64_t n_pairs, int E,
                                           int R, int64_t warp_base, int* cnt, int (&er)[RMAX],
                                           int32_t* status) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const unsigned lt = (1u << lane) - 1u;
    int* my = cnt + w * cnt_stride(E);
    bool bad = false;
    // all of this lane's ids first, in one batch of loads (er[r] holds the raw id until
    // round r replaces it with the packed expert and rank)
#pragma unroll
    for (int r = 0; r < RMAX; r++) {
        const int64_t i = warp_base + r * 32 + lane;
        er[r] = (r < R && i < n_pairs) ? read_id(ids, ids64, i) : -1;
    }
#pragma unroll
    for (int r = 0; r < RMAX; r++) {
        if (r < R) {
            const int64_t i = warp_base + r * 32 + lane;
            int e = er[r];
            er[r] = pack_er(-1, 0);
            if (i < n_pairs) {
                if (ids_out != nullptr) ids_out[i] = e;
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
            er[r] = pack_er(e, base + __popc(peers & lt));
        } else {
            er[r] = pack_er(-1, 0);
        }
    }
    if (__any_sync(kFullMask, bad) && lane == 0) set_status(status, MOE_ERR_BAD_EXPERT_ID);
}

// Exclusive scan of cnt[w][e] over the 32 warps, per expert; block totals go to hist.
// Warp v scans the columns e = v, v+32, ...: lane l holds warp l's count, a 5-step
// shuffle scan gives every lane its exclusive prefix, lane 31 the column total.
__device__ __forceinline__ void scan_warps(int* cnt, int* hist, int E) {
    constexpr int kCols = 4;  // columns scanned together, so their shuffles overlap
    const int lane = threadIdx.x & 31, v = threadIdx.x >> 5;
    const int S = cnt_stride(E);
    for (int e0 = v; e0 < E; e0 += kWarps * kCols) {
        int c[kCols], x[kCols];
#pragma unroll
        for (int j = 0; j < kCols; j++) {
            const int e = e0 + j * kWarps;
            c[j] = e < E ? cnt[lane * S + e] : 0;
            x[j] = c[j];
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
            for (int j = 0; j < kCols; j++) {
                const int y = __shfl_up_sync(kFullMask, x[j], o);
                if (lane >= o) x[j] += y;
            }
        }
#pragma unroll
        for (int j = 0; j < kCols; j++) {
            const int e = e0 + j * kWarps;
            if (e < E) {
                cnt[lane * S + e] = x[j] - c[j];
                if (lane == 31) hist[e] = x[j];
            }
        }
    }
}

struct RouteArgs {
    const int32_t* ids;    // int32 ids, or
    const int64_t* ids64;  // int64 ids (exactly one of the two is set)
    int32_t* ids_out;      // optional int32 copy of the ids
    int64_t n_pairs;
    int E, P, M, R;
    int A;  // expert alignment of the segments (1 = none)
    int64_t* seg_indptr;
    int32_t* src2dst;
    int32_t* reorder;
    int32_t* masked_m;
    int32_t* partition_counts;
    int32_t* table;  // [B][E]
    int32_t* status;
};

// shared memory: cnt[32][S] | hist[E] | seg[E+1] | warp_sums[32] | one spare int
__host__ __device__ constexpr size_t route_smem_bytes(int E) {
    return sizeof(int) * (size_t(kWarps) * cnt_stride(E) + E + (E + 1) + 32 + 1);
}

// One block for all pairs.
template <int RMAX>
__global__ void __launch_bounds__(kRouteThreads, 1) route_meta_single_kernel(RouteArgs a) {
    extern __shared__ int smem[];
    const int E = a.E;
    const int S = cnt_stride(E);
    int* cnt = smem;
    int* hist = cnt + kWarps * S;
    int* seg = hist + E;
    int* warp_sums = seg + E + 1;
    for (int j = threadIdx.x; j < kWarps * S; j += blockDim.x) cnt[j] = 0;
    __syncthreads();
    pdl_wait();

    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t warp_base = int64_t(w) * 32 * a.R;
    int er[RMAX];
    warp_ranks<RMAX>(a.ids, a.ids64, a.ids_out, a.n_pairs, E, a.R, warp_base, cnt, er, a.status);
    __syncthreads();
    scan_warps(cnt, hist, E);
    __syncthreads();
    finish_histogram(hist, seg, warp_sums, E, a.P, a.M, a.A, a.seg_indptr, a.masked_m,
                     a.partition_counts, a.status);
    write_padding(hist, seg, E, a.A, a.reorder, 0, 1);
    // finish_histogram ends with __syncthreads: seg[] and the warp offsets in cnt are final
#pragma unroll
    for (int r = 0; r < RMAX; r++) {
        if (r < a.R) {
            const int64_t i = warp_base + r * 32 + lane;
            if (i < a.n_pairs) {
                const int e = er_expert(er[r]);
                if (e >= 0) {
                    const int d = seg[e] + cnt[w * S + e] + er_rank(er[r]);
                    a.src2dst[i] = d;
                    a.reorder[d] = e;
                } else {
                    a.src2dst[i] = -1;
                }
            }
        }
    }
}

// Several blocks, kernel 1: block ranks + histogram rows.
template <int RMAX>
__global__ void __launch_bounds__(kRouteThreads, 1) route_meta_count_kernel(RouteArgs a) {
    extern __shared__ int smem[];
    const int E = a.E;
    const int S = cnt_stride(E);
    int* cnt = smem;
    int* hist = cnt + kWarps * S;
    for (int j = threadIdx.x; j < kWarps * S; j += blockDim.x) cnt[j] = 0;
    __syncthreads();
    pdl_wait();

    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t block_base = int64_t(blockIdx.x) * kRouteThreads * a.R;
    const int64_t warp_base = block_base + int64_t(w) * 32 * a.R;
    int er[RMAX];
    warp_ranks<RMAX>(a.ids, a.ids64, a.ids_out, a.n_pairs, E, a.R, warp_base, cnt, er, a.status);
    __syncthreads();
    scan_warps(cnt, hist, E);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) a.table[size_t(blockIdx.x) * E + e] = hist[e];
#pragma unroll
    for (int r = 0; r < RMAX; r++) {
        if (r < a.R) {
            const int64_t i = warp_base + r * 32 + lane;
            const int e = er_expert(er[r]);
            if (i < a.n_pairs) a.src2dst[i] = e >= 0 ? cnt[w * S + e] + er_rank(er[r]) : -1;
        }
    }
}

// Threads per table column in the column sums (blockDim == kRouteThreads).
__host__ __device__ constexpr int table_cols_g(int E) {
    return kRouteThreads / E < kWarps ? kRouteThreads / E : kWarps;
}

// Column sums of the [B][E] table, read from L2: pre[e] = sum of rows < b (block b's
// per-expert offsets), tot[e] = sum of all rows (the histogram). Every block reads the whole
// table: G threads per column, each a contiguous run of rows fetched kColBatch loads at a
// time. part_pre / part_tot: shared [G][E]. Ends with __syncthreads.
__device__ void table_column_sums(const int32_t* table, int B, int b, int E, int* part_pre, int* part_tot,
                                  int* pre, int* tot) {
    constexpr int kColBatch = 16;
    const int tid = threadIdx.x, G = table_cols_g(E);
    const int rows_per = (B + G - 1) / G;
    const int col = tid % E, g = tid / E;
    if (tid < G * E) {
        const int b0 = g * rows_per, b1 = min(B, b0 + rows_per);
        int p = 0, q = 0;
        for (int c0 = b0; c0 < b1; c0 += kColBatch) {
            int v[kColBatch];
#pragma unroll
            for (int j = 0; j < kColBatch; j++)
                v[j] = c0 + j < b1 ? __ldcg(table + size_t(c0 + j) * E + col) : 0;
#pragma unroll
            for (int j = 0; j < kColBatch; j++) {
                q += v[j];
                p += c0 + j < b ? v[j] : 0;
            }
        }
        part_pre[g * E + col] = p;
        part_tot[g * E + col] = q;
    }
    __syncthreads();
    if (tid < E) {
        int p = 0, q = 0;
        for (int g2 = 0; g2 < G; g2++) {
            p += part_pre[g2 * E + tid];
            q += part_tot[g2 * E + tid];
        }
        pre[tid] = p;
        tot[tid] = q;
    }
    __syncthreads();
}

// Several blocks, kernel 2: column sums of the table -> offsets and seg_indptr; final positions.
// shared memory: part_pre[G][E] | part_tot[G][E] | tot[E] | pre[E] | seg[E+1] | warp_sums[32]
__global__ void __launch_bounds__(kRouteThreads) route_meta_place_kernel(RouteArgs a) {
    extern __shared__ int smem[];
    pdl_wait();
    const int E = a.E, B = gridDim.x, b = blockIdx.x, tid = threadIdx.x;
    const int G = table_cols_g(E);
    int* part_pre = smem;
    int* part_tot = part_pre + G * E;
    int* tot = part_tot + G * E;
    int* pre = tot + E;
    int* seg = pre + E;
    int* warp_sums = seg + E + 1;

    // this thread's first pair (in-block rank and expert) is fetched before the table work
    const int64_t i0 = int64_t(b) * kRouteThreads * a.R;
    const int64_t i1 = min(a.n_pairs, i0 + int64_t(kRouteThreads) * a.R);
    int d_first = -1, e_first = -1;
    if (i0 + tid < i1) {
        d_first = a.src2dst[i0 + tid];
        e_first = read_id(a.ids, a.ids64, i0 + tid);
    }

    table_column_sums(a.table, B, b, E, part_pre, part_tot, pre, tot);
    finish_histogram(tot, seg, warp_sums, E, a.P, a.M, a.A, a.seg_indptr, a.masked_m, a.partition_counts,
                     a.status, b == 0);
    write_padding(tot, seg, E, a.A, a.reorder, b, B);

    for (int64_t i = i0 + tid; i < i1; i += blockDim.x) {
        const bool first = i == i0 + tid;
        const int d = first ? d_first : a.src2dst[i];
        const int e = first ? e_first : read_id(a.ids, a.ids64, i);
        if (d >= 0) {
            const int dst = seg[e] + pre[e] + d;
            a.src2dst[i] = dst;
            a.reorder[dst] = e;
        }
    }
}

template <int RMAX>
cudaError_t launch_single(const LaunchCtx& ctx, const RouteArgs& a, int E) {
    const size_t smem = route_smem_bytes(E);
    auto k = route_meta_single_kernel<RMAX>;
    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (err != cudaSuccess) return err;
    }
    return launch_pdl(ctx, k, dim3(1), dim3(kRouteThreads), smem, a);
}

template <int RMAX>
cudaError_t launch_rmax(const LaunchCtx& ctx, const RoutePlan& plan, const RouteArgs& a, int E) {
    const size_t smem = route_smem_bytes(E);
    if (plan.single) return launch_single<RMAX>(ctx, a, E);
    auto k1 = route_meta_count_kernel<RMAX>;
    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (err != cudaSuccess) return err;
    }
    cudaError_t err = launch_pdl(ctx, k1, dim3(plan.blocks), dim3(kRouteThreads), smem, a);
    if (err != cudaSuccess) return err;
    // kernel 2's launch overlaps kernel 1's tail; griddepcontrol.wait orders its reads
    const int G = table_cols_g(E);
    const size_t smem2 = sizeof(int) * (size_t(2 * G) * E + 3 * size_t(E) + 1 + 32);
    return launch_pdl(ctx, route_meta_place_kernel, dim3(plan.blocks), dim3(kRouteThreads), smem2, a);
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
    // the workspace is the int32 table [B][E]; every block writes its whole row before the
    // place kernel reads any of it, so the table needs no initial contents
    p.ws_bytes = sizeof(int32_t) * size_t(p.blocks) * size_t(num_experts);
    return p;
}

cudaError_t launch_route_meta(const LaunchCtx& ctx, const RoutePlan& plan, const int32_t* topk_ids,
                              int64_t n_pairs, int K, int E, int P, int M, int64_t* seg_indptr,
                              int32_t* src2dst, int32_t* reorder_topk_ids, int32_t* masked_m,
                              int32_t* partition_counts, void* workspace, int32_t* dev_status, int A,
                              const int64_t* topk_ids64, int32_t* ids_out) {
    (void)K;
    RouteArgs a{};
    a.A = A;
    a.ids = topk_ids64 ? nullptr : topk_ids;
    a.ids64 = topk_ids64;
    a.ids_out = ids_out;
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
    if (!plan.single) a.table = static_cast<int32_t*>(workspace);
    if (plan.rounds <= 1) return launch_rmax<1>(ctx, plan, a, E);
    if (plan.rounds <= 2) return launch_rmax<2>(ctx, plan, a, E);
    if (plan.rounds <= 4) return launch_rmax<4>(ctx, plan, a, E);
    if (plan.rounds <= 8) return launch_rmax<8>(ctx, plan, a, E);
    return launch_rmax<16>(ctx, plan, a, E);
}

}  // namespace moe

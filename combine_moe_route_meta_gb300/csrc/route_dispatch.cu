// route_dispatch.cu -- routing metadata and dispatch in one call (moe_route_dispatch).
//
// The call computes what moe_route_meta followed by moe_dispatch compute (histogram,
// exclusive scan and stable rank of deepep_run_moe_deep_preprocess, then the PreReorder /
// low_latency_dispatch gather with fused quantisation -- "sglang 0.4.4.post2 -> 0.4.4.post4,
// ep_moe/token_dispatcher.py" diff, _deepep_permute; "sglang token_dispatcher/deepep.py"
// page, _DeepEPDispatcherImplLowLatency._dispatch_core).
//
// Small batches (the decode regime: T*K <= kFusedMaxPairs, T <= kFusedMaxTokens) run as
// ONE kernel with no communication between blocks. Blocks 0..T-1 each own one token:
//  1. the block issues the loads of its token's row slices first (after griddepcontrol.wait,
//     so the previous kernel's hidden_states and topk_ids are complete);
//  2. for each of its K pairs (expert e_k, flattened index i_k) it needs only two counts
//     over all T*K ids: #{valid ids < e_k} = seg_indptr[e_k] and #{j < i_k : id_j = e_k},
//     the stable rank. The ids are staged in shared memory in one round of loads; all
//     threads then take both counts in one strided pass (register counters), reduce them
//     with the hardware warp reduction and one shared-memory step;
//  3. it writes its K entries of src2dst / reorder_topk_ids, and quantises and stores its
//     row slices into the K destination rows (dispatch_slice.cuh).
// Block T builds the full histogram and its exclusive scan and writes seg_indptr,
// masked_m and the partition counts, in parallel with the token blocks.
// Every block re-reads the T*K ids (at most 16 KB, from L2), which costs far less than a
// second launch and a grid-wide dependency.
// Larger batches: moe_route_meta's kernels, then the dispatch kernel.
#include <cstdint>

#include "dispatch_slice.cuh"
#include "moe_device.cuh"
#include "moe_launch.h"

namespace moe {
namespace {

constexpr int kSlice = 512;
constexpr int kLaneElems = 16;

struct FusedArgs {
    const uint16_t* x;
    const int32_t* ids;
    int T, H, K, E, P, M;
    int n_pairs;
    int units_per_row;
    float g;
    int64_t* seg_indptr;
    int32_t* src2dst;
    int32_t* reorder;
    int32_t* masked_m;
    int32_t* partition_counts;
    void* out_q;
    void* out_s;
    int32_t* status;
};

// In-place exclusive scan of data[0..n) by the whole block (blockDim a multiple of 32).
// Returns the total; data[n] is not touched. warp_sums: 32 ints of shared memory.
__device__ int block_scan_inplace(int* data, int n, int* warp_sums) {
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, nw = blockDim.x >> 5;
    const int per = (n + blockDim.x - 1) / blockDim.x;
    const int b0 = min(n, tid * per), b1 = min(n, b0 + per);
    int local = 0;
    for (int j = b0; j < b1; j++) local += data[j];
    int x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFullMask, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[w] = x;
    __syncthreads();
    if (w == 0) {
        int s = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFullMask, s, o);
            if (lane >= o) s += y;
        }
        warp_sums[lane] = s;  // inclusive over warps
    }
    __syncthreads();
    int run = x - local + (w > 0 ? warp_sums[w - 1] : 0);
    for (int j = b0; j < b1; j++) {
        const int c = data[j];
        data[j] = run;
        run += c;
    }
    const int total = warp_sums[nw - 1];
    __syncthreads();
    return total;
}

// Block T of the fused kernel: histogram, exclusive scan and the per-expert outputs.
__device__ void fused_global_metadata(const FusedArgs& a, int* smem) {
    const int tid = threadIdx.x, lane = tid & 31, E = a.E;
    int* warp_sums = smem;        // [32]
    int* s_seg = smem + 32;       // [E + 1]
    int* s_ids = s_seg + E + 1;   // [n_pairs]
    for (int e = tid; e < E; e += blockDim.x) s_seg[e] = 0;
    stage_to_shared(a.ids, s_ids, a.n_pairs);
    __syncthreads();
    bool bad = false;
    for (int j = tid; j < a.n_pairs; j += blockDim.x) {
        const int v = s_ids[j];
        if (v >= 0 && v < E) atomicAdd(&s_seg[v], 1);
        else if (v != -1) bad = true;
    }
    if (__any_sync(kFullMask, bad) && lane == 0) set_status(a.status, MOE_ERR_BAD_EXPERT_ID);
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) {
        int cnt = s_seg[e];
        if (a.M > 0 && cnt > a.M) {
            cnt = a.M;
            set_status(a.status, MOE_ERR_CAPACITY);
        }
        a.masked_m[e] = cnt;
    }
    const int total = block_scan_inplace(s_seg, E, warp_sums);
    if (tid == 0) s_seg[E] = total;
    __syncthreads();
    for (int e = tid; e <= E; e += blockDim.x) a.seg_indptr[e] = s_seg[e];
    if (a.partition_counts != nullptr) {
        const int ep = E / a.P;
        for (int p = tid; p < a.P; p += blockDim.x) a.partition_counts[p] = s_seg[(p + 1) * ep] - s_seg[p * ep];
    }
}

template <int QUANT, bool MASKED, int KMAX>
__global__ void route_dispatch_small_kernel(FusedArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    pdl_wait();               // the previous kernel's writes (ids, hidden_states) are visible
    if (blockIdx.x == unsigned(a.T)) {
        fused_global_metadata(a, reinterpret_cast<int*>(smem_raw));
        return;
    }
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    int64_t* s_row = reinterpret_cast<int64_t*>(smem_raw);         // [MOE_MAX_TOPK]
    int* s_part = reinterpret_cast<int*>(s_row + MOE_MAX_TOPK);     // [warps][2 * KMAX]
    int* s_ids = s_part + nw * 2 * KMAX;                            // [n_pairs]
    const int t = blockIdx.x, H = a.H, K = a.K, E = a.E;

    // 1. this warp's first row slice, in flight during the counting
    int c = warp;
    int col = c * kSlice + lane * kLaneElems;
    bool active = c < a.units_per_row && col < H;
    LaneSlice sl{make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    if (active) sl = load_slice(a.x + int64_t(t) * H + col);

    // 2. per pair k: less[k] = #{valid ids < e_k}, rank[k] = #{j < i_k : id_j == e_k}
    stage_to_shared(a.ids, s_ids, a.n_pairs);
    __syncthreads();
    const int base = t * K;
    int ek[KMAX], less[KMAX], rank[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; k++) {
        ek[k] = k < K ? s_ids[base + k] : -2;
        less[k] = 0;
        rank[k] = 0;
    }
    for (int j = tid; j < a.n_pairs; j += blockDim.x) {
        const int v = s_ids[j];
        const bool ok = v >= 0;
#pragma unroll
        for (int k = 0; k < KMAX; k++) {
            less[k] += (ok && v < ek[k]) ? 1 : 0;
            rank[k] += (v == ek[k] && j < base + k) ? 1 : 0;
        }
    }
#pragma unroll
    for (int k = 0; k < KMAX; k++) {
        if (k < K) {
            const int l = __reduce_add_sync(kFullMask, less[k]);  // hardware warp reduction
            const int r = __reduce_add_sync(kFullMask, rank[k]);
            if (lane == 0) {
                s_part[warp * 2 * KMAX + k] = l;
                s_part[warp * 2 * KMAX + KMAX + k] = r;
            }
        }
    }
    __syncthreads();

    // 3. this token's metadata entries and destination rows
    if (tid < K) {
        const int k = tid, i = base + k, e = s_ids[i];
        int64_t row = -1;
        if (e >= 0 && e < E) {
            int seg_e = 0, r = 0;
            for (int w = 0; w < nw; w++) {
                seg_e += s_part[w * 2 * KMAX + k];
                r += s_part[w * 2 * KMAX + KMAX + k];
            }
            const int d = seg_e + r;
            a.src2dst[i] = d;
            a.reorder[d] = e;
            row = MASKED ? (r < a.M ? int64_t(e) * a.M + r : -1) : int64_t(d);
        } else {
            a.src2dst[i] = -1;
        }
        s_row[k] = row;
    }
    __syncthreads();

    const int64_t my_row = lane < K ? s_row[lane] : -1;
    while (c < a.units_per_row) {
        quantise_store<QUANT>(sl, active, lane, col, H, K, my_row, a.g, a.out_q, a.out_s);
        c += nw;
        col = c * kSlice + lane * kLaneElems;
        active = c < a.units_per_row && col < H;
        if (active) sl = load_slice(a.x + int64_t(t) * H + col);
    }
}

template <int QUANT, bool MASKED>
cudaError_t launch_fused(const LaunchCtx& ctx, const FusedArgs& a) {
    // K <= 8 (the pages' top-8 routing) gets a specialisation with half the counters
    auto kern = a.K <= 8 ? route_dispatch_small_kernel<QUANT, MASKED, 8>
                         : route_dispatch_small_kernel<QUANT, MASKED, MOE_MAX_TOPK>;
    int threads = a.units_per_row * 32;
    threads = threads < 128 ? 128 : (threads > 512 ? 512 : threads);
    const int kmax = a.K <= 8 ? 8 : MOE_MAX_TOPK;
    const size_t token_smem = sizeof(int64_t) * MOE_MAX_TOPK + sizeof(int) * size_t(threads / 32) * 2 * kmax +
                              sizeof(int) * size_t(a.n_pairs);
    const size_t meta_smem = sizeof(int) * (32 + size_t(a.E) + 1 + size_t(a.n_pairs));
    const size_t smem = token_smem > meta_smem ? token_smem : meta_smem;
    // blocks 0..T-1: one token each; block T: the per-expert outputs
    return launch_pdl(ctx, kern, dim3(a.T + 1), dim3(threads), smem, a);
}

}  // namespace

bool route_dispatch_fusable(int64_t T, int K) {
    return T > 0 && T <= kFusedMaxTokens && T * K <= kFusedMaxPairs;
}

cudaError_t launch_route_dispatch_small(const LaunchCtx& ctx, int mode, int quant, const uint16_t* x,
                                        int64_t T, int H, const int32_t* topk_ids, int K, int E, int P,
                                        int M, float global_scale, int64_t* seg_indptr, int32_t* src2dst,
                                        int32_t* reorder_topk_ids, int32_t* masked_m,
                                        int32_t* partition_counts, void* out_q, void* out_scales,
                                        int32_t* dev_status) {
    FusedArgs a{};
    a.x = x;
    a.ids = topk_ids;
    a.T = int(T);
    a.H = H;
    a.K = K;
    a.E = E;
    a.P = P;
    a.M = M;
    a.n_pairs = int(T * K);
    a.units_per_row = (H + kSlice - 1) / kSlice;
    a.g = global_scale;
    a.seg_indptr = seg_indptr;
    a.src2dst = src2dst;
    a.reorder = reorder_topk_ids;
    a.masked_m = masked_m;
    a.partition_counts = partition_counts;
    a.out_q = out_q;
    a.out_s = out_scales;
    a.status = dev_status;
    const bool masked = mode == MOE_MODE_MASKED;
    switch (quant) {
        case MOE_QUANT_NONE:
            return masked ? launch_fused<MOE_QUANT_NONE, true>(ctx, a) : launch_fused<MOE_QUANT_NONE, false>(ctx, a);
        case MOE_QUANT_FP8_G128:
            return masked ? launch_fused<MOE_QUANT_FP8_G128, true>(ctx, a)
                          : launch_fused<MOE_QUANT_FP8_G128, false>(ctx, a);
        case MOE_QUANT_FP8_G128_UE8M0:
            return masked ? launch_fused<MOE_QUANT_FP8_G128_UE8M0, true>(ctx, a)
                          : launch_fused<MOE_QUANT_FP8_G128_UE8M0, false>(ctx, a);
        default:
            return masked ? launch_fused<MOE_QUANT_NVFP4_B16, true>(ctx, a)
                          : launch_fused<MOE_QUANT_NVFP4_B16, false>(ctx, a);
    }
}

}  // namespace moe

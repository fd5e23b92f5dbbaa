// combine.cu -- weighted reduction of expert outputs back to token order.
//
// Operation (deepep_post_reorder in combine_a, "sglang 0.4.4.post2 -> 0.4.4.post4,
// ep_moe/token_dispatcher.py" diff; low_latency_combine in
// _DeepEPDispatcherImplLowLatency._combine_core, "sglang token_dispatcher/deepep.py" page):
//   out[t, :] = bf16_rn( sum_{k valid, ascending} topk_weights[t,k] * expert_out[row(t,k), :] )
// row = src2dst (normal) or e*M + rank (masked); fp32 fused multiply-add accumulation.
//
// Design: HBM-bound K-way gather. One warp per (token, 512-column slice); each lane owns
// 16 columns, as two runs of 8 placed 256 columns apart so that each warp-wide 16-byte load
// covers 512 contiguous bytes. Lanes 0..K-1 fetch the slot metadata (row, weight) and
// broadcast it by shuffle (the masked layout reads seg_indptr from a shared-memory copy).
// Each lane then issues the loads of up to 8 source rows (2 x 16 B per row, ld.global.nc
// with L1::no_allocate) before consuming any, so a warp keeps 8 KB in flight, and the next
// unit's slot metadata is fetched alongside. Accumulation order is fixed (k ascending)
// and the result is rounded once to bf16 (cvt.rn.bf16x2). A token with no valid slot
// gets zeros. Small grids use smaller blocks so that every SM gets a similar share.
#include <cstdint>

#include "moe_device.cuh"
#include "moe_launch.h"

namespace moe {
namespace {

constexpr int kCombineThreads = 256;
constexpr int kSlice = 512;
constexpr int kLaneElems = 16;  // per lane and slice: two runs of kHalfElems
constexpr int kHalfElems = 8;
constexpr int kBatch = 8;  // source rows in flight per lane

struct CombineArgs {
    const uint16_t* eo;
    int64_t T;
    int H, K, E, M;
    const int32_t* ids;
    const int32_t* src2dst;
    const int64_t* seg;
    const float* w;
    uint16_t* out;
    int32_t* status;
    int units_per_row;
    int64_t n_units;
    int64_t max_row;
};

// Slot metadata of pair t*K + lane as loaded from memory (lanes >= K hold d = -1).
struct SlotMeta {
    int d;    // src2dst
    int e;    // expert id (masked layout only)
    float w;  // topk weight
};

template <bool MASKED>
__device__ __forceinline__ SlotMeta load_slot(const CombineArgs& a, int64_t t, int lane) {
    SlotMeta m{-1, -1, 0.0f};
    if (lane < a.K) {
        const int64_t i = t * a.K + lane;
        m.d = __ldg(a.src2dst + i);
        m.w = __ldg(a.w + i);
        if (MASKED) m.e = __ldg(a.ids + i);
    }
    return m;
}

template <bool MASKED>
__device__ __forceinline__ int64_t slot_row(const CombineArgs& a, const int* s_seg, const SlotMeta& m) {
    if (m.d < 0) return -1;
    if (MASKED) {
        if (m.e < 0 || m.e >= a.E) {
            set_status(a.status, MOE_ERR_BAD_EXPERT_ID);
            return -1;
        }
        const int rank = m.d - s_seg[m.e];
        return (rank >= 0 && rank < a.M) ? int64_t(m.e) * a.M + rank : -1;
    }
    if (m.d < a.max_row) return m.d;
    set_status(a.status, MOE_ERR_INVALID_ARG);
    return -1;
}

template <bool MASKED>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(CombineArgs a) {
    extern __shared__ int s_seg[];  // [E] in masked mode
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const int H = a.H;

    // the first unit's slot metadata is in flight while seg_indptr is staged
    int64_t u = warp;
    SlotMeta meta = load_slot<MASKED>(a, u < a.n_units ? u / a.units_per_row : 0, u < a.n_units ? lane : 32);
    if (MASKED) {
        stage_to_shared(a.seg, s_seg, a.E);
        __syncthreads();
    }

    for (; u < a.n_units; u += nwarps) {
        const int64_t t = u / a.units_per_row;
        // lane l owns columns [8l, 8l+8) and [256+8l, 256+8l+8) of the slice, so each of the
        // warp's two 16-byte loads per row reads 512 contiguous bytes (whole 32-byte sectors)
        const int col0 = int(u - t * a.units_per_row) * kSlice + lane * kHalfElems;
        const int col1 = col0 + kSlice / 2;
        const bool act0 = col0 < H, act1 = col1 < H;  // act1 implies act0
        const int64_t my_row = slot_row<MASKED>(a, s_seg, meta);
        const float my_w = meta.w;

        float acc[kLaneElems];
#pragma unroll
        for (int j = 0; j < kLaneElems; j++) acc[j] = 0.0f;

        for (int k0 = 0; k0 < a.K; k0 += kBatch) {
            int64_t rows[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; j++) {
                const int k = k0 + j;
                rows[j] = __shfl_sync(kFullMask, my_row, k & 31);
                if (k >= a.K || !act0) rows[j] = -1;
            }
            uint4 v[kBatch][2];
#pragma unroll
            for (int j = 0; j < kBatch; j++) {
                v[j][0] = make_uint4(0, 0, 0, 0);
                v[j][1] = v[j][0];
                if (rows[j] >= 0) {
                    const uint16_t* p = a.eo + rows[j] * H;
                    v[j][0] = ld_stream_v4(p + col0);
                    if (act1) v[j][1] = ld_stream_v4(p + col1);
                }
            }
            // the weights are shuffled only now: the row loads above do not wait for them
            // (a weight load may still be in flight from memory when the rows are addressed)
            float wk[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; j++) wk[j] = __shfl_sync(kFullMask, my_w, (k0 + j) & 31);
            // the next unit's slot metadata rides along with this unit's row loads
            if (k0 + kBatch >= a.K) {
                const int64_t un = u + nwarps;
                meta = load_slot<MASKED>(a, un < a.n_units ? un / a.units_per_row : 0, un < a.n_units ? lane : 32);
            }
#pragma unroll
            for (int j = 0; j < kBatch; j++) {
                if (rows[j] >= 0) {
                    float f[16];
                    unpack8(v[j][0], f);
                    unpack8(v[j][1], f + 8);
#pragma unroll
                    for (int e = 0; e < kLaneElems; e++) acc[e] = fmaf(wk[j], f[e], acc[e]);
                }
            }
        }
        uint16_t* dst = a.out + t * H;
        if (act0)
            st_v4(dst + col0, make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                         pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7])));
        if (act1)
            st_v4(dst + col1, make_uint4(pack_bf16x2(acc[8], acc[9]), pack_bf16x2(acc[10], acc[11]),
                                         pack_bf16x2(acc[12], acc[13]), pack_bf16x2(acc[14], acc[15])));
    }
}

template <bool MASKED>
cudaError_t launch_variant(const LaunchCtx& ctx, const CombineArgs& a) {
    auto kern = combine_kernel<MASKED>;
    const size_t smem = MASKED ? sizeof(int) * size_t(a.E) : 0;
    // one wave or less of 256-thread blocks leaves SMs unevenly loaded: use 64 threads
    const int threads = a.n_units < int64_t(ctx.num_sms) * 16 ? 64 : kCombineThreads;
    int per_sm = 0;
    cudaError_t err = blocks_per_sm(ctx, kern, threads, smem, &per_sm);
    if (err != cudaSuccess) return err;
    const int64_t warps_per_block = threads / 32;
    const int64_t need = (a.n_units + warps_per_block - 1) / warps_per_block;
    const int64_t cap = int64_t(ctx.num_sms) * (per_sm > 0 ? per_sm : 1);
    const int grid = int(need < cap ? need : cap);

    return launch_pdl(ctx, kern, dim3(grid), dim3(threads), smem, a);
}

}  // namespace

cudaError_t launch_combine(const LaunchCtx& ctx, int mode, const uint16_t* expert_out, int64_t T,
                           int H, int K, int E, int M, const int32_t* topk_ids,
                           const int32_t* src2dst, const int64_t* seg_indptr,
                           const float* topk_weights, uint16_t* out, int32_t* dev_status,
                           int64_t expert_out_rows) {
    CombineArgs a{};
    a.eo = expert_out;
    a.T = T;
    a.H = H;
    a.K = K;
    a.E = E;
    a.M = M;
    a.ids = topk_ids;
    a.src2dst = src2dst;
    a.seg = seg_indptr;
    a.w = topk_weights;
    a.out = out;
    a.status = dev_status;
    a.units_per_row = (H + kSlice - 1) / kSlice;
    a.n_units = T * a.units_per_row;
    a.max_row = expert_out_rows > 0 ? expert_out_rows : T * K;
    return mode == MOE_MODE_MASKED ? launch_variant<true>(ctx, a) : launch_variant<false>(ctx, a);
}

}  // namespace moe

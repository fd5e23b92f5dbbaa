// dispatch.cu -- gather token rows into expert order, optionally fused with quantisation.
//
// Operation: out[row(i)] = Q(hidden_states[t]) for every valid pair i = t*K + k, with
//   row(i) = src2dst[i]                              (normal: the PreReorder permute of
//            _DeepEPDispatcherImplNormal._deepep_permute, "sglang 0.4.4.post2 -> 0.4.4.post4,
//            ep_moe/token_dispatcher.py" diff)
//   row(i) = e*M + (src2dst[i] - seg_indptr[e])      (masked: the layout of
//            low_latency_dispatch, "sglang token_dispatcher/deepep.py" page)
// and Q one of
//   none     identity (bf16 rows)
//   fp8g128  per 128-element group: s = max(amax, 1e-10) / 448, q = e4m3(x / s)
//            (sglang_per_token_group_quant_fp8 in _DeepEPDispatcherImplNormal.dispatch_a)
//   nvfp4b16 per 16-element block: sf = e4m3((amax / 6) * g), q = e2m1(x * (g / sf))
//            (fp4_quantize in FlashinferDispatcher.dispatch, "sglang
//            token_dispatcher/flashinfer.py" page; use_nvfp4 of low_latency_dispatch)
//
// Design: HBM-bound gather; the read of each token row happens once and the K
// destination rows are written from registers.
//  * Work unit = (token t, a 512-element column slice). One warp per unit; each lane
//    owns 16 consecutive elements (two 16-byte loads with L1::no_allocate).
//  * The K destination rows of the token are resolved by lanes 0..K-1 and broadcast
//    with shuffles while the row loads are in flight.
//  * FP8: a 128-element group spans 8 lanes; its amax is a 3-step xor-shuffle. NVFP4:
//    a 16-element block is one lane, so its amax needs no shuffle.
//  * Every division and multiplication of the quantiser is an explicit
//    round-to-nearest binary32 operation (__fdiv_rn / __fmul_rn), and the conversions
//    are the hardware cvt.rn.satfinite instructions, so the codes are a deterministic
//    function of the input bits.
//  * Stores are 16-byte (bf16, e4m3) or 8-byte (e2m1) vectors; a warp writes a
//    contiguous 1 KB / 512 B / 256 B span of each destination row.
//  * Grid-stride over units with a grid of (SMs x resident blocks); the warp-to-unit
//    order walks a token's slices with neighbouring warps.
#include <cstdint>

#include "moe_device.cuh"
#include "moe_launch.h"

namespace moe {
namespace {

constexpr int kDispatchThreads = 256;
constexpr int kSlice = 512;       // elements per warp unit
constexpr int kLaneElems = 16;    // elements per lane

struct DispatchArgs {
    const uint16_t* x;
    int64_t T;
    int H, K, E, M;
    const int32_t* ids;
    const int32_t* src2dst;
    const int64_t* seg;
    float g;
    void* out_q;
    void* out_s;
    int32_t* status;
    int units_per_row;
    int64_t n_units;
    int64_t max_row;  // exclusive bound on normal-mode rows (T*K)
};

// destination row of pair t*K + lane (lanes >= K return -1)
template <bool MASKED>
__device__ __forceinline__ int64_t dest_row(const DispatchArgs& a, int64_t t, int lane) {
    int64_t row = -1;
    if (lane < a.K) {
        const int64_t i = t * a.K + lane;
        const int d = __ldg(a.src2dst + i);
        if (d >= 0) {
            if (MASKED) {
                const int e = __ldg(a.ids + i);
                if (e >= 0 && e < a.E) {
                    const int64_t rank = int64_t(d) - __ldg(a.seg + e);
                    if (rank >= 0 && rank < a.M) row = int64_t(e) * a.M + rank;
                } else {
                    set_status(a.status, MOE_ERR_BAD_EXPERT_ID);
                }
            } else if (d < a.max_row) {
                row = d;
            } else {
                set_status(a.status, MOE_ERR_INVALID_ARG);
            }
        }
    }
    return row;
}

template <int QUANT, bool MASKED>
__global__ void __launch_bounds__(kDispatchThreads) dispatch_kernel(DispatchArgs a) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const int H = a.H;

    for (int64_t u = warp; u < a.n_units; u += nwarps) {
        const int64_t t = u / a.units_per_row;
        const int col = int(u - t * a.units_per_row) * kSlice + lane * kLaneElems;
        const bool active = col < H;
        uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0;
        if (active) {
            const uint16_t* src = a.x + t * H + col;
            v0 = ld_stream_v4(src);
            v1 = ld_stream_v4(src + 8);
        }
        const int64_t my_row = dest_row<MASKED>(a, t, lane);

        if constexpr (QUANT == MOE_QUANT_NONE) {
            uint16_t* out = static_cast<uint16_t*>(a.out_q);
            for (int k = 0; k < a.K; k++) {
                const int64_t row = __shfl_sync(kFullMask, my_row, k);
                if (row >= 0 && active) {
                    uint16_t* dst = out + row * H + col;
                    st_v4(dst, v0);
                    st_v4(dst + 8, v1);
                }
            }
        } else if constexpr (QUANT == MOE_QUANT_FP8_G128) {
            float f[16];
            unpack8(v0, f);
            unpack8(v1, f + 8);
            float amax = 0.0f;
#pragma unroll
            for (int j = 0; j < 16; j++) amax = fmaxf(amax, fabsf(f[j]));
            // a 128-element group is 8 aligned lanes
            amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 2));
            amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 4));
            const float s = __fdiv_rn(fmaxf(amax, 1e-10f), 448.0f);
            uint32_t w[4];
#pragma unroll
            for (int p = 0; p < 4; p++) {
                const uint32_t lo = e4m3x2(__fdiv_rn(f[4 * p], s), __fdiv_rn(f[4 * p + 1], s));
                const uint32_t hi = e4m3x2(__fdiv_rn(f[4 * p + 2], s), __fdiv_rn(f[4 * p + 3], s));
                w[p] = lo | (hi << 16);
            }
            const uint4 q = make_uint4(w[0], w[1], w[2], w[3]);
            uint8_t* out = static_cast<uint8_t*>(a.out_q);
            float* scales = static_cast<float*>(a.out_s);
            const int groups = H / 128;
            for (int k = 0; k < a.K; k++) {
                const int64_t row = __shfl_sync(kFullMask, my_row, k);
                if (row >= 0 && active) {
                    st_v4(out + row * H + col, q);
                    if ((lane & 7) == 0) scales[row * groups + col / 128] = s;
                }
            }
        } else {  // MOE_QUANT_NVFP4_B16
            float f[16];
            unpack8(v0, f);
            unpack8(v1, f + 8);
            float amax = 0.0f;
#pragma unroll
            for (int j = 0; j < 16; j++) amax = fmaxf(amax, fabsf(f[j]));
            const float tsf = __fmul_rn(__fdiv_rn(amax, 6.0f), a.g);
            const uint32_t sf = e4m3x2(tsf, 0.0f) & 0xffu;
            const float sff = e4m3_value(sf);
            uint2 q = make_uint2(0, 0);
            if (sff != 0.0f) {
                const float r = __fdiv_rn(a.g, sff);
                uint32_t b[8];
#pragma unroll
                for (int p = 0; p < 8; p++) b[p] = e2m1x2(__fmul_rn(f[2 * p], r), __fmul_rn(f[2 * p + 1], r));
                q.x = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
                q.y = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
            }
            uint8_t* out = static_cast<uint8_t*>(a.out_q);
            uint8_t* sfo = static_cast<uint8_t*>(a.out_s);
            for (int k = 0; k < a.K; k++) {
                const int64_t row = __shfl_sync(kFullMask, my_row, k);
                if (row >= 0 && active) {
                    st_v2(out + row * (H / 2) + col / 2, q);
                    sfo[row * (H / 16) + col / 16] = uint8_t(sf);
                }
            }
        }
    }
}

template <int QUANT, bool MASKED>
cudaError_t launch_variant(const LaunchCtx& ctx, const DispatchArgs& a) {
    auto kern = dispatch_kernel<QUANT, MASKED>;
    int per_sm = 0;
    cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDispatchThreads, 0);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) per_sm = 1;
    const int64_t warps_per_block = kDispatchThreads / 32;
    const int64_t need = (a.n_units + warps_per_block - 1) / warps_per_block;
    const int64_t cap = int64_t(ctx.num_sms) * per_sm;
    const int grid = int(need < cap ? need : cap);

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kDispatchThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = ctx.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

__global__ void convert_probe_kernel(const float* __restrict__ in, int64_t n_pairs, uint8_t* e4m3,
                                     uint8_t* e2m1, float* e4m3_val) {
    for (int64_t j = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; j < n_pairs;
         j += int64_t(gridDim.x) * blockDim.x) {
        const float lo = in[2 * j], hi = in[2 * j + 1];
        const uint32_t w = e4m3x2(lo, hi);
        if (e4m3 != nullptr) {
            e4m3[2 * j] = uint8_t(w & 0xffu);
            e4m3[2 * j + 1] = uint8_t(w >> 8);
        }
        if (e2m1 != nullptr) e2m1[j] = uint8_t(e2m1x2(lo, hi));
        if (e4m3_val != nullptr) {
            e4m3_val[2 * j] = e4m3_value(w & 0xffu);
            e4m3_val[2 * j + 1] = e4m3_value(w >> 8);
        }
    }
}

}  // namespace

cudaError_t launch_convert_probe(const LaunchCtx& ctx, const float* in, int64_t n, uint8_t* e4m3,
                                 uint8_t* e2m1, float* e4m3_value) {
    const int64_t pairs = n / 2;
    int64_t blocks = (pairs + 255) / 256;
    if (blocks > int64_t(ctx.num_sms) * 8) blocks = int64_t(ctx.num_sms) * 8;
    if (blocks < 1) blocks = 1;
    convert_probe_kernel<<<int(blocks), 256, 0, ctx.stream>>>(in, pairs, e4m3, e2m1, e4m3_value);
    return cudaGetLastError();
}

cudaError_t launch_dispatch(const LaunchCtx& ctx, int mode, int quant, const uint16_t* x, int64_t T,
                            int H, const int32_t* topk_ids, int K, int E, int M,
                            const int32_t* src2dst, const int64_t* seg_indptr, float global_scale,
                            void* out_q, void* out_scales, int32_t* dev_status) {
    DispatchArgs a{};
    a.x = x;
    a.T = T;
    a.H = H;
    a.K = K;
    a.E = E;
    a.M = M;
    a.ids = topk_ids;
    a.src2dst = src2dst;
    a.seg = seg_indptr;
    a.g = global_scale;
    a.out_q = out_q;
    a.out_s = out_scales;
    a.status = dev_status;
    a.units_per_row = (H + kSlice - 1) / kSlice;
    a.n_units = T * a.units_per_row;
    a.max_row = T * K;
    const bool masked = mode == MOE_MODE_MASKED;
    switch (quant) {
        case MOE_QUANT_NONE:
            return masked ? launch_variant<MOE_QUANT_NONE, true>(ctx, a)
                          : launch_variant<MOE_QUANT_NONE, false>(ctx, a);
        case MOE_QUANT_FP8_G128:
            return masked ? launch_variant<MOE_QUANT_FP8_G128, true>(ctx, a)
                          : launch_variant<MOE_QUANT_FP8_G128, false>(ctx, a);
        default:
            return masked ? launch_variant<MOE_QUANT_NVFP4_B16, true>(ctx, a)
                          : launch_variant<MOE_QUANT_NVFP4_B16, false>(ctx, a);
    }
}

}  // namespace moe

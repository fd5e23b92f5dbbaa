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
//  * Work unit = (token t, a 512-element column slice). One warp per unit; each lane owns
//    16 consecutive elements (two 16-byte loads with L1::no_allocate).
//  * The K destination rows of the token are resolved by lanes 0..K-1 and broadcast
//    with shuffles while the row loads are in flight. In the masked layout the block
//    first stages seg_indptr in shared memory, so a slot index costs no dependent load.
//  * FP8: a 128-element group spans 8 lanes; its amax is a 3-step xor-shuffle. NVFP4:
//    a 16-element block is one lane, so its amax needs no shuffle (dispatch_slice.cuh).
//  * Stores are 16-byte (bf16, e4m3) or 8-byte (e2m1) vectors; a warp writes a
//    contiguous 1 KB / 512 B / 256 B span of each destination row.
//  * Grid-stride over units with a grid of (SMs x resident blocks); the warp-to-unit
//    order walks a token's slices with neighbouring warps.
#include <algorithm>
#include <cstdint>

#include "dispatch_slice.cuh"
#include "moe_device.cuh"
#include "moe_launch.h"

namespace moe {
namespace {

constexpr int kDispatchThreads = 256;
constexpr int kSlice = 512;       // elements per warp unit
constexpr int kLaneElems = 16;    // elements per lane
constexpr int64_t kBulkMinTokens = 1024;  // the bulk (TMA) path for batches this large

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
    int64_t max_row;  // exclusive bound on normal-mode rows (the output's row capacity)
    ScaleLayout L;
    // one-row-per-partition destinations (FlashInfer layout, bulk kernels with PART): row
    // p*S + t for every partition p < P owning one of token t's experts, plus the receive ids
    // (sanitised to invalid_id) and weights of every partition's row of the token
    int P, ep;
    int64_t S;
    int32_t invalid_id;
    const float* w;
    int32_t* recv_ids;
    float* recv_w;
    // the scale rows are read back by a later kernel of the call (the swizzled layout's
    // in-place interleave): bulk kernels store them with an L2 evict-last policy
    bool keep_scales_in_l2;
};

// destination row of pair t*K + lane (lanes >= K return -1); s_seg: seg_indptr in smem
template <bool MASKED>
__device__ __forceinline__ int64_t dest_row(const DispatchArgs& a, const int* s_seg, int64_t t, int lane) {
    int64_t row = -1;
    if (lane < a.K) {
        const int64_t i = t * a.K + lane;
        const int d = __ldg(a.src2dst + i);
        if (d >= 0) {
            if (MASKED) {
                const int e = __ldg(a.ids + i);
                if (e >= 0 && e < a.E) {
                    const int rank = d - s_seg[e];
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
    extern __shared__ int s_seg[];  // [E] in masked mode
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const int H = a.H;

    // the first unit's row slice is in flight while seg_indptr is staged
    int64_t u = warp;
    int64_t t = u < a.n_units ? u / a.units_per_row : 0;
    int col = int(u - t * a.units_per_row) * kSlice + lane * kLaneElems;
    bool active = u < a.n_units && col < H;
    LaneSlice sl{make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    if (active) sl = load_slice(a.x + t * H + col);
    if (MASKED) {
        stage_to_shared(a.seg, s_seg, a.E);
        __syncthreads();
    }

    while (u < a.n_units) {
        const int64_t my_row = dest_row<MASKED>(a, s_seg, t, lane);
        quantise_store<QUANT>(sl, active, lane, col, H, a.K, my_row, a.g, a.out_q, a.out_s, a.L);
        u += nwarps;
        if (u >= a.n_units) break;
        t = u / a.units_per_row;
        col = int(u - t * a.units_per_row) * kSlice + lane * kLaneElems;
        active = col < H;
        if (active) sl = load_slice(a.x + t * H + col);
    }
}

// ---------------------------------------------------------------------------
// Bulk (TMA) path for large batches: one token row at a time per CTA. The row is
// bulk-loaded into a shared-memory ring (mbarrier completion, loads issued NS-1 tokens
// ahead); the quantising modes turn it into the quantised row + scale row in shared
// memory; then one bulk store per destination row (and per scale row) writes whole rows.
// Whole-row bulk stores keep each destination's bytes together in DRAM (a probe of this
// pattern ran at 5.8 TB/s against 5.0 TB/s for 512-byte warp slices).
// ---------------------------------------------------------------------------
// Warp-collective (all 32 lanes): lane p's destination row for token t in the partition
// layout, p*S + t when partition p (< P) owns one of the token's experts, else -1. my_id /
// my_w: the token's id and weight of slot `lane` (lanes >= K: -1 / 0), loaded by the caller.
// The same warp writes the token's receive ids (ids the partition does not own ->
// invalid_id) and weights (routed partitions only) for every partition.
__device__ __forceinline__ int64_t partition_row(const DispatchArgs& a, int64_t t, int lane, int my_id,
                                                 float my_w) {
    const bool valid = my_id >= 0 && my_id < a.E;
    if (!valid && my_id != -1 && lane < a.K) set_status(a.status, MOE_ERR_BAD_EXPERT_ID);
    bool routed = false;
    for (int k = 0; k < a.K; k++) {
        const int e = __shfl_sync(kFullMask, my_id, k);
        routed |= e >= 0 && e < a.E && e / a.ep == lane;
    }
    routed = routed && lane < a.P;
    for (int p = 0; p < a.P; p++) {
        const bool rp = __shfl_sync(kFullMask, routed, p);
        if (lane < a.K) {
            const int64_t r = (int64_t(p) * a.S + t) * a.K + lane;
            a.recv_ids[r] = (rp && valid && my_id / a.ep == p) ? my_id : a.invalid_id;
            if (rp) a.recv_w[r] = my_w;
        }
    }
    return routed ? int64_t(lane) * a.S + t : -1;
}

// Token metadata of the partition layout, loaded one token ahead by the warp that resolves
// the destination rows: the ids and weights are inputs that no earlier kernel of the call
// has brought into L2, so each token would otherwise wait a DRAM round trip for them.
struct PartMeta {
    int id = -1;
    float w = 0.0f;
    __device__ __forceinline__ void load(const DispatchArgs& a, int64_t t, int lane) {
        if (lane < a.K) {
            id = __ldg(a.ids + t * a.K + lane);
            w = __ldg(a.w + t * a.K + lane);
        }
    }
};

// Warp-collective destination row of lane `lane` for token t in the bulk kernels: pair
// t*K + lane of the expert layouts, or partition `lane` of the partition layout (PART; `pm`
// holds token t's metadata on entry and the next token's, tn < T, on return).
template <bool MASKED, bool PART>
__device__ __forceinline__ int64_t bulk_dest_row(const DispatchArgs& a, const int* s_seg, int64_t t, int lane,
                                                 PartMeta& pm, int64_t tn) {
    if constexpr (PART) {
        const PartMeta cur = pm;
        if (tn < a.T) pm.load(a, tn, lane);
        return partition_row(a, t, lane, cur.id, cur.w);
    } else {
        return dest_row<MASKED>(a, s_seg, t, lane);
    }
}

// Token metadata of the partition layout staged in shared memory by warp 0 of the quantising
// bulk kernel, so that the receive ids and weights of the token's P rows are written after the
// block barrier by P*K threads at once, not by warp 0 in a loop on the token's critical path.
struct PartStage {
    int id[16];      // the token's K expert ids
    float w[16];     // and weights
    unsigned routed;  // bit p: partition p receives the token
    int pad;
};

// Warp-collective (warp 0): lane p's destination row for token t (p*S + t when partition p owns
// one of the token's experts, else -1); stages ids, weights and the routed mask in `ps`.
__device__ __forceinline__ int64_t partition_row_staged(const DispatchArgs& a, int64_t t, int lane, int my_id,
                                                        float my_w, PartStage* ps) {
    const bool valid = my_id >= 0 && my_id < a.E;
    if (!valid && my_id != -1 && lane < a.K) set_status(a.status, MOE_ERR_BAD_EXPERT_ID);
    bool routed = false;
    for (int k = 0; k < a.K; k++) {
        const int e = __shfl_sync(kFullMask, my_id, k);
        routed |= e >= 0 && e < a.E && e / a.ep == lane;
    }
    routed = routed && lane < a.P;
    const unsigned mask = __ballot_sync(kFullMask, routed);
    if (lane < a.K) {
        ps->id[lane] = my_id;
        ps->w[lane] = my_w;
    }
    if (lane == 0) ps->routed = mask;
    return routed ? int64_t(lane) * a.S + t : -1;
}

// The receive ids (ids the partition does not own -> invalid_id) and weights (routed
// partitions only) of token t's P rows, from the staged metadata: entry j < P*K (slot
// k = j % K of partition p = j / K) by thread j % nthreads.
__device__ __forceinline__ void partition_meta_store(const DispatchArgs& a, int64_t t, const PartStage* ps, int tid,
                                                     int nthreads) {
    for (int j = tid; j < a.P * a.K; j += nthreads) {
        const int p = j / a.K, k = j - p * a.K;
        const int id = ps->id[k];
        const bool rp = (ps->routed >> p) & 1u;
        const int64_t r = (int64_t(p) * a.S + t) * a.K + k;
        a.recv_ids[r] = (rp && id >= 0 && id < a.E && id / a.ep == p) ? id : a.invalid_id;
        if (rp) a.recv_w[r] = ps->w[k];
    }
}

// Partition layout: the receive ids of the padding slots t in [T, S) of every partition are
// invalid_id (grid-stride over all threads of the grid).
__device__ __forceinline__ void partition_padding_ids(const DispatchArgs& a) {
    const int64_t per_p = (a.S - a.T) * a.K;
    const int64_t pad = per_p * a.P;
    for (int64_t j = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; j < pad; j += int64_t(gridDim.x) * blockDim.x) {
        const int64_t p = j / per_p, rem = j - p * per_p;
        a.recv_ids[(p * a.S + a.T) * a.K + rem] = a.invalid_id;
    }
}

struct BulkGeom {
    uint32_t in_bytes;   // 2H: one bf16 row
    uint32_t q_bytes;    // quantised row (2H for the copy)
    uint32_t s_bytes;    // scale row (0 for the copy)
    uint32_t in_off;     // shared offsets
    uint32_t out_off;
    int stages;
    int ts;  // scales stored by the threads (TS kernels), s_bytes then only sizes the staging
};

constexpr int kBulkCopyThreads = 32;
constexpr int kBulkQuantThreads = 256;
// shared-memory header of the bulk kernels: mbarriers (8 B each) at 0, destination rows
// (2 x 32 x 8 B) at 256; the partition layout adds the staged token metadata at 768
// (PartStage, 2 x 136 B)
constexpr uint32_t kBulkHeader = 768;
constexpr uint32_t kBulkHeaderPart = 1152;
constexpr uint32_t kPartStageOff = 768;
constexpr int kBulkRows = 32;          // destination rows per token: K <= 16 pairs, or P <= 32 partitions

template <bool MASKED>
__device__ __forceinline__ void stage_seg(const DispatchArgs& a, int* s_seg) {
    if (MASKED)
        stage_to_shared(a.seg, s_seg, a.E);
}

// TS kernels: the staged scale row `so` of the current token, written by all threads to each
// destination row in rows[0..nd) (< 0: none) in the output's scale layout. Swizzled NVFP4 (a
// buffer the in-place interleave cannot take, its tiles cleared first): 4 consecutive columns
// of a row are 4 contiguous bytes of the 128 x 4 tile layout, so each row takes H/64 word stores. FP8 fp32 scales: one word per group (column-major, or a
// row-major array whose rows are not 16-byte multiples). UE8M0 and row-major NVFP4 scales:
// one byte per group, at the index the register path writes.
template <int QUANT>
__device__ __forceinline__ void store_scales_from_stage(const DispatchArgs& a, const unsigned char* so,
                                                        const int64_t* rows, int nd, int H, int tid, int nthreads) {
    uint8_t* out = static_cast<uint8_t*>(a.out_s);
    if constexpr (QUANT == MOE_QUANT_NVFP4_B16) {
        if (a.L.kind == MOE_SCALES_SWIZZLED_128X4) {
            const int C4 = H / 64;
            for (int j = tid; j < nd * C4; j += nthreads) {
                const int k = j / C4, c4 = j - k * C4;
                const int64_t row = rows[k];
                if (row >= 0)
                    *reinterpret_cast<uint32_t*>(out + swizzled_128x4_index(row, 4 * c4, H / 16)) =
                        *reinterpret_cast<const uint32_t*>(so + 4 * c4);
            }
            return;
        }
    }
    if constexpr (QUANT == MOE_QUANT_FP8_G128) {
        const int G = H / 128;
        for (int j = tid; j < nd * G; j += nthreads) {
            const int k = j / G, g = j - k * G;
            const int64_t row = rows[k];
            if (row >= 0)
                reinterpret_cast<uint32_t*>(out)[scale_index(a.L, row, g, G, false)] =
                    reinterpret_cast<const uint32_t*>(so)[g];
        }
    } else {
        const int G = QUANT == MOE_QUANT_NVFP4_B16 ? H / 16 : H / 128;
        for (int j = tid; j < nd * G; j += nthreads) {
            const int k = j / G, g = j - k * G;
            const int64_t row = rows[k];
            if (row >= 0) out[scale_index(a.L, row, g, G, true)] = so[g];
        }
    }
}

// copy mode: lane 0 drives the ring, lanes < K (partitions < P) resolve the destination rows
template <bool MASKED, bool PART>
__global__ void __launch_bounds__(kBulkCopyThreads) dispatch_bulk_copy_kernel(DispatchArgs a, BulkGeom geo) {
    extern __shared__ __align__(128) unsigned char smem[];
    pdl_wait();
    if constexpr (PART) partition_padding_ids(a);
    const int nd = PART ? a.P : a.K;
    const int lane = threadIdx.x & 31, NS = geo.stages;
    const uint32_t bar0 = smem_addr(smem), in0 = smem_addr(smem + geo.in_off);
    int* s_seg = reinterpret_cast<int*>(smem + geo.out_off);
    if (lane == 0) {
        for (int s = 0; s < NS; s++) mbar_init(bar0 + 8 * s, 1);
        mbar_fence_init();
    }
    stage_seg<MASKED>(a, s_seg);
    __syncwarp();
    const int64_t G = gridDim.x;
    const int64_t ntok = a.T > blockIdx.x ? (a.T - 1 - blockIdx.x) / G + 1 : 0;
    PartMeta pm;  // PART: the first token's ids and weights (warp 0), then one token ahead
    if (PART && threadIdx.x < 32 && ntok > 0) pm.load(a, blockIdx.x, threadIdx.x & 31);
    int64_t issued = 0, consumed = 0;  // lane 0's counts of loads issued / completed
    auto issue = [&](int64_t i) {
        const int s = int(i % NS);
        bulk_load(in0 + s * geo.in_bytes, a.x + (blockIdx.x + i * G) * a.H, geo.in_bytes, bar0 + 8 * s);
        issued = i + 1;
    };
    if (lane == 0)
        for (int64_t i = 0; i < NS - 1 && i < ntok; i++) issue(i);
    for (int64_t i = 0; i < ntok; i++) {
        const int64_t t = blockIdx.x + i * G;
        const int s = int(i % NS);
        const int64_t my_row = bulk_dest_row<MASKED, PART>(a, s_seg, t, lane, pm, t + G);
        int ok = 1;
        if (lane == 0) {
            if (i + NS - 1 < ntok) {
                bulk_wait_read<0>();  // the stage being refilled was the source of token i-1's stores
                issue(i + NS - 1);
            }
            ok = mbar_wait(bar0 + 8 * s, uint32_t((i / NS) & 1));
            consumed += ok;
        }
        ok = __shfl_sync(kFullMask, ok, 0);
        if (!ok) {
            if (lane == 0) set_status(a.status, MOE_ERR_TIMEOUT);
            break;
        }
        for (int k = 0; k < nd; k++) {
            const int64_t row = __shfl_sync(kFullMask, my_row, k);
            if (lane == 0 && row >= 0)
                bulk_store(static_cast<uint8_t*>(a.out_q) + row * geo.q_bytes, in0 + s * geo.in_bytes, geo.q_bytes);
        }
        if (lane == 0) bulk_commit();
    }
    if (lane == 0) {
        bulk_wait_all();
        // after a timeout, loads still in flight are waited for (bounded) before shared memory is released
        for (int64_t j = consumed; j < issued; j++) mbar_wait(bar0 + 8 * int(j % NS), uint32_t((j / NS) & 1), kDrainLimitNs);
    }
}

// How the bulk quantising kernel writes scale rows: one bulk store per row; by its threads
// (layouts a bulk row store cannot write); or one bulk store per row with an L2 evict-last
// policy (rows a later kernel of the same call reads back: the swizzled layout's interleave).
constexpr int kScalesBulk = 0, kScalesThreads = 1, kScalesBulkKeep = 2;

// quantising modes: 256 threads quantise shared -> shared; thread 0 drives the copies
// The partition layout's variants are held to five CTAs per SM (48 registers with 224-thread
// blocks: 59.4 against 60.3 us for the NVFP4 workload at 64 registers and four CTAs); the others
// keep the compiler's choice (a minimum of one block per SM measured 2 us slower there).
template <int QUANT, bool MASKED, bool PART, int SCALES>
__global__ void __launch_bounds__(kBulkQuantThreads, PART ? 5 : 0) dispatch_bulk_quant_kernel(DispatchArgs a, BulkGeom geo) {
    constexpr bool TS = SCALES == kScalesThreads;
    extern __shared__ __align__(128) unsigned char smem[];
    pdl_wait();
    if constexpr (PART) partition_padding_ids(a);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthreads = blockDim.x;
    const int NS = geo.stages, H = a.H, nd = PART ? a.P : a.K;
    const uint32_t bar0 = smem_addr(smem);
    int64_t* s_rows = reinterpret_cast<int64_t*>(smem + 256);  // [2][kBulkRows]
    PartStage* s_part = reinterpret_cast<PartStage*>(smem + kPartStageOff);  // [2], PART only
    unsigned char* in_base = smem + geo.in_off;
    unsigned char* out_base = smem + geo.out_off;                // [2][q_bytes + s_bytes]
    int* s_seg = reinterpret_cast<int*>(out_base + 2 * (geo.q_bytes + geo.s_bytes));
    const uint32_t in0 = smem_addr(in_base), out0 = smem_addr(out_base);
    const uint32_t out_bytes = geo.q_bytes + geo.s_bytes;
    if (tid == 0) {
        for (int s = 0; s < NS; s++) mbar_init(bar0 + 8 * s, 1);
        mbar_fence_init();
    }
    stage_seg<MASKED>(a, s_seg);
    __syncthreads();
    const int64_t G = gridDim.x;
    const int64_t ntok = a.T > blockIdx.x ? (a.T - 1 - blockIdx.x) / G + 1 : 0;
    PartMeta pm;  // PART: the first token's ids and weights (warp 0), then one token ahead
    if (PART && threadIdx.x < 32 && ntok > 0) pm.load(a, blockIdx.x, threadIdx.x & 31);
    int64_t issued = 0, consumed = 0;  // thread 0's counts of loads issued / completed
    auto issue = [&](int64_t i) {
        const int s = int(i % NS);
        bulk_load(in0 + s * geo.in_bytes, a.x + (blockIdx.x + i * G) * H, geo.in_bytes, bar0 + 8 * s);
        issued = i + 1;
    };
    if (tid == 0)
        for (int64_t i = 0; i < NS - 1 && i < ntok; i++) issue(i);
    const int nslices = H / kLaneElems;
    for (int64_t i = 0; i < ntok; i++) {
        const int64_t t = blockIdx.x + i * G;
        const int s = int(i % NS), o = int(i & 1);
        if (warp == 0) {
            int64_t r;
            if constexpr (PART) {
                const PartMeta cur = pm;
                if (t + G < a.T) pm.load(a, t + G, lane);
                r = partition_row_staged(a, t, lane, cur.id, cur.w, s_part + o);
            } else {
                r = bulk_dest_row<MASKED, PART>(a, s_seg, t, lane, pm, t + G);
            }
            if (lane < nd) s_rows[o * kBulkRows + lane] = r;
        }
        if (tid == 0) {
            if (i + NS - 1 < ntok) issue(i + NS - 1);  // its stage was last read before the previous barrier
            bulk_wait_read<1>();                       // out stage o was the source of token i-2's stores
        }
        const int ok = __syncthreads_and(mbar_wait(bar0 + 8 * s, uint32_t((i / NS) & 1)));
        if (!ok) {
            if (tid == 0) set_status(a.status, MOE_ERR_TIMEOUT);
            break;
        }
        consumed = i + 1;
        if constexpr (PART) partition_meta_store(a, t, s_part + o, tid, nthreads);
        const unsigned char* src = in_base + size_t(s) * geo.in_bytes;
        unsigned char* qo = out_base + size_t(o) * out_bytes;
        unsigned char* so = qo + geo.q_bytes;
        for (int base = warp * 32; base < nslices; base += nthreads) {
            const int slice = base + lane;
            const bool active = slice < nslices;
            LaneSlice sl{make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
            if (active) {
                sl.v0 = *reinterpret_cast<const uint4*>(src + slice * 32);
                sl.v1 = *reinterpret_cast<const uint4*>(src + slice * 32 + 16);
            }
            const LaneCodes c = quantise16<QUANT>(sl, a.g);
            if (active) {
                if constexpr (QUANT == MOE_QUANT_NVFP4_B16) {
                    *reinterpret_cast<uint2*>(qo + slice * 8) = make_uint2(c.q.x, c.q.y);
                    so[slice] = uint8_t(c.scale);
                } else {
                    *reinterpret_cast<uint4*>(qo + slice * 16) = c.q;
                    if ((lane & 7) == 0) {
                        if constexpr (QUANT == MOE_QUANT_FP8_G128)
                            reinterpret_cast<uint32_t*>(so)[slice / 8] = c.scale;
                        else
                            so[slice / 8] = uint8_t(c.scale);
                    }
                }
            }
        }
        fence_proxy_async();
        __syncthreads();
        // TS: the scale rows are stored by the threads below (layouts a bulk row cannot write)
        if (tid == 0) {
            for (int k = 0; k < nd; k++) {
                const int64_t row = s_rows[o * kBulkRows + k];
                if (row < 0) continue;
                bulk_store(static_cast<uint8_t*>(a.out_q) + row * geo.q_bytes, out0 + o * out_bytes, geo.q_bytes);
                if constexpr (SCALES == kScalesBulk)
                    bulk_store(static_cast<uint8_t*>(a.out_s) + row * geo.s_bytes, out0 + o * out_bytes + geo.q_bytes,
                               geo.s_bytes);
                if constexpr (SCALES == kScalesBulkKeep)
                    bulk_store_hint(static_cast<uint8_t*>(a.out_s) + row * geo.s_bytes,
                                    out0 + o * out_bytes + geo.q_bytes, geo.s_bytes, l2_policy_evict_last());
            }
            bulk_commit();
        }
        if constexpr (TS) store_scales_from_stage<QUANT>(a, so, s_rows + o * kBulkRows, nd, H, tid, nthreads);
    }
    if (tid == 0) {
        bulk_wait_all();
        // after a timeout, loads still in flight are waited for (bounded) before shared memory is released
        for (int64_t j = consumed; j < issued; j++) mbar_wait(bar0 + 8 * int(j % NS), uint32_t((j / NS) & 1), kDrainLimitNs);
    }
}

// Row geometry of the bulk path, or stages = 0 when it does not apply (rows or scale rows
// that are not 16-byte multiples, unaligned bases, column-major scales, shared memory).
BulkGeom bulk_geometry(int quant, const DispatchArgs& a, bool part) {
    BulkGeom g{};
    const int H = a.H;
    g.in_bytes = uint32_t(2 * H);
    switch (quant) {
        case MOE_QUANT_NONE: g.q_bytes = uint32_t(2 * H); g.s_bytes = 0; break;
        case MOE_QUANT_FP8_G128: g.q_bytes = uint32_t(H); g.s_bytes = uint32_t(H / 32); break;
        case MOE_QUANT_FP8_G128_UE8M0: g.q_bytes = uint32_t(H); g.s_bytes = uint32_t(H / 128); break;
        default: g.q_bytes = uint32_t(H / 2); g.s_bytes = uint32_t(H / 16); break;
    }
    // A scale row goes out as one bulk store when it is row-major, a 16-byte multiple and
    // 16-byte aligned; otherwise (swizzled or column-major layouts, short or unaligned rows)
    // the threads store it (TS) and s_bytes only sizes its staging, rounded up to 16 bytes so
    // that every stage's code row stays 16-byte aligned for its bulk store.
    const bool aligned16 = (reinterpret_cast<uintptr_t>(a.out_s) & 15) == 0;
    const bool ts = quant != MOE_QUANT_NONE &&
                    (a.L.kind != MOE_SCALES_ROW_MAJOR || g.s_bytes % 16 != 0 || !aligned16);
    if (g.q_bytes % 16) return g;
    if (ts) g.s_bytes = (g.s_bytes + 15) / 16 * 16;
    g.ts = ts;
    const bool masked = a.M > 0;  // the masked layout stages seg_indptr after the stages
    const uint32_t seg_bytes = masked ? uint32_t(sizeof(int)) * uint32_t(a.E) : 0u;
    // ring depth, measured on GB300 (prefill / qwen3 / nvfp4 shapes): the copy mode is flat
    // from 2 to 6 stages; FP8 is best at 3; NVFP4 is best at 2, where its smaller footprint
    // lets 5 CTAs share an SM (61.8 us against 67.7 us at 3 stages for 8192 x 7168)
    const int stages = quant == MOE_QUANT_NONE ? 4 : (quant == MOE_QUANT_NVFP4_B16 ? 2 : 3);
    g.in_off = part ? kBulkHeaderPart : kBulkHeader;
    g.out_off = g.in_off + uint32_t(stages) * g.in_bytes;
    const size_t smem = size_t(g.out_off) + (quant == MOE_QUANT_NONE ? 0 : 2 * (g.q_bytes + g.s_bytes)) + seg_bytes;
    if (smem > 200 * 1024) return g;
    g.stages = stages;
    return g;
}

size_t bulk_smem(int quant, const BulkGeom& g, int E, bool masked) {
    return size_t(g.out_off) + (quant == MOE_QUANT_NONE ? 0 : 2 * (g.q_bytes + g.s_bytes)) +
           (masked ? sizeof(int) * size_t(E) : 0);
}

template <int QUANT, bool MASKED, bool PART = false>
cudaError_t launch_bulk(const LaunchCtx& ctx, const DispatchArgs& a, const BulkGeom& geo) {
    const size_t smem = bulk_smem(QUANT, geo, a.E, MASKED);
    int threads;
    int per_sm = 0;
    cudaError_t err;
    if constexpr (QUANT == MOE_QUANT_NONE) {
        auto kern = dispatch_bulk_copy_kernel<MASKED, PART>;
        threads = kBulkCopyThreads;
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (err == cudaSuccess) err = blocks_per_sm(ctx, kern, threads, smem, &per_sm);
        if (err != cudaSuccess) return err;
        const int grid = int(std::min<int64_t>(a.T, int64_t(ctx.num_sms) * (per_sm > 0 ? per_sm : 1)));
        return launch_pdl(ctx, kern, dim3(grid), dim3(threads), smem, a, geo);
    } else {
        auto kern = geo.ts ? dispatch_bulk_quant_kernel<QUANT, MASKED, PART, kScalesThreads>
                           : dispatch_bulk_quant_kernel<QUANT, MASKED, PART, kScalesBulk>;
        if constexpr (QUANT == MOE_QUANT_NVFP4_B16)
            if (!geo.ts && a.keep_scales_in_l2) kern = dispatch_bulk_quant_kernel<QUANT, MASKED, PART, kScalesBulkKeep>;
        // as many passes over the row's 16-element slices as 256 threads need, with the block
        // sized so that every pass is full (H = 7168: 448 slices = 2 x 224, not 256 + 192)
        const int nslices = a.H / kLaneElems;
        const int passes = (nslices + kBulkQuantThreads - 1) / kBulkQuantThreads;
        threads = ((nslices + passes - 1) / passes + 31) / 32 * 32;
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (err == cudaSuccess) err = blocks_per_sm(ctx, kern, threads, smem, &per_sm);
        if (err != cudaSuccess) return err;
        const int grid = int(std::min<int64_t>(a.T, int64_t(ctx.num_sms) * (per_sm > 0 ? per_sm : 1)));
        return launch_pdl(ctx, kern, dim3(grid), dim3(threads), smem, a, geo);
    }
}

template <int QUANT, bool MASKED>
cudaError_t launch_variant(const LaunchCtx& ctx, const DispatchArgs& a) {
    // large batches: the bulk path when its geometry applies
    if (a.T >= kBulkMinTokens) {
        const BulkGeom geo = bulk_geometry(QUANT, a, false);
        if (geo.stages > 0) return launch_bulk<QUANT, MASKED>(ctx, a, geo);
    }
    auto kern = dispatch_kernel<QUANT, MASKED>;
    const size_t smem = MASKED ? sizeof(int) * size_t(a.E) : 0;
    // one wave or less of 256-thread blocks leaves SMs unevenly loaded: use 64 threads
    const int threads = a.n_units < int64_t(ctx.num_sms) * 16 ? 64 : kDispatchThreads;
    int per_sm = 0;
    cudaError_t err = blocks_per_sm(ctx, kern, threads, smem, &per_sm);
    if (err != cudaSuccess) return err;
    const int64_t warps_per_block = threads / 32;
    const int64_t need = (a.n_units + warps_per_block - 1) / warps_per_block;
    const int64_t cap = int64_t(ctx.num_sms) * (per_sm > 0 ? per_sm : 1);
    const int grid = int(need < cap ? need : cap);

    return launch_pdl(ctx, kern, dim3(grid), dim3(threads), smem, a);
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

// Exhaustive check of div_by_scale against the IEEE division over the FP8 quantiser's
// domain: amax = every non-negative finite bf16 (bit patterns 0 .. 0x7F7F, increasing in
// value; 0 is clamped to 1e-10 as the quantiser does), s = max(amax, 1e-10) / 448, and every
// bf16 x of either sign with |x| <= amax.
//   result[0]  pairs whose e4m3 codes differ (the quantiser's output)
//   result[1]  the first such pair: x bits << 32 | s bits
//   result[2]  pairs whose quotients differ while |x / s| >= 2^-12 (codes there are not zero)
//   result[3]  pairs whose quotients differ at all (only where the remainder x - q*s falls
//              below the normal range, |x| < 2^-103, so |x / s| < 2^-61 and the code is a zero)
__global__ void __launch_bounds__(256) fp8_division_check_kernel(unsigned long long* result) {
    for (int a = blockIdx.x; a <= 0x7F7F; a += gridDim.x) {
        const float amax = __uint_as_float(uint32_t(a) << 16);
        const float sc = __fdiv_rn(fmaxf(amax, 1e-10f), 448.0f);
        const float y = __frcp_rn(sc);
        for (int xb = threadIdx.x; xb <= a; xb += blockDim.x) {
#pragma unroll
            for (int sign = 0; sign < 2; sign++) {
                const float x = __uint_as_float((uint32_t(xb) << 16) | (sign ? 0x80000000u : 0u));
                const float want = __fdiv_rn(x, sc), got = div_by_scale(x, sc, y);
                if (__float_as_uint(want) == __float_as_uint(got)) continue;
                atomicAdd(result + 3, 1ull);
                if (fabsf(want) >= 0x1p-12f) atomicAdd(result + 2, 1ull);
                const uint32_t codes = e4m3x2(want, got);  // low byte: IEEE quotient's code
                if ((codes & 0xffu) != (codes >> 8)) {
                    if (atomicAdd(result, 1ull) == 0ull)
                        result[1] = (static_cast<unsigned long long>(__float_as_uint(x)) << 32) | __float_as_uint(sc);
                }
            }
        }
    }
}

// The bulk kernels' bounded ring wait on one mbarrier of count 1: arrived at first
// (complete = 1), or never arrived at (complete = 0), when the wait has to give up.
__global__ void wait_timeout_check_kernel(int32_t* status, uint64_t limit_ns, int complete) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_addr(&bar);
    mbar_init(b, 1);
    mbar_fence_init();
    if (complete) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(b) : "memory");
    if (!mbar_wait(b, 0, limit_ns)) set_status(status, MOE_ERR_TIMEOUT);
}

cudaError_t launch_wait_timeout_check(const LaunchCtx& ctx, int32_t* status, uint64_t limit_ns, int complete) {
    wait_timeout_check_kernel<<<1, 1, 0, ctx.stream>>>(status, limit_ns, complete);
    return cudaGetLastError();
}

cudaError_t launch_fp8_division_check(const LaunchCtx& ctx, unsigned long long* result) {
    cudaError_t err = cudaMemsetAsync(result, 0, 4 * sizeof(unsigned long long), ctx.stream);
    if (err != cudaSuccess) return err;
    fp8_division_check_kernel<<<ctx.num_sms * 8, 256, 0, ctx.stream>>>(result);
    return cudaGetLastError();
}

cudaError_t launch_convert_probe(const LaunchCtx& ctx, const float* in, int64_t n, uint8_t* e4m3,
                                 uint8_t* e2m1, float* e4m3_value) {
    const int64_t pairs = n / 2;
    int64_t blocks = (pairs + 255) / 256;
    if (blocks > int64_t(ctx.num_sms) * 8) blocks = int64_t(ctx.num_sms) * 8;
    if (blocks < 1) blocks = 1;
    convert_probe_kernel<<<int(blocks), 256, 0, ctx.stream>>>(in, pairs, e4m3, e2m1, e4m3_value);
    return cudaGetLastError();
}

cudaError_t launch_dispatch_partitioned_bulk(const LaunchCtx& ctx, int quant, const uint16_t* x, int64_t T,
                                             int64_t S, int H, const int32_t* ids, const float* w, int K, int E,
                                             int P, int32_t invalid_id, float g, void* recv_x, uint8_t* recv_sf,
                                             int32_t* recv_ids, float* recv_w, int32_t* dev_status,
                                             int scale_layout, bool* launched, bool keep_scales_in_l2) {
    *launched = false;
    if (T < kBulkMinTokens || (quant != MOE_QUANT_NONE && quant != MOE_QUANT_NVFP4_B16)) return cudaSuccess;
    DispatchArgs a{};
    a.x = x;
    a.T = T;
    a.H = H;
    a.K = K;
    a.E = E;
    a.ids = ids;
    a.g = g;
    a.out_q = recv_x;
    a.out_s = recv_sf;
    a.status = dev_status;
    a.units_per_row = (H + kSlice - 1) / kSlice;
    a.n_units = T * a.units_per_row;
    a.max_row = int64_t(P) * S;
    a.L = ScaleLayout{scale_layout, 0, 0};
    a.P = P;
    a.ep = E / P;
    a.S = S;
    a.invalid_id = invalid_id;
    a.w = w;
    a.recv_ids = recv_ids;
    a.recv_w = recv_w;
    a.keep_scales_in_l2 = keep_scales_in_l2;
    const BulkGeom geo = bulk_geometry(quant, a, true);
    if (geo.stages == 0) return cudaSuccess;
    *launched = true;
    return quant == MOE_QUANT_NVFP4_B16 ? launch_bulk<MOE_QUANT_NVFP4_B16, false, true>(ctx, a, geo)
                                        : launch_bulk<MOE_QUANT_NONE, false, true>(ctx, a, geo);
}

cudaError_t launch_dispatch(const LaunchCtx& ctx, int mode, int quant, const uint16_t* x, int64_t T,
                            int H, const int32_t* topk_ids, int K, int E, int M,
                            const int32_t* src2dst, const int64_t* seg_indptr, float global_scale,
                            void* out_q, void* out_scales, int32_t* dev_status, int scale_layout,
                            int64_t out_rows) {
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
    a.max_row = out_rows > 0 ? out_rows : T * K;
    const bool masked = mode == MOE_MODE_MASKED;
    a.L.kind = scale_layout;
    a.L.M = masked ? M : 0;
    a.L.rows_al = ((masked ? int64_t(M) : a.max_row) + 3) / 4 * 4;
    // swizzled NVFP4 scales: when the buffer allows it, the scale rows go out row-major and the
    // touched tiles are interleaved in place afterwards (the interleave zeroing the rows the
    // dispatch does not write, or a clear of the touched tiles first where it cannot tell them);
    // else the touched tiles are cleared and every scale word is stored at its tile position
    SfTiles tiles{};
    bool by_tiles = false;
    if (scale_layout == MOE_SCALES_SWIZZLED_128X4) {
        tiles.sf = static_cast<uint8_t*>(out_scales);
        tiles.R = masked ? int64_t(E) * M : a.max_row;
        tiles.C = H / 16;
        tiles.kind = masked ? kSfTilesMasked : kSfTilesAll;
        tiles.seg = seg_indptr;
        tiles.E = E;
        tiles.M = M;
        tiles.n_blocks = (tiles.R + 127) / 128;
        // a group's run: a quarter above the mean pairs per expert (longer runs loop), at most M
        tiles.q_per_group = sf_tiles_q_per_group(std::min<int64_t>(M, (5 * T * K / E + 3) / 4), E);
        tiles.status = dev_status;
        by_tiles = sf_tiles_interleavable(tiles);
        cudaError_t err = sf_tiles_interleave_zeroes(tiles) ? cudaSuccess : launch_sf_tiles_clear(ctx, tiles);
        if (err != cudaSuccess) return err;
        if (by_tiles) {
            a.L.kind = MOE_SCALES_ROW_MAJOR;
            a.keep_scales_in_l2 = true;
        }
    }
    cudaError_t err;
    switch (quant) {
        case MOE_QUANT_NONE:
            err = masked ? launch_variant<MOE_QUANT_NONE, true>(ctx, a) : launch_variant<MOE_QUANT_NONE, false>(ctx, a);
            break;
        case MOE_QUANT_FP8_G128:
            err = masked ? launch_variant<MOE_QUANT_FP8_G128, true>(ctx, a)
                         : launch_variant<MOE_QUANT_FP8_G128, false>(ctx, a);
            break;
        case MOE_QUANT_FP8_G128_UE8M0:
            err = masked ? launch_variant<MOE_QUANT_FP8_G128_UE8M0, true>(ctx, a)
                         : launch_variant<MOE_QUANT_FP8_G128_UE8M0, false>(ctx, a);
            break;
        default:
            err = masked ? launch_variant<MOE_QUANT_NVFP4_B16, true>(ctx, a)
                         : launch_variant<MOE_QUANT_NVFP4_B16, false>(ctx, a);
            break;
    }
    if (err != cudaSuccess || !by_tiles) return err;
    return launch_sf_tiles_interleave(ctx, tiles);
}

}  // namespace moe

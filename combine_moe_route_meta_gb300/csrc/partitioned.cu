// partitioned.cu -- per-partition routing layout and the FlashInfer all-to-all layout.
//
// moe_dispatch_layout: buffer.get_dispatch_layout(topk_ids, num_experts) of
//   _DeepEPDispatcherImplNormal._dispatch_core ("sglang token_dispatcher/deepep.py" page):
//   is_token_in_rank [T, P], num_tokens_per_rank [P], num_tokens_per_expert [E], with the
//   E experts split into P partitions of E/P.
// moe_dispatch_partitioned / moe_combine_partitioned: FlashinferDispatcher.dispatch and
//   .combine ("sglang token_dispatcher/flashinfer.py" page) for one source rank. The
//   payload (bf16 row, or NVFP4 codes + e4m3 block scales, plus topk_ids and topk_weights)
//   goes once to each partition owning one of the token's experts, into
//   [P, num_slots, .] receive rows (slot = token index; num_slots plays
//   runtime_max_tokens_per_rank). Receive ids of experts the partition does not own, of
//   tokens it does not receive and of padding slots are set to invalid_expert_id. The
//   combine sums, per token, the (already weighted) partial outputs of the partitions the
//   token was sent to.
//
// Design: batches of at least 1024 tokens whose rows suit whole-row bulk copies go to the
// bulk (TMA) dispatch kernels of dispatch.cu with partition destinations. Smaller ones, and
// the combine, use the same warp-per-(token, 512-column slice) structure as dispatch.cu /
// combine.cu. Lanes 0..K-1 hold the token's expert ids; lane p (< P <= 32) tests every id
// against its partition's expert range, so the destination row of lane p is p*num_slots + t
// or -1, and the row broadcast of the shared quantise_store serves P candidate rows.
#include <cstdint>

#include "dispatch_slice.cuh"
#include "moe_device.cuh"
#include "moe_launch.h"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kSlice = 512;
constexpr int kLaneElems = 16;

// ---------------------------------------------------------------------------
// layout: one thread per token
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) dispatch_layout_kernel(const int32_t* __restrict__ ids, int64_t T,
                                                                    int K, int E, int P, int32_t* ntr,
                                                                    uint8_t* itr, int32_t* nte, int32_t* status) {
    extern __shared__ int s_cnt[];  // [P] tokens per partition, then [E] pairs per expert
    pdl_wait();
    int* s_rank = s_cnt;
    int* s_exp = s_cnt + P;
    for (int j = threadIdx.x; j < P + E; j += blockDim.x) s_cnt[j] = 0;
    __syncthreads();
    const int ep = E / P;
    bool bad = false;
    for (int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; t < T; t += int64_t(gridDim.x) * blockDim.x) {
        uint8_t* row = itr + t * P;
        for (int p = 0; p < P; p++) row[p] = 0;
        for (int k = 0; k < K; k++) {
            const int e = __ldg(ids + t * K + k);
            if (e < 0 || e >= E) {
                bad |= e != -1;
                continue;
            }
            atomicAdd(&s_exp[e], 1);
            const int p = e / ep;
            bool seen = false;  // an earlier slot of this token in the same partition
            for (int k2 = 0; k2 < k; k2++) {
                const int e2 = __ldg(ids + t * K + k2);
                seen |= e2 >= 0 && e2 < E && e2 / ep == p;
            }
            if (!seen) {
                row[p] = 1;
                atomicAdd(&s_rank[p], 1);
            }
        }
    }
    if (__any_sync(kFullMask, bad) && (threadIdx.x & 31) == 0) set_status(status, MOE_ERR_BAD_EXPERT_ID);
    __syncthreads();
    for (int p = threadIdx.x; p < P; p += blockDim.x)
        if (s_rank[p]) atomicAdd(ntr + p, s_rank[p]);
    if (nte != nullptr)
        for (int e = threadIdx.x; e < E; e += blockDim.x)
            if (s_exp[e]) atomicAdd(nte + e, s_exp[e]);
}

// One block for batches whose T*K ids fit in shared memory (<= kLayoutSingleMaxPairs): the
// ids are staged in one round of loads, the counters live in shared memory and are written
// out whole at the end, so there is no global atomic and no clearing of the outputs first.
constexpr int kLayoutSingleThreads = 1024;
__global__ void __launch_bounds__(kLayoutSingleThreads)
    dispatch_layout_single_kernel(const int32_t* __restrict__ ids, int T, int K, int E, int P, int32_t* ntr,
                                  uint8_t* itr, int32_t* nte, int32_t* status) {
    extern __shared__ int s_lay[];  // [P] tokens per partition | [E] pairs per expert | [T*K] ids
    int* s_rank = s_lay;
    int* s_exp = s_rank + P;
    int* s_ids = s_exp + E;
    for (int j = threadIdx.x; j < P + E; j += blockDim.x) s_lay[j] = 0;
    pdl_wait();
    stage_to_shared(ids, s_ids, T * K);
    __syncthreads();
    const int ep = E / P;
    bool bad = false;
    for (int t = threadIdx.x; t < T; t += blockDim.x) {
        const int* tid_ids = s_ids + t * K;
        uint8_t* row = itr + int64_t(t) * P;
        for (int p = 0; p < P; p++) row[p] = 0;
        for (int k = 0; k < K; k++) {
            const int e = tid_ids[k];
            if (e < 0 || e >= E) {
                bad |= e != -1;
                continue;
            }
            atomicAdd(&s_exp[e], 1);
            const int p = e / ep;
            bool seen = false;  // an earlier slot of this token in the same partition
            for (int k2 = 0; k2 < k; k2++) {
                const int e2 = tid_ids[k2];
                seen |= e2 >= 0 && e2 < E && e2 / ep == p;
            }
            if (!seen) {
                row[p] = 1;
                atomicAdd(&s_rank[p], 1);
            }
        }
    }
    if (__any_sync(kFullMask, bad) && (threadIdx.x & 31) == 0) set_status(status, MOE_ERR_BAD_EXPERT_ID);
    __syncthreads();
    for (int p = threadIdx.x; p < P; p += blockDim.x) ntr[p] = s_rank[p];
    if (nte != nullptr)
        for (int e = threadIdx.x; e < E; e += blockDim.x) nte[e] = s_exp[e];
}

struct PartArgs {
    const uint16_t* x;
    const int32_t* ids;
    const float* w;
    int64_t T, S;  // tokens, slots per partition
    int H, K, E, P, ep;
    int32_t invalid_id;
    float g;
    void* recv_x;
    uint8_t* recv_sf;
    int32_t* recv_ids;
    float* recv_w;
    const uint16_t* partial;
    uint16_t* out;
    int32_t* status;
    int units_per_row;
    int64_t n_units;
    ScaleLayout L;  // of recv_sf: row-major [P*S, H/16] or 128 x 4 swizzled over the P*S rows
};

// lane p: whether token t sends to partition p; all lanes return the same K ids in e_out
__device__ __forceinline__ bool token_in_partition(const PartArgs& a, int64_t t, int lane, int& my_id) {
    my_id = lane < a.K ? __ldg(a.ids + t * a.K + lane) : -1;
    bool routed = false;
    for (int k = 0; k < a.K; k++) {
        const int e = __shfl_sync(kFullMask, my_id, k);
        routed |= e >= 0 && e < a.E && e / a.ep == lane;
    }
    return routed && lane < a.P;
}

template <int QUANT>
__global__ void __launch_bounds__(kThreads) dispatch_partitioned_kernel(PartArgs a) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const int H = a.H;
    for (int64_t u = warp; u < a.n_units; u += nwarps) {
        const int64_t t = u / a.units_per_row;
        const int slice = int(u - t * a.units_per_row);
        const int col = slice * kSlice + lane * kLaneElems;
        const bool active = col < H;
        LaneSlice sl{make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
        if (active) sl = load_slice(a.x + t * H + col);
        int my_id;
        const bool routed = token_in_partition(a, t, lane, my_id);
        const int64_t my_row = routed ? int64_t(lane) * a.S + t : -1;
        if (slice == 0) {
            // the sanitised ids and the weights of every partition's receive row
            const float my_w = lane < a.K ? __ldg(a.w + t * a.K + lane) : 0.0f;
            const bool valid = my_id >= 0 && my_id < a.E;
            if (!valid && my_id != -1 && lane < a.K) set_status(a.status, MOE_ERR_BAD_EXPERT_ID);
            for (int p = 0; p < a.P; p++) {
                const bool rp = __shfl_sync(kFullMask, routed, p);
                if (lane < a.K) {
                    const int64_t r = (int64_t(p) * a.S + t) * a.K + lane;
                    a.recv_ids[r] = (rp && valid && my_id / a.ep == p) ? my_id : a.invalid_id;
                    if (rp) a.recv_w[r] = my_w;
                }
            }
        }
        if constexpr (QUANT == MOE_QUANT_NVFP4_B16)
            quantise_store<QUANT>(sl, active, lane, col, H, a.P, my_row, a.g, a.recv_x, a.recv_sf, a.L);
        else
            quantise_store<QUANT>(sl, active, lane, col, H, a.P, my_row, a.g, a.recv_x, nullptr);
    }
    // padding slots t in [T, S): every partition's ids are the invalid id
    const int64_t pad = (a.S - a.T) * a.P * a.K;
    for (int64_t j = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; j < pad; j += int64_t(gridDim.x) * blockDim.x) {
        const int64_t per_p = (a.S - a.T) * a.K;
        const int64_t p = j / per_p, rem = j - p * per_p;
        a.recv_ids[(p * a.S + a.T) * a.K + rem] = a.invalid_id;
    }
}

// The NVFP4 quantiser's per-block ratio g / value(sf) for the e4m3 code sf: the same correctly
// rounded quotient quantise16 divides out per block (0 for the two zero codes, whose blocks get
// zero codes). A kernel that tabulates it for all 256 codes once replaces a division per block
// by a shared-memory load (quantise16_nvfp4_lut).
__device__ __forceinline__ float nvfp4_ratio(float g, uint32_t code) {
    const float sff = e4m3_value(code);
    return sff != 0.0f ? __fdiv_rn(g, sff) : 0.0f;
}

// quantise16<MOE_QUANT_NVFP4_B16> with the ratio looked up in s_ratio[256] (nvfp4_ratio of
// every code) and the block amax taken on the packed bf16 pairs (abs and max of bf16 values
// are exact, and max returns the non-NaN operand as fmaxf does): the same codes and scale.
__device__ __forceinline__ LaneCodes quantise16_nvfp4_lut(const LaneSlice& s, float g, const float* s_ratio) {
    uint32_t m;
    asm("{\n\t.reg .b32 a, b, c, d;\n\t"
        "abs.bf16x2 a, %1;\n\tabs.bf16x2 b, %2;\n\tabs.bf16x2 c, %3;\n\tabs.bf16x2 d, %4;\n\t"
        "max.bf16x2 a, a, b;\n\tmax.bf16x2 c, c, d;\n\tmax.bf16x2 a, a, c;\n\t"
        "abs.bf16x2 b, %5;\n\tabs.bf16x2 c, %6;\n\tabs.bf16x2 d, %7;\n\t"
        "max.bf16x2 a, a, b;\n\tmax.bf16x2 c, c, d;\n\tmax.bf16x2 a, a, c;\n\t"
        "abs.bf16x2 b, %8;\n\tmax.bf16x2 %0, a, b;\n\t}"
        : "=r"(m)
        : "r"(s.v0.x), "r"(s.v0.y), "r"(s.v0.z), "r"(s.v0.w), "r"(s.v1.x), "r"(s.v1.y), "r"(s.v1.z), "r"(s.v1.w));
    const float amax = fmaxf(fmaxf(bf16_lo(m), bf16_hi(m)), 0.0f);  // 0 when all 16 are NaN, as in quantise16
    const float tsf = __fmul_rn(__fdiv_rn(amax, 6.0f), g);
    LaneCodes out;
    out.scale = e4m3x2(tsf, 0.0f) & 0xffu;
    out.q = make_uint4(0, 0, 0, 0);
    if (out.scale & 0x7fu) {  // not one of the two zero codes
        const float r = s_ratio[out.scale];
        float f[16];
        unpack8(s.v0, f);
        unpack8(s.v1, f + 8);
        uint32_t b[8];
#pragma unroll
        for (int p = 0; p < 8; p++) b[p] = e2m1x2(__fmul_rn(f[2 * p], r), __fmul_rn(f[2 * p + 1], r));
        out.q.x = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
        out.q.y = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
    }
    return out;
}

// NVFP4 with 128 x 4 swizzled scales when every 128-row tile lies in one partition (S % 128 ==
// 0): the scale tiles are built in shared memory and written as whole 16-byte lines, so there is
// neither a clear nor an interleave pass. Line L of a tile holds rows L, L+32, L+64 and L+96 (4
// scale columns each), so the 128 slots of a group split into two halves that share no line: half
// h takes the rows whose L lies in [16h, 16h + 16). Unit = (group of 128 tokens, half, 512-column
// slice), 64 tokens: warp w quantises 8 of them (lane = 16 columns = one block; the row slices of
// kTileBatch tokens in flight, the next batch loaded while the current one is quantised), stores
// each token's codes (256 bytes) into the row of every partition it goes to and its block scales
// into the 8 staged tiles of the slice. A token's scales are the same for every partition, and so
// is their place in a tile (slot t sits at row t % 128 of its partition's tile), so one staged
// copy serves all P partitions: the threads then write the half's 16-byte lines for every
// partition, with the words of slots the partition does not receive (or past T) zeroed. The
// receive ids and weights are written by the slice-0 units.
constexpr int kTileTokens = 128;     // slots per tile
constexpr int kTileThreads = 256;  // also one thread per e4m3 code for the ratio table
constexpr int kTileUnitTokens = 64;  // one half of a group
constexpr int kTileParts = kTileTokens / kTileUnitTokens;     // units per group
constexpr int kTileLines = kTileUnitTokens / 4;               // lines of a tile per unit
constexpr int kTileWarpTokens = kTileUnitTokens / (kTileThreads / 32);  // 8
constexpr int kTileBatch = 4;
constexpr int kTilesPerSlice = kSlice / 64;  // tile columns (4 scale columns of 16 elements each)
// staged tile stride: 512 bytes + 16, so that the 8 tiles of a slice start in different banks
constexpr int kTileStride = 528;
static_assert(kTileThreads == 256, "one thread per e4m3 code fills the ratio table");
static_assert(kTileUnitTokens % 4 == 0 && 32 % kTileLines == 0 && kTileUnitTokens <= kTileThreads,
              "a unit is whole lines of a tile, its masks built by one thread per token");
static_assert(kTileWarpTokens % kTileBatch == 0, "whole batches per warp");
static_assert(kTileThreads % (kTilesPerSlice * kTileLines) == 0, "whole partition phases in the tile output");

// row in its group of token j (< kTileUnitTokens) of part h
__device__ __forceinline__ int tile_half_row(int h, int j) {
    return kTileLines * h + (j % kTileLines) + 32 * (j / kTileLines);
}

__global__ void __launch_bounds__(kTileThreads, 4) dispatch_partitioned_tiles_kernel(PartArgs a) {
    __shared__ unsigned s_mask[kTileTokens];  // bit p: partition p receives the token of row i
    __shared__ __align__(16) unsigned char s_tiles[kTilesPerSlice * kTileStride];
    __shared__ float s_ratio[256];  // nvfp4_ratio of every e4m3 code
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    s_ratio[tid] = nvfp4_ratio(a.g, uint32_t(tid));  // read after the first barrier below
    pdl_wait();
    const int H = a.H, K = a.K, P = a.P;
    const int C4 = H / 64;  // tile columns per 128-row block
    const int nsl = a.units_per_row;
    uint8_t* recv_q = static_cast<uint8_t*>(a.recv_x);
    // padding slots t in [T, S): every partition's ids are the invalid id
    {
        const int64_t per_p = (a.S - a.T) * K;
        for (int64_t j = int64_t(blockIdx.x) * blockDim.x + tid; j < per_p * P; j += int64_t(gridDim.x) * blockDim.x) {
            const int64_t p = j / per_p, rem = j - p * per_p;
            a.recv_ids[(p * a.S + a.T) * K + rem] = a.invalid_id;
        }
    }
    const LaneSlice zero{make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    for (int64_t u = blockIdx.x; u < a.n_units; u += gridDim.x) {
        const int64_t gh = u / nsl;  // (group, part); the slices of one part are neighbours
        const int c = int(u - gh * nsl);
        const int64_t t0 = (gh / kTileParts) * kTileTokens;
        const int h = int(gh % kTileParts);
        const int ntg = a.T - t0 < kTileTokens ? int(a.T - t0) : kTileTokens;  // rows holding tokens
        const int col = c * kSlice + lane * kLaneElems;
        const bool active = col < H;
        const int jw = warp * kTileWarpTokens;
        // the first batch of row slices is in flight while the routing masks are built
        LaneSlice sl[kTileBatch];
#pragma unroll
        for (int b = 0; b < kTileBatch; b++) {
            const int i = tile_half_row(h, jw + b);
            sl[b] = zero;
            if (active && i < ntg) sl[b] = load_slice(a.x + (t0 + i) * H + col);
        }
        if (tid < kTileUnitTokens) {
            const int i = tile_half_row(h, tid);
            unsigned m = 0;
            if (i < ntg) {
                const int32_t* ip = a.ids + (t0 + i) * K;
                bool bad = false;
                for (int k = 0; k < K; k++) {
                    const int e = __ldg(ip + k);
                    if (e >= 0 && e < a.E)
                        m |= 1u << (e / a.ep);
                    else
                        bad |= e != -1;
                }
                if (bad && c == 0) set_status(a.status, MOE_ERR_BAD_EXPERT_ID);
            }
            s_mask[i] = m;
        }
        __syncthreads();
        for (int jb = 0; jb < kTileWarpTokens; jb += kTileBatch) {
            if (jb > 0) {
#pragma unroll
                for (int b = 0; b < kTileBatch; b++) {
                    const int i = tile_half_row(h, jw + jb + b);
                    if (active && i < ntg) sl[b] = load_slice(a.x + (t0 + i) * H + col);
                }
            }
#pragma unroll
            for (int b = 0; b < kTileBatch; b++) {
                const int i = tile_half_row(h, jw + jb + b);
                if (i >= ntg || !active) continue;
                const LaneCodes q = quantise16_nvfp4_lut(sl[b], a.g, s_ratio);
                unsigned m = s_mask[i];
                while (m) {
                    const int p = __ffs(m) - 1;
                    m &= m - 1;
                    st_v2(recv_q + (int64_t(p) * a.S + t0 + i) * (H / 2) + col / 2, make_uint2(q.q.x, q.q.y));
                }
                // scale column 4*(lane/4) + lane%4 of the slice, row i of the tile
                s_tiles[(lane >> 2) * kTileStride + (i & 31) * 16 + (i >> 5) * 4 + (lane & 3)] = uint8_t(q.scale);
            }
        }
        if (c == 0) {
            // the receive ids (ids the partition does not own -> invalid_id) and weights (routed
            // partitions only) of every partition's row of the unit's tokens
            for (int jj = tid; jj < kTileUnitTokens * K; jj += kTileThreads) {
                const int j = jj / K, k = jj - j * K;
                const int i = tile_half_row(h, j);
                if (i >= ntg) continue;
                const int64_t t = t0 + i;
                const int id = __ldg(a.ids + t * K + k);
                const float w = __ldg(a.w + t * K + k);
                const unsigned m = s_mask[i];
                const bool valid = id >= 0 && id < a.E;
                for (int p = 0; p < P; p++) {
                    const bool rp = (m >> p) & 1u;
                    const int64_t r = (int64_t(p) * a.S + t) * K + k;
                    a.recv_ids[r] = (rp && valid && id / a.ep == p) ? id : a.invalid_id;
                    if (rp) a.recv_w[r] = w;
                }
            }
        }
        __syncthreads();
        // the part's lines of the slice's tiles: thread -> (tile q, line L), partitions p0,
        // p0 + kPStep, ...
        constexpr int kPStep = kTileThreads / (kTilesPerSlice * kTileLines);
        const int nq = min(kTilesPerSlice, C4 - c * kTilesPerSlice);
        const int q = (tid / kTileLines) % kTilesPerSlice, L = kTileLines * h + tid % kTileLines;
        const int p0 = tid / (kTilesPerSlice * kTileLines);
        if (q < nq) {
            const uint4 v = *reinterpret_cast<const uint4*>(s_tiles + q * kTileStride + L * 16);
            const unsigned m0 = s_mask[L], m1 = s_mask[L + 32], m2 = s_mask[L + 64], m3 = s_mask[L + 96];
            const int64_t tile0 = (gh / kTileParts) * C4 + c * kTilesPerSlice + q;  // the tile of partition 0
            const int64_t tiles_per_p = (a.S / kTileTokens) * C4;
            for (int p = p0; p < P; p += kPStep) {
                uint4 o;
                o.x = (m0 >> p) & 1u ? v.x : 0u;
                o.y = (m1 >> p) & 1u ? v.y : 0u;
                o.z = (m2 >> p) & 1u ? v.z : 0u;
                o.w = (m3 >> p) & 1u ? v.w : 0u;
                st_v4(a.recv_sf + (tile0 + int64_t(p) * tiles_per_p) * 512 + L * 16, o);
            }
        }
        __syncthreads();  // s_mask and s_tiles are rebuilt by the next unit
    }
}

// NVFP4 with row-major scales, >= 1024 tokens: the dispatch as a warp-specialised ring. Warp 0
// (producer) bulk-copies token rows into kDRingIn row slots, kDRingIn tokens ahead. Warps
// 2 .. 2+kDRingConsumerWarps-1 (consumers) quantise a token's 16-element blocks from its row slot
// into one of kDRingOut code-row slots (codes, then the row's scales). Warp 1 (stores) finds the
// partitions each token goes to, writes the receive ids and weights of its P rows, and once the
// code row is complete stores it, with its scale row, to every routed partition by bulk copies.
// Full / empty mbarriers hand each slot from one role to the next (row slot: producer ->
// consumers -> producer; code-row slot: consumers -> stores -> consumers), so no role waits on a
// block-wide barrier. Every wait is bounded; a role that gives up reports MOE_ERR_TIMEOUT and
// the others give up in turn.
constexpr int kDRingConsumerWarps = 7;  // 224 threads: two passes over a 7168-element row
constexpr int kDRingThreads = (2 + kDRingConsumerWarps) * 32;
constexpr int kDRingIn = 2;
constexpr int kDRingOut = 3;

size_t dring_smem(int H) {
    return size_t(kDRingIn) * 2 * H + size_t(kDRingOut) * (H / 2 + H / 16) + 8 * 2 * (kDRingIn + kDRingOut);
}

__global__ void __launch_bounds__(kDRingThreads) dispatch_partitioned_ring_kernel(PartArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = a.H, K = a.K, P = a.P;
    const uint32_t in_bytes = uint32_t(2 * H), qb = uint32_t(H / 2), sb = uint32_t(H / 16), ob = qb + sb;
    const uint32_t in0 = smem_addr(smem), out0 = in0 + kDRingIn * in_bytes;
    const uint32_t bars = out0 + kDRingOut * ob;
    auto in_full = [&](int s) { return bars + 8 * s; };
    auto in_empty = [&](int s) { return bars + 8 * (kDRingIn + s); };
    auto out_full = [&](int o) { return bars + 8 * (2 * kDRingIn + o); };
    auto out_empty = [&](int o) { return bars + 8 * (2 * kDRingIn + kDRingOut + o); };
    if (tid == 0) {
        for (int s = 0; s < kDRingIn; s++) {
            mbar_init(in_full(s), 1);
            mbar_init(in_empty(s), kDRingConsumerWarps);
        }
        for (int o = 0; o < kDRingOut; o++) {
            mbar_init(out_full(o), kDRingConsumerWarps);
            mbar_init(out_empty(o), 1);
        }
        mbar_fence_init();
    }
    __syncthreads();
    pdl_wait();
    // padding slots t in [T, S): every partition's ids are the invalid id
    {
        const int64_t per_p = (a.S - a.T) * K;
        for (int64_t j = int64_t(blockIdx.x) * blockDim.x + tid; j < per_p * P; j += int64_t(gridDim.x) * blockDim.x) {
            const int64_t p = j / per_p, rem = j - p * per_p;
            a.recv_ids[(p * a.S + a.T) * K + rem] = a.invalid_id;
        }
    }
    const int64_t G = gridDim.x;
    const int64_t ntok = a.T > blockIdx.x ? (a.T - 1 - blockIdx.x) / G + 1 : 0;
    if (warp == 0) {
        // producer
        if (lane == 0) {
            bool ok = true;
            int64_t issued = 0;
            for (int64_t i = 0; i < ntok; i++) {
                const int s = int(i % kDRingIn);
                if (i >= kDRingIn) ok = mbar_wait(in_empty(s), uint32_t((i / kDRingIn - 1) & 1));
                if (!ok) break;
                bulk_load(in0 + s * in_bytes, a.x + (blockIdx.x + i * G) * H, in_bytes, in_full(s));
                issued = i + 1;
            }
            if (!ok) set_status(a.status, MOE_ERR_TIMEOUT);
            // the copies still in flight land before the CTA's shared memory is released
            for (int64_t j = issued > kDRingIn ? issued - kDRingIn : 0; j < issued; j++)
                mbar_wait(in_full(int(j % kDRingIn)), uint32_t((j / kDRingIn) & 1), kDrainLimitNs);
        }
        return;
    }
    if (warp == 1) {
        // stores: routing, receive ids and weights, bulk stores of the code and scale rows
        uint8_t* recv_q = static_cast<uint8_t*>(a.recv_x);
        int nid = -1;
        float nw = 0.0f;
        if (ntok > 0 && lane < K) {
            nid = __ldg(a.ids + int64_t(blockIdx.x) * K + lane);
            nw = __ldg(a.w + int64_t(blockIdx.x) * K + lane);
        }
        bool ok = true;
        const int rounds = (P * K + 31) / 32;
        for (int64_t i = 0; i < ntok; i++) {
            const int64_t t = blockIdx.x + i * G;
            const int o = int(i % kDRingOut);
            const int my_id = nid;
            const float my_w = nw;
            if (i + 1 < ntok && lane < K) {  // the next token's ids and weights, one token ahead
                nid = __ldg(a.ids + (t + G) * K + lane);
                nw = __ldg(a.w + (t + G) * K + lane);
            }
            const bool valid = my_id >= 0 && my_id < a.E;
            if (!valid && my_id != -1 && lane < K) set_status(a.status, MOE_ERR_BAD_EXPERT_ID);
            bool routed = false;
            for (int k = 0; k < K; k++) {
                const int e = __shfl_sync(kFullMask, my_id, k);
                routed |= e >= 0 && e < a.E && e / a.ep == lane;
            }
            const unsigned mask = __ballot_sync(kFullMask, routed && lane < P);
            for (int r = 0; r < rounds; r++) {
                const int j = r * 32 + lane;
                const int p = j / K, k = j - p * K;
                const int id = __shfl_sync(kFullMask, my_id, k & 31);
                const float wk = __shfl_sync(kFullMask, my_w, k & 31);
                if (j < P * K) {
                    const bool rp = (mask >> p) & 1u;
                    const int64_t rr = (int64_t(p) * a.S + t) * K + k;
                    a.recv_ids[rr] = (rp && id >= 0 && id < a.E && id / a.ep == p) ? id : a.invalid_id;
                    if (rp) a.recv_w[rr] = wk;
                }
            }
            int got = 1;
            if (lane == 0) got = mbar_wait(out_full(o), uint32_t((i / kDRingOut) & 1));
            ok = __shfl_sync(kFullMask, got, 0) != 0;
            if (!ok) break;
            if (lane == 0) {
                for (unsigned m = mask; m; m &= m - 1) {
                    const int64_t row = int64_t(__ffs(m) - 1) * a.S + t;
                    bulk_store(recv_q + row * qb, out0 + o * ob, qb);
                    bulk_store(a.recv_sf + row * sb, out0 + o * ob + qb, sb);
                }
                bulk_commit();
                // the stores of token i - (kDRingOut - 1) have read their slot: hand it back
                bulk_wait_read<kDRingOut - 1>();
                if (i >= kDRingOut - 1)
                    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(out_empty(int((i - kDRingOut + 1) % kDRingOut)))
                                 : "memory");
            }
        }
        if (lane == 0) {
            bulk_wait_all();
            if (!ok) set_status(a.status, MOE_ERR_TIMEOUT);
        }
        return;
    }
    // consumers: thread ct quantises the 16-element blocks ct, ct + nct, ... of each row
    const int ct = tid - 64, nct = kDRingConsumerWarps * 32, nslices = H / 16;
    bool ok = true;
    for (int64_t i = 0; i < ntok; i++) {
        const int s = int(i % kDRingIn), o = int(i % kDRingOut);
        ok = mbar_wait(in_full(s), uint32_t((i / kDRingIn) & 1));
        if (ok && i >= kDRingOut) ok = mbar_wait(out_empty(o), uint32_t((i / kDRingOut - 1) & 1));
        if (!__all_sync(kFullMask, ok)) {
            ok = false;
            break;
        }
        const unsigned char* src = smem + size_t(s) * in_bytes;
        unsigned char* qo = smem + size_t(kDRingIn) * in_bytes + size_t(o) * ob;
        for (int slice = ct; slice < nslices; slice += nct) {
            const LaneSlice sl{*reinterpret_cast<const uint4*>(src + slice * 32),
                               *reinterpret_cast<const uint4*>(src + slice * 32 + 16)};
            const LaneCodes c = quantise16<MOE_QUANT_NVFP4_B16>(sl, a.g);
            *reinterpret_cast<uint2*>(qo + slice * 8) = make_uint2(c.q.x, c.q.y);
            qo[qb + slice] = uint8_t(c.scale);
        }
        fence_proxy_async();  // this thread's code and scale bytes become visible to the bulk stores
        __syncwarp();
        if (lane == 0) {
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(in_empty(s)) : "memory");
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(out_full(o)) : "memory");
        }
    }
    if (!ok && lane == 0) set_status(a.status, MOE_ERR_TIMEOUT);
}

__global__ void __launch_bounds__(kThreads) combine_partitioned_kernel(PartArgs a) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const int H = a.H;
    constexpr int kBatch = 8;
    for (int64_t u = warp; u < a.n_units; u += nwarps) {
        const int64_t t = u / a.units_per_row;
        // lane l owns columns [8l, 8l+8) and [256+8l, 256+8l+8) of the slice: each warp-wide
        // 16-byte load reads 512 contiguous bytes
        const int col0 = int(u - t * a.units_per_row) * kSlice + lane * 8;
        const int col1 = col0 + kSlice / 2;
        const bool act0 = col0 < H, act1 = col1 < H;  // act1 implies act0
        int my_id;
        const bool routed = token_in_partition(a, t, lane, my_id);
        const int64_t my_row = routed ? int64_t(lane) * a.S + t : -1;
        float acc[kLaneElems];
#pragma unroll
        for (int j = 0; j < kLaneElems; j++) acc[j] = 0.0f;
        for (int p0 = 0; p0 < a.P; p0 += kBatch) {
            int64_t rows[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; j++) {
                rows[j] = __shfl_sync(kFullMask, my_row, (p0 + j) & 31);
                if (p0 + j >= a.P || !act0) rows[j] = -1;
            }
            uint4 v[kBatch][2];
#pragma unroll
            for (int j = 0; j < kBatch; j++) {
                v[j][0] = make_uint4(0, 0, 0, 0);
                v[j][1] = v[j][0];
                if (rows[j] >= 0) {
                    const uint16_t* src = a.partial + rows[j] * H;
                    v[j][0] = ld_stream_v4(src + col0);
                    if (act1) v[j][1] = ld_stream_v4(src + col1);
                }
            }
#pragma unroll
            for (int j = 0; j < kBatch; j++) {
                if (rows[j] >= 0) {
                    float f[16];
                    unpack8(v[j][0], f);
                    unpack8(v[j][1], f + 8);
#pragma unroll
                    for (int e = 0; e < kLaneElems; e++) acc[e] += f[e];
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

// The combine for large batches: a ring of whole partial rows in shared memory. One producer warp
// walks the CTA's tokens and, for each partition the token was sent to (ascending p), bulk-copies
// the partial row p*S + t into the next ring slot (mbarrier "full" per slot, transaction bytes);
// eight consumer warps add each token's rows slot by slot (fp32, ascending p, as the register
// kernel), release every slot on its "empty" mbarrier (one arrival per consumer warp) and write
// the token's bf16 row. The register kernel keeps at most 8 row slices of 1 KB in flight per warp
// and uses only the routed ones (about 5.25 of 8 in the nvfp4 workload); the rings hold routed
// rows only, several small rings per SM. All waits are bounded; a CTA gives up with MOE_ERR_TIMEOUT.
constexpr int kRingConsumerWarps = 8;
constexpr int kRingThreads = (kRingConsumerWarps + 1) * 32;
constexpr int kRingMaxVecs = 4;  // 8-column vectors per consumer thread: H <= 8 * 4 * 256
constexpr int kRingMaxSlots = 16;
constexpr int kRingMinSlots = 2;
constexpr int64_t kRingMinTokens = 1024;
// Ring size: about 28 KB (two 14 KB rows at H = 7168). Measured on the nvfp4 tokens (P = 8): one
// 200 KB ring per SM 141.3 us, 100 KB 137.2, 70 KB 131.1, 44 KB 129.0, 28 KB 127.0 us (from 44 KB
// down, four CTAs per SM, held there by 56 registers x 288 threads); four consumer warps instead
// of eight 128.0-129.0; a single slot 147.4 us.
constexpr size_t kRingTargetBytes = 28 * 1024;

// Partitions of the CTA's tokens i0 + lane (stride G from blockIdx.x), one token per lane, as bit
// masks: every lane loads its token's K ids at once, so a warp pays one round trip for 32 tokens.
__device__ __forceinline__ unsigned lane_token_partitions(const PartArgs& a, int64_t i0, int64_t ntok, int lane) {
    const int64_t i = i0 + lane;
    if (i >= ntok) return 0;
    const int64_t t = blockIdx.x + i * gridDim.x;
    int id[MOE_MAX_TOPK];
#pragma unroll
    for (int k = 0; k < MOE_MAX_TOPK; k++) id[k] = k < a.K ? __ldg(a.ids + t * a.K + k) : -1;
    unsigned mask = 0;
#pragma unroll
    for (int k = 0; k < MOE_MAX_TOPK; k++)
        if (id[k] >= 0 && id[k] < a.E) mask |= 1u << (id[k] / a.ep);
    return mask;
}

__global__ void __launch_bounds__(kRingThreads) combine_partitioned_ring_kernel(PartArgs a, int NS) {
    extern __shared__ __align__(128) unsigned char smem[];  // [NS][2H] rows | full[NS] | empty[NS]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t row_bytes = uint32_t(2 * a.H);
    const uint32_t rows0 = smem_addr(smem), bars = rows0 + uint32_t(NS) * row_bytes;
    if (tid == 0) {
        for (int s = 0; s < NS; s++) {
            mbar_init(bars + 8 * s, 1);
            mbar_init(bars + 8 * (NS + s), kRingConsumerWarps);
        }
        mbar_fence_init();
    }
    __syncthreads();
    pdl_wait();
    const int64_t G = gridDim.x;
    const int64_t ntok = a.T > blockIdx.x ? (a.T - 1 - blockIdx.x) / G + 1 : 0;
    uint32_t cnt = 0;  // ring slots used so far (the same count in every warp)
    bool ok = true;
    if (warp == kRingConsumerWarps) {
        // producer
        unsigned lane_mask = 0;
        for (int64_t i = 0; i < ntok && ok; i++) {
            const int64_t t = blockIdx.x + i * G;
            if ((i & 31) == 0) lane_mask = lane_token_partitions(a, i, ntok, lane);
            unsigned mask = __shfl_sync(kFullMask, lane_mask, int(i & 31));
            while (mask && ok) {
                const int p = __ffs(mask) - 1;
                mask &= mask - 1;
                const int s = int(cnt % uint32_t(NS));
                if (lane == 0) {
                    if (cnt >= uint32_t(NS)) ok = mbar_wait(bars + 8 * (NS + s), ((cnt / NS) - 1) & 1);
                    if (ok)
                        bulk_load(rows0 + uint32_t(s) * row_bytes, a.partial + (int64_t(p) * a.S + t) * a.H, row_bytes,
                                  bars + 8 * s);
                }
                ok = __shfl_sync(kFullMask, ok, 0);
                if (ok) cnt++;
            }
        }
        if (lane == 0) {
            if (!ok) set_status(a.status, MOE_ERR_TIMEOUT);
            // the loads still in flight land before the CTA releases its shared memory
            for (uint32_t c = cnt > uint32_t(NS) ? cnt - NS : 0; c < cnt; c++)
                mbar_wait(bars + 8 * (c % NS), (c / NS) & 1, kDrainLimitNs);
        }
        return;
    }
    // consumers: thread c owns the 8-column vectors c, c + 256, ...
    const int nvec = a.H / 8, nct = kRingConsumerWarps * 32;
    unsigned lane_mask = 0;
    for (int64_t i = 0; i < ntok && ok; i++) {
        const int64_t t = blockIdx.x + i * G;
        if ((i & 31) == 0) lane_mask = lane_token_partitions(a, i, ntok, lane);
        unsigned mask = __shfl_sync(kFullMask, lane_mask, int(i & 31));
        float acc[kRingMaxVecs][8];
#pragma unroll
        for (int j = 0; j < kRingMaxVecs; j++)
#pragma unroll
            for (int e = 0; e < 8; e++) acc[j][e] = 0.0f;
        while (mask) {
            mask &= mask - 1;
            const int s = int(cnt % uint32_t(NS));
            ok = mbar_wait(bars + 8 * s, (cnt / NS) & 1);
            if (!__all_sync(kFullMask, ok)) {
                ok = false;
                break;
            }
            const unsigned char* row = smem + size_t(s) * row_bytes;
#pragma unroll
            for (int j = 0; j < kRingMaxVecs; j++) {
                const int v = tid + j * nct;
                if (v < nvec) {
                    float f[8];
                    unpack8(*reinterpret_cast<const uint4*>(row + 16 * v), f);
#pragma unroll
                    for (int e = 0; e < 8; e++) acc[j][e] += f[e];
                }
            }
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bars + 8 * (NS + s)) : "memory");
            cnt++;
        }
        if (!ok) break;
        uint16_t* dst = a.out + t * a.H;
#pragma unroll
        for (int j = 0; j < kRingMaxVecs; j++) {
            const int v = tid + j * nct;
            if (v < nvec)
                st_v4(dst + 8 * v, make_uint4(pack_bf16x2(acc[j][0], acc[j][1]), pack_bf16x2(acc[j][2], acc[j][3]),
                                              pack_bf16x2(acc[j][4], acc[j][5]), pack_bf16x2(acc[j][6], acc[j][7])));
        }
    }
    if (!ok && lane == 0) set_status(a.status, MOE_ERR_TIMEOUT);
}

template <typename Kernel>
cudaError_t launch_units(const LaunchCtx& ctx, Kernel kern, const PartArgs& a, int64_t extra_threads) {
    int per_sm = 0;
    cudaError_t err = blocks_per_sm(ctx, kern, kThreads, 0, &per_sm);
    if (err != cudaSuccess) return err;
    const int64_t need = std::max((a.n_units * 32 + kThreads - 1) / kThreads, (extra_threads + kThreads - 1) / kThreads);
    const int64_t cap = int64_t(ctx.num_sms) * (per_sm > 0 ? per_sm : 1);
    const int grid = int(std::max<int64_t>(1, std::min(need, cap)));
    return launch_pdl(ctx, kern, dim3(grid), dim3(kThreads), 0, a);
}

}  // namespace

cudaError_t launch_dispatch_layout(const LaunchCtx& ctx, const int32_t* ids, int64_t T, int K, int E, int P,
                                   int32_t* num_tokens_per_rank, uint8_t* is_token_in_rank,
                                   int32_t* num_tokens_per_expert, int32_t* dev_status) {
    if (T * K <= kLayoutSingleMaxPairs) {
        const size_t smem = sizeof(int) * size_t(P + E + T * K);
        if (smem > 48 * 1024) {
            cudaError_t err = cudaFuncSetAttribute(dispatch_layout_single_kernel,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
            if (err != cudaSuccess) return err;
        }
        return launch_pdl(ctx, dispatch_layout_single_kernel, dim3(1), dim3(kLayoutSingleThreads), smem, ids,
                          int(T), K, E, P, num_tokens_per_rank, is_token_in_rank, num_tokens_per_expert, dev_status);
    }
    cudaError_t err = cudaMemsetAsync(num_tokens_per_rank, 0, sizeof(int32_t) * size_t(P), ctx.stream);
    if (err == cudaSuccess && num_tokens_per_expert)
        err = cudaMemsetAsync(num_tokens_per_expert, 0, sizeof(int32_t) * size_t(E), ctx.stream);
    if (err != cudaSuccess || T == 0) return err;
    const int64_t blocks = std::min<int64_t>((T + kThreads - 1) / kThreads, int64_t(ctx.num_sms) * 4);
    return launch_pdl(ctx, dispatch_layout_kernel, dim3(int(blocks)), dim3(kThreads),
                      sizeof(int) * size_t(P + E), ids, T, K, E, P, num_tokens_per_rank, is_token_in_rank,
                      num_tokens_per_expert, dev_status);
}

cudaError_t launch_dispatch_partitioned(const LaunchCtx& ctx, int quant, const uint16_t* x, int64_t T, int64_t S,
                                        int H, const int32_t* ids, const float* w, int K, int E, int P,
                                        int32_t invalid_id, float g, void* recv_x, uint8_t* recv_sf,
                                        int32_t* recv_ids, float* recv_w, int32_t* dev_status, int scale_layout) {
    PartArgs a{};
    a.x = x;
    a.ids = ids;
    a.w = w;
    a.T = T;
    a.S = S;
    a.H = H;
    a.K = K;
    a.E = E;
    a.P = P;
    a.ep = E / P;
    a.invalid_id = invalid_id;
    a.g = g;
    a.recv_x = recv_x;
    a.recv_sf = recv_sf;
    a.recv_ids = recv_ids;
    a.recv_w = recv_w;
    a.status = dev_status;
    a.units_per_row = (H + kSlice - 1) / kSlice;
    a.n_units = T * a.units_per_row;
    a.L = ScaleLayout{scale_layout, 0, 0};
    // swizzled NVFP4 scales whose 128-row tiles each lie in one partition: one launch writes
    // the codes and the whole tiles (dispatch_partitioned_tiles_kernel)
    if (quant == MOE_QUANT_NVFP4_B16 && scale_layout == MOE_SCALES_SWIZZLED_128X4 && S % kTileTokens == 0 &&
        (reinterpret_cast<uintptr_t>(recv_sf) & 15) == 0) {
        a.n_units = (T + kTileTokens - 1) / kTileTokens * kTileParts * a.units_per_row;
        const int64_t pad = (S - T) * P * K;
        if (a.n_units == 0 && pad == 0) return cudaSuccess;
        int per_sm = 0;
        cudaError_t err = blocks_per_sm(ctx, dispatch_partitioned_tiles_kernel, kTileThreads, 0, &per_sm);
        if (err != cudaSuccess) return err;
        const int64_t cap = int64_t(ctx.num_sms) * (per_sm > 0 ? per_sm : 1);
        // every CTA takes the same number of units
        int64_t grid = std::min(cap, (pad + kTileThreads - 1) / kTileThreads);
        if (a.n_units > 0) {
            const int64_t per_cta = (a.n_units + cap - 1) / cap;
            grid = (a.n_units + per_cta - 1) / per_cta;
        }
        return launch_pdl(ctx, dispatch_partitioned_tiles_kernel, dim3(unsigned(std::max<int64_t>(1, grid))),
                          dim3(kTileThreads), 0, a);
    }
    // swizzled NVFP4 scales otherwise: when the buffer allows it, the scale rows go out row-major and the
    // touched tiles are interleaved in place afterwards (the interleave zeroing the rows the
    // dispatch does not write, or a clear of the touched tiles first where it cannot tell them);
    // else the touched tiles are cleared and every scale word is stored at its tile position
    SfTiles tiles{};
    bool by_tiles = false;
    if (quant == MOE_QUANT_NVFP4_B16 && scale_layout == MOE_SCALES_SWIZZLED_128X4) {
        tiles.sf = recv_sf;
        tiles.R = int64_t(P) * S;
        tiles.C = H / 16;
        tiles.kind = kSfTilesPartitioned;
        tiles.P = P;
        tiles.S = S;
        tiles.T = T;
        tiles.n_blocks = (tiles.R + 127) / 128;
        tiles.q_per_group = sf_tiles_q_per_group(T, P);
        tiles.status = dev_status;
        tiles.ids = ids;
        tiles.K = K;
        tiles.E = E;
        tiles.ep = E / P;
        by_tiles = sf_tiles_interleavable(tiles);
        cudaError_t err = sf_tiles_interleave_zeroes(tiles) ? cudaSuccess : launch_sf_tiles_clear(ctx, tiles);
        if (err != cudaSuccess) return err;
        if (by_tiles) {
            scale_layout = MOE_SCALES_ROW_MAJOR;
            a.L.kind = MOE_SCALES_ROW_MAJOR;
        }
    }
    // NVFP4 with row-major scale rows (the caller's layout, not the swizzled layout's row-major
    // stage) that bulk copies can store: the warp-specialised ring
    constexpr bool kDRing = true;
    if (kDRing && quant == MOE_QUANT_NVFP4_B16 && scale_layout == MOE_SCALES_ROW_MAJOR && !by_tiles && T >= 1024 &&
        H % 256 == 0 &&
        (reinterpret_cast<uintptr_t>(recv_sf) & 15) == 0 && dring_smem(H) <= 200 * 1024) {
        const size_t smem = dring_smem(H);
        cudaError_t err = cudaFuncSetAttribute(dispatch_partitioned_ring_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        int per_sm = 0;
        if (err == cudaSuccess) err = blocks_per_sm(ctx, dispatch_partitioned_ring_kernel, kDRingThreads, smem, &per_sm);
        if (err != cudaSuccess) return err;
        const int grid = int(std::min<int64_t>(T, int64_t(ctx.num_sms) * (per_sm > 0 ? per_sm : 1)));
        return launch_pdl(ctx, dispatch_partitioned_ring_kernel, dim3(grid), dim3(kDRingThreads), smem, a);
    }
    bool bulk = false;
    cudaError_t err = launch_dispatch_partitioned_bulk(ctx, quant, x, T, S, H, ids, w, K, E, P, invalid_id, g,
                                                       recv_x, recv_sf, recv_ids, recv_w, dev_status, scale_layout,
                                                       &bulk, by_tiles);
    if (err == cudaSuccess && !bulk) {
        const int64_t pad = (S - T) * P * K;
        if (a.n_units > 0 || pad > 0)
            err = quant == MOE_QUANT_NVFP4_B16 ? launch_units(ctx, dispatch_partitioned_kernel<MOE_QUANT_NVFP4_B16>, a, pad)
                                               : launch_units(ctx, dispatch_partitioned_kernel<MOE_QUANT_NONE>, a, pad);
    }
    if (err != cudaSuccess || !by_tiles) return err;
    return launch_sf_tiles_interleave(ctx, tiles);
}

cudaError_t launch_combine_partitioned(const LaunchCtx& ctx, const uint16_t* partial, int64_t T, int64_t S, int H,
                                       const int32_t* ids, int K, int E, int P, uint16_t* out, int32_t* dev_status) {
    PartArgs a{};
    a.partial = partial;
    a.ids = ids;
    a.T = T;
    a.S = S;
    a.H = H;
    a.K = K;
    a.E = E;
    a.P = P;
    a.ep = E / P;
    a.out = out;
    a.status = dev_status;
    a.units_per_row = (H + kSlice - 1) / kSlice;
    a.n_units = T * a.units_per_row;
    if (a.n_units == 0) return cudaSuccess;
    // large batches whose rows fit a consumer thread's registers (H <= 8192): the ring
    const size_t row_bytes = 2 * size_t(H);
    const int NS = int(std::max<size_t>(kRingMinSlots, std::min<size_t>(kRingMaxSlots, kRingTargetBytes / row_bytes)));
    if (T >= kRingMinTokens && H / 8 <= kRingMaxVecs * kRingConsumerWarps * 32) {
        const size_t smem = size_t(NS) * row_bytes + 16 * size_t(NS);
        cudaError_t err =
            cudaFuncSetAttribute(combine_partitioned_ring_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        int per_sm = 0;
        if (err == cudaSuccess) err = blocks_per_sm(ctx, combine_partitioned_ring_kernel, kRingThreads, smem, &per_sm);
        if (err != cudaSuccess) return err;
        const int grid = int(std::min<int64_t>(T, int64_t(ctx.num_sms) * (per_sm > 0 ? per_sm : 1)));
        return launch_pdl(ctx, combine_partitioned_ring_kernel, dim3(grid), dim3(kRingThreads), smem, a, NS);
    }
    return launch_units(ctx, combine_partitioned_kernel, a, 0);
}

}  // namespace moe

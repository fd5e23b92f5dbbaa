// sf_swizzle.cu -- NVFP4 block scales in the 128 x 4 tile layout of the block-scaled MMA.
//
// The flashinfer.py page ("sglang token_dispatcher/flashinfer.py", FlashinferDispatcher.dispatch)
// passes the received row-major e4m3 block scales [R, C] (C = H/16) through
// nvfp4_block_scale_interleave before the CUTLASS MoE: 128-row x 4-column tiles of 512 bytes in
// row-tile-major order, row i / column c of a tile at byte (i % 32) * 16 + (i / 32) * 4 + c.
//
// Row block b (rows 128b .. 128b+127) occupies bytes [128 b C, 128 (b+1) C) in the row-major
// layout and exactly the same bytes in the tile layout (its C/4 tiles of 512 bytes). So the
// dispatch kernels write the scale rows row-major, whole rows at a time, into the caller's
// swizzled buffer, and one pass per touched row block turns the block into its tiles in place:
// the block's rows are bulk-copied (TMA) into shared memory, then written back as whole 16-byte
// lines (a line holds rows i, i+32, i+64, i+96 of four columns; a warp writes 512 contiguous
// bytes). The rows of a touched block that no pair maps to end up as zeros, and so do the
// padding rows R .. roundup(R, 128) - 1: in the masked and partitioned layouts the interleave
// itself writes zeros for them (it knows which rows the dispatch writes: the ranks below each
// expert's segment length, the slots of tokens a partition receives); in the contiguous layout
// the touched blocks are cleared before the dispatch. A buffer that is not 16-byte aligned, or
// whose block does not fit in shared memory, is cleared the same way and then receives each
// scale word straight at its tile position from the dispatch.
//
// Touched row blocks: every block of the contiguous layout [0, roundup(R, 128)); in the masked
// layout the blocks overlapping rows e*M + [0, min(M, seg_indptr[e+1] - seg_indptr[e])) of some
// expert e (a group); in the partitioned layout those overlapping p*S + [0, T) of some partition
// p (a group); and, in every layout, the last block when R is not a multiple of 128 (its padding
// rows). Blocks not touched keep their previous bytes.
//
// Work split: CTA (g, q) of the Q CTAs of group g takes blocks first + q, first + q + Q, ... of
// the group's run of blocks; one more CTA takes the padding block. A block that two groups
// touch (only a group's first block can also belong to an earlier group) is interleaved by the
// earlier group only; the clear may zero it twice, which is harmless.
#include <algorithm>
#include <cstdint>

#include "moe_device.cuh"
#include "moe_launch.h"

namespace moe {
namespace {

constexpr int kSfThreads = 256;

// Run of blocks [*fb, *lb] of group g (empty when *lb < *fb). Masked groups read seg_indptr.
__device__ __forceinline__ void group_run(const SfTiles& a, int64_t g, int64_t* fb, int64_t* lb) {
    int64_t lo, n;
    if (a.kind == kSfTilesMasked) {
        lo = g * a.M;
        n = __ldg(a.seg + g + 1) - __ldg(a.seg + g);
        if (n > a.M) n = a.M;
    } else {
        lo = g * a.S;
        n = a.T;
    }
    *fb = lo / 128;
    *lb = n > 0 ? (lo + n - 1) / 128 : *fb - 1;
}

__host__ __device__ inline int64_t sf_groups(const SfTiles& a) {
    return a.kind == kSfTilesMasked ? a.E : (a.kind == kSfTilesPartitioned ? a.P : 0);
}

// Whether block b belongs to the run of some group g' < g_end among those whose rows can reach
// it (groups from the one holding row 128b).
__device__ bool block_in_earlier_run(const SfTiles& a, int64_t b, int64_t g_end) {
    const int64_t span = a.kind == kSfTilesMasked ? a.M : a.S;
    for (int64_t g = (b * 128) / span; g < g_end; g++) {
        int64_t fb, lb;
        group_run(a, g, &fb, &lb);
        if (lb >= fb && fb <= b && b <= lb) return true;
    }
    return false;
}

// The blocks CTA blockIdx.x handles: *b0, *b0 + *step, ... up to *b1. With `owned` the block a
// group shares with an earlier one is left to the earlier one (interleave); the clear takes all.
__device__ void cta_blocks(const SfTiles& a, bool owned, int64_t* b0, int64_t* b1, int64_t* step) {
    *b0 = 0;
    *b1 = -1;
    *step = 1;
    const int64_t c = blockIdx.x;
    if (a.kind == kSfTilesAll) {  // grid-stride over every block
        *b0 = c;
        *b1 = a.n_blocks - 1;
        *step = gridDim.x;
        return;
    }
    const int64_t G = sf_groups(a), Q = a.q_per_group;
    if (c < G * Q) {
        const int64_t g = c / Q, q = c - g * Q;
        int64_t fb, lb;
        group_run(a, g, &fb, &lb);
        if (lb < fb) return;
        if (owned && g > 0 && block_in_earlier_run(a, fb, g)) fb++;
        *b0 = fb + q;
        *b1 = lb;
        *step = Q;
        return;
    }
    // the padding block, unless a group's run holds it
    if (c == G * Q && (a.R % 128) != 0) {
        const int64_t pb = a.n_blocks - 1;
        if (!owned || !block_in_earlier_run(a, pb, G)) *b0 = *b1 = pb;
    }
}

// Zeros of every touched block; 16-byte stores when the buffer is 16-byte aligned, else 4-byte ones.
template <bool VEC16>
__global__ void __launch_bounds__(kSfThreads) sf_tiles_clear_kernel(SfTiles a) {
    pdl_wait();
    int64_t b0, b1, step;
    cta_blocks(a, false, &b0, &b1, &step);
    const int64_t block_bytes = int64_t(a.C) * 128;
    // the interleave reads these lines back after the dispatch: kept in L2 ahead of the code rows
    const uint64_t keep = l2_policy_evict_last();
    for (int64_t b = b0; b <= b1; b += step) {
        uint8_t* base = a.sf + b * block_bytes;
        if constexpr (VEC16) {
            for (int64_t o = 16 * int64_t(threadIdx.x); o < block_bytes; o += 16 * int64_t(blockDim.x))
                st_v4_hint(base + o, make_uint4(0, 0, 0, 0), keep);
        } else {
            for (int64_t o = 4 * int64_t(threadIdx.x); o < block_bytes; o += 4 * int64_t(blockDim.x))
                *reinterpret_cast<uint32_t*>(base + o) = 0u;
        }
    }
}

// Shared-memory row stride of the interleave: C rounded up to an odd number of 16-byte units, so
// that eight consecutive rows' 16-byte reads at one column fall in eight different bank groups.
__host__ __device__ constexpr int sf_row_stride(int C) { return ((C + 15) / 16 | 1) * 16; }

// Whether row r of the scale matrix holds scales the dispatch wrote, for the layouts whose
// interleave zeroes the other rows: masked, rank < min(M, seg_indptr[e+1] - seg_indptr[e]) (the
// dispatch writes ranks below the expert's pair count, which these segment lengths are for
// metadata without expert alignment); partitioned, slot t < T of a partition that receives token t.
__device__ bool row_written(const SfTiles& a, int64_t r) {
    if (r >= a.R) return false;  // padding rows
    if (a.kind == kSfTilesMasked) {
        const int64_t e = r / a.M, rank = r - e * a.M;
        int64_t n = __ldg(a.seg + e + 1) - __ldg(a.seg + e);
        if (n > a.M) n = a.M;
        return rank < n;
    }
    if (a.kind == kSfTilesPartitioned) {
        const int64_t p = r / a.S, t = r - p * a.S;
        if (t >= a.T) return false;
        bool routed = false;
        for (int k = 0; k < a.K; k++) {
            const int e = __ldg(a.ids + t * a.K + k);
            routed |= e >= 0 && e < a.E && e / a.ep == p;
        }
        return routed;
    }
    return true;  // contiguous layout: cleared before the dispatch, every row is taken as it is
}

// Row-major -> 128 x 4 tiles, in place (C % 16 == 0). The block's 128 rows arrive by bulk copies
// into rows of sf_row_stride(C) bytes; thread (c16, i) then reads rows i, i+32, i+64, i+96 at
// columns 16*c16 .. 16*c16+15 (four 16-byte reads) and writes the four lines (4*c16 + k, i),
// k = 0..3, line k taking word k of each of the four rows. Rows the dispatch did not write
// (row_written) go out as zeros.
__global__ void __launch_bounds__(kSfThreads) sf_tiles_interleave_kernel(SfTiles a) {
    // [128][stride] rows, then the mbarrier (8 bytes), then 128 row flags
    extern __shared__ __align__(128) unsigned char s_rows[];
    const int C = a.C, stride = sf_row_stride(C), C16 = C / 16;
    const uint32_t bar = smem_addr(s_rows + 128 * stride);
    int* s_keep = reinterpret_cast<int*>(s_rows + 128 * stride + 8);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        mbar_fence_init();
    }
    __syncthreads();
    pdl_wait();
    int64_t b0, b1, step;
    cta_blocks(a, true, &b0, &b1, &step);
    uint32_t phase = 0;
    int64_t issued = 0, done = 0;  // thread 0's counts of block loads issued / completed
    for (int64_t b = b0; b <= b1; b += step) {
        uint8_t* base = a.sf + b * 128 * int64_t(C);
        // warp 0 issues the 128 row copies, four per lane, after lane 0 has set the byte count
        if (threadIdx.x < 32) {
            if (threadIdx.x == 0) {
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                             "r"(uint32_t(128 * C))
                             : "memory");
                issued++;
            }
            __syncwarp();
            for (int r = threadIdx.x; r < 128; r += 32)
                asm volatile(
                    "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                        smem_addr(s_rows + r * stride)),
                    "l"(base + int64_t(r) * C), "r"(uint32_t(C)), "r"(bar)
                    : "memory");
        } else if (threadIdx.x < 32 + 128) {
            // while the rows are in flight: which of them the dispatch wrote
            const int r = threadIdx.x - 32;
            s_keep[r] = row_written(a, b * 128 + r) ? -1 : 0;
        }
        const int ok = __syncthreads_and(mbar_wait(bar, phase));
        if (!ok) {
            if (threadIdx.x == 0) set_status(a.status, MOE_ERR_TIMEOUT);
            break;
        }
        done++;
        phase ^= 1;
        for (int L = threadIdx.x; L < 32 * C16; L += blockDim.x) {
            const int c16 = L >> 5, i = L & 31;
            uint4 r[4];
#pragma unroll
            for (int q = 0; q < 4; q++) {
                r[q] = *reinterpret_cast<const uint4*>(s_rows + (i + 32 * q) * stride + 16 * c16);
                const uint32_t m = uint32_t(s_keep[i + 32 * q]);
                r[q] = make_uint4(r[q].x & m, r[q].y & m, r[q].z & m, r[q].w & m);
            }
            uint8_t* dst = base + int64_t(4 * c16) * 512 + i * 16;
            st_v4(dst, make_uint4(r[0].x, r[1].x, r[2].x, r[3].x));
            st_v4(dst + 512, make_uint4(r[0].y, r[1].y, r[2].y, r[3].y));
            st_v4(dst + 1024, make_uint4(r[0].z, r[1].z, r[2].z, r[3].z));
            st_v4(dst + 1536, make_uint4(r[0].w, r[1].w, r[2].w, r[3].w));
        }
        // the rows are overwritten by the next block's copies: every read above happens first
        __syncthreads();
    }
    // after a timeout, a load still in flight is waited for (bounded) before shared memory is released
    if (threadIdx.x == 0 && issued > done) mbar_wait(bar, phase, kDrainLimitNs);
}

// Row-major -> 128 x 4 tiles, in place, for C % 16 != 0 (C % 4 == 0): word loads through
// registers into rows of an odd number of words.
constexpr int kLoadBatch = 16;
__host__ __device__ constexpr int sf_stride_words(int C) { return (C / 4) | 1; }

__global__ void __launch_bounds__(kSfThreads) sf_tiles_interleave_words_kernel(SfTiles a) {
    extern __shared__ uint32_t s_blk[];  // [128][stride] words
    const int C4 = a.C / 4, stride = sf_stride_words(a.C);
    pdl_wait();
    int64_t b0, b1, step;
    cta_blocks(a, true, &b0, &b1, &step);
    const int tid = threadIdx.x, nt = blockDim.x;
    for (int64_t b = b0; b <= b1; b += step) {
        uint8_t* base = a.sf + b * 128 * a.C;
        const int nw = 128 * C4;
        for (int w0 = tid; w0 < nw; w0 += kLoadBatch * nt) {
            uint32_t x[kLoadBatch];
#pragma unroll
            for (int u = 0; u < kLoadBatch; u++)
                if (w0 + u * nt < nw) x[u] = __ldcs(reinterpret_cast<const unsigned int*>(base) + w0 + u * nt);
#pragma unroll
            for (int u = 0; u < kLoadBatch; u++) {
                const int w = w0 + u * nt;
                if (w < nw) {
                    const int row = w / C4, col = w - row * C4;
                    s_blk[row * stride + col] = x[u];
                }
            }
        }
        __syncthreads();
        // line (c4, i): rows i, i+32, i+64, i+96 of columns 4c4 .. 4c4+3, at c4*512 + i*16
        for (int L = tid; L < 32 * C4; L += nt) {
            const int c4 = L >> 5, i = L & 31;
            const uint32_t* s = s_blk + i * stride + c4;
            st_v4(base + int64_t(c4) * 512 + i * 16, make_uint4(s[0], s[32 * stride], s[64 * stride], s[96 * stride]));
        }
        __syncthreads();
    }
}

size_t interleave_smem(const SfTiles& a) {
    if (a.C % 16 == 0) return 128 * size_t(sf_row_stride(a.C)) + 8 + 128 * sizeof(int);
    return sizeof(uint32_t) * 128 * size_t(sf_stride_words(a.C));
}

// Grid: Q CTAs per group plus one for the padding block; for the contiguous layout, every block
// with what fits on the device at once.
int64_t sf_grid(const LaunchCtx& ctx, const SfTiles& a, int per_sm) {
    if (a.kind == kSfTilesAll)
        return std::max<int64_t>(1, std::min(a.n_blocks, int64_t(ctx.num_sms) * (per_sm > 0 ? per_sm : 1)));
    return sf_groups(a) * a.q_per_group + 1;
}

template <typename Kernel>
cudaError_t launch_sf(const LaunchCtx& ctx, Kernel kern, const SfTiles& a, size_t smem) {
    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (err != cudaSuccess) return err;
    }
    int per_sm = 0;
    cudaError_t err = blocks_per_sm(ctx, kern, kSfThreads, smem, &per_sm);
    if (err != cudaSuccess) return err;
    return launch_pdl(ctx, kern, dim3(unsigned(sf_grid(ctx, a, per_sm))), dim3(kSfThreads), smem, a);
}

}  // namespace

bool sf_tiles_interleave_zeroes(const SfTiles& a) {
    return sf_tiles_interleavable(a) && a.C % 16 == 0 && a.kind != kSfTilesAll;
}

bool sf_tiles_interleavable(const SfTiles& a) {
    return a.C % 4 == 0 && (reinterpret_cast<uintptr_t>(a.sf) & 15) == 0 && interleave_smem(a) <= 200 * 1024;
}

cudaError_t launch_sf_tiles_clear(const LaunchCtx& ctx, const SfTiles& a) {
    if (a.n_blocks == 0) return cudaSuccess;
    if ((reinterpret_cast<uintptr_t>(a.sf) & 15) == 0) return launch_sf(ctx, sf_tiles_clear_kernel<true>, a, 0);
    return launch_sf(ctx, sf_tiles_clear_kernel<false>, a, 0);
}

cudaError_t launch_sf_tiles_interleave(const LaunchCtx& ctx, const SfTiles& a) {
    if (a.n_blocks == 0) return cudaSuccess;
    if (a.C % 16 == 0) return launch_sf(ctx, sf_tiles_interleave_kernel, a, interleave_smem(a));
    return launch_sf(ctx, sf_tiles_interleave_words_kernel, a, interleave_smem(a));
}

int64_t sf_tiles_q_per_group(int64_t rows_per_group_guess, int64_t groups) {
    // enough CTAs per group for a run of that many rows (rows / 128, plus one block for a run
    // that does not start on a block boundary), within a grid of at most 2^20 CTAs; longer
    // runs loop
    const int64_t q = (std::max<int64_t>(rows_per_group_guess, 1) + 127) / 128 + 1;
    const int64_t cap = std::max<int64_t>(1, (int64_t(1) << 20) / std::max<int64_t>(groups, 1));
    return std::min(q, cap);
}

}  // namespace moe

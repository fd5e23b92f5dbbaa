// dispatch_slice.cuh -- quantise one lane's 16 elements of a token row and store them into
// the K destination rows (shared by the dispatch kernels).
//
// Q = identity, FP8 e4m3 per 128-element group (sglang_per_token_group_quant_fp8 in
// _DeepEPDispatcherImplNormal.dispatch_a, "sglang token_dispatcher/deepep.py" page; with
// round_scale / use_ue8m0 the scale is rounded up to a power of two, kept as a UE8M0 byte), or
// NVFP4 e2m1 with an e4m3 scale per 16-element block (fp4_quantize in
// FlashinferDispatcher.dispatch, "sglang token_dispatcher/flashinfer.py" page):
//   fp8:   s = max(amax, 1e-10) / 448,           q = e4m3(x / s)
//   nvfp4: sf = e4m3((amax / 6) * g),             q = e2m1(x * (g / value(sf))), 0 if sf == 0
// Every division and multiplication is an explicit round-to-nearest binary32 operation
// (__fdiv_rn / __fmul_rn; x / s as a correctly rounded quotient from the reciprocal, see
// div_by_scale) and the conversions are cvt.rn.satfinite, so the codes are a deterministic
// function of the input bits.
#pragma once

#include "moe_device.cuh"

namespace moe {

// Where the scales of a destination row go (moe_scale_layout_t).
struct ScaleLayout {
    int kind;         // MOE_SCALES_ROW_MAJOR: [rows, G]; MOE_SCALES_COL_MAJOR: MN-major with rows
                      // padded to a multiple of 4; MOE_SCALES_SWIZZLED_128X4: 128 x 4 tiles
    int64_t rows_al;  // column-major: padded rows (normal layout) or padded slots M (masked)
    int M;            // masked layout: slots per expert; 0 for the contiguous layout
};

// Byte offset of scale column g (of G, a multiple of 4) of row r in the 128 x 4 tile layout
// of the block-scaled MMA (nvfp4_block_scale_interleave): tiles of 128 rows x 4 columns,
// 512 bytes each, in row-tile-major order; inside a tile, row i and column c at
// (i % 32) * 16 + (i / 32) * 4 + c.
__host__ __device__ __forceinline__ int64_t swizzled_128x4_index(int64_t r, int g, int G) {
    const int64_t tile = (r >> 7) * (G >> 2) + (g >> 2);
    const int i = int(r & 127);
    return tile * 512 + (i & 31) * 16 + (i >> 5) * 4 + (g & 3);
}

// Element index of group g's scale for destination `row`: fp32 elements, or bytes when
// `packed4` (UE8M0: four groups per int32 word, little-endian) or for the swizzled layout.
__device__ __forceinline__ int64_t scale_index(const ScaleLayout& L, int64_t row, int g, int G, bool packed4) {
    if (L.kind == MOE_SCALES_ROW_MAJOR) return row * G + g;
    if (L.kind == MOE_SCALES_SWIZZLED_128X4) return swizzled_128x4_index(row, g, G);
    int64_t e = 0, r = row;
    if (L.M > 0) {
        e = row / L.M;
        r = row - e * L.M;
    }
    if (!packed4) return (e * G + g) * L.rows_al + r;
    const int G4 = (G + 3) / 4;
    return ((e * G4 + g / 4) * L.rows_al + r) * 4 + (g & 3);
}

// x / s rounded to nearest even in binary32, given y = 1/s rounded to nearest even, by one
// correction step after P. W. Markstein ("Computation of elementary functions on the IBM
// RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990): q = x*y lies within an ulp of
// x/s, the remainder x - q*s is exact in one fused multiply-add, and q + remainder*y rounded
// once is the correctly rounded quotient -- unless the remainder leaves the normal range
// (|x| < 2^-103 here), where |x/s| < 2^-61 and the e4m3 code is a signed zero either way.
// moe_fp8_division_check compares the codes with those of the IEEE division over every
// (x, s) pair the FP8 quantiser can meet.
__device__ __forceinline__ float div_by_scale(float x, float s, float y) {
    const float q = __fmul_rn(x, y);
    const float r = __fmaf_rn(-q, s, x);
    // a zero remainder means q is exact; adding it would also turn -0 into +0
    return r == 0.0f ? q : __fmaf_rn(r, y, q);
}

// One lane's payload: 16 bf16 elements (two 16-byte vectors) of a token row.
struct LaneSlice {
    uint4 v0, v1;
};

__device__ __forceinline__ LaneSlice load_slice(const uint16_t* src) {
    LaneSlice s;
    s.v0 = ld_stream_v4(src);
    s.v1 = ld_stream_v4(src + 8);
    return s;
}

// The quantised form of one lane's 16 elements.
//   FP8 (both scale kinds): q = 16 e4m3 codes; scale = fp32 scale bits or the UE8M0 byte
//   NVFP4: q.x, q.y = 16 e2m1 codes (8 bytes); scale = the e4m3 block-scale byte
struct LaneCodes {
    uint4 q;
    uint32_t scale;
};

// Quantise the lane's 16 elements. FP8 modes reduce amax over the 8 aligned lanes of a
// 128-element group with shuffles, so all 32 lanes of the warp must call this together
// (inactive lanes hold zeros, and a group is never split between active and inactive lanes).
template <int QUANT>
__device__ __forceinline__ LaneCodes quantise16(const LaneSlice& s, float g) {
    float f[16];
    unpack8(s.v0, f);
    unpack8(s.v1, f + 8);
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; j++) amax = fmaxf(amax, fabsf(f[j]));
    LaneCodes out;
    if constexpr (QUANT == MOE_QUANT_FP8_G128 || QUANT == MOE_QUANT_FP8_G128_UE8M0) {
        amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 2));
        amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 4));
        const float sc = __fdiv_rn(fmaxf(amax, 1e-10f), 448.0f);
        uint32_t w[4];
        if constexpr (QUANT == MOE_QUANT_FP8_G128) {
            const float y = __frcp_rn(sc);
#pragma unroll
            for (int p = 0; p < 4; p++) {
                const uint32_t lo = e4m3x2(div_by_scale(f[4 * p], sc, y), div_by_scale(f[4 * p + 1], sc, y));
                const uint32_t hi = e4m3x2(div_by_scale(f[4 * p + 2], sc, y), div_by_scale(f[4 * p + 3], sc, y));
                w[p] = lo | (hi << 16);
            }
            out.scale = __float_as_uint(sc);
        } else {
            // the scale rounded up to a power of two 2^(ex-127): dividing by it is exact, so
            // x * 2^(127-ex) gives the same binary32 value as x / 2^(ex-127)
            const uint32_t bits = __float_as_uint(sc);
            const uint32_t ex = (bits >> 23) + ((bits & 0x7fffffu) ? 1u : 0u);
            const float inv = __uint_as_float((254u - ex) << 23);
#pragma unroll
            for (int p = 0; p < 4; p++) {
                const uint32_t lo = e4m3x2(__fmul_rn(f[4 * p], inv), __fmul_rn(f[4 * p + 1], inv));
                const uint32_t hi = e4m3x2(__fmul_rn(f[4 * p + 2], inv), __fmul_rn(f[4 * p + 3], inv));
                w[p] = lo | (hi << 16);
            }
            out.scale = ex;
        }
        out.q = make_uint4(w[0], w[1], w[2], w[3]);
    } else {  // MOE_QUANT_NVFP4_B16: the lane's 16 elements are one block
        const float tsf = __fmul_rn(__fdiv_rn(amax, 6.0f), g);
        const uint32_t sf = e4m3x2(tsf, 0.0f) & 0xffu;
        const float sff = e4m3_value(sf);
        out.q = make_uint4(0, 0, 0, 0);
        if (sff != 0.0f) {
            const float r = __fdiv_rn(g, sff);
            uint32_t b[8];
#pragma unroll
            for (int p = 0; p < 8; p++) b[p] = e2m1x2(__fmul_rn(f[2 * p], r), __fmul_rn(f[2 * p + 1], r));
            out.q.x = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
            out.q.y = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
        }
        out.scale = sf;
    }
    return out;
}

// Quantise `s` (the lane's 16 elements starting at column `col`, lane index `lane`) and
// write it to every destination row: row k of the token is __shfl(my_row, k), -1 = none.
// All 32 lanes of the warp must call this together (the FP8 group amax and the row
// broadcast are warp shuffles); `active` is false for lanes past the end of the row.
template <int QUANT>
__device__ __forceinline__ void quantise_store(const LaneSlice& s, bool active, int lane, int col, int H,
                                               int K, int64_t my_row, float g, void* out_q,
                                               void* out_s, const ScaleLayout& L = ScaleLayout{MOE_SCALES_ROW_MAJOR, 0, 0}) {
    if constexpr (QUANT == MOE_QUANT_NONE) {
        uint16_t* out = static_cast<uint16_t*>(out_q);
        for (int k = 0; k < K; k++) {
            const int64_t row = __shfl_sync(kFullMask, my_row, k);
            if (row >= 0 && active) {
                uint16_t* dst = out + row * H + col;
                st_v4(dst, s.v0);
                st_v4(dst + 8, s.v1);
            }
        }
    } else {
        const LaneCodes c = quantise16<QUANT>(s, g);
        uint8_t* out = static_cast<uint8_t*>(out_q);
        const int groups = H / 128;
        for (int k = 0; k < K; k++) {
            const int64_t row = __shfl_sync(kFullMask, my_row, k);
            if (row < 0 || !active) continue;
            if constexpr (QUANT == MOE_QUANT_FP8_G128) {
                st_v4(out + row * H + col, c.q);
                if ((lane & 7) == 0)
                    static_cast<float*>(out_s)[scale_index(L, row, col / 128, groups, false)] = __uint_as_float(c.scale);
            } else if constexpr (QUANT == MOE_QUANT_FP8_G128_UE8M0) {
                st_v4(out + row * H + col, c.q);
                if ((lane & 7) == 0)
                    static_cast<uint8_t*>(out_s)[scale_index(L, row, col / 128, groups, true)] = uint8_t(c.scale);
            } else {
                st_v2(out + row * (H / 2) + col / 2, make_uint2(c.q.x, c.q.y));
                static_cast<uint8_t*>(out_s)[scale_index(L, row, col / 16, H / 16, true)] = uint8_t(c.scale);
            }
        }
    }
}

}  // namespace moe

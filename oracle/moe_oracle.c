/*
 * moe_oracle.c -- CPU oracle for the MoE token dispatch / combine hot path.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the independent reference that the CUDA
 * library is checked against. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load it; the product path never does. It shares no
 * code, header, table or constant generator with the CUDA library.
 *
 * Style: plain, single-threaded, obviously correct. Every function restates the
 * definition it implements; nothing is blocked, fused or reordered beyond it.
 * Floating point: quantisation runs in IEEE binary32 with round-to-nearest-even,
 * one operation at a time, in the order written (the pages fix no precision, so
 * the oracle takes the decision in the kernel's precision); the combine
 * accumulates in binary64 and rounds once to bf16. Build with
 * -ffp-contract=off and without -ffast-math so no operation is fused or reassociated.
 *
 * Sources (the SGLang dispatcher pages):
 *  - "sglang 0.4.4.post2 -> 0.4.4.post4, ep_moe/token_dispatcher.py" diff:
 *    _DeepEPDispatcherImplNormal._deepep_permute (deepep_run_moe_deep_preprocess
 *    returns reorder_topk_ids, src2dst, seg_indptr; the PreReorder kernel copies each
 *    token row to its src2dst rows), dispatch_b (empty batch: seg_indptr is zeros of
 *    length num_experts+1, int64), combine_a (deepep_post_reorder: output[t] is the
 *    topk_weights-weighted sum of the rows src2dst[t, k]).
 *  - "sglang token_dispatcher/deepep.py" page: _DeepEPDispatcherImplNormal.dispatch_a
 *    (per-token-group-128 FP8 quantisation before dispatch),
 *    _DeepEPDispatcherImplLowLatency.dispatch_a (expected_m) and _dispatch_core
 *    (low_latency_dispatch into the masked layout with packed_recv_count = masked_m,
 *    num_max_dispatch_tokens_per_rank, use_nvfp4 with x_global_scale).
 *  - "sglang token_dispatcher/flashinfer.py" page: FlashinferDispatcher.__init__
 *    (dispatch payload bytes per token) and dispatch (fp4_quantize with
 *    input_global_scale, non-swizzled e4m3 block scales; nvfp4_block_scale_interleave
 *    of the received scales for the CUTLASS MoE).
 *
 * Readings where the pages are silent (the metadata routine's body, the exact
 * quantisation arithmetic, the masked slot order) are listed beside each function.
 *
 * Parity pins: every function here is checked by the CPU tests against brute force,
 * closed forms, library conversions or invariants that do not reuse this code.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* oracle-local status bits (returned by oracle_route_meta / oracle_dispatch) */
#define ORACLE_BAD_ID   1   /* an id outside [-1, E) was seen and skipped          */
#define ORACLE_CAPACITY 2   /* an expert received more than M pairs (masked mode) */

/* ------------------------------------------------------------------------- */
/* number formats                                                             */
/* ------------------------------------------------------------------------- */

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static float bf16_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

float oracle_bf16_to_float(uint16_t h) { return bf16_to_float(h); }

/*
 * Round a real number (given exactly as a binary64) to the nearest bf16,
 * ties to even. bf16: 1 sign, 8 exponent (bias 127), 7 stored mantissa bits;
 * normal values 2^(e-127) * (1 + m/128), subnormals m * 2^-133.
 * The quotient a / quantum below is an exact power-of-two scaling, so nearbyint
 * (round-half-even in the default rounding mode) performs the only rounding.
 */
uint16_t oracle_bf16_from_double(double d)
{
    if (isnan(d)) return 0x7FC0;
    uint16_t sign = signbit(d) ? 0x8000 : 0x0000;
    double a = fabs(d);
    if (a == 0.0) return sign;
    double r;
    if (a < 0x1p-126) {
        r = nearbyint(a * 0x1p133) * 0x1p-133;
    } else {
        int ex;
        (void)frexp(a, &ex);                   /* a in [2^(ex-1), 2^ex) */
        double quantum = ldexp(1.0, ex - 1 - 7);
        r = nearbyint(a / quantum) * quantum;
    }
    if (r > 0x1.FEp127) return (uint16_t)(sign | 0x7F80);   /* rounds past the largest finite */
    float f = (float)r;                                      /* exact: r is a bf16 value */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (u >> 16));
}

/*
 * FP8 E4M3 ("fn" flavour: no infinities, 0x7F/0xFF are NaN, largest finite 448).
 * Code layout s.eeee.mmm, bias 7:
 *   e == 0 : value = m * 2^-9            (subnormal)
 *   e >= 1 : value = 2^(e-7) * (1 + m/8)
 */
double oracle_e4m3_to_double(uint8_t c)
{
    int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = m * 0x1p-9;
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/*
 * Nearest E4M3 value to v, ties to even, saturating to +-448 ("satfinite"):
 * magnitudes that would round above 448 become 448. The sign is kept, so a
 * negative value that rounds to zero gives the negative zero code 0x80.
 * Within one binade [2^k, 2^(k+1)) the E4M3 values are evenly spaced by
 * 2^(k-3); below 2^-6 the spacing is the subnormal quantum 2^-9. Codes are
 * monotone in value, so code = (biased exponent)*8 + (multiple of the quantum) - 8.
 */
uint8_t oracle_e4m3_from_float(float v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    if (isnan(v)) return (uint8_t)(sign | 0x7F);
    double a = fabs((double)v);
    if (isinf(a)) return (uint8_t)(sign | 0x7E);
    long code;
    if (a < 0x1p-6) {
        code = (long)nearbyint(a * 0x1p9);                  /* 0..8; 8 is the smallest normal */
    } else {
        int ex;
        (void)frexp(a, &ex);                                /* a in [2^(ex-1), 2^ex) */
        long e = (ex - 1) + 7;                              /* biased exponent */
        double q = nearbyint(a / ldexp(1.0, ex - 1 - 3));   /* 8..16 */
        code = e * 8 + (long)q - 8;
    }
    if (code > 0x7E) code = 0x7E;
    return (uint8_t)(sign | (uint8_t)code);
}

/*
 * FP4 E2M1: s.ee.m, bias 1, values {0, 0.5, 1, 1.5, 2, 3, 4, 6} with sign.
 *   e == 0 : value = m * 0.5
 *   e >= 1 : value = 2^(e-1) * (1 + m/2)
 */
double oracle_e2m1_to_double(uint8_t c)
{
    int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    double v = (e == 0) ? m * 0.5 : ldexp(1.0 + m / 2.0, e - 1);
    return s ? -v : v;
}

/* Nearest E2M1 value, ties to even, saturating to +-6, sign kept (see E4M3). */
uint8_t oracle_e2m1_from_float(float v)
{
    uint8_t sign = signbit(v) ? 0x8 : 0x0;
    double a = fabs((double)v);
    if (isnan(v) || isinf(a)) return (uint8_t)(sign | 0x7);
    long code;
    if (a < 1.0) {
        code = (long)nearbyint(a * 2.0);                     /* 0..2; 2 is the smallest normal */
    } else {
        int ex;
        (void)frexp(a, &ex);
        long e = (ex - 1) + 1;
        double q = nearbyint(a / ldexp(1.0, ex - 1 - 1));    /* 2..4 */
        code = e * 2 + (long)q - 2;
    }
    if (code > 7) code = 7;
    return (uint8_t)(sign | (uint8_t)code);
}

/* array forms of the encoders, for comparing many values at once */
void oracle_e4m3_from_float_array(const float *v, int64_t n, uint8_t *out)
{
    for (int64_t j = 0; j < n; j++) out[j] = oracle_e4m3_from_float(v[j]);
}

void oracle_e2m1_from_float_array(const float *v, int64_t n, uint8_t *out)
{
    for (int64_t j = 0; j < n; j++) out[j] = oracle_e2m1_from_float(v[j]);
}

/* ------------------------------------------------------------------------- */
/* step a1-a3: routing metadata                                               */
/* ------------------------------------------------------------------------- */

/*
 * deepep_run_moe_deep_preprocess(topk_ids, num_experts) -> (reorder_topk_ids,
 * src2dst, seg_indptr), as its outputs are used on the diff page's
 * _deepep_permute / combine_a: seg_indptr has num_experts+1 int64 entries (its
 * empty-batch value is all zeros), src2dst has one entry per (token, k) pair
 * (num_tokens = src2dst.numel() / router_topk), reorder_topk_ids.numel() rows
 * are gathered. Reading: a stable counting sort of the flattened pairs
 * i = t*K + k by expert id --
 *   count[e]       = #{i valid : id_i = e}                            (histogram)
 *   seg_indptr[0]  = 0, seg_indptr[e+1] = seg_indptr[e] + count[e]    (exclusive scan)
 *   src2dst[i]     = seg_indptr[id_i] + #{j < i valid : id_j = id_i}  (stable rank)
 *   src2dst[i]     = -1 for an invalid pair
 *   reorder_topk_ids[src2dst[i]] = id_i
 * A pair is valid iff 0 <= id < E. id == -1 is the pages' invalid-slot marker
 * (DeepEPDispatcher.__init__ comment); any other out-of-range id is skipped too
 * and reported with ORACLE_BAD_ID.
 * Low-latency extras: masked_m[e] = min(count[e], M) when M > 0 (count[e] when
 * M == 0), ORACLE_CAPACITY when count[e] > M; partition_counts[p] = number of
 * valid pairs whose expert lies in [p*E/P, (p+1)*E/P).
 * The running cursor below visits pairs in ascending i, so cursor[e] - seg[e]
 * equals #{j < i valid : id_j = e} at the moment pair i is placed.
 */
int oracle_route_meta(const int32_t *topk_ids, int64_t T, int K, int E, int P, int M,
                      int64_t *seg_indptr, int32_t *src2dst, int32_t *reorder_topk_ids,
                      int32_t *masked_m, int32_t *partition_counts)
{
    int status = 0;
    int64_t n_pairs = T * (int64_t)K;
    int64_t *count = (int64_t *)calloc((size_t)E, sizeof(int64_t));
    int64_t *cursor = (int64_t *)calloc((size_t)E, sizeof(int64_t));

    for (int64_t i = 0; i < n_pairs; i++) {
        int32_t e = topk_ids[i];
        if (e >= 0 && e < E) count[e]++;
        else if (e != -1) status |= ORACLE_BAD_ID;
    }

    seg_indptr[0] = 0;
    for (int e = 0; e < E; e++) seg_indptr[e + 1] = seg_indptr[e] + count[e];

    for (int e = 0; e < E; e++) cursor[e] = seg_indptr[e];
    for (int64_t i = 0; i < n_pairs; i++) {
        int32_t e = topk_ids[i];
        if (e >= 0 && e < E) {
            src2dst[i] = (int32_t)cursor[e];
            reorder_topk_ids[cursor[e]] = e;
            cursor[e]++;
        } else {
            src2dst[i] = -1;
        }
    }

    for (int e = 0; e < E; e++) {
        int64_t c = count[e];
        if (M > 0 && c > M) {
            status |= ORACLE_CAPACITY;
            c = M;
        }
        if (masked_m) masked_m[e] = (int32_t)c;
    }
    if (partition_counts && P > 0) {
        int ep = E / P;
        for (int p = 0; p < P; p++)
            partition_counts[p] = (int32_t)(seg_indptr[(p + 1) * ep] - seg_indptr[p * ep]);
    }
    free(count);
    free(cursor);
    return status;
}

/* expected_m = (T * group_size * K + E) // E, group_size = 1 (one source rank):
 * _DeepEPDispatcherImplLowLatency.dispatch_a on the deepep.py page. */
int64_t oracle_expected_m(int64_t T, int K, int E)
{
    return (T * (int64_t)K + E) / E;
}

/* FlashinferDispatcher.__init__ (flashinfer.py page): bytes per token of the
 * dispatch payload -- NVFP4: H/2 e2m1 + H/16 e4m3 scales + K int32 ids + K fp32
 * weights; otherwise 2H bf16 + 4K + 4K. Combine payload: 2H. */
int64_t oracle_dispatch_payload_bytes(int H, int K, int nvfp4)
{
    if (nvfp4) return H / 2 + H / 16 + (int64_t)K * 4 + (int64_t)K * 4;
    return (int64_t)H * 2 + (int64_t)K * 4 + (int64_t)K * 4;
}

/* ------------------------------------------------------------------------- */
/* step a6: FP8 E4M3 per-token-group-128 quantisation                         */
/* ------------------------------------------------------------------------- */

/*
 * sglang_per_token_group_quant_fp8(x, 128) on one token row (deepep.py page,
 * _DeepEPDispatcherImplNormal.dispatch_a). For each group g of 128 consecutive
 * elements:  amax = max_j |x_j|;  a = max(amax, 1e-10);  s = a / 448;
 * q_j = E4M3(x_j / s);  scale[g] = s  (fp32, row-major [H/128]).
 * All arithmetic in binary32, round-to-nearest-even, in this order.
 */
void oracle_quant_fp8_g128_row(const uint16_t *x, int H, uint8_t *q, float *scales)
{
    for (int g = 0; g < H / 128; g++) {
        const uint16_t *xg = x + (size_t)g * 128;
        float amax = 0.0f;
        for (int j = 0; j < 128; j++) {
            float v = fabsf(bf16_to_float(xg[j]));
            if (v > amax) amax = v;
        }
        float a = amax > 1e-10f ? amax : 1e-10f;
        float s = a / 448.0f;
        for (int j = 0; j < 128; j++) q[(size_t)g * 128 + j] = oracle_e4m3_from_float(bf16_to_float(xg[j]) / s);
        scales[g] = s;
    }
}

/* ------------------------------------------------------------------------- */
/* step a7: NVFP4 (E2M1 + E4M3 block-16 scale) quantisation                    */
/* ------------------------------------------------------------------------- */

/*
 * fp4_quantize(x, input_global_scale, is_sf_swizzled_layout=False) on one token
 * row (flashinfer.py page, FlashinferDispatcher.dispatch; also DeepEP's use_nvfp4
 * with x_global_scale). For each block b of 16 consecutive elements, with g the
 * global scale:
 *   amax = max_j |x_j|;  t = (amax / 6) * g;  sf = E4M3(t);  sff = value(sf);
 *   if sff == 0: every code is 0;  else r = g / sff and q_j = E2M1(x_j * r).
 * Packing: byte j of the row holds element 2j in its low nibble and element 2j+1
 * in its high nibble; sf is row-major [H/16] (non-swizzled).
 */
void oracle_quant_nvfp4_b16_row(const uint16_t *x, int H, float g, uint8_t *q, uint8_t *sf)
{
    uint8_t code[16];
    for (int b = 0; b < H / 16; b++) {
        const uint16_t *xb = x + (size_t)b * 16;
        float amax = 0.0f;
        for (int j = 0; j < 16; j++) {
            float v = fabsf(bf16_to_float(xb[j]));
            if (v > amax) amax = v;
        }
        float t = (amax / 6.0f) * g;
        uint8_t s = oracle_e4m3_from_float(t);
        float sff = (float)oracle_e4m3_to_double(s);
        if (sff == 0.0f) {
            memset(code, 0, sizeof code);
        } else {
            float r = g / sff;
            for (int j = 0; j < 16; j++) code[j] = oracle_e2m1_from_float(bf16_to_float(xb[j]) * r);
        }
        for (int j = 0; j < 8; j++) q[(size_t)b * 8 + j] = (uint8_t)(code[2 * j] | (code[2 * j + 1] << 4));
        sf[b] = s;
    }
}

/* ------------------------------------------------------------------------- */
/* steps a4/a5: gather into the expert-contiguous or the masked layout         */
/* ------------------------------------------------------------------------- */

/* destination row of pair i, or -1 when the pair carries no row */
static int64_t dest_row(int mode, int64_t i, const int32_t *topk_ids, int E, int M,
                        const int32_t *src2dst, const int64_t *seg_indptr)
{
    int32_t d = src2dst[i];
    if (d < 0) return -1;
    if (mode == 0) return d;                       /* normal: row src2dst[i] of [N, .] */
    int32_t e = topk_ids[i];                       /* masked: row e*M + rank of [E, M, .] */
    int64_t rank = (int64_t)d - seg_indptr[e];
    if (rank >= M) return -1;
    return (int64_t)e * M + rank;
}

/*
 * Normal mode (mode 0): out[src2dst[i], :] = Q(x[t, :]) for every valid pair
 * i = t*K + k -- the PreReorder gather of _deepep_permute (diff page), with the
 * quantisation of dispatch_a fused in. Masked mode (mode 1): the low-latency layout
 * [E, M, .] of low_latency_dispatch (deepep.py page); pair i lands in slot
 * rank = src2dst[i] - seg_indptr[e] of expert e (the same stable order as normal
 * mode), slots >= M are dropped. quant: 0 none (bf16 rows), 1 FP8 g128
 * (q rows of H bytes + fp32 scales [.., H/128]), 2 NVFP4 b16 (q rows of H/2 bytes +
 * e4m3 scales [.., H/16]), 4 rows that already hold one-byte codes (per-tensor FP8: the
 * diff page's _deepep_permute allocates gateup_input with fp8_dtype when use_fp8_w8a8 and
 * not use_block_quant) copied as H bytes; x is then read as [T, H] bytes. Each destination
 * quantises its token afresh.
 */
void oracle_dispatch(int mode, int quant, const uint16_t *x, int64_t T, int H,
                     const int32_t *topk_ids, int K, int E, int M,
                     const int32_t *src2dst, const int64_t *seg_indptr, float global_scale,
                     void *out_q, void *out_scales)
{
    for (int64_t t = 0; t < T; t++) {
        const uint16_t *row = x + (size_t)t * H;
        for (int k = 0; k < K; k++) {
            int64_t r = dest_row(mode, t * K + k, topk_ids, E, M, src2dst, seg_indptr);
            if (r < 0) continue;
            if (quant == 4) {
                memcpy((uint8_t *)out_q + (size_t)r * H, (const uint8_t *)x + (size_t)t * H, (size_t)H);
            } else if (quant == 0) {
                memcpy((uint16_t *)out_q + (size_t)r * H, row, (size_t)H * 2);
            } else if (quant == 1) {
                oracle_quant_fp8_g128_row(row, H, (uint8_t *)out_q + (size_t)r * H,
                                          (float *)out_scales + (size_t)r * (H / 128));
            } else {
                oracle_quant_nvfp4_b16_row(row, H, global_scale,
                                           (uint8_t *)out_q + (size_t)r * (H / 2),
                                           (uint8_t *)out_scales + (size_t)r * (H / 16));
            }
        }
    }
}

/* ------------------------------------------------------------------------- */
/* step a8: weighted combine                                                   */
/* ------------------------------------------------------------------------- */

/*
 * deepep_post_reorder (diff page, combine_a) / low_latency_combine (deepep.py
 * page, _combine_core): output[t, h] = sum over valid k of
 * topk_weights[t, k] * expert_out[row(t, k), h], where row is src2dst (normal) or
 * e*M + rank (masked). Sum in binary64 over k ascending, then one rounding to
 * bf16 (nearest, ties to even). A token with no valid pair gives zeros.
 */
void oracle_combine(int mode, const uint16_t *expert_out, int64_t T, int H, int K, int E, int M,
                    const int32_t *topk_ids, const int32_t *src2dst, const int64_t *seg_indptr,
                    const float *topk_weights, uint16_t *out)
{
    double *acc = (double *)malloc(sizeof(double) * (size_t)(H > 0 ? H : 1));
    for (int64_t t = 0; t < T; t++) {
        for (int h = 0; h < H; h++) acc[h] = 0.0;
        for (int k = 0; k < K; k++) {
            int64_t i = t * K + k;
            int64_t r = dest_row(mode, i, topk_ids, E, M, src2dst, seg_indptr);
            if (r < 0) continue;
            double w = (double)topk_weights[i];
            const uint16_t *src = expert_out + (size_t)r * H;
            for (int h = 0; h < H; h++) acc[h] = acc[h] + w * (double)bf16_to_float(src[h]);
        }
        for (int h = 0; h < H; h++) out[(size_t)t * H + h] = oracle_bf16_from_double(acc[h]);
    }
    free(acc);
}

/* ------------------------------------------------------------------------- */
/* dispatch layout per expert-parallel partition (get_dispatch_layout)          */
/* ------------------------------------------------------------------------- */

/*
 * buffer.get_dispatch_layout(topk_ids, num_experts) in
 * _DeepEPDispatcherImplNormal._dispatch_core ("sglang token_dispatcher/deepep.py" page)
 * returns num_tokens_per_rank, num_tokens_per_expert and is_token_in_rank (the RDMA-rank
 * counts belong to the inter-node transport, which has no counterpart here). With P
 * partitions of E/P experts each:
 *   is_token_in_rank[t][p]  = 1 iff some valid pair of token t names an expert of p
 *   num_tokens_per_rank[p]  = #{t : is_token_in_rank[t][p]}
 *   num_tokens_per_expert[e] = #{valid pairs with id e}
 */
void oracle_dispatch_layout(const int32_t *topk_ids, int64_t T, int K, int E, int P,
                            int32_t *num_tokens_per_rank, uint8_t *is_token_in_rank,
                            int32_t *num_tokens_per_expert)
{
    int ep = E / P;
    for (int p = 0; p < P; p++) num_tokens_per_rank[p] = 0;
    if (num_tokens_per_expert)
        for (int e = 0; e < E; e++) num_tokens_per_expert[e] = 0;
    for (int64_t t = 0; t < T; t++) {
        for (int p = 0; p < P; p++) is_token_in_rank[t * P + p] = 0;
        for (int k = 0; k < K; k++) {
            int32_t e = topk_ids[t * K + k];
            if (e < 0 || e >= E) continue;
            is_token_in_rank[t * P + e / ep] = 1;
            if (num_tokens_per_expert) num_tokens_per_expert[e]++;
        }
        for (int p = 0; p < P; p++) num_tokens_per_rank[p] += is_token_in_rank[t * P + p];
    }
}

/* ------------------------------------------------------------------------- */
/* FlashInfer all-to-all layout, one source rank (f1)                           */
/* ------------------------------------------------------------------------- */

/*
 * FlashinferDispatcher.dispatch ("sglang token_dispatcher/flashinfer.py" page): the payload
 * list [x (or its NVFP4 codes), x_sf, topk_ids, topk_weights] is sent once to every EP rank
 * that owns at least one of the token's experts, into receive buffers shaped
 * [ep_size, runtime_max_tokens_per_rank, ...]; the receiver's topk_ids are sanitised so that
 * experts it does not own, and padding slots, carry invalid_token_expert_id. With one
 * source rank and P partitions, partition p's receive rows are recv[p][slot] for
 * slot < num_slots (num_slots = runtime_max_tokens_per_rank >= T). Reading: token t uses
 * slot t.
 *   token t routed to p: recv_x[p][t] = Q(x[t]) (quant 0 bf16 copy, 2 NVFP4 codes + sf),
 *                        recv_ids[p][t][k] = id if id is an expert of p else invalid_id,
 *                        recv_w[p][t][k] = topk_weights[t][k]
 *   token not routed to p, and slots t >= T: recv_ids[p][t][k] = invalid_id for all k
 *                        (the payload and weights of those slots are left untouched).
 */
void oracle_dispatch_partitioned(int quant, const uint16_t *x, int64_t T, int64_t num_slots, int H,
                                 const int32_t *topk_ids, const float *topk_weights, int K, int E, int P,
                                 int32_t invalid_id, float global_scale, void *recv_x, uint8_t *recv_sf,
                                 int32_t *recv_ids, float *recv_w)
{
    int ep = E / P;
    size_t row_bytes = quant == 2 ? (size_t)H / 2 : (size_t)H * 2;
    for (int p = 0; p < P; p++) {
        for (int64_t t = 0; t < num_slots; t++) {
            int32_t *ids_out = recv_ids + ((size_t)p * num_slots + t) * K;
            int routed = 0;
            if (t < T)
                for (int k = 0; k < K; k++) {
                    int32_t e = topk_ids[t * K + k];
                    if (e >= 0 && e < E && e / ep == p) routed = 1;
                }
            if (!routed) {
                for (int k = 0; k < K; k++) ids_out[k] = invalid_id;
                continue;
            }
            for (int k = 0; k < K; k++) {
                int32_t e = topk_ids[t * K + k];
                ids_out[k] = (e >= 0 && e < E && e / ep == p) ? e : invalid_id;
                recv_w[((size_t)p * num_slots + t) * K + k] = topk_weights[t * K + k];
            }
            unsigned char *dst = (unsigned char *)recv_x + ((size_t)p * num_slots + t) * row_bytes;
            if (quant == 2)
                oracle_quant_nvfp4_b16_row(x + (size_t)t * H, H, global_scale, dst,
                                           recv_sf + ((size_t)p * num_slots + t) * (H / 16));
            else
                memcpy(dst, x + (size_t)t * H, row_bytes);
        }
    }
}

/*
 * FlashinferDispatcher.combine (flashinfer.py page): moe_a2a.combine takes each rank's
 * output [ep_size, runtime_max_tokens_per_rank, H] (already weighted by the MoE runner)
 * back to the source tokens and sums over the ranks. One source: out[t] = bf16( sum over
 * the partitions p that received token t, ascending, of partial[p][t] ), binary64
 * accumulation, one rounding. A token routed nowhere gives zeros.
 */
void oracle_combine_partitioned(const uint16_t *partial, int64_t T, int64_t num_slots, int H,
                                const int32_t *topk_ids, int K, int E, int P, uint16_t *out)
{
    int ep = E / P;
    double *acc = (double *)malloc(sizeof(double) * (size_t)(H > 0 ? H : 1));
    for (int64_t t = 0; t < T; t++) {
        for (int h = 0; h < H; h++) acc[h] = 0.0;
        for (int p = 0; p < P; p++) {
            int routed = 0;
            for (int k = 0; k < K; k++) {
                int32_t e = topk_ids[t * K + k];
                if (e >= 0 && e < E && e / ep == p) routed = 1;
            }
            if (!routed) continue;
            const uint16_t *src = partial + ((size_t)p * num_slots + t) * H;
            for (int h = 0; h < H; h++) acc[h] = acc[h] + (double)bf16_to_float(src[h]);
        }
        for (int h = 0; h < H; h++) out[(size_t)t * H + h] = oracle_bf16_from_double(acc[h]);
    }
    free(acc);
}

/* ------------------------------------------------------------------------- */
/* consumer formats for DeepGEMM (f3)                                          */
/* ------------------------------------------------------------------------- */

/*
 * Routing metadata with expert_alignment A (buffer.dispatch(..., expert_alignment=128 if
 * DeepGEMM), _DeepEPDispatcherImplNormal._dispatch_core, "sglang token_dispatcher/deepep.py"
 * page). Reading: every expert's segment of the contiguous layout starts at a multiple of A:
 *   seg_indptr[e+1] = seg_indptr[e] + roundup(count[e], A)
 *   src2dst[i]      = seg_indptr[id_i] + #{j < i valid : id_j = id_i}
 *   reorder_topk_ids[r] = expert of row r, or -1 for the padding rows of a segment
 *                          (seg_indptr[E] entries; capacity T*K + E*(A-1))
 *   masked_m[e] = count[e] (or min(count[e], M)), partition_counts[p] = valid pairs in p.
 * A = 1 gives oracle_route_meta's result.
 */
int oracle_route_meta_aligned(const int32_t *topk_ids, int64_t T, int K, int E, int P, int M, int A,
                              int64_t *seg_indptr, int32_t *src2dst, int32_t *reorder_topk_ids,
                              int32_t *masked_m, int32_t *partition_counts)
{
    int status = 0;
    int64_t n_pairs = T * (int64_t)K;
    int64_t *count = (int64_t *)calloc((size_t)E, sizeof(int64_t));
    int64_t *cursor = (int64_t *)calloc((size_t)E, sizeof(int64_t));
    for (int64_t i = 0; i < n_pairs; i++) {
        int32_t e = topk_ids[i];
        if (e >= 0 && e < E) count[e]++;
        else if (e != -1) status |= ORACLE_BAD_ID;
    }
    seg_indptr[0] = 0;
    for (int e = 0; e < E; e++) seg_indptr[e + 1] = seg_indptr[e] + (count[e] + A - 1) / A * A;
    for (int64_t r = 0; r < seg_indptr[E]; r++) reorder_topk_ids[r] = -1;
    for (int e = 0; e < E; e++) cursor[e] = seg_indptr[e];
    for (int64_t i = 0; i < n_pairs; i++) {
        int32_t e = topk_ids[i];
        if (e >= 0 && e < E) {
            src2dst[i] = (int32_t)cursor[e];
            reorder_topk_ids[cursor[e]] = e;
            cursor[e]++;
        } else {
            src2dst[i] = -1;
        }
    }
    for (int e = 0; e < E; e++) {
        int64_t c = count[e];
        if (M > 0 && c > M) {
            status |= ORACLE_CAPACITY;
            c = M;
        }
        if (masked_m) masked_m[e] = (int32_t)c;
    }
    if (partition_counts && P > 0) {
        int ep = E / P;
        for (int p = 0; p < P; p++) {
            int64_t c = 0;
            for (int e = p * ep; e < (p + 1) * ep; e++) c += count[e];
            partition_counts[p] = (int32_t)c;
        }
    }
    free(count);
    free(cursor);
    return status;
}

/*
 * FP8 group-128 quantisation with power-of-two UE8M0 scales (round_scale / use_ue8m0 of
 * low_latency_dispatch and scale_ue8m0 of sglang_per_token_group_quant_fp8, deepep.py page).
 * Reading: s = max(amax, 1e-10) / 448 as in oracle_quant_fp8_g128_row, rounded UP to a
 * power of two s2 = 2^ceil(log2 s) (so |x / s2| <= 448); q = E4M3(x / s2); the stored
 * scale is the UE8M0 byte log2(s2) + 127. Four consecutive groups' bytes form one
 * little-endian int32 ("int32-packed").
 */
void oracle_quant_fp8_g128_ue8m0_row(const uint16_t *x, int H, uint8_t *q, uint8_t *scale_exp)
{
    for (int g = 0; g < H / 128; g++) {
        const uint16_t *xg = x + (size_t)g * 128;
        float amax = 0.0f;
        for (int j = 0; j < 128; j++) {
            float v = fabsf(bf16_to_float(xg[j]));
            if (v > amax) amax = v;
        }
        float a = amax > 1e-10f ? amax : 1e-10f;
        float s = a / 448.0f;
        int ex;
        double m = frexp((double)s, &ex);            /* s = m * 2^ex, m in [0.5, 1) */
        int k = (m == 0.5) ? ex - 1 : ex;             /* smallest k with 2^k >= s */
        float s2 = (float)ldexp(1.0, k);
        for (int j = 0; j < 128; j++) q[(size_t)g * 128 + j] = oracle_e4m3_from_float(bf16_to_float(xg[j]) / s2);
        scale_exp[g] = (uint8_t)(k + 127);
    }
}

/*
 * nvfp4_block_scale_interleave(x_sf) (flashinfer.py page, FlashinferDispatcher.dispatch, applied
 * to the received block scales, flattened to [rows, cols], before the CUTLASS MoE).
 * Reading (the page names the call only): the scale-factor layout of the block-scaled tensor-core
 * MMA as publicly documented for NVFP4 -- the [rows, cols] byte matrix is padded with zeros to
 * rows a multiple of 128 and cols a multiple of 4, cut into 128 x 4 tiles stored one after the
 * other in row-tile-major order (512 bytes each), and inside a tile the scale of tile row i
 * (0..127) and tile column c (0..3) sits at byte (i % 32) * 16 + (i / 32) * 4 + c: each
 * 16-byte line holds rows j, j+32, j+64, j+96 for the tile's 4 columns.
 * out: ((rows + 127) / 128 * 128) * ((cols + 3) / 4 * 4) bytes.
 */
void oracle_nvfp4_sf_interleave(const uint8_t *sf, int64_t rows, int cols, uint8_t *out)
{
    const int64_t row_tiles = (rows + 127) / 128;
    const int64_t col_tiles = (cols + 3) / 4;
    memset(out, 0, (size_t)(row_tiles * 128 * col_tiles * 4));
    for (int64_t r = 0; r < rows; r++) {
        for (int c = 0; c < cols; c++) {
            int64_t tile = (r / 128) * col_tiles + c / 4;
            int64_t i = r % 128;
            int64_t at = tile * 512 + (i % 32) * 16 + (i / 32) * 4 + c % 4;
            out[at] = sf[r * cols + c];
        }
    }
}

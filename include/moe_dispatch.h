/*
 * moe_dispatch.h -- C ABI of the GB300 (sm_103a) MoE token dispatch / combine library.
 *
 * Three stream-ordered calls cover the hot path of the SGLang dispatcher pages:
 *
 *   moe_route_meta  top-k routing -> per-expert metadata (histogram, exclusive scan,
 *                   stable per-pair rank): seg_indptr, src2dst, reorder_topk_ids,
 *                   masked_m. This is deepep_run_moe_deep_preprocess as consumed by
 *                   _DeepEPDispatcherImplNormal._deepep_permute ("sglang 0.4.4.post2 ->
 *                   0.4.4.post4, ep_moe/token_dispatcher.py" diff), plus the
 *                   low-latency counts of _DeepEPDispatcherImplLowLatency.dispatch_a
 *                   ("sglang token_dispatcher/deepep.py" page).
 *   moe_dispatch    gathers token rows into the expert-contiguous layout [N, .]
 *                   (the PreReorder permute) or into the low-latency masked layout
 *                   [E, M, .] (low_latency_dispatch), optionally fused with FP8 e4m3
 *                   per-token-group-128 quantisation (sglang_per_token_group_quant_fp8,
 *                   deepep.py page, _DeepEPDispatcherImplNormal.dispatch_a) or NVFP4
 *                   block-16 quantisation (fp4_quantize, "sglang
 *                   token_dispatcher/flashinfer.py" page, FlashinferDispatcher.dispatch).
 *   moe_combine     topk_weights-weighted, fp32-accumulated reduction of expert outputs
 *                   back to token order (deepep_post_reorder on the diff page,
 *                   low_latency_combine on the deepep.py page).
 *
 * Conventions (all calls):
 *  - Every pointer argument is a DEVICE pointer unless its name ends in _host.
 *    The caller allocates and owns every buffer, including the workspace; the
 *    library keeps no pointer after a call returns.
 *  - Calls are asynchronous on `stream` (NULL = the legacy default stream) and
 *    never synchronise the host.
 *  - Argument errors are detected on the host before anything is launched and
 *    returned as a moe_status_t; nothing is written in that case.
 *  - Data-dependent errors are written by the kernels into the caller's device word
 *    *dev_status, first error wins (atomic compare-and-swap from MOE_OK). The caller
 *    sets *dev_status = 0 before use and reads it whenever it chooses; the kernels
 *    never trap, never assert and never spin without a bound.
 *  - bf16 tensors are passed as their 16-bit patterns (uint16_t), row-major.
 *  - Notation: T tokens, H hidden size, K top-k slots per token, E experts,
 *    M = num_max_dispatch_tokens_per_rank (slots per expert in the masked layout),
 *    pair i = t*K + k, a pair is valid iff 0 <= topk_ids[i] < E, N = #valid pairs.
 */
#ifndef MOE_DISPATCH_H
#define MOE_DISPATCH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; NULL selects the legacy default stream. */
typedef struct CUstream_st *moe_stream_t;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,    /* host-side: bad size, null or misaligned pointer     */
    MOE_ERR_UNSUPPORTED = 2,    /* host-side: a size beyond the limits below           */
    MOE_ERR_CAPACITY = 3,       /* device: an expert received more than M pairs        */
    MOE_ERR_BAD_EXPERT_ID = 4,  /* device: an id outside [-1, E) was seen (skipped)    */
    MOE_ERR_TIMEOUT = 5,        /* device: a bounded wait gave up                      */
    MOE_ERR_CUDA = 6            /* host-side: a CUDA launch or runtime call failed     */
} moe_status_t;

typedef enum { MOE_MODE_NORMAL = 0, MOE_MODE_MASKED = 1 } moe_mode_t;

typedef enum {
    MOE_QUANT_NONE = 0,        /* bf16 rows                                                  */
    MOE_QUANT_FP8_G128 = 1,    /* e4m3 rows [.., H] + fp32 scales [.., H/128]                */
    MOE_QUANT_NVFP4_B16 = 2,   /* e2m1 rows [.., H/2] (2 per byte) + e4m3 scales [.., H/16]  */
    MOE_QUANT_FP8_G128_UE8M0 = 3, /* e4m3 rows [.., H] + power-of-two scales as UE8M0 bytes
                                    [.., H/128] (four groups = one little-endian int32)      */
    MOE_QUANT_FP8_PASSTHROUGH = 4 /* hidden_states already hold one-byte codes ([T, H] bytes,
                                    per-tensor FP8): rows of H bytes are copied, no scales   */
} moe_quant_t;

/* Layout of the scale arrays (moe_dispatch_ex, moe_dispatch_partitioned_ex). */
typedef enum {
    MOE_SCALES_ROW_MAJOR = 0,  /* [rows, G]: group g of row r at r*G + g                      */
    MOE_SCALES_COL_MAJOR = 1,  /* FP8 only. MN-major, TMA-aligned: group g of row r at g*R4 + r
                                  with R4 = rows rounded up to a multiple of 4 (per expert
                                  [E, G, R4] in the masked layout, R4 from M); UE8M0 bytes:
                                  int32 word (r, g/4) at (g/4)*R4 + r, byte g%4 of the word   */
    MOE_SCALES_SWIZZLED_128X4 = 2 /* NVFP4 only, H % 64 == 0. The e4m3 block scales of all R
                                  destination rows as one [R, C] matrix (C = H/16) in the 128 x 4
                                  tile layout of the block-scaled MMA, as nvfp4_block_scale_interleave
                                  produces it for the CUTLASS MoE (flashinfer.py page,
                                  FlashinferDispatcher.dispatch): scale (r, c) at byte
                                  ((r/128)*(C/4) + c/4)*512 + (r%32)*16 + ((r%128)/32)*4 + c%4.
                                  R = out_rows (normal), E*M (masked) or P*num_slots (partitioned);
                                  the buffer holds roundup(R, 128)*C bytes, 4-byte aligned
                                  (16-byte aligned: the fast path, whole tiles written at once).
                                  Every 128-row tile the call touches is written in full: its
                                  destination rows hold their scales, all its other rows (and the
                                  padding rows R..roundup(R, 128)-1) zeros. Touched tiles: every
                                  tile (normal); those overlapping rows e*M + [0, min(M,
                                  seg_indptr[e+1] - seg_indptr[e])) of some expert e (masked);
                                  those overlapping slots p*num_slots + [0, T) of some partition p
                                  (partitioned); and the tile holding the padding rows. Other
                                  tiles keep their previous bytes. Masked layout: seg_indptr must
                                  come without expert alignment (moe_route_meta, or
                                  expert_alignment 1); with aligned segments the rows between an
                                  expert's pair count and its segment length are unspecified.  */
} moe_scale_layout_t;

#define MOE_MAX_EXPERTS 1024   /* E <= 1024                                  */
#define MOE_MAX_TOPK 16        /* 1 <= K <= 16                               */
#define MOE_ABI_VERSION 1

/* Version of this ABI (MOE_ABI_VERSION of the built library). */
int moe_abi_version(void);

/* Human-readable name of a status code; never NULL. */
const char *moe_status_string(moe_status_t status);

/*
 * Bytes of scratch that moe_route_meta needs for num_tokens x topk pairs and
 * num_experts experts (0 when one thread block handles all pairs, i.e. up to 2048 pairs).
 * The scratch holds one int32 histogram row per thread block of the count kernel
 * ([B][E], B = the block count); each call writes every row before it reads any, so
 * its initial contents do not matter (no clearing, neither at allocation nor per call).
 * Calls that share a workspace must not overlap on the GPU.
 * Returns 0 for arguments moe_route_meta would reject.
 */
size_t moe_route_meta_workspace_size(int64_t num_tokens, int topk, int num_experts);

/*
 * moe_route_meta -- routing metadata: histogram, exclusive scan, stable rank.
 *
 * Operation (deepep_run_moe_deep_preprocess as used by _deepep_permute on the diff
 * page; masked_m / expected_m as in _DeepEPDispatcherImplLowLatency.dispatch_a on the
 * deepep.py page; invalid slots marked -1 as noted in DeepEPDispatcher.__init__):
 *   count[e]       = #{i valid : topk_ids[i] = e}
 *   seg_indptr[0]  = 0,  seg_indptr[e+1] = seg_indptr[e] + count[e]
 *   src2dst[i]     = seg_indptr[id_i] + #{j < i valid : id_j = id_i}, or -1 if invalid
 *   reorder_topk_ids[src2dst[i]] = id_i            (first N entries, non-decreasing)
 *   masked_m[e]    = count[e] if M == 0, else min(count[e], M)
 *   partition_counts[p] = seg_indptr[(p+1)*E/P] - seg_indptr[p*E/P]
 *   *expected_m_host = (T*K + E) / E                (host value, computed without a sync)
 *
 * Arguments:
 *   topk_ids            [T, K] int32, row-major. -1 = empty slot (skipped silently);
 *                       any other id outside [0, E) is skipped and reported as
 *                       MOE_ERR_BAD_EXPERT_ID in *dev_status.
 *   num_tokens (T)      >= 0; T*K <= INT32_MAX. T = 0 is legal (outputs zeroed).
 *   topk (K)            1..MOE_MAX_TOPK.
 *   num_experts (E)     1..MOE_MAX_EXPERTS.
 *   num_partitions (P)  >= 1, E % P == 0 (logical expert-parallel ranks of E/P experts).
 *   max_tokens_per_expert (M)  >= 0. M > 0 enables the capacity check: an expert with
 *                       more than M pairs sets MOE_ERR_CAPACITY; its extra pairs keep
 *                       their src2dst but land in no masked slot.
 *   seg_indptr          [E+1] int64 out.
 *   src2dst             [T*K] int32 out.
 *   reorder_topk_ids    [T*K] int32 out (capacity; the first N entries are written).
 *   masked_m            [E] int32 out.
 *   partition_counts    [P] int32 out, or NULL.
 *   expected_m_host     host int32 out, or NULL.
 *   workspace           moe_route_meta_workspace_size(T, K, E) bytes, 256-byte aligned
 *                       (as cudaMalloc returns), any contents; may be NULL when that size is 0.
 *   dev_status          [1] int32 device status word (see conventions).
 * Returns MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED or MOE_ERR_CUDA.
 */
moe_status_t moe_route_meta(const int32_t *topk_ids, int64_t num_tokens, int topk,
                            int num_experts, int num_partitions, int max_tokens_per_expert,
                            int64_t *seg_indptr, int32_t *src2dst, int32_t *reorder_topk_ids,
                            int32_t *masked_m, int32_t *partition_counts,
                            int32_t *expected_m_host, void *workspace, size_t workspace_bytes,
                            int32_t *dev_status, moe_stream_t stream);

/*
 * moe_route_meta_ex -- moe_route_meta with expert-aligned segments.
 *
 * buffer.dispatch(..., expert_alignment=128 if DeepGEMM else 1) in
 * _DeepEPDispatcherImplNormal._dispatch_core ("sglang token_dispatcher/deepep.py" page):
 * every expert's segment of the contiguous layout starts at a multiple of
 * expert_alignment A (1..1024):
 *   seg_indptr[e+1]     = seg_indptr[e] + roundup(count[e], A)
 *   src2dst[i]          = seg_indptr[id_i] + #{j < i valid : id_j = id_i}
 *   reorder_topk_ids[r] = the expert of row r, -1 on the padding rows of each segment
 *                         (seg_indptr[E] entries; capacity T*K + E*(A-1))
 *   masked_m[e] and partition_counts[p] count valid pairs (no padding).
 * A = 1 is moe_route_meta. Padding rows of a dispatched buffer are never written.
 *
 * topk_ids may be int32 (topk_ids_bytes = 4) or int64 (8; the pages convert topk_ids with
 * .to(torch.int64) before dispatch). An int64 id outside [-1, E) is skipped and reported
 * like any bad id. topk_ids_i32_out ([T*K] int32, or NULL) receives the ids as int32 for the
 * calls that read int32 ids (ids outside the int32 range become INT32_MIN / INT32_MAX,
 * which those calls skip and report).
 * Other arguments, workspace and errors as moe_route_meta; T*K + E*(A-1) <= INT32_MAX.
 */
moe_status_t moe_route_meta_ex(const void *topk_ids, int topk_ids_bytes, int64_t num_tokens, int topk,
                               int num_experts, int num_partitions, int max_tokens_per_expert,
                               int expert_alignment, int64_t *seg_indptr, int32_t *src2dst,
                               int32_t *reorder_topk_ids, int32_t *masked_m, int32_t *partition_counts,
                               int32_t *topk_ids_i32_out, int32_t *expected_m_host, void *workspace,
                               size_t workspace_bytes, int32_t *dev_status, moe_stream_t stream);

/*
 * moe_route_meta_noalloc -- moe_route_meta without a caller-provided workspace.
 *
 * The pages have no counterpart: this is an addition for callers that cannot allocate
 * device memory at the point they need the metadata -- for example an engine that has
 * already reserved the GPU's memory for its own pool, a plugin interface that hands over
 * only input and output pointers, or a path where cudaMalloc's implicit synchronisation
 * is not acceptable. It computes exactly what moe_route_meta computes, with the same
 * arguments minus workspace / workspace_bytes, and allocates nothing.
 *
 * Scratch: a fixed 1 MiB array in the library's own device memory (every GPU that loads
 * the library holds it until the process exits). Sizes whose moe_route_meta workspace
 * would exceed 1 MiB are rejected with MOE_ERR_UNSUPPORTED before anything is launched:
 * with 1024 experts it covers up to 4,194,304 (token, k) pairs, with 256 experts up to
 * 16,777,216, with 128 experts up to 33,554,432. Up to 2048 pairs need no scratch at all.
 * First call on a device: looks up the array's device address with that device current;
 * make that first call before any stream capture. A call issues exactly the kernels of
 * moe_route_meta and nothing else (no memset, no copy).
 * Every call shares the one array, which keeps the previous call's contents (no call
 * depends on them: each writes every cell it reads). Calls whose kernels may overlap on
 * the GPU (different streams, no ordering between them) race and must not be issued.
 * Returns the statuses of moe_route_meta.
 */
moe_status_t moe_route_meta_noalloc(const int32_t *topk_ids, int64_t num_tokens, int topk,
                                    int num_experts, int num_partitions, int max_tokens_per_expert,
                                    int64_t *seg_indptr, int32_t *src2dst, int32_t *reorder_topk_ids,
                                    int32_t *masked_m, int32_t *partition_counts,
                                    int32_t *expected_m_host, int32_t *dev_status,
                                    moe_stream_t stream);

/*
 * moe_dispatch -- gather (and optionally quantise) token rows into expert order.
 *
 * Operation (the PreReorder permute of _deepep_permute on the diff page; the masked
 * layout of low_latency_dispatch on the deepep.py page):
 *   normal: row r = src2dst[i]                            of out [T*K (capacity N), .]
 *   masked: row r = e*M + (src2dst[i] - seg_indptr[e])    of out [E, M, .], e = topk_ids[i];
 *           pairs with rank >= M are dropped (moe_route_meta reported them).
 *   out[r] = Q(hidden_states[t]) for every valid pair i = t*K + k. Rows no pair maps
 *   to (rows >= N, masked slots >= masked_m[e]) are left untouched.
 *   Q = identity (MOE_QUANT_NONE), or per group of 128 consecutive elements
 *   (MOE_QUANT_FP8_G128):  amax = max|x|, s = max(amax, 1e-10) / 448,
 *       q = e4m3_rn_satfinite(x / s), scale = s (fp32);
 *   or per block of 16 consecutive elements with g = input_global_scale
 *   (MOE_QUANT_NVFP4_B16):  sf = e4m3_rn_satfinite((amax / 6) * g),
 *       q = e2m1_rn_satfinite(x * (g / sf)), all codes 0 when sf decodes to 0;
 *       two codes per byte, the even element in the low nibble; sf row-major [H/16].
 *   MOE_QUANT_FP8_G128_UE8M0 is FP8_G128 with s rounded up to a power of two 2^k
 *   (round_scale / use_ue8m0 on the deepep.py page): q = e4m3_rn_satfinite(x / 2^k),
 *   scale byte = k + 127, [rows, H/128] bytes (= [rows, H/512] little-endian int32).
 *   MOE_QUANT_FP8_PASSTHROUGH: hidden_states are [T, H] one-byte codes (per-tensor FP8,
 *   the diff page's gateup_input of fp8_dtype) and each destination row is a copy of H bytes.
 *   All arithmetic is binary32 with round-to-nearest-even, in the order written.
 *
 * Arguments:
 *   hidden_states  [T, H] bf16 ([T, H] bytes for MOE_QUANT_FP8_PASSTHROUGH), 16-byte aligned.
 *   hidden (H)     > 0, H % 16 == 0; H % 128 == 0 for the FP8 modes; H % 32 == 0 for
 *                  MOE_QUANT_FP8_PASSTHROUGH.
 *   topk_ids       [T, K] int32 (read in masked mode; may be NULL in normal mode).
 *   max_tokens_per_expert (M)  >= 1 in masked mode; ignored in normal mode.
 *   src2dst        [T*K] int32 and seg_indptr [E+1] int64 from moe_route_meta
 *                  (seg_indptr is read in masked mode only; may be NULL otherwise).
 *   out_q          rows as above, 16-byte aligned. bf16 rows hold H uint16, FP8 rows
 *                  H bytes, NVFP4 rows H/2 bytes.
 *   out_scales     FP8: fp32 [rows, H/128] (4-byte aligned); NVFP4: uint8 [rows, H/16];
 *                  NULL for MOE_QUANT_NONE.
 * Returns MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED or MOE_ERR_CUDA.
 */
moe_status_t moe_dispatch(moe_mode_t mode, moe_quant_t quant, const uint16_t *hidden_states,
                          int64_t num_tokens, int hidden, const int32_t *topk_ids, int topk,
                          int num_experts, int max_tokens_per_expert, const int32_t *src2dst,
                          const int64_t *seg_indptr, float input_global_scale, void *out_q,
                          void *out_scales, int32_t *dev_status, moe_stream_t stream);

/*
 * moe_dispatch_ex -- moe_dispatch with a scale layout and an explicit row capacity.
 *
 * For the DeepGEMM consumers of the deepep.py page (sglang_per_token_group_quant_fp8 with
 * column_major_scales / scale_tma_aligned / scale_ue8m0 in
 * _DeepEPDispatcherImplNormal.dispatch_a; round_scale / use_ue8m0 in
 * _DeepEPDispatcherImplLowLatency._dispatch_core):
 *   scale_layout  MOE_SCALES_ROW_MAJOR (as moe_dispatch) or MOE_SCALES_COL_MAJOR (FP8 modes
 *                 only): group g of row r at g*R4 + r, R4 = roundup(out_rows, 4) in the
 *                 normal layout; per expert [E, G, R4] with R4 = roundup(M, 4) in the masked
 *                 layout. UE8M0 bytes are grouped four per int32 word, the words laid out
 *                 the same way ([G/4 rounded up, R4] words per expert / buffer).
 *                 MOE_SCALES_SWIZZLED_128X4 (NVFP4 only): see moe_scale_layout_t, with the
 *                 destination rows (row-capacity out_rows, or E*M in the masked layout) as R.
 *   out_rows      normal layout: the row capacity of out_q (>= T*K; T*K + E*(A-1) for
 *                 metadata from moe_route_meta_ex); 0 means T*K. Ignored in masked mode.
 * Everything else as moe_dispatch.
 */
moe_status_t moe_dispatch_ex(moe_mode_t mode, moe_quant_t quant, moe_scale_layout_t scale_layout,
                             const uint16_t *hidden_states, int64_t num_tokens, int hidden,
                             const int32_t *topk_ids, int topk, int num_experts, int max_tokens_per_expert,
                             int64_t out_rows, const int32_t *src2dst, const int64_t *seg_indptr,
                             float input_global_scale, void *out_q, void *out_scales, int32_t *dev_status,
                             moe_stream_t stream);

/*
 * moe_route_dispatch -- moe_route_meta followed by moe_dispatch, in one call.
 *
 * Same results as the two calls (all their outputs are written), for the dispatch
 * sequence of _DeepEPDispatcherImplNormal._deepep_permute (diff page: preprocess, then
 * PreReorder) and of low_latency_dispatch (deepep.py page: counts and the masked layout in
 * one step). Arguments are the union of the two calls' arguments, with the same meaning
 * and limits; max_tokens_per_expert is the masked capacity (>= 1 in masked mode; >= 0 in
 * normal mode, where M > 0 only enables the capacity check of masked_m).
 * Small batches (T <= 512 and T*K <= 4096 pairs) run as a single kernel that needs no
 * workspace (workspace may be NULL); larger ones need moe_route_meta_workspace_size(T, K, E)
 * bytes of workspace, exactly as moe_route_meta.
 * Returns MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED or MOE_ERR_CUDA.
 */
moe_status_t moe_route_dispatch(moe_mode_t mode, moe_quant_t quant, const uint16_t *hidden_states,
                                int64_t num_tokens, int hidden, const int32_t *topk_ids, int topk,
                                int num_experts, int num_partitions, int max_tokens_per_expert,
                                float input_global_scale, int64_t *seg_indptr, int32_t *src2dst,
                                int32_t *reorder_topk_ids, int32_t *masked_m,
                                int32_t *partition_counts, int32_t *expected_m_host, void *workspace,
                                size_t workspace_bytes, void *out_q, void *out_scales,
                                int32_t *dev_status, moe_stream_t stream);

/*
 * moe_combine -- weighted reduction of expert outputs back to token order.
 *
 * Operation (deepep_post_reorder in combine_a on the diff page; low_latency_combine in
 * _DeepEPDispatcherImplLowLatency._combine_core on the deepep.py page):
 *   out[t, :] = bf16_rn( sum_{k valid, k ascending} topk_weights[t, k] * expert_out[row(t,k), :] )
 *   with row as in moe_dispatch; fp32 fused multiply-add accumulation. A token with
 *   no valid slot gets zeros.
 *
 * Arguments:
 *   expert_out     bf16 [N (capacity T*K), H] (normal) or [E, M, H] (masked), 16-byte aligned.
 *   topk_ids       [T, K] int32 (read in masked mode; may be NULL in normal mode).
 *   src2dst, seg_indptr  from moe_route_meta (seg_indptr read in masked mode only).
 *   topk_weights   [T, K] fp32.
 *   out            [T, H] bf16 out, 16-byte aligned, must not overlap expert_out.
 *   hidden (H)     > 0, H % 16 == 0.
 * Returns MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED or MOE_ERR_CUDA.
 */
moe_status_t moe_combine(moe_mode_t mode, const uint16_t *expert_out, int64_t num_tokens,
                         int hidden, int topk, int num_experts, int max_tokens_per_expert,
                         const int32_t *topk_ids, const int32_t *src2dst,
                         const int64_t *seg_indptr, const float *topk_weights, uint16_t *out,
                         int32_t *dev_status, moe_stream_t stream);

/*
 * moe_dispatch_layout -- which expert-parallel partitions each token is sent to.
 *
 * buffer.get_dispatch_layout(topk_ids, num_experts) in _DeepEPDispatcherImplNormal._dispatch_core
 * ("sglang token_dispatcher/deepep.py" page), with the E experts split into P partitions
 * of E/P consecutive experts (the RDMA-rank counts of the inter-node transport have no
 * counterpart on one GPU):
 *   is_token_in_rank[t][p]   = 1 iff some valid slot of token t names an expert of p
 *   num_tokens_per_rank[p]   = #{t : is_token_in_rank[t][p]}
 *   num_tokens_per_expert[e] = #{valid (t, k) with topk_ids[t][k] = e}
 * Arguments: topk_ids [T, K] int32; num_partitions (P) >= 1 with E % P == 0;
 * num_tokens_per_rank [P] int32 out; is_token_in_rank [T, P] uint8 out (0/1);
 * num_tokens_per_expert [E] int32 out or NULL. Ids outside [-1, E) are skipped and reported
 * as MOE_ERR_BAD_EXPERT_ID in *dev_status. Every output is written in full (the caller need not
 * clear them): up to 4096 (token, k) pairs by one block that writes the counts at the end,
 * above that by clearing the counts on `stream` and accumulating them with atomics.
 * Returns MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED or MOE_ERR_CUDA.
 */
moe_status_t moe_dispatch_layout(const int32_t *topk_ids, int64_t num_tokens, int topk, int num_experts,
                                 int num_partitions, int32_t *num_tokens_per_rank,
                                 uint8_t *is_token_in_rank, int32_t *num_tokens_per_expert,
                                 int32_t *dev_status, moe_stream_t stream);

/*
 * moe_dispatch_partitioned -- the FlashInfer all-to-all dispatch layout, one source rank.
 *
 * FlashinferDispatcher.dispatch ("sglang token_dispatcher/flashinfer.py" page): the payload
 * [x or its NVFP4 codes, NVFP4 block scales, topk_ids, topk_weights] of token t goes once to
 * every partition p that owns one of its experts, into slot t of p's receive rows:
 *   recv_x[p][t]             = hidden_states[t] (bf16) or its NVFP4 codes (as moe_dispatch)
 *   recv_scales[p][t]        = the e4m3 block scales [H/16] (NVFP4 only)
 *   recv_topk_ids[p][t][k]   = topk_ids[t][k] if that expert belongs to p, else invalid_expert_id
 *   recv_topk_weights[p][t][k] = topk_weights[t][k]
 * Slots of tokens p does not receive, and padding slots t in [T, num_slots), get
 * invalid_expert_id in every recv_topk_ids entry; their other payload is left untouched.
 * num_slots plays runtime_max_tokens_per_rank (>= T). quant: MOE_QUANT_NONE or
 * MOE_QUANT_NVFP4_B16 (input_global_scale as in moe_dispatch). Limits: P <= 32, H % 16 == 0,
 * hidden_states / recv_x 16-byte aligned. Shapes: recv_x [P, num_slots, H] bf16 or
 * [P, num_slots, H/2] uint8; recv_scales [P, num_slots, H/16]; recv_topk_ids / weights
 * [P, num_slots, K].
 * Returns MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED or MOE_ERR_CUDA.
 */
moe_status_t moe_dispatch_partitioned(moe_quant_t quant, const uint16_t *hidden_states, int64_t num_tokens,
                                      int64_t num_slots, int hidden, const int32_t *topk_ids,
                                      const float *topk_weights, int topk, int num_experts, int num_partitions,
                                      int32_t invalid_expert_id, float input_global_scale, void *recv_x,
                                      uint8_t *recv_scales, int32_t *recv_topk_ids, float *recv_topk_weights,
                                      int32_t *dev_status, moe_stream_t stream);

/*
 * moe_dispatch_partitioned_ex -- moe_dispatch_partitioned with a block-scale layout.
 *
 * scale_layout MOE_SCALES_SWIZZLED_128X4 writes recv_scales already interleaved, as
 * FlashinferDispatcher.dispatch (flashinfer.py page) obtains them by applying
 * nvfp4_block_scale_interleave to the received scales viewed as [P*num_slots, H/16] before the
 * CUTLASS MoE: R = P*num_slots rows, roundup(R, 128)*H/16 bytes. The tiles holding slots
 * t < T of some partition, and the one holding the padding rows, are written in full: slots a
 * partition does not receive are zero there, like the padding rows (moe_scale_layout_t); tiles
 * of padding slots only keep their bytes. NVFP4 only, H % 64 == 0, recv_scales 4-byte aligned.
 * Launches: with num_slots % 128 == 0 and recv_scales 16-byte aligned, one (every tile lies in
 * one partition and is written whole from shared memory); otherwise a clear of the touched
 * tiles, the dispatch, and (recv_scales 16-byte aligned) an in-place interleave of the
 * row-major scale rows the dispatch wrote there.
 * MOE_SCALES_ROW_MAJOR is moe_dispatch_partitioned.
 * Everything else as moe_dispatch_partitioned.
 */
moe_status_t moe_dispatch_partitioned_ex(moe_quant_t quant, moe_scale_layout_t scale_layout,
                                         const uint16_t *hidden_states, int64_t num_tokens, int64_t num_slots,
                                         int hidden, const int32_t *topk_ids, const float *topk_weights, int topk,
                                         int num_experts, int num_partitions, int32_t invalid_expert_id,
                                         float input_global_scale, void *recv_x, uint8_t *recv_scales,
                                         int32_t *recv_topk_ids, float *recv_topk_weights, int32_t *dev_status,
                                         moe_stream_t stream);

/*
 * moe_combine_partitioned -- the FlashInfer all-to-all combine, one source rank.
 *
 * FlashinferDispatcher.combine (flashinfer.py page): each partition's output rows
 * [P, num_slots, H] bf16 (already weighted by its experts) are summed back per token over
 * the partitions the token was sent to, in ascending p, fp32 accumulation, one rounding:
 *   out[t] = bf16_rn( sum_{p : token t sent to p} partial[p][t] ),   zeros if sent nowhere.
 * Arguments as moe_dispatch_partitioned; out [T, H] bf16, 16-byte aligned.
 * Returns MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED or MOE_ERR_CUDA.
 */
moe_status_t moe_combine_partitioned(const uint16_t *partial, int64_t num_tokens, int64_t num_slots, int hidden,
                                     const int32_t *topk_ids, int topk, int num_experts, int num_partitions,
                                     uint16_t *out, int32_t *dev_status, moe_stream_t stream);

/*
 * moe_combine_ex -- moe_combine with the row capacity of expert_out in the normal layout
 * (>= T*K; T*K + E*(A-1) for metadata from moe_route_meta_ex; 0 means T*K), so that rows of
 * expert-aligned segments are accepted. Everything else as moe_combine.
 */
moe_status_t moe_combine_ex(moe_mode_t mode, const uint16_t *expert_out, int64_t num_tokens, int hidden,
                            int topk, int num_experts, int max_tokens_per_expert, int64_t expert_out_rows,
                            const int32_t *topk_ids, const int32_t *src2dst, const int64_t *seg_indptr,
                            const float *topk_weights, uint16_t *out, int32_t *dev_status, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_DISPATCH_H */

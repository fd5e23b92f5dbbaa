/*
 * moe_diag.h -- diagnostics entry points of libmoe_dispatch.so (test hooks, not the hot path).
 *
 * These calls have no counterpart on the SGLang dispatcher pages. They expose pieces of the
 * kernels of moe_dispatch.h -- the FP8 quantiser's division, the e4m3 / e2m1 conversions and
 * the bounded device wait of the bulk (TMA) dispatch -- so that tests can check them against
 * independent definitions without a fault. Conventions (device pointers, stream order,
 * status codes) are those of moe_dispatch.h.
 */
#ifndef MOE_DIAG_H
#define MOE_DIAG_H

#include "moe_dispatch.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * moe_fp8_division_check -- diagnostics: the FP8 quantiser divides by its group scale with
 * the scale's reciprocal and one correction step (after Markstein) instead of a division per
 * element. This call checks that choice exhaustively on the GPU: for every non-negative finite
 * bf16 amax (0 clamped to 1e-10), s = amax/448, and every bf16 x with |x| <= amax, it compares
 * the result with the IEEE division.
 * (No counterpart on the pages: a test hook for sglang_per_token_group_quant_fp8's x / s.)
 *   result  [4] uint64 device out (cleared on `stream` first):
 *           [0] pairs whose e4m3 codes differ, [1] the first one as (x bits << 32) | s bits,
 *           [2] pairs whose quotients differ while |x / s| >= 2^-12,
 *           [3] pairs whose quotients differ at all (expected only for |x| < 2^-103, where the
 *               correction's remainder leaves the normal range and the code is a zero anyway).
 * Returns MOE_OK, MOE_ERR_INVALID_ARG or MOE_ERR_CUDA.
 */
moe_status_t moe_fp8_division_check(unsigned long long *result, moe_stream_t stream);

/*
 * moe_wait_timeout_check -- diagnostics: runs the bounded wait of the bulk (TMA) dispatch
 * kernels on one shared-memory mbarrier of arrival count 1, so that its give-up path can be
 * checked without any fault. With complete = 1 the kernel arrives at the barrier first and
 * the wait returns at once; with complete = 0 nothing ever arrives, the wait gives up after
 * limit_ns of wall-clock time and the kernel writes MOE_ERR_TIMEOUT to dev_status (first
 * error wins) and exits. The dispatch kernels wait the same way with a limit of 1 s per ring
 * stage (0.1 s for draining their loads after a timeout).
 * (No counterpart on the pages: a test hook for the library's own bounded waits.)
 *   dev_status  [1] int32 device status word.
 *   limit_ns    1 .. 10^10.
 *   complete    0 or 1.
 * Returns MOE_OK, MOE_ERR_INVALID_ARG or MOE_ERR_CUDA.
 */
moe_status_t moe_wait_timeout_check(int32_t *dev_status, int64_t limit_ns, int complete, moe_stream_t stream);

/*
 * moe_convert_probe -- diagnostics: run the number-format conversions of the quantising
 * kernels on arbitrary fp32 inputs, so their rounding, saturation, signed zeros and
 * packing order can be checked against an independent implementation of the formats.
 * (No counterpart on the pages: a test hook for the e4m3 / e2m1 codecs used by
 * sglang_per_token_group_quant_fp8 and fp4_quantize.)
 *   in          [n] fp32, n even.
 *   e4m3        [n] uint8 out: e4m3_rn_satfinite(in[j]), converted in pairs
 *               (in[2j], in[2j+1]) exactly as the FP8 kernel packs them; or NULL.
 *   e2m1        [n/2] uint8 out: byte j = e2m1(in[2j]) | e2m1(in[2j+1]) << 4, as the NVFP4
 *               kernel packs them; or NULL.
 *   e4m3_value  [n] fp32 out: the value of the e4m3 code of in[j], decoded as the NVFP4
 *               kernel decodes its block scales; or NULL.
 * Returns MOE_OK, MOE_ERR_INVALID_ARG or MOE_ERR_CUDA.
 */
moe_status_t moe_convert_probe(const float *in, int64_t n, uint8_t *e4m3, uint8_t *e2m1,
                               float *e4m3_value, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_DIAG_H */

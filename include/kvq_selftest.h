/*
 * kvq_selftest.h -- device self-tests of the arithmetic the quantizer
 * kernels rely on, and of the bounded device wait. Part of the same C ABI
 * library as kvq.h (same conventions: a status is returned, nothing aborts;
 * work is asynchronous on `stream`; the library allocates nothing).
 *
 * The quantizer decides each code as rne((x - z) / s) in fp32
 * ([TurboQuant-3bit] "TurboQuant 3-bit KV-cache quantization",
 * dpshk.com/news/6341316, §3.1: offset = group minimum, scale =
 * (max - min) / (2^b - 1)); the kernels reach the IEEE quotient without a
 * division on the common path. These entry points run the kernels' own
 * device functions over exhaustive or adversarial inputs and count where
 * they differ from the IEEE division (__fdiv_rn, then round to nearest even).
 *
 * Result buffer: `dev_result` is caller-owned device memory of two uint64
 * (16 bytes, 8-byte aligned). The call first sets result[0] = 0 and
 * result[1] = UINT64_MAX on `stream`; the kernel adds every mismatch to
 * result[0] and lowers result[1] to the smallest mismatching input key
 * (defined per entry point). Read it after the stream has finished.
 */
#ifndef KVQ_SELFTEST_H
#define KVQ_SELFTEST_H

#include "kvq.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Scale of a group from its range, (max - min) / L with L = 2^b - 1 in
 * {3, 7, 15, 127, 255} (b = 2, 3, 4, 7, 8), as the prefill computes it: a
 * product with RN(1/L) corrected once by a fused multiply-add (Markstein's
 * division correction). Compares it bit for bit with __fdiv_rn(a, L) for
 * every fp32 bit pattern a in [a_first, a_last] (a_first <= a_last; the
 * prefill's ranges are fp16 max - min <= 131008, below 2^17 = bit pattern
 * 0x48000000). Input key: the bit pattern of a.
 * Errors: KVQ_ERR_INVALID_ARG for another L, a_first > a_last or a NULL or
 * misaligned dev_result. */
KVQ_API kvq_status kvq_selftest_div_levels(int32_t levels, uint32_t a_first, uint32_t a_last,
                                           void* dev_result, void* stream);

/* Codes near rounding ties. For every positive finite fp16 scale s (bit
 * patterns 0x0001..0x7BFF; method 1: normal ones only, 0x0400..0x7BFF),
 * every k in [k_first, k_last] and every offset j in [-ulps, ulps], the
 * dividend d is RN32((k + 1/2) * s) moved by j units in the last place
 * (zero and non-finite d are skipped). The code
 * under test is compared with rne(__fdiv_rn(d, s)):
 *  method 0: the append / per-token kernels' quant_step(d, s, RN(1/s))
 *            (product with the rounded reciprocal, exact division only
 *            within 2^-20 of a half-integer);
 *  method 1: the prefill's bracketed reciprocal: rne(d * r_lo) and
 *            rne(d * r_hi) from a bracket of 1/s, and where they differ the
 *            exact-residual settle d - (k + 1/2) s.
 * Input key: (s bits << 32) | ((k - k_first) << 8) | (j + ulps).
 * Ranges: method 0 takes -4096 <= k_first <= k_last <= 4096; method 1 takes
 * 0 <= k_first <= k_last <= 255 (the prefill's codes: d >= 0, at most 8 bits).
 * Errors: KVQ_ERR_INVALID_ARG for another method, a k range outside these,
 * ulps outside [0, 64], or a NULL or misaligned dev_result. */
KVQ_API kvq_status kvq_selftest_code_rounding(int32_t method, int32_t k_first, int32_t k_last,
                                              int32_t ulps, void* dev_result, void* stream);

/* The codebook quantizer's quotients (KVQ_CODEBOOK_PER_TOKEN: the group
 * scale absmax / max|level| and each value's x / s16, KVQuant page,
 * cf-1.com/news/2306543, §2.2 item 2), formed as RN(x * RN(1/s)) corrected
 * once by a fused multiply-add (Markstein's division correction). Compares
 * them as values (+0 equals -0) with __fdiv_rn(x, s) for every finite fp16
 * x (bit patterns 0x0000..0xFFFF) and every positive finite fp16 s (bit
 * patterns 0x0001..0x7BFF): about 2.0e9 pairs. Input key:
 * (s bits << 16) | x bits.
 * Errors: KVQ_ERR_INVALID_ARG for a NULL or misaligned dev_result. */
KVQ_API kvq_status kvq_selftest_codebook_quotient(void* dev_result, void* stream);

/* The kernels' bounded wait, made to give up: one CTA initializes an
 * mbarrier that nothing ever completes and waits on it through the same
 * bounded-poll loop the kernels use, with `polls` polls (1..100000) of at
 * most 10 us each instead of the kernels' ~1 s budget. When the wait gives
 * up, the kernel raises the timeout bit of `cache`'s device status word and
 * returns, as a kernel does after a wait that gave up; the next
 * kvq_cache_status on the cache then reports KVQ_ERR_TIMEOUT and clears the
 * word. The cache's contents are untouched. The cache's device must be
 * current. Errors: KVQ_ERR_INVALID_ARG for a NULL cache or polls out of range. */
KVQ_API kvq_status kvq_selftest_wait_timeout(kvq_cache* cache, int32_t polls, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_SELFTEST_H */

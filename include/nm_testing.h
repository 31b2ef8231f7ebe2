/*
 * nm_testing.h - test and measurement entry points of the library (not part
 * of the product workflow in nm.h).  They exist so that failure paths which
 * must never hang or fault a GPU can be exercised on one, and so that a
 * benchmark can measure an instruction rate that no published figure gives.
 */
#ifndef NM_TESTING_H_
#define NM_TESTING_H_

#include "nm.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * nm_test_spmm_wait_timeout - runs the 2:4 sparse tensor-core product of
 * `desc` (SPARSE_A, F16/BF16, NM_META_TC, K > 0; the same operands as nm_spmm
 * with alpha = 1, beta = 0) with one difference: the MMA-issuing lane first
 * waits on a barrier that nothing arrives at, with a wait budget of
 * `budget_cycles` GPU clock cycles.  The wait gives up, the kernel writes
 * NM_ERR_TIMEOUT to *d_status (device int32, caller-owned), every role of the
 * kernel drains its outstanding asynchronous work and frees its tensor
 * memory, and the kernel returns; D is left unspecified.  The context stays
 * usable.  plan_unused must be NULL.  Returns NM_ERR_INVALID_ARG for a bad
 * description, NM_ERR_CUDA if the launch fails, NM_OK otherwise.
 */
nm_status_t nm_test_spmm_wait_timeout(nm_spmm_plan_t plan_unused, const nm_spmm_desc_t* desc, const void* A,
                                      const void* A_meta, const void* B, void* D, int32_t* d_status,
                                      long long budget_cycles, nm_stream_t stream);

/*
 * nm_test_i8_sparse_mma_rate - instruction-rate probe of the warp-level 2:4
 * sparse int8 MMA that the int8 product uses (mma.sp m16n8k64, s8 x s8 ->
 * s32): one CTA of eight warps per SM, each warp `iters` times four
 * independent MMAs on register operands (no memory traffic), timed with CUDA
 * events around the second of two launches on the legacy default stream,
 * which the call synchronises.  Writes the elapsed milliseconds to *ms and
 * the dense-equivalent operations performed (2 * 16 * 8 * 64 per MMA) to
 * *ops, both host memory; ops / ms is the roofline denominator of the int8
 * sparse product (the cuSPARSELt blog names INT8 among the sparse tensor-core
 * inputs; no rate for this part is published).  Allocates and frees a small
 * device buffer.  Returns NM_ERR_INVALID_ARG for iters < 1 or > 10^6 or a
 * NULL output, NM_ERR_CUDA if a CUDA call fails, NM_OK otherwise.
 */
nm_status_t nm_test_i8_sparse_mma_rate(int iters, float* ms, double* ops);

#ifdef __cplusplus
}
#endif

#endif /* NM_TESTING_H_ */

/*
 * fpd_testing.h — diagnostic entry points of libfpd used by the test-suite to check single kernels in
 * isolation.  They are not part of the drafter hot path and no paper passage defines them; the hot-path
 * entry points are declared in fpd.h.
 */
#ifndef FPD_TESTING_H_
#define FPD_TESTING_H_

#include "fpd.h"

#ifdef __cplusplus
extern "C" {
#endif

/* C[M, N] (fp32, row-major) = A[M, K] . B[N, K]^T with A, B bf16 row-major device matrices, computed by the
 * library's GEMM kernels.  impl 0: the tcgen05 tensor-core kernel with the production plan for this shape
 * (placement -1), or with the token tile on the 128-row MMA operand (placement 0), or with the weight tile
 * there (placement 1); impl 1: the CUDA-core tile kernel.  K must be a multiple of 64.  workspace holds the
 * split-K partial sums: at least fpd_test_gemm_workspace_bytes(M, N, K) bytes.  Asynchronous on stream. */
fpd_status fpd_test_gemm(int impl, int placement, int M, int N, int K, const void* A, const void* B, float* C,
                         void* workspace, size_t workspace_bytes, void* stream);
size_t fpd_test_gemm_workspace_bytes(int M, int N, int K);

/* hmid[M, F] (bf16) = silu(X . Wg^T) * (X . Wu^T) for X [M, K] and W = [Wg; Wu] ([2F, K]) bf16 row-major device
 * matrices, with the gate/up tcgen05 kernel and its SwiGLU epilogue (weight-tile placement for M <= 64, token
 * tiles above).  Asynchronous on stream. */
fpd_status fpd_test_swiglu(int M, int F, int K, const void* X, const void* W, void* hmid, void* stream);

/* Selects the pipeline shape of the 16-token weight-tile GEMM kernels for tuning sweeps: 0 (default) = one
 * 64-element K atom per stage, 6 stages, 2 CTAs per SM; 1 = 2 atoms x 6 stages, 1 CTA/SM; 2 = 4 atoms x 3 stages,
 * 1 CTA/SM; 3 = 2 atoms x 3 stages, 2 CTAs/SM; 4 = 1 atom x 12 stages, 1 CTA/SM.  Affects plans (and so
 * workspace sizes) made afterwards: set it before fpd_workspace_bytes. */
void fpd_test_set_variant(int variant);

#ifdef __cplusplus
}
#endif
#endif /* FPD_TESTING_H_ */

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

#ifdef __cplusplus
}
#endif
#endif /* FPD_TESTING_H_ */

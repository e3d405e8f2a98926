// fpd_testing.cu — diagnostic entry points declared in include/fpd_testing.h (single-kernel checks).
#include "../../include/fpd_testing.h"
#include "fpd_kernels.cuh"

using namespace fpd;

namespace {
int current_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return n;
}
}  // namespace

extern "C" {

size_t fpd_test_gemm_workspace_bytes(int M, int N, int K) {
  if (M < 1 || N < 1 || K < 64) return 0;
  const int sms = current_sms();
  if (!sms) return 0;
  size_t best = (size_t)M * N;
  for (int pl = -1; pl <= 1; pl++) {
    TcPlan p = tc_plan_force(M, N, K, sms, pl);
    best = std::max(best, (size_t)p.splits * M * N);
  }
  return best * sizeof(float);
}

fpd_status fpd_test_gemm(int impl, int placement, int M, int N, int K, const void* A, const void* B, float* C,
                         void* workspace, size_t workspace_bytes, void* stream) {
  if (M < 1 || N < 1 || K < 64 || K % 64 || impl < 0 || impl > 1 || placement < -1 || placement > 1)
    return FPD_ERR_SHAPE;
  if (!A || !B || !C || !workspace) return FPD_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  GemmArgs g{};
  g.a[0] = (const bf16*)A;
  g.seg_k = K;
  g.lda = K;
  g.b = (const bf16*)B;
  g.ldb = K;
  g.ldc = N;
  g.M = M;
  g.N = N;
  g.K = K;
  if (impl == 1) {
    g.c = C;
    g.k_split = K;
    return launch_gemm_simt(g, st) == cudaSuccess ? FPD_OK : FPD_ERR_CUDA;
  }
  const int sms = current_sms();
  if (!sms) return FPD_ERR_CUDA;
  static cudaError_t init_err = tc_init_attributes();
  if (init_err != cudaSuccess) return FPD_ERR_CUDA;
  const TcPlan pl = tc_plan_force(M, N, K, sms, placement);
  if ((size_t)pl.splits * M * N * sizeof(float) > workspace_bytes) return FPD_ERR_CAPACITY;
  g.c = (float*)workspace;
  g.c_split_stride = (size_t)M * N;
  g.k_split = pl.k_split;
  if (launch_tc_gemm(g, pl, st) != cudaSuccess) return FPD_ERR_CUDA;
  return launch_sum_splits(C, (const float*)workspace, pl.splits, (size_t)M * N, st) == cudaSuccess ? FPD_OK : FPD_ERR_CUDA;
}

fpd_status fpd_test_swiglu(int M, int F, int K, const void* X, const void* W, void* hmid, void* stream) {
  if (M < 1 || F < 1 || K < 64 || K % 64) return FPD_ERR_SHAPE;
  if (!X || !W || !hmid) return FPD_ERR_INVALID_ARG;
  const int sms = current_sms();
  if (!sms) return FPD_ERR_CUDA;
  static cudaError_t init_err = tc_init_attributes();
  if (init_err != cudaSuccess) return FPD_ERR_CUDA;
  const TcPlan pl = tc_plan_swiglu(M, F, K, sms);
  return launch_tc_swiglu((const bf16*)X, M, K, (const bf16*)W, F, (bf16*)hmid, pl, (cudaStream_t)stream) == cudaSuccess
             ? FPD_OK
             : FPD_ERR_CUDA;
}

void fpd_test_set_variant(int variant) { tc_set_swap_variant(variant); }

}  // extern "C"

// k_gemm_simt.cu — CUDA-core tiled GEMM  C[split][m][n] = sum_{k in split} A[m][k] * B[n][k]  (fp32 out).
//
// A plain 64x64x32 shared-memory tile kernel.  It serves shapes the tensor-core path does not take and is
// the cross-check for it in the tests.  A may be split into K-segments held in separate buffers (the
// concatenated target-layer features of the context fusion, VFlash paper (zh) §2.1: the n_f feature
// matrices are never copied into one buffer).
#include "fpd_kernels.cuh"

namespace fpd {

namespace {
constexpr int TM = 64, TN = 64, TK = 32;

__global__ void __launch_bounds__(256) gemm_simt_kernel(GemmArgs g) {
  pdl_trigger();
  pdl_wait();
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
  const int k_begin = blockIdx.z * g.k_split, k_end = min(g.K, k_begin + g.k_split);
  float acc[4][4] = {};
  const int lr = tid >> 2, lk = (tid & 3) * 8;   // loader: row lr, k chunk lk..lk+7
  for (int k0 = k_begin; k0 < k_end; k0 += TK) {
    {
      const int m = m0 + lr, k = k0 + lk;
      uint4 u = make_uint4(0, 0, 0, 0);
      if (m < g.M) {
        const int seg = k / g.seg_k, kk = k - seg * g.seg_k;
        u = *reinterpret_cast<const uint4*>(g.a[seg] + (size_t)m * g.lda + kk);
      }
      const bf16* e = reinterpret_cast<const bf16*>(&u);
#pragma unroll
      for (int i = 0; i < 8; i++) As[lk + i][lr] = __bfloat162float(e[i]);
    }
    {
      const int n = n0 + lr, k = k0 + lk;
      uint4 u = make_uint4(0, 0, 0, 0);
      if (n < g.N) u = *reinterpret_cast<const uint4*>(g.b + (size_t)n * g.ldb + k);
      const bf16* e = reinterpret_cast<const bf16*>(&u);
#pragma unroll
      for (int i = 0; i < 8; i++) Bs[lk + i][lr] = __bfloat162float(e[i]);
    }
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < TK; k++) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; i++) a[i] = As[k][ty * 4 + i];
#pragma unroll
      for (int i = 0; i < 4; i++) b[i] = Bs[k][tx * 4 + i];
#pragma unroll
      for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  float* C = g.c + (size_t)blockIdx.z * g.c_split_stride;
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const int m = m0 + ty * 4 + i;
    if (m >= g.M) continue;
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const int n = n0 + tx * 4 + j;
      if (n < g.N) C[(size_t)m * g.ldc + n] = acc[i][j];
    }
  }
}
}  // namespace

cudaError_t launch_gemm_simt(const GemmArgs& g, cudaStream_t st) {
  if (g.M <= 0 || g.N <= 0) return cudaSuccess;
  dim3 grid(ceil_div(g.N, TN), ceil_div(g.M, TM), ceil_div(g.K, g.k_split));
  return launch_k(gemm_simt_kernel, grid, 256, 0, st, g);
}

}  // namespace fpd

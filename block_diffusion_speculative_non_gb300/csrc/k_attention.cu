// k_attention.cu — a5: bidirectional grouped-query block attention over [context K/V ; block K/V], as standalone
// kernels (the work units are in attn_body.cuh: one query tile of one kv-head group over one KV split, and the
// fixed-order merge of the splits).
#include "attn_body.cuh"

namespace fpd {

namespace {
using namespace attn;

struct CtaSync {
  __device__ void operator()() const { __syncthreads(); }
};

template <int H>
__global__ void __launch_bounds__(NWARP * 32) attn_mma_kernel(AttnArgs a, bf16* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(128) unsigned char smem_raw[];
  attn_tile<H>(a, out, blockIdx.x, blockIdx.y, blockIdx.z, threadIdx.x, smem_raw, CtaSync{});
}

// one warp per (row, q head), 8 per block
template <int H>
__global__ void __launch_bounds__(256) attn_merge_kernel(bf16* __restrict__ out, const float* __restrict__ o_part,
                                                         const float2* __restrict__ ml, int nsplit, int rows, int nq) {
  pdl_trigger();
  pdl_wait();
  const int wid = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (wid >= rows * nq) return;
  attn_merge_warp<H>(out, o_part, ml, nsplit, rows, nq, wid / nq, wid % nq, threadIdx.x & 31);
}
}  // namespace

void attn_plan(int batch, int L, int nq, int nkv, int t_cap, int num_sms, int* splits, int* chunk) {
  const int grp = nq / nkv;
  const int q_tiles = ceil_div(L * grp, QT);
  const int base = q_tiles * batch * nkv;
  const int max_keys = t_cap + L;
  const int max_splits = ceil_div(max_keys, KT);
  int s = ceil_div(num_sms, base);   // about one CTA per SM
  s = s < 1 ? 1 : (s > max_splits ? max_splits : s);
  s = s > 128 ? 128 : s;
  const int ch = ceil_div(ceil_div(max_keys, s), KT) * KT;
  *chunk = ch;
  *splits = ceil_div(max_keys, ch);
}

cudaError_t attn_init_attributes() {
  cudaError_t e = cudaFuncSetAttribute(attn_mma_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sizeof(Smem<128>));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_mma_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(Smem<64>));
  return e;
}

cudaError_t launch_attn_merge(const AttnArgs& a, bf16* out, cudaStream_t st) {
  const int blocks = ceil_div(a.rows * a.nq, 8);
  if (a.head_dim == 128)
    return launch_k(attn_merge_kernel<128>, blocks, 256, 0, st, out, (const float*)a.o_part, (const float2*)a.ml,
                    a.splits, a.rows, a.nq);
  return launch_k(attn_merge_kernel<64>, blocks, 256, 0, st, out, (const float*)a.o_part, (const float2*)a.ml,
                  a.splits, a.rows, a.nq);
}

cudaError_t launch_attention(const AttnArgs& a, bf16* out, cudaStream_t st) {
  const int grp = a.nq / a.nkv;
  dim3 grid(ceil_div(a.L * grp, QT), a.batch * a.nkv, a.splits);
  cudaError_t err;
  if (a.head_dim == 128)
    err = launch_k(attn_mma_kernel<128>, grid, NWARP * 32, sizeof(Smem<128>), st, a, out);
  else
    err = launch_k(attn_mma_kernel<64>, grid, NWARP * 32, sizeof(Smem<64>), st, a, out);
  if (err != cudaSuccess || a.splits == 1) return err;
  return launch_attn_merge(a, out, st);
}

}  // namespace fpd

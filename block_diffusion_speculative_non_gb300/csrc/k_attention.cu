// k_attention.cu — a5: bidirectional grouped-query block attention over [context K/V ; block K/V].
//
// VFlash paper (zh), §2.1: the fused target features enter every drafter layer as keys and values, and
// the masked positions are predicted in one BIDIRECTIONAL pass — so there is no mask at all inside a
// request: every block query sees all ctx_len[b] context keys of its layer and all L block keys.
// VFlash blog, "Key claims": the drafter is a non-causal transformer.
//
// Work split: (query tile of 64 rows of one kv-head group) x (request, kv head) x (KV split).  The rows of a
// tile are the L positions x H_q/H_kv q heads that share one kv head, so every K/V row loaded is used by the
// whole group.  Each CTA runs an online softmax over its key range and writes an unnormalised partial
// (o, m, l); a merge kernel combines the splits in fixed order (deterministic, no atomics).
#include "fpd_kernels.cuh"

namespace fpd {

namespace {
constexpr int QT = 64, KT = 64;

template <int H>
struct AttnSmem {
  float q[QT][H];
  float k[KT][H + 1];
  float v[KT][H];
  float s[QT][KT + 1];
  float corr[QT];
};

template <int H>
__global__ void __launch_bounds__(256) attn_simt_kernel(AttnArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  AttnSmem<H>& sm = *reinterpret_cast<AttnSmem<H>*>(smem_raw);
  const int tid = threadIdx.x;
  const int qt = blockIdx.x, bg = blockIdx.y, split = blockIdx.z;
  const int b = bg / a.nkv, g = bg % a.nkv;
  const int grp = a.nq / a.nkv, nrows = a.L * grp;
  int T = a.ctx_len[b];
  T = T < 0 ? 0 : (T > a.t_cap ? a.t_cap : T);
  const int n_keys = T + a.L;
  const int k_begin = split * a.chunk, k_end = min(n_keys, k_begin + a.chunk);
  const float scale = rsqrtf((float)H);

  // query rows of this tile
  for (int idx = tid; idx < QT * H; idx += blockDim.x) {
    const int rr = idx / H, e = idx % H, qi = qt * QT + rr;
    float v = 0.f;
    if (qi < nrows) {
      const int j = qi / grp, i = g * grp + qi % grp;
      v = __bfloat162float(a.q[(((size_t)b * a.L + j) * a.nq + i) * H + e]) * scale;
    }
    sm.q[rr][e] = v;
  }
  const int orow = tid >> 2, oc0 = (tid & 3) * (H / 4);
  float o[H / 4];
#pragma unroll
  for (int c = 0; c < H / 4; c++) o[c] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;   // valid in threads tid < QT (row tid)

  const bf16* kctx = a.store + ((((size_t)a.layer * a.batch + b) * 2 + 0) * a.nkv + g) * (size_t)a.t_cap * H;
  const bf16* vctx = a.store + ((((size_t)a.layer * a.batch + b) * 2 + 1) * a.nkv + g) * (size_t)a.t_cap * H;
  const bf16* kb = a.kblk + ((size_t)b * a.nkv + g) * a.L * H;
  const bf16* vb = a.vblk + ((size_t)b * a.nkv + g) * a.L * H;

  for (int k0 = k_begin; k0 < k_end; k0 += KT) {
    __syncthreads();
    for (int idx = tid; idx < KT * H; idx += blockDim.x) {
      const int kk = idx / H, e = idx % H, t = k0 + kk;
      float kv = 0.f, vv = 0.f;
      if (t < k_end) {
        if (t < T) {
          kv = __bfloat162float(kctx[(size_t)t * H + e]);
          vv = __bfloat162float(vctx[(size_t)t * H + e]);
        } else {
          kv = __bfloat162float(kb[(size_t)(t - T) * H + e]);
          vv = __bfloat162float(vb[(size_t)(t - T) * H + e]);
        }
      }
      sm.k[kk][e] = kv;
      sm.v[kk][e] = vv;
    }
    __syncthreads();
    {
      const int ty = tid >> 4, tx = tid & 15;
      float acc[4][4] = {};
      for (int e = 0; e < H; e++) {
        float qa[4], kbv[4];
#pragma unroll
        for (int i = 0; i < 4; i++) qa[i] = sm.q[ty * 4 + i][e];
#pragma unroll
        for (int j = 0; j < 4; j++) kbv[j] = sm.k[tx * 4 + j][e];
#pragma unroll
        for (int i = 0; i < 4; i++)
#pragma unroll
          for (int j = 0; j < 4; j++) acc[i][j] = fmaf(qa[i], kbv[j], acc[i][j]);
      }
#pragma unroll
      for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) sm.s[ty * 4 + i][tx * 4 + j] = (k0 + tx * 4 + j < k_end) ? acc[i][j] : -INFINITY;
    }
    __syncthreads();
    if (tid < QT) {
      float mx = -INFINITY;
      for (int kk = 0; kk < KT; kk++) mx = fmaxf(mx, sm.s[tid][kk]);
      const float m_new = fmaxf(m_run, mx);
      const float corr = m_run == -INFINITY ? 0.f : expf(m_run - m_new);
      float sum = 0.f;
      for (int kk = 0; kk < KT; kk++) {
        const float sv = sm.s[tid][kk];
        const float pv = sv == -INFINITY ? 0.f : expf(sv - m_new);
        sm.s[tid][kk] = pv;
        sum += pv;
      }
      l_run = l_run * corr + sum;
      m_run = m_new;
      sm.corr[tid] = corr;
    }
    __syncthreads();
    {
      const float corr = sm.corr[orow];
#pragma unroll
      for (int c = 0; c < H / 4; c++) o[c] *= corr;
      for (int kk = 0; kk < KT; kk++) {
        const float pv = sm.s[orow][kk];
#pragma unroll
        for (int c = 0; c < H / 4; c++) o[c] = fmaf(pv, sm.v[kk][oc0 + c], o[c]);
      }
    }
  }
  // partial outputs
  const int qi = qt * QT + orow;
  if (qi < nrows) {
    const int j = qi / grp, i = g * grp + qi % grp;
    const size_t row = (size_t)b * a.L + j;
    float* dst = a.o_part + (((size_t)split * a.rows + row) * a.nq + i) * H + oc0;
#pragma unroll
    for (int c = 0; c < H / 4; c++) dst[c] = o[c];
  }
  if (tid < QT) {
    const int qi2 = qt * QT + tid;
    if (qi2 < nrows) {
      const int j = qi2 / grp, i = g * grp + qi2 % grp;
      const size_t row = (size_t)b * a.L + j;
      a.ml[((size_t)split * a.rows + row) * a.nq + i] = make_float2(m_run, l_run);
    }
  }
}

template <int H>
__global__ void attn_merge_kernel(bf16* __restrict__ out, const float* __restrict__ o_part,
                                  const float2* __restrict__ ml, int nsplit, int rows, int nq) {
  const int r = blockIdx.x, i = blockIdx.y, e = threadIdx.x;
  float M = -INFINITY;
  for (int s = 0; s < nsplit; s++) {
    const float2 v = ml[((size_t)s * rows + r) * nq + i];
    if (v.y > 0.f) M = fmaxf(M, v.x);
  }
  float den = 0.f, num = 0.f;
  for (int s = 0; s < nsplit; s++) {
    const float2 v = ml[((size_t)s * rows + r) * nq + i];
    if (v.y > 0.f) {
      const float w = expf(v.x - M);
      den += v.y * w;
      num += o_part[(((size_t)s * rows + r) * nq + i) * H + e] * w;
    }
  }
  out[((size_t)r * nq + i) * H + e] = __float2bfloat16_rn(den > 0.f ? num / den : 0.f);
}
}  // namespace

void attn_plan(int batch, int L, int nq, int nkv, int t_cap, int num_sms, int* splits, int* chunk) {
  const int grp = nq / nkv;
  const int q_tiles = ceil_div(L * grp, QT);
  const int base = q_tiles * batch * nkv;
  const int max_keys = t_cap + L;
  const int max_splits = ceil_div(max_keys, KT);
  int s = ceil_div(2 * num_sms, base);
  s = s < 1 ? 1 : (s > max_splits ? max_splits : s);
  int ch = ceil_div(ceil_div(max_keys, s), KT) * KT;
  *chunk = ch;
  *splits = ceil_div(max_keys, ch);
}

cudaError_t attn_init_attributes() {
  cudaError_t e = cudaFuncSetAttribute(attn_simt_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sizeof(AttnSmem<128>));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_simt_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(AttnSmem<64>));
  return e;
}

cudaError_t launch_attention(const AttnArgs& a, bf16* out, cudaStream_t st) {
  const int grp = a.nq / a.nkv;
  dim3 grid(ceil_div(a.L * grp, QT), a.batch * a.nkv, a.splits);
  cudaError_t err;
  if (a.head_dim == 128) {
    const size_t smem = sizeof(AttnSmem<128>);
    attn_simt_kernel<128><<<grid, 256, smem, st>>>(a);
    count_launch();
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    attn_merge_kernel<128><<<dim3(a.rows, a.nq), 128, 0, st>>>(out, a.o_part, a.ml, a.splits, a.rows, a.nq);
  } else {
    const size_t smem = sizeof(AttnSmem<64>);
    attn_simt_kernel<64><<<grid, 256, smem, st>>>(a);
    count_launch();
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    attn_merge_kernel<64><<<dim3(a.rows, a.nq), 64, 0, st>>>(out, a.o_part, a.ml, a.splits, a.rows, a.nq);
  }
  count_launch();
  return cudaGetLastError();
}

}  // namespace fpd

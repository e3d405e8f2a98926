// k_rowops.cu — row-wise kernels of the drafter pass: embedding gather + RMSNorm, residual add + RMSNorm (which
// also reduces the split-K partial sums), the q/k RMSNorm + RoPE epilogue of the QKV projection, and the context
// K/V epilogue.  (SwiGLU runs in the gate/up GEMM epilogue, k_gemm_tc.cu.)
//
// Method: VFlash paper (zh) §2.1-§2.2 (one anchor + L-1 mask tokens through a bidirectional layer stack
// conditioned on per-layer context K/V); layer form = pre-norm transformer layer with per-head q/k RMSNorm
// and rotate-half RoPE, SwiGLU MLP (the reading of the five-layer non-causal drafter of the VFlash blog,
// "Key claims").  All of these are HBM/latency-bound (a few MB per call): one thread block or one warp per
// row or head, 16-byte vector loads, fp32 arithmetic, bf16 stores at the storage points.
#include "fpd_kernels.cuh"

namespace fpd {

__device__ int32_t g_device_check = 0;

// ---- block reduction helper ------------------------------------------------------------------------------------
__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = blockDim.x >> 5;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float t = l < nw ? red[l] : 0.f;
  return warp_sum(t);
}

// ---- RMSNorm of fp32 split-K partial sums -> bf16 (fused context) -------------------------------------------------
// Thread t holds the float4 groups t, t + 256, ... (VPT of them) of row blockIdx.x: the split-K partials are read
// once (one round trip per split, every thread's groups of a split in flight together), summed in split order,
// then normed from registers.
template <int VPT>
__global__ void __launch_bounds__(256) rmsnorm_partials_kernel(bf16* __restrict__ out, const float* __restrict__ part,
                                                               int nsplit, size_t split_stride,
                                                               const bf16* __restrict__ g, int d, float eps) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[32];
  const int r = blockIdx.x, n4 = d / 4;
  const float4* src = reinterpret_cast<const float4*>(part + (size_t)r * d);
  const size_t s4 = split_stride / 4;
  float4 v[VPT];
#pragma unroll
  for (int k = 0; k < VPT; k++) {
    const int i = threadIdx.x + k * 256;
    v[k] = i < n4 ? __ldcg(src + i) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int s = 1; s < nsplit; s++) {
    float4 t[VPT];
#pragma unroll
    for (int k = 0; k < VPT; k++) {
      const int i = threadIdx.x + k * 256;
      t[k] = i < n4 ? __ldcg(src + s * s4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < VPT; k++) {
      v[k].x += t[k].x;
      v[k].y += t[k].y;
      v[k].z += t[k].z;
      v[k].w += t[k].w;
    }
  }
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; k++) ss += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
  const float inv = rsqrtf(block_sum(ss, red) / (float)d + eps);
#pragma unroll
  for (int k = 0; k < VPT; k++) {
    const int i = threadIdx.x + k * 256;
    if (i < n4) {
      const uint2 gu = reinterpret_cast<const uint2*>(g)[i];
      const float2 g01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gu.x));
      const float2 g23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gu.y));
      const __nv_bfloat162 o01 = __floats2bfloat162_rn(v[k].x * inv * g01.x, v[k].y * inv * g01.y);
      const __nv_bfloat162 o23 = __floats2bfloat162_rn(v[k].z * inv * g23.x, v[k].w * inv * g23.y);
      uint2 o;
      o.x = *reinterpret_cast<const uint32_t*>(&o01);
      o.y = *reinterpret_cast<const uint32_t*>(&o23);
      reinterpret_cast<uint2*>(out + (size_t)r * d)[i] = o;
    }
  }
}

cudaError_t launch_rmsnorm_partials(bf16* out, const float* part, int nsplit, size_t split_stride, const bf16* g,
                                    int rows, int d, float eps, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  if (d % 4 || split_stride % 4 || d > 16384) return cudaErrorInvalidValue;
  const int n4 = d / 4;
  if (n4 <= 256) return launch_k(rmsnorm_partials_kernel<1>, rows, 256, 0, st, out, part, nsplit, split_stride, g, d, eps);
  if (n4 <= 512) return launch_k(rmsnorm_partials_kernel<2>, rows, 256, 0, st, out, part, nsplit, split_stride, g, d, eps);
  if (n4 <= 1024) return launch_k(rmsnorm_partials_kernel<4>, rows, 256, 0, st, out, part, nsplit, split_stride, g, d, eps);
  if (n4 <= 2048) return launch_k(rmsnorm_partials_kernel<8>, rows, 256, 0, st, out, part, nsplit, split_stride, g, d, eps);
  return launch_k(rmsnorm_partials_kernel<16>, rows, 256, 0, st, out, part, nsplit, split_stride, g, d, eps);
}

// ---- a4 epilogue: sum split-K partials of [q | k | v], q/k RMSNorm + RoPE at pos = ctx_len[b] + j ------------------
// grid (B*L, Hq + 2 Hkv), one warp per (row, head).
template <int H>
__global__ void qkv_post_kernel(bf16* __restrict__ q_out, bf16* __restrict__ kblk, bf16* __restrict__ vblk,
                                const float* __restrict__ part, int nsplit, size_t split_stride,
                                const bf16* __restrict__ q_norm, const bf16* __restrict__ k_norm,
                                const float2* __restrict__ rope, const int32_t* __restrict__ ctx_len, int t_cap,
                                int L, int nq, int nkv, float eps) {
  pdl_trigger();
  pdl_wait();
  constexpr int NV = H / 32;
  const int r = blockIdx.x, hd = blockIdx.y, lane = threadIdx.x;
  const int b = r / L, j = r % L;
  const int ncol = (nq + 2 * nkv) * H;
  float v[NV];
#pragma unroll
  for (int k = 0; k < NV; k++) v[k] = 0.f;
  const float* pr = part + (size_t)r * ncol + hd * H + lane;
  for (int s0 = 0; s0 < nsplit; s0 += 4) {
    float t[4][NV];
#pragma unroll
    for (int u = 0; u < 4; u++)
#pragma unroll
      for (int k = 0; k < NV; k++) t[u][k] = s0 + u < nsplit ? __ldcg(pr + (size_t)(s0 + u) * split_stride + 32 * k) : 0.f;
#pragma unroll
    for (int u = 0; u < 4; u++)
#pragma unroll
      for (int k = 0; k < NV; k++) v[k] += t[u][k];
  }
  int cl = ctx_len[b];
  cl = clamp_ctx(cl, t_cap);
  const float2* rope_row = rope + (size_t)(cl + j) * (H / 2);
  bf16* dst;
  if (hd < nq) {
    head_norm_rope<H>(v, q_norm, eps, rope_row, true, true);
    dst = q_out + ((size_t)r * nq + hd) * H;
  } else if (hd < nq + nkv) {
    head_norm_rope<H>(v, k_norm, eps, rope_row, true, true);
    dst = kblk + (((size_t)b * nkv + (hd - nq)) * L + j) * H;
  } else {
    dst = vblk + (((size_t)b * nkv + (hd - nq - nkv)) * L + j) * H;
  }
#pragma unroll
  for (int k = 0; k < NV; k++) dst[lane + 32 * k] = __float2bfloat16_rn(v[k]);
}

cudaError_t launch_qkv_post(bf16* q, bf16* kblk, bf16* vblk, const float* part, int nsplit, size_t split_stride,
                            const bf16* q_norm, const bf16* k_norm, const float2* rope, const int32_t* ctx_len,
                            int t_cap, int B, int L, int nq, int nkv, int h, float eps, cudaStream_t st) {
  dim3 grid(B * L, nq + 2 * nkv);
  if (h == 128)
    return launch_k(qkv_post_kernel<128>, grid, 32, 0, st, q, kblk, vblk, part, nsplit, split_stride, q_norm, k_norm,
                    rope, ctx_len, t_cap, L, nq, nkv, eps);
  return launch_k(qkv_post_kernel<64>, grid, 32, 0, st, q, kblk, vblk, part, nsplit, split_stride, q_norm, k_norm,
                  rope, ctx_len, t_cap, L, nq, nkv, eps);
}

// ---- a2 epilogue: context K (k-norm + RoPE at its context position) and V into the KV store -----------------------
// part: [rows, 2*nkv*H] fp32 = ctx . [Wk; Wv]^T for `rows` packed rows starting at global row row0.
// Store layout [layer][b][K|V][g][t_cap][H].
template <int H>
__global__ void kv_post_kernel(bf16* __restrict__ store, const float* __restrict__ part, int nsplit,
                               size_t split_stride, const bf16* __restrict__ k_norm, const float2* __restrict__ rope,
                               const int32_t* __restrict__ row_off, const int32_t* __restrict__ row_cnt,
                               const int32_t* __restrict__ pos_start, int batch, int layer, int t_cap, int row0, int nkv,
                               float eps) {
  pdl_trigger();
  pdl_wait();
  constexpr int NV = H / 32;
  const int r = blockIdx.x, hd = blockIdx.y, lane = threadIdx.x;
  const int grow = row0 + r;
  int lo = 0, hi = batch;                       // request b with row_off[b] <= grow < row_off[b+1]
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (row_off[mid] <= grow) lo = mid; else hi = mid;
  }
  const int b = lo;
  if (grow >= row_off[batch] || (row_cnt && grow - row_off[b] >= row_cnt[b])) return;   // rows past the count
  const int pos = (pos_start ? pos_start[b] : 0) + grow - row_off[b];
  if (pos < 0 || pos >= t_cap) {                // caller contract violated: skip the store, record it
    if (lane == 0 && hd == 0) record_check(kCheckBadPosition);
    return;
  }
  const int ncol = 2 * nkv * H;
  float v[NV];
#pragma unroll
  for (int k = 0; k < NV; k++) {
    float a = 0.f;
    for (int s = 0; s < nsplit; s++) a += part[s * split_stride + (size_t)r * ncol + hd * H + lane + 32 * k];
    v[k] = a;
  }
  const int is_v = hd >= nkv, g = is_v ? hd - nkv : hd;
  if (!is_v) head_norm_rope<H>(v, k_norm, eps, rope + (size_t)pos * (H / 2), true, true);
  bf16* dst = store + (((((size_t)layer * batch + b) * 2 + is_v) * nkv + g) * (size_t)t_cap + pos) * H;
#pragma unroll
  for (int k = 0; k < NV; k++) dst[lane + 32 * k] = __float2bfloat16_rn(v[k]);
}

cudaError_t launch_kv_post(bf16* store, const float* part, int nsplit, size_t split_stride, const bf16* k_norm,
                           const float2* rope, const int32_t* row_off, const int32_t* row_cnt, const int32_t* pos_start,
                           int batch, int layer, int t_cap, int row0, int rows, int nkv, int h, float eps,
                           cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  dim3 grid(rows, 2 * nkv);
  if (h == 128)
    return launch_k(kv_post_kernel<128>, grid, 32, 0, st, store, part, nsplit, split_stride, k_norm, rope, row_off,
                    row_cnt, pos_start, batch, layer, t_cap, row0, nkv, eps);
  return launch_k(kv_post_kernel<64>, grid, 32, 0, st, store, part, nsplit, split_stride, k_norm, rope, row_off,
                  row_cnt, pos_start, batch, layer, t_cap, row0, nkv, eps);
}

// ---- residual add fused with the next RMSNorm: one block per row ------------------------------------------------
// x = bf16(x + sum_s part[s]);  xn = bf16(x / sqrt(mean(x^2) + eps) * g)   (g == nullptr: residual only).
// The norm reads the bf16-rounded x, exactly what an unfused norm kernel would read back.
template <int VPT>
__global__ void residual_norm_kernel(bf16* __restrict__ x, bf16* __restrict__ xn, const float* __restrict__ part,
                                     int nsplit, size_t split_stride, const bf16* __restrict__ g, int d, float eps) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[32];
  const int r = blockIdx.x;
  bf16* xr = x + (size_t)r * d;
  const float* pr = part + (size_t)r * d;
  float acc[VPT];
#pragma unroll
  for (int k = 0; k < VPT; k++) acc[k] = 0.f;
  // split-K partials: four splits' loads in flight at once, summed in split order (bit-reproducible)
  for (int s0 = 0; s0 < nsplit; s0 += 4) {
    float t[4][VPT];
#pragma unroll
    for (int u = 0; u < 4; u++)
#pragma unroll
      for (int k = 0; k < VPT; k++) {
        const int i = threadIdx.x + k * blockDim.x;
        t[u][k] = (s0 + u < nsplit && i < d) ? __ldcg(pr + (size_t)(s0 + u) * split_stride + i) : 0.f;
      }
#pragma unroll
    for (int u = 0; u < 4; u++)
#pragma unroll
      for (int k = 0; k < VPT; k++) acc[k] += t[u][k];
  }
  float v[VPT];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; k++) {
    const int i = threadIdx.x + k * blockDim.x;
    v[k] = 0.f;
    if (i < d) {
      const bf16 nb = __float2bfloat16_rn(__bfloat162float(xr[i]) + acc[k]);
      xr[i] = nb;
      v[k] = __bfloat162float(nb);
      ss += v[k] * v[k];
    }
  }
  if (!g) return;
  const float inv = rsqrtf(block_sum(ss, red) / (float)d + eps);
#pragma unroll
  for (int k = 0; k < VPT; k++) {
    const int i = threadIdx.x + k * blockDim.x;
    if (i < d) xn[(size_t)r * d + i] = __float2bfloat16_rn(v[k] * inv * __bfloat162float(g[i]));
  }
}

cudaError_t launch_residual_norm(bf16* x, bf16* xn, const float* part, int nsplit, size_t split_stride, const bf16* g,
                                 int rows, int d, float eps, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  if (d <= 256 * 4) return launch_k(residual_norm_kernel<4>, rows, 256, 0, st, x, xn, part, nsplit, split_stride, g, d, eps);
  if (d <= 512 * 8) return launch_k(residual_norm_kernel<8>, rows, 512, 0, st, x, xn, part, nsplit, split_stride, g, d, eps);
  return launch_k(residual_norm_kernel<16>, rows, 1024, 0, st, x, xn, part, nsplit, split_stride, g, d, eps);
}

// ---- RMSNorm of rows whose sums of squares were left by the residual GEMM epilogue: one block per row -----------
// One 128-thread block per row: warp 0 loads the row's column-tile partials of sum(x^2) (lane t holds part t) and
// adds them in part order, while every thread already holds its chunks of x and g; one round trip for the loads.
template <int CPT>
__global__ void __launch_bounds__(128) norm_rows_kernel(bf16* __restrict__ xn, const bf16* __restrict__ x,
                                                        const float* __restrict__ ss_part, int n_part,
                                                        const bf16* __restrict__ g, int M, int d, float eps) {
  pdl_trigger();
  pdl_wait();
  __shared__ float s_inv;
  const int r = blockIdx.x, tid = threadIdx.x, n8 = d / 8;
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)r * d);
  const uint4* gs = reinterpret_cast<const uint4*>(g);
  uint4 u[CPT], gu[CPT];
#pragma unroll
  for (int k = 0; k < CPT; k++) {
    const int c = tid + k * 128;
    if (c < n8) {
      u[k] = src[c];
      gu[k] = gs[c];
    }
  }
  if (tid < 32) {
    float ss = 0.f;   // sequential in part order: the same fp32 sum as a one-thread loop
    for (int t0 = 0; t0 < n_part; t0 += 32) {
      const float v = t0 + tid < n_part ? __ldcg(ss_part + (size_t)(t0 + tid) * M + r) : 0.f;
      for (int j = 0; j < 32 && t0 + j < n_part; j++) ss += __shfl_sync(0xffffffffu, v, j);
    }
    if (tid == 0) s_inv = rsqrtf(ss / (float)d + eps);
  }
  __syncthreads();
  const float inv = s_inv;
  uint4* dst = reinterpret_cast<uint4*>(xn + (size_t)r * d);
#pragma unroll
  for (int k = 0; k < CPT; k++) {
    const int c = tid + k * 128;
    if (c < n8) {
      __nv_bfloat162* e = reinterpret_cast<__nv_bfloat162*>(&u[k]);
      const __nv_bfloat162* ge = reinterpret_cast<const __nv_bfloat162*>(&gu[k]);
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const float2 xf = __bfloat1622float2(e[i]), gf = __bfloat1622float2(ge[i]);
        e[i] = __floats2bfloat162_rn(xf.x * inv * gf.x, xf.y * inv * gf.y);
      }
      dst[c] = u[k];
    }
  }
}

cudaError_t launch_norm_rows(bf16* xn, const bf16* x, const float* ss_part, int n_part, const bf16* g, int M, int d,
                             float eps, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  if (d % 8 || d > 16384) return cudaErrorInvalidValue;
  const int n8 = d / 8;
  if (n8 <= 128) return launch_k(norm_rows_kernel<1>, M, 128, 0, st, xn, x, ss_part, n_part, g, M, d, eps);
  if (n8 <= 256) return launch_k(norm_rows_kernel<2>, M, 128, 0, st, xn, x, ss_part, n_part, g, M, d, eps);
  if (n8 <= 512) return launch_k(norm_rows_kernel<4>, M, 128, 0, st, xn, x, ss_part, n_part, g, M, d, eps);
  if (n8 <= 1024) return launch_k(norm_rows_kernel<8>, M, 128, 0, st, xn, x, ss_part, n_part, g, M, d, eps);
  return launch_k(norm_rows_kernel<16>, M, 128, 0, st, xn, x, ss_part, n_part, g, M, d, eps);
}

// ---- embedding gather fused with the first RMSNorm ----------------------------------------------------------------
__global__ void embed_norm_kernel(bf16* __restrict__ x, bf16* __restrict__ xn, const bf16* __restrict__ embed,
                                  const int32_t* __restrict__ anchor, int32_t mask_id, const bf16* __restrict__ g,
                                  int L, int d, int V, float eps) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[32];
  const int r = blockIdx.x, b = r / L, j = r % L;
  int id = j == 0 ? anchor[b] : mask_id;
  const bool bad = id < 0 || id >= V;
  if (bad) {
    if (threadIdx.x == 0) record_check(kCheckBadToken);
    id = 0;
  }
  const uint4* src = reinterpret_cast<const uint4*>(embed + (size_t)id * d);
  uint4* dx = reinterpret_cast<uint4*>(x + (size_t)r * d);
  float ss = 0.f;
  for (int i = threadIdx.x; i < d / 8; i += blockDim.x) {
    uint4 u = bad ? make_uint4(0, 0, 0, 0) : src[i];
    dx[i] = u;
    const bf16* e = reinterpret_cast<const bf16*>(&u);
#pragma unroll
    for (int k = 0; k < 8; k++) {
      const float f = __bfloat162float(e[k]);
      ss += f * f;
    }
  }
  const float inv = rsqrtf(block_sum(ss, red) / (float)d + eps);
  const uint4* gs = reinterpret_cast<const uint4*>(g);
  uint4* dn = reinterpret_cast<uint4*>(xn + (size_t)r * d);
  for (int i = threadIdx.x; i < d / 8; i += blockDim.x) {
    uint4 u = bad ? make_uint4(0, 0, 0, 0) : src[i], gu = gs[i], o;
    const bf16* e = reinterpret_cast<const bf16*>(&u);
    const bf16* ge = reinterpret_cast<const bf16*>(&gu);
    bf16* oe = reinterpret_cast<bf16*>(&o);
#pragma unroll
    for (int k = 0; k < 8; k++) oe[k] = __float2bfloat16_rn(__bfloat162float(e[k]) * inv * __bfloat162float(ge[k]));
    dn[i] = o;
  }
}

cudaError_t launch_embed_norm(bf16* x, bf16* xn, const bf16* embed, const int32_t* anchor, int32_t mask_id,
                              const bf16* g, int B, int L, int d, int V, float eps, cudaStream_t st) {
  return launch_k(embed_norm_kernel, B * L, 256, 0, st, x, xn, embed, anchor, mask_id, g, L, d, V, eps);
}

}  // namespace fpd

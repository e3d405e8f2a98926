// k_attention_short.cu — a5 for few-token blocks: bidirectional grouped-query attention of at most 64 query rows
// per (request, kv head) (e.g. one request's 16-position text block x 4 q heads) over [context K/V ; block K/V].
//
// VFlash paper (zh) §2.1: every block query sees all ctx_len[b] context keys and all L block keys of its layer (no
// mask inside a request).  With 16 positions the work is a read of the context K/V (8.4 MB per layer at T = 2048,
// the 4B shape), so the keys of one (request, kv head) are split over the CTAs of a thread-block cluster and the
// splits are merged through distributed shared memory inside the same kernel: no fp32 partials go to global memory
// and no merge kernel follows.
//
//   - CTA `rank` of the cluster takes 64-key tiles [rank * tiles / C, (rank + 1) * tiles / C) of [0, T + L); a last
//     tile of at most 16 keys runs the 16-key tile math.
//   - Tiles that hold only context keys are fetched (cp.async, 3-tile ring) before griddepcontrol.wait: the store
//     and ctx_len are written before the call, and the call's first kernel lets its successors launch only after
//     its own wait, so they are complete.  Q and the block K/V come from the call's QKV kernel: after the wait.
//   - Per tile: S = Q K^T, base-2 online softmax and O += (P_hi + P_lo) V on mma.sync (attn_tile_math).
//   - Each CTA leaves its unnormalised partial (o [64][h] fp32, running max m and sum l per row) in its own shared
//     memory; after a cluster barrier CTA `rank` merges rows [rank * rpc, ...) over all C partials in rank order
//     (weights 2^(m_c - max), fixed order: bit-reproducible) and writes bf16 O; a second cluster barrier keeps
//     every partial alive until all readers are done.
#include "attn_body.cuh"

namespace fpd {

namespace {
using namespace attn;

constexpr int SNS = 3;   // K/V ring depth (64-key tiles)

template <int H>
struct ShortSmem {
  bf16 q[QT * H];
  bf16 k[SNS][KT * H];
  bf16 v[SNS][KT * H];
};
// the partial (o [QT][H] fp32, then (m, l) [QT]) reuses the K/V ring once the key loop is over
template <int H>
constexpr bool partial_fits() {
  return (size_t)QT * H * 4 + (size_t)QT * 8 <= sizeof(bf16) * 2 * SNS * KT * H;
}
static_assert(partial_fits<128>() && partial_fits<64>(), "the cluster partial must fit in the K/V ring");

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// Cluster-wide barrier: this CTA's shared-memory writes before it are visible to the cluster's reads after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of this CTA's shared-memory location `p` as seen in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_rank(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ float2 ld_cluster_f2(uint32_t a) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ float2 ld_cluster_f2x(uint32_t a, float& z, float& w) {
  float2 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(z), "=f"(w) : "r"(a));
  return v;
}
// waits until at most n cp.async groups of this thread are pending (n in [0, SNS + 1])
__device__ __forceinline__ void cp_async_wait_n(int n) {
  switch (n) {
    case 0: cp_async_wait<0>(); break;
    case 1: cp_async_wait<1>(); break;
    case 2: cp_async_wait<2>(); break;
    case 3: cp_async_wait<3>(); break;
    default: cp_async_wait<4>(); break;
  }
}

constexpr int kMaxCluster = 16;

template <int H>
__global__ void __launch_bounds__(NWARP * 32) attn_short_kernel(const __grid_constant__ AttnArgs a,
                                                                 bf16* __restrict__ out) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  ShortSmem<H>& sm = *reinterpret_cast<ShortSmem<H>*>(smem_raw);
  constexpr int CH = H / 8, NKS = H / 16, NOT = H / 8;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = (int)cluster_size(), rank = (int)cluster_rank();
  const int bg = blockIdx.x / C;
  const int b = bg / a.nkv, g = bg % a.nkv, grp = a.nq / a.nkv, nrows = a.L * grp;
  pdl_trigger();

  int T = a.ctx_len[b];
  T = clamp_ctx(T, a.t_cap);
  const int n_keys = T + a.L;
  // tiles spread as evenly as the count allows, the extra ones to the last ranks: with 2048 + 16 keys every CTA
  // walks 2 full tiles and the last one also the 16-key tail, which takes the short tile math
  const int nt = ceil_div(n_keys, KT);
  const int t0 = rank * nt / C, t1 = (rank + 1) * nt / C, nts = t1 - t0;
  const int k_begin = t0 * KT, k_end = min(n_keys, t1 * KT);
  const float sl2 = rsqrtf((float)H) * 1.4426950408889634f;   // 1/sqrt(h) * log2(e): softmax in base 2

  const bf16* kctx = a.store + ((((size_t)a.layer * a.batch + b) * 2 + 0) * a.nkv + g) * (size_t)a.t_cap * H;
  const bf16* vctx = a.store + ((((size_t)a.layer * a.batch + b) * 2 + 1) * a.nkv + g) * (size_t)a.t_cap * H;
  const bf16* kbk = a.kblk + ((size_t)b * a.nkv + g) * a.L * H;
  const bf16* vbk = a.vblk + ((size_t)b * a.nkv + g) * a.L * H;

  auto load_kv = [&](int slot, int k0) {
    const uint32_t ks = smem_addr(sm.k[slot]), vs = smem_addr(sm.v[slot]);
    for (int idx = tid; idx < KT * CH; idx += NWARP * 32) {
      const int r = idx / CH, c = idx % CH, t = k0 + r;
      const bool ok = t < k_end;
      const bf16 *ksrc = kctx, *vsrc = vctx;
      if (ok) {
        if (t < T) {
          ksrc = kctx + (size_t)t * H + c * 8;
          vsrc = vctx + (size_t)t * H + c * 8;
        } else {
          ksrc = kbk + (size_t)(t - T) * H + c * 8;
          vsrc = vbk + (size_t)(t - T) * H + c * 8;
        }
      }
      cp_async16(swz<H>(ks, r, c), ksrc, ok);
      cp_async16(swz<H>(vs, r, c), vsrc, ok);
    }
    cp_async_commit();
  };

  // cp.async groups in commit order: the context-only tiles of the first ring (n_pre), Q, the rest of the first
  // ring, then one refill per consumed tile.  Tile i is group i + (i >= n_pre); Q is group n_pre.
  const int first = min(SNS, nts);
  int n_pre = 0;
  while (n_pre < first && (t0 + n_pre + 1) * KT <= T) {
    load_kv(n_pre, k_begin + n_pre * KT);
    n_pre++;
  }
  pdl_wait();
  const uint32_t q_s = smem_addr(sm.q);
  for (int idx = tid; idx < QT * CH; idx += NWARP * 32) {
    const int r = idx / CH, c = idx % CH;
    const bool ok = r < nrows;
    const bf16* src = a.q;
    if (ok) {
      const int j = r / grp, i = g * grp + r % grp;
      src = a.q + (((size_t)b * a.L + j) * a.nq + i) * H + c * 8;
    }
    cp_async16(swz<H>(q_s, r, c), src, ok);
  }
  cp_async_commit();
  for (int i = n_pre; i < first; i++) load_kv(i, k_begin + i * KT);
  int committed = first + 1;

  float o[NOT][4];
#pragma unroll
  for (int n = 0; n < NOT; n++) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // rows lane/4 and lane/4 + 8 of the warp's 16
  uint32_t qf[NKS][4];

  for (int it = 0; it < nts; it++) {
    const int slot = it % SNS;
    const int need = max(it + (it >= n_pre ? 1 : 0), n_pre);   // tile it and Q
    cp_async_wait_n(committed - 1 - need);
    __syncthreads();
    if (it == 0) {
      const int r = warp * 16 + (lane & 15);
#pragma unroll
      for (int kk = 0; kk < NKS; kk++)
        ldsm_x4(swz<H>(q_s, r, kk * 2 + (lane >> 4)), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
    }
    if (k_end - (k_begin + it * KT) <= 16)   // a tail of at most 16 keys: a quarter of the products
      attn_tile_math<H, 16>(smem_addr(sm.k[slot]), smem_addr(sm.v[slot]), qf, o, m0, m1, l0, l1, k_begin + it * KT,
                            k_end, lane, sl2);
    else
      attn_tile_math<H>(smem_addr(sm.k[slot]), smem_addr(sm.v[slot]), qf, o, m0, m1, l0, l1, k_begin + it * KT, k_end,
                        lane, sl2);
    __syncthreads();   // slot is refilled next
    if (it + SNS < nts) {
      load_kv(slot, k_begin + (it + SNS) * KT);
      committed++;
    }
  }
  cp_async_wait<0>();
  __syncthreads();

  // ---- this CTA's partial into its own shared memory ----
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  float* o_s = reinterpret_cast<float*>(sm.k);
  float2* ml_s = reinterpret_cast<float2*>(o_s + QT * H);
#pragma unroll
  for (int half = 0; half < 2; half++) {
    const int row = warp * 16 + (lane >> 2) + half * 8;
#pragma unroll
    for (int n = 0; n < NOT; n++)
      *reinterpret_cast<float2*>(o_s + row * H + n * 8 + (lane & 3) * 2) =
          make_float2(o[n][half * 2], o[n][half * 2 + 1]);
    if ((lane & 3) == 0) ml_s[row] = half ? make_float2(m1, l1) : make_float2(m0, l0);
  }
  cluster_sync();

  // ---- merge rows [rank * rpc, ...) over the C partials, in rank order ----
  constexpr int DPL = H / 32;   // output dims per lane (4 or 2)
  const int rpc = ceil_div(nrows, C);
  const int r0 = rank * rpc, r1 = min(nrows, r0 + rpc);
  for (int row = r0 + warp; row < r1; row += NWARP) {
    float mc[kMaxCluster], lc[kMaxCluster], ox[kMaxCluster][DPL];
#pragma unroll
    for (int c = 0; c < kMaxCluster; c++) {   // every load issued before any use
      if (c < C) {
        const float2 v = ld_cluster_f2(map_rank(ml_s + row, c));
        mc[c] = v.x;
        lc[c] = v.y;
        if constexpr (DPL == 4) {
          float z, w;
          const float2 xy = ld_cluster_f2x(map_rank(o_s + row * H + lane * DPL, c), z, w);
          ox[c][0] = xy.x;
          ox[c][1] = xy.y;
          ox[c][2] = z;
          ox[c][3] = w;
        } else {
          const float2 xy = ld_cluster_f2(map_rank(o_s + row * H + lane * DPL, c));
          ox[c][0] = xy.x;
          ox[c][1] = xy.y;
        }
      }
    }
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < kMaxCluster; c++) {
      if (c < C) {
        mc[c] = lc[c] > 0.f ? mc[c] : -INFINITY;
        mx = fmaxf(mx, mc[c]);
      }
    }
    float den = 0.f, num[DPL];
#pragma unroll
    for (int e = 0; e < DPL; e++) num[e] = 0.f;
#pragma unroll
    for (int c = 0; c < kMaxCluster; c++) {
      if (c < C && mc[c] != -INFINITY) {
        const float wgt = exp2f(mc[c] - mx);
        den += lc[c] * wgt;
#pragma unroll
        for (int e = 0; e < DPL; e++) num[e] += ox[c][e] * wgt;
      }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    const int j = row / grp, i = g * grp + row % grp;
    bf16* dst = out + (((size_t)b * a.L + j) * a.nq + i) * H + lane * DPL;
#pragma unroll
    for (int e = 0; e < DPL; e += 2)
      *reinterpret_cast<__nv_bfloat162*>(dst + e) = __floats2bfloat162_rn(num[e] * inv, num[e + 1] * inv);
  }
  cluster_sync();   // every partial stays in place until the whole cluster has read it
}

int g_short_cluster = 0;   // cluster size chosen at initialisation (16 where the GPU schedules it, else 8)

template <int H>
cudaError_t launch_short(const AttnArgs& a, bf16* out, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.batch * a.nkv * g_short_cluster);
  cfg.blockDim = dim3(NWARP * 32);
  cfg.dynamicSmemBytes = sizeof(ShortSmem<H>);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = g_short_cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  count_launch();
  return cudaLaunchKernelEx(&cfg, attn_short_kernel<H>, a, out);
}

template <int H>
cudaError_t init_short() {
  cudaError_t e = cudaFuncSetAttribute(attn_short_kernel<H>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sizeof(ShortSmem<H>));
  if (e == cudaSuccess) e = cudaFuncSetAttribute(attn_short_kernel<H>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

// Largest cluster (16, else 8) of which the GPU can hold at least one.
template <int H>
int pick_cluster() {
  for (int c : {16, 8}) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(c);
    cfg.blockDim = dim3(NWARP * 32);
    cfg.dynamicSmemBytes = sizeof(ShortSmem<H>);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, attn_short_kernel<H>, &cfg) == cudaSuccess && n > 0) return c;
    cudaGetLastError();
  }
  return 8;
}

}  // namespace

bool attn_short_supported(int head_dim, int L, int nq, int nkv) {
  return (head_dim == 128 || head_dim == 64) && L * (nq / nkv) <= QT;
}

cudaError_t attn_short_init_attributes() {
  cudaError_t e = init_short<128>();
  if (e == cudaSuccess) e = init_short<64>();
  if (e == cudaSuccess) g_short_cluster = pick_cluster<128>();
  return e;
}

cudaError_t launch_attention_short(const AttnArgs& a, bf16* out, cudaStream_t st) {
  if (!attn_short_supported(a.head_dim, a.L, a.nq, a.nkv) || g_short_cluster < 1) return cudaErrorInvalidValue;
  return a.head_dim == 128 ? launch_short<128>(a, out, st) : launch_short<64>(a, out, st);
}

}  // namespace fpd

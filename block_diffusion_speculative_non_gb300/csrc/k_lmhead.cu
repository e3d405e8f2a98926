// k_lmhead.cu — a8: planning, final-norm gather and decoding around the tensor-core LM head.
//
// VFlash paper (zh), §2.5 "Inference": per-position constraints limit coordinates and delimiters to their
// legal vocabulary and act on logits, adding no neural compute.  Here illegal columns are never computed at
// all: positions are grouped by class on the device (a stable counting sort), and work items pair one
// 128-id tile of one legal id range with one tile of the positions of that range's class (k_gemm_tc.cu,
// EPI_ARGMAX).  Each work item folds its (logit, id) maxima into a per-position 64-bit word with atomicMax,
// where the packing makes a larger word mean a larger fp32 logit and, for equal logits, a smaller id, so the
// result is the argmax with lowest-id ties whatever the order of work items.
#include "fpd_kernels.cuh"

namespace fpd {

__device__ __forceinline__ int block_excl_scan_flag(int flag, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const unsigned m = __ballot_sync(0xffffffffu, flag);
  const int in_warp = __popc(m & ((1u << lane) - 1u));
  __syncthreads();
  if (lane == 0) warp_tot[w] = __popc(m);
  __syncthreads();
  if (w == 0) {
    int v = lane < nw ? warp_tot[lane] : 0, incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane < nw) warp_tot[lane] = incl - v;
    if (lane == 31) *total = incl;
  }
  __syncthreads();
  return warp_tot[w] + in_warp;
}

// One CTA: rows grouped by class (stable), the work-item list, argmax words cleared.
__global__ void __launch_bounds__(1024) lm_plan_kernel(LmPlan p, const int16_t* __restrict__ pos_class,
                                                        int* __restrict__ rows_sorted, int* __restrict__ inv_sorted,
                                                        int* __restrict__ class_row_off, int4* __restrict__ items,
                                                        int* __restrict__ n_items,
                                                        unsigned long long* __restrict__ packed,
                                                        unsigned long long* __restrict__ packed2, int max_items) {
  pdl_trigger();
  pdl_wait();
  __shared__ int warp_tot[32];
  __shared__ int s_total;
  __shared__ int s_off[FPD_MAX_CLASSES + 1];
  __shared__ int s_item_off[FPD_MAX_RANGES + 1];
  const int tid = threadIdx.x;
  for (int r = tid; r < p.n_rows; r += blockDim.x) {
    packed[r] = 0ull;
    packed2[r] = 0ull;
    inv_sorted[r] = -1;
    rows_sorted[r] = -1;
  }
  __syncthreads();
  if (!pos_class) {
    for (int r = tid; r < p.n_rows; r += blockDim.x) {
      rows_sorted[r] = r;
      inv_sorted[r] = r;
    }
    if (tid == 0) { s_off[0] = 0; s_off[1] = p.n_rows; }
  } else {
    int base = 0;
    for (int c = 0; c < p.n_class; c++) {
      if (tid == 0) s_off[c] = base;
      for (int r0 = 0; r0 < p.n_rows; r0 += blockDim.x) {
        const int r = r0 + tid;
        int cls = -1;
        if (r < p.n_rows) {
          const int b = r / (p.L - 1), j = r % (p.L - 1) + 1;
          cls = pos_class[(size_t)b * p.L + j];
          if (c == 0 && (cls < 0 || cls >= p.n_class)) record_check(kCheckBadClass);
        }
        const int flag = cls == c;
        const int pos = block_excl_scan_flag(flag, warp_tot, &s_total);
        if (flag) {
          rows_sorted[base + pos] = r;
          inv_sorted[r] = base + pos;
        }
        base += s_total;
        __syncthreads();
      }
    }
    if (tid == 0) s_off[p.n_class] = base;
  }
  __syncthreads();
  const int nc = pos_class ? p.n_class : 1;
  if (tid <= nc) class_row_off[tid] = s_off[tid];
  if (tid == 0) {
    int acc = 0;
    for (int q = 0; q < p.n_range; q++) {
      const int c = pos_class ? p.range_class[q] : 0;
      const int cnt = s_off[c + 1] - s_off[c];
      acc += ceil_div(cnt, p.rt) * ceil_div(p.range_hi[q] - p.range_lo[q], p.ct);
      s_item_off[q + 1] = acc;
    }
    s_item_off[0] = 0;
    if (acc > max_items) record_check(kCheckNoLegalId);
    *n_items = acc < max_items ? acc : max_items;
  }
  __syncthreads();
  // items of one range are id-tile major: the row tiles of one 128-id weight tile are consecutive, so the
  // persistent CTAs working on them at the same time share that weight tile through L2
  for (int q = 0; q < p.n_range; q++) {
    const int c = pos_class ? p.range_class[q] : 0;
    const int cnt = s_off[c + 1] - s_off[c];
    const int rowtiles = ceil_div(cnt, p.rt);
    const int n_q = s_item_off[q + 1] - s_item_off[q];
    for (int i = tid; i < n_q; i += blockDim.x) {
      const int t = i / rowtiles, k = i % rowtiles;
      const int dst = s_item_off[q] + i;
      if (dst < max_items)
        items[dst] = make_int4(q, p.range_lo[q] + t * p.ct, s_off[c] + k * p.rt, min(p.rt, cnt - k * p.rt));
    }
  }
}

cudaError_t launch_lm_plan(const LmPlan& p, const int16_t* pos_class, int* rows_sorted, int* inv_sorted,
                           int* class_row_off, int4* items, int* n_items, unsigned long long* packed,
                           unsigned long long* packed2, int max_items, cudaStream_t st) {
  return launch_k(lm_plan_kernel, 1, 1024, 0, st, p, pos_class, rows_sorted, inv_sorted, class_row_off, items, n_items,
                  packed, packed2, max_items);
}

// ---- final RMSNorm into sorted order -------------------------------------------------------------------------------
__global__ void rmsnorm_gather_kernel(bf16* __restrict__ out, const bf16* __restrict__ in, const bf16* __restrict__ g,
                                      const int* __restrict__ rows_sorted, int d, float eps, int L) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[32];
  const int i = blockIdx.x;
  const int r = rows_sorted[i];
  uint4* dst = reinterpret_cast<uint4*>(out + (size_t)i * d);
  if (r < 0) {   // slot past the placed rows (a position with an invalid class): zeros
    for (int k = threadIdx.x; k < d / 8; k += blockDim.x) dst[k] = make_uint4(0, 0, 0, 0);
    return;
  }
  const int rin = (r / (L - 1)) * L + r % (L - 1) + 1;   // drop the anchor row of every block
  const uint4* src = reinterpret_cast<const uint4*>(in + (size_t)rin * d);
  float ss = 0.f;
  for (int k = threadIdx.x; k < d / 8; k += blockDim.x) {
    uint4 u = src[k];
    const bf16* e = reinterpret_cast<const bf16*>(&u);
#pragma unroll
    for (int t = 0; t < 8; t++) {
      const float f = __bfloat162float(e[t]);
      ss += f * f;
    }
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = (threadIdx.x & 31) < (blockDim.x >> 5) ? red[threadIdx.x & 31] : 0.f;
  tot = warp_sum(tot);
  const float inv = rsqrtf(tot / (float)d + eps);
  const uint4* gs = reinterpret_cast<const uint4*>(g);
  for (int k = threadIdx.x; k < d / 8; k += blockDim.x) {
    uint4 u = src[k], gu = gs[k], o;
    const bf16* e = reinterpret_cast<const bf16*>(&u);
    const bf16* ge = reinterpret_cast<const bf16*>(&gu);
    bf16* oe = reinterpret_cast<bf16*>(&o);
#pragma unroll
    for (int t = 0; t < 8; t++) oe[t] = __float2bfloat16_rn(__bfloat162float(e[t]) * inv * __bfloat162float(ge[t]));
    dst[k] = o;
  }
}

cudaError_t launch_rmsnorm_gather(bf16* out, const bf16* in, const bf16* g, const int* rows_sorted, int rows, int d,
                                  float eps, int L, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  return launch_k(rmsnorm_gather_kernel, rows, 256, 0, st, out, in, g, rows_sorted, d, eps, L);
}

// ---- decode the packed argmax words into ids (and the top-2 margin when asked) ------------------------------------
__device__ __forceinline__ float unpack_value(unsigned long long p) {
  uint32_t u = (uint32_t)(p >> 32);
  u = (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u;
  return __uint_as_float(u);
}

__global__ void lm_decode_kernel(int32_t* __restrict__ tokens, float* __restrict__ margin,
                                 const unsigned long long* __restrict__ packed,
                                 const unsigned long long* __restrict__ packed2, const int* __restrict__ inv_sorted,
                                 int n) {
  pdl_trigger();
  pdl_wait();
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < n; r += gridDim.x * blockDim.x) {
    const int i = inv_sorted[r];
    const unsigned long long p = i >= 0 ? packed[i] : 0ull;
    if (!p) record_check(kCheckNoLegalId);
    tokens[r] = p ? unpack_argmax_id(p) : -1;
    if (margin) {
      const unsigned long long p2 = i >= 0 ? packed2[i] : 0ull;
      margin[r] = !p ? 0.f : (p2 ? (float)((double)unpack_value(p) - (double)unpack_value(p2)) : INFINITY);
    }
  }
}

// ---- cross-position rule (f3): off-screen coordinates in pairs -----------------------------------------------
// VFlash paper (zh) §2.5: a cross-position rule pairs off-screen coordinates, on the computed logits.  One warp per
// (request, pair): o_x = z_x . W[off_id] (fp32, fixed order) for both positions, a_x = the best legal logit other
// than off_id (the top-1 word, or the top-2 word when the top-1 is off_id); both positions take off_id when
// o_p + o_q > a_p + a_q, else their best other id.  The margin of both becomes the smaller of their own and
// |(o_p + o_q) - (a_p + a_q)|.
__global__ void pair_offscreen_kernel(int32_t* __restrict__ tokens, float* __restrict__ margin,
                                      const unsigned long long* __restrict__ packed,
                                      const unsigned long long* __restrict__ packed2,
                                      const int* __restrict__ inv_sorted, const bf16* __restrict__ z,
                                      const bf16* __restrict__ w_lm, int d, int L, int B, PairTable pt) {
  pdl_trigger();
  pdl_wait();
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (gw >= B * pt.n) return;
  const int b = gw / pt.n, k = gw % pt.n;
  const int rp = b * (L - 1) + pt.p[k] - 1, rq = b * (L - 1) + pt.q[k] - 1;
  const int ip = inv_sorted[rp], iq = inv_sorted[rq];
  if (ip < 0 || iq < 0) return;
  const bf16* wo = w_lm + (size_t)pt.off_id * d;
  const bf16* zp = z + (size_t)ip * d;
  const bf16* zq = z + (size_t)iq * d;
  float op = 0.f, oq = 0.f;
  for (int c = lane * 8; c < d; c += 256) {
    const uint4 uw = *reinterpret_cast<const uint4*>(wo + c), up = *reinterpret_cast<const uint4*>(zp + c),
                uq = *reinterpret_cast<const uint4*>(zq + c);
    const __nv_bfloat162* ew = reinterpret_cast<const __nv_bfloat162*>(&uw);
    const __nv_bfloat162* ep = reinterpret_cast<const __nv_bfloat162*>(&up);
    const __nv_bfloat162* eq = reinterpret_cast<const __nv_bfloat162*>(&uq);
#pragma unroll
    for (int e = 0; e < 4; e++) {
      const float2 fw = __bfloat1622float2(ew[e]), fp = __bfloat1622float2(ep[e]), fq = __bfloat1622float2(eq[e]);
      op = fmaf(fp.x, fw.x, fmaf(fp.y, fw.y, op));
      oq = fmaf(fq.x, fw.x, fmaf(fq.y, fw.y, oq));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    op += __shfl_xor_sync(0xffffffffu, op, o);
    oq += __shfl_xor_sync(0xffffffffu, oq, o);
  }
  if (lane != 0) return;
  unsigned long long bp = packed[ip], bq = packed[iq];
  if (bp && unpack_argmax_id(bp) == pt.off_id) bp = packed2[ip];
  if (bq && unpack_argmax_id(bq) == pt.off_id) bq = packed2[iq];
  if (!bp || !bq) return;   // a position whose only legal id is off_id keeps it
  const float on = unpack_value(bp) + unpack_value(bq), off = op + oq;
  const bool take_off = off > on;
  tokens[rp] = take_off ? pt.off_id : unpack_argmax_id(bp);
  tokens[rq] = take_off ? pt.off_id : unpack_argmax_id(bq);
  if (margin) {
    const float gap = fabsf(off - on);
    margin[rp] = fminf(margin[rp], gap);
    margin[rq] = fminf(margin[rq], gap);
  }
}

cudaError_t launch_pair_offscreen(int32_t* tokens, float* margin, const unsigned long long* packed,
                                  const unsigned long long* packed2, const int* inv_sorted, const bf16* z,
                                  const bf16* w_lm, int d, int L, int B, const PairTable& pt, cudaStream_t st) {
  if (pt.n <= 0) return cudaSuccess;
  const int warps = B * pt.n;
  return launch_k(pair_offscreen_kernel, ceil_div(warps, 8), 256, 0, st, tokens, margin, packed, packed2, inv_sorted,
                  z, w_lm, d, L, B, pt);
}

cudaError_t launch_lm_decode(int32_t* tokens, float* margin, const unsigned long long* packed,
                             const unsigned long long* packed2, const int* inv_sorted, int n, cudaStream_t st) {
  const int grid = std::min(ceil_div(n, 256), 1024);
  return launch_k(lm_decode_kernel, grid, 256, 0, st, tokens, margin, packed, packed2, inv_sorted, n);
}

}  // namespace fpd

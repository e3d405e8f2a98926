#pragma once

#include "fpd_kernels.cuh"

// attn_body.cuh — the attention work units (one query tile over one KV split; the merge of the splits of one
// (row, head)), written as device functions of 128 threads with a caller-supplied barrier.  Internal to libfpd.
//
// VFlash paper (zh), §2.1: the fused target features enter every drafter layer as keys and values, and
// the masked positions are predicted in one BIDIRECTIONAL pass — so there is no mask at all inside a
// request: every block query sees all ctx_len[b] context keys of its layer and all L block keys.
// VFlash blog, "Key claims": the drafter is a non-causal transformer.
//
// Work split: (query tile of 64 rows of one kv-head group) x (request, kv head) x (KV split).  The rows of a
// tile are the L positions x H_q/H_kv q heads that share one kv head, so every K/V row loaded is used by the
// whole group.  Four warps each own 16 query rows; Q stays in registers as mma fragments; K/V tiles of 64
// keys are staged in shared memory with cp.async (double buffered, 16-byte chunks XOR-swizzled so ldmatrix
// is conflict free); S = Q K^T and O += P V run on the tensor cores (mma.sync m16n8k16, bf16 in, fp32
// accumulate; P enters the second product as two bf16 terms hi + lo, see split_bf16x2); the online softmax
// works in base 2 on the fp32 accumulators.  With one split the CTA writes the normalised bf16 output; with several it writes
// an unnormalised partial (o, m, l) and a merge kernel combines the splits in fixed order (deterministic,
// no atomics).

namespace fpd {
namespace attn {

constexpr int QT = 64, KT = 64, NWARP = 4;

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;   // 0 source bytes: the 16 destination bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// 2^x on the special-function unit (ex2.approx, flush-to-zero): relative error near 2^-22 for the arguments used
// here (<= 0), and 2^-inf = 0 for masked keys.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Tile of rows x H bf16 in shared memory; 16-byte chunk c of row r lives at chunk c ^ (r & 7).
template <int H>
__device__ __forceinline__ uint32_t swz(uint32_t base, int r, int c) {
  return base + (uint32_t)(r * H * 2 + ((c ^ (r & 7)) << 4));
}

template <int H>
struct Smem {
  bf16 q[QT * H];
  bf16 k[2][KT * H];
  bf16 v[2][KT * H];
};

// One tile of NK keys (64, or 16 for a short last tile: a quarter of the products) of the online softmax for one
// warp's 16 query rows (rows lane/4 and lane/4 + 8 of its m16 fragment): S = Q K^T on mma.sync from the swizzled K
// tile at ks, keys at or past k_end masked, running maximum (m0, m1) and sum (l0, l1) in base 2, O += (P_hi + P_lo)
// V from the V tile at vs.  k0: the tile's first key.
template <int H, int NK = KT>
__device__ __forceinline__ void attn_tile_math(uint32_t ks, uint32_t vs, const uint32_t (&qf)[H / 16][4],
                                               float (&o)[H / 8][4], float& m0, float& m1, float& l0, float& l1,
                                               int k0, int k_end, int lane, float sl2) {
  constexpr int NKS = H / 16;   // k-steps over the head dimension
  constexpr int NOT = H / 8;    // 8-wide n-tiles of O
  // ---- S = Q K^T: 16 rows x NK keys per warp ----
  static_assert(NK % 16 == 0 && NK <= KT, "tile keys");
  float s[NK / 8][4];
#pragma unroll
  for (int n = 0; n < NK / 8; n++) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
  for (int kp = 0; kp < NK / 16; kp++) {
#pragma unroll
    for (int kk = 0; kk < NKS; kk++) {
      // 8x8 matrices: (keys +0..7, dims lo), (keys +0..7, dims hi), (keys +8..15, dims lo), (keys +8..15, dims hi)
      const int key = kp * 16 + (lane & 7) + ((lane >> 4) << 3);
      const int c = kk * 2 + ((lane >> 3) & 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4(swz<H>(ks, key, c), b0, b1, b2, b3);
      mma_bf16(s[2 * kp], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b0, b1);
      mma_bf16(s[2 * kp + 1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b2, b3);
    }
  }
  // ---- online softmax (base 2) ----
  if (k0 + NK > k_end) {   // a partial tile (warp-uniform): keys past the end get 2^-inf = 0
#pragma unroll
    for (int n = 0; n < NK / 8; n++) {
      const int key = k0 + n * 8 + (lane & 3) * 2;
      if (key >= k_end) s[n][0] = s[n][2] = -INFINITY;
      if (key + 1 >= k_end) s[n][1] = s[n][3] = -INFINITY;
    }
  }
  float mx0 = -INFINITY, mx1 = -INFINITY;   // raw maxima, scaled once below (sl2 > 0)
#pragma unroll
  for (int n = 0; n < NK / 8; n++) {
    mx0 = fmaxf(mx0, fmaxf(s[n][0], s[n][1]));
    mx1 = fmaxf(mx1, fmaxf(s[n][2], s[n][3]));
  }
  mx0 *= sl2;
  mx1 *= sl2;
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
  const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);   // finite: every tile holds at least one valid key
  const float c0 = m0 == -INFINITY ? 0.f : ex2_approx(m0 - mn0);
  const float c1 = m1 == -INFINITY ? 0.f : ex2_approx(m1 - mn1);
  m0 = mn0;
  m1 = mn1;
  float ps0 = 0.f, ps1 = 0.f;
  const float n0 = -mn0, n1 = -mn1;
#pragma unroll
  for (int n = 0; n < NK / 8; n++) {
    s[n][0] = ex2_approx(fmaf(s[n][0], sl2, n0));
    s[n][1] = ex2_approx(fmaf(s[n][1], sl2, n0));
    s[n][2] = ex2_approx(fmaf(s[n][2], sl2, n1));
    s[n][3] = ex2_approx(fmaf(s[n][3], sl2, n1));
    ps0 += s[n][0] + s[n][1];
    ps1 += s[n][2] + s[n][3];
  }
  l0 = l0 * c0 + ps0;
  l1 = l1 * c1 + ps1;
#pragma unroll
  for (int n = 0; n < NOT; n++) {
    o[n][0] *= c0;
    o[n][1] *= c0;
    o[n][2] *= c1;
    o[n][3] *= c1;
  }
  // ---- O += (P_hi + P_lo) V ----
#pragma unroll
  for (int kk = 0; kk < NK / 16; kk++) {
    uint32_t h0, h1, h2, h3, l0_, l1_, l2_, l3_;
    split_bf16x2(s[2 * kk][0], s[2 * kk][1], h0, l0_);
    split_bf16x2(s[2 * kk][2], s[2 * kk][3], h1, l1_);
    split_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1], h2, l2_);
    split_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3], h3, l3_);
#pragma unroll
    for (int np = 0; np < NOT / 2; np++) {
      // transposed 8x8 matrices: (keys +0..7, dims lo), (keys +8..15, dims lo), (keys +0..7, dims hi), (keys +8..15, dims hi)
      const int key = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
      const int c = np * 2 + (lane >> 4);
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(swz<H>(vs, key, c), b0, b1, b2, b3);
      mma_bf16(o[2 * np], h0, h1, h2, h3, b0, b1);
      mma_bf16(o[2 * np + 1], h0, h1, h2, h3, b2, b3);
      mma_bf16(o[2 * np], l0_, l1_, l2_, l3_, b0, b1);
      mma_bf16(o[2 * np + 1], l0_, l1_, l2_, l3_, b2, b3);
    }
  }
}

// One (query tile, request x kv head, KV split) unit of the attention, run by 128 threads (tid 0..127) that
// synchronise with `sync` (the whole CTA in the standalone kernel, a named barrier inside the persistent kernel).
template <int H, class Sync>
__device__ __forceinline__ void attn_tile(const AttnArgs& a, bf16* __restrict__ out, int qt, int bg, int split,
                                          int tid, unsigned char* smem_raw, Sync sync) {
  constexpr int CH = H / 8;     // 16-byte chunks per row
  constexpr int NKS = H / 16;   // k-steps over the head dimension
  constexpr int NOT = H / 8;    // 8-wide n-tiles of O
  Smem<H>& sm = *reinterpret_cast<Smem<H>*>(smem_raw);
  const int warp = tid >> 5, lane = tid & 31;
  const int b = bg / a.nkv, g = bg % a.nkv;
  const int grp = a.nq / a.nkv, nrows = a.L * grp;
  int T = a.ctx_len[b];
  T = clamp_ctx(T, a.t_cap);
  const int n_keys = T + a.L;
  const int k_begin = split * a.chunk, k_end = min(n_keys, k_begin + a.chunk);
  const float sl2 = rsqrtf((float)H) * 1.4426950408889634f;   // 1/sqrt(h) * log2(e): softmax in base 2

  const bf16* kctx = a.store + ((((size_t)a.layer * a.batch + b) * 2 + 0) * a.nkv + g) * (size_t)a.t_cap * H;
  const bf16* vctx = a.store + ((((size_t)a.layer * a.batch + b) * 2 + 1) * a.nkv + g) * (size_t)a.t_cap * H;
  const bf16* kbk = a.kblk + ((size_t)b * a.nkv + g) * a.L * H;
  const bf16* vbk = a.vblk + ((size_t)b * a.nkv + g) * a.L * H;

  const uint32_t q_s = smem_addr(sm.q);
  for (int idx = tid; idx < QT * CH; idx += NWARP * 32) {
    const int r = idx / CH, c = idx % CH, qi = qt * QT + r;
    const bool ok = qi < nrows;
    const bf16* src = a.q;
    if (ok) {
      const int j = qi / grp, i = g * grp + qi % grp;
      src = a.q + (((size_t)b * a.L + j) * a.nq + i) * H + c * 8;
    }
    cp_async16(swz<H>(q_s, r, c), src, ok);
  }
  cp_async_commit();

  auto load_kv = [&](int buf, int k0) {
    const uint32_t ks = smem_addr(sm.k[buf]), vs = smem_addr(sm.v[buf]);
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

  const int n_tiles = k_end > k_begin ? (k_end - k_begin + KT - 1) / KT : 0;
  if (n_tiles > 0) load_kv(0, k_begin);

  float o[NOT][4];
#pragma unroll
  for (int n = 0; n < NOT; n++) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // rows lane/4 and lane/4 + 8 of the warp
  uint32_t qf[NKS][4];

  if (n_tiles > 0)
    cp_async_wait<1>();   // Q has landed; the first K/V tile may still be in flight
  else
    cp_async_wait<0>();
  sync();
  {
    const int r = warp * 16 + (lane & 15);
#pragma unroll
    for (int kk = 0; kk < NKS; kk++) ldsm_x4(swz<H>(q_s, r, kk * 2 + (lane >> 4)), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
  }

  for (int it = 0; it < n_tiles; it++) {
    const int buf = it & 1, k0 = k_begin + it * KT;
    if (it + 1 < n_tiles) {
      load_kv(buf ^ 1, k0 + KT);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    sync();
    attn_tile_math<H>(smem_addr(sm.k[buf]), smem_addr(sm.v[buf]), qf, o, m0, m1, l0, l1, k0, k_end, lane, sl2);
    sync();   // this buffer is refilled by the next iteration's prefetch
  }

  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const int rlo = qt * QT + warp * 16 + (lane >> 2);
#pragma unroll
  for (int half = 0; half < 2; half++) {
    const int qi = rlo + half * 8;
    if (qi >= nrows) continue;
    const int j = qi / grp, i = g * grp + qi % grp;
    const size_t row = (size_t)b * a.L + j;
    const float m = half ? m1 : m0, l = half ? l1 : l0;
    if (a.splits == 1) {
      const float inv = l > 0.f ? 1.f / l : 0.f;
      bf16* dst = out + (row * a.nq + i) * H + (lane & 3) * 2;
#pragma unroll
      for (int n = 0; n < NOT; n++)
        *reinterpret_cast<__nv_bfloat162*>(dst + n * 8) =
            __floats2bfloat162_rn(o[n][half * 2] * inv, o[n][half * 2 + 1] * inv);
    } else {
      float* dst = a.o_part + (((size_t)split * a.rows + row) * a.nq + i) * H + (lane & 3) * 2;
#pragma unroll
      for (int n = 0; n < NOT; n++)
        *reinterpret_cast<float2*>(dst + n * 8) = make_float2(o[n][half * 2], o[n][half * 2 + 1]);
      if ((lane & 3) == 0) a.ml[((size_t)split * a.rows + row) * a.nq + i] = make_float2(m, l);
    }
  }
}

// Combines the splits of one (row, q head) in one warp; running maxima are in base-2 units.  Lane s of a 32-split
// chunk holds split s's (m, l): the warp takes the maximum M of the split maxima (empty splits, l = 0, carry no
// weight and their partial is never read), the denominator sum_s l_s 2^(m_s - M) in a fixed xor tree per chunk,
// chunks in order; then every lane sums its H/32 columns over the splits in split order (8 splits' loads in flight
// at a time) and divides by the denominator.  Bit-reproducible.
template <int H>
__device__ __forceinline__ void attn_merge_warp(bf16* __restrict__ out, const float* __restrict__ o_part,
                                                const float2* __restrict__ ml, int nsplit, int rows, int nq, int r,
                                                int i, int lane) {
  constexpr int DPL = H / 32;
  const size_t mstride = (size_t)rows * nq;
  const float2* mp = ml + (size_t)r * nq + i;
  float mx = -INFINITY;
  for (int s0 = 0; s0 < nsplit; s0 += 32) {
    const int s = s0 + lane;
    const float2 v = s < nsplit ? __ldcg(mp + (size_t)s * mstride) : make_float2(-INFINITY, 0.f);
    mx = fmaxf(mx, warp_max(v.y > 0.f ? v.x : -INFINITY));
  }
  float den = 0.f;
  for (int s0 = 0; s0 < nsplit; s0 += 32) {
    const int s = s0 + lane;
    const float2 v = s < nsplit ? __ldcg(mp + (size_t)s * mstride) : make_float2(-INFINITY, 0.f);
    den += warp_sum(v.y > 0.f ? v.y * exp2f(v.x - mx) : 0.f);
  }
  const float* op = o_part + ((size_t)r * nq + i) * H + lane * DPL;
  const size_t ostride = mstride * H;
  float num[DPL];
#pragma unroll
  for (int e = 0; e < DPL; e++) num[e] = 0.f;
  for (int s0 = 0; s0 < nsplit; s0 += 8) {
    float t[8][DPL], wgt[8];
#pragma unroll
    for (int u = 0; u < 8; u++) {
      const int s = s0 + u;
      wgt[u] = 0.f;
#pragma unroll
      for (int e = 0; e < DPL; e++) t[u][e] = 0.f;
      if (s < nsplit) {
        const float2 v = __ldcg(mp + (size_t)s * mstride);
        wgt[u] = v.y > 0.f ? exp2f(v.x - mx) : 0.f;
      }
      if (wgt[u] != 0.f) {
        if constexpr (DPL == 4) {
          const float4 f = __ldcg(reinterpret_cast<const float4*>(op + (size_t)s * ostride));
          t[u][0] = f.x;
          t[u][1] = f.y;
          t[u][2] = f.z;
          t[u][3] = f.w;
        } else {
          const float2 f = __ldcg(reinterpret_cast<const float2*>(op + (size_t)s * ostride));
          t[u][0] = f.x;
          t[u][1] = f.y;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 8; u++)
      if (wgt[u] != 0.f)
#pragma unroll
        for (int e = 0; e < DPL; e++) num[e] += t[u][e] * wgt[u];
  }
  bf16* dst = out + ((size_t)r * nq + i) * H + lane * DPL;
#pragma unroll
  for (int e = 0; e < DPL; e += 2)
    *reinterpret_cast<__nv_bfloat162*>(dst + e) =
        __floats2bfloat162_rn(den > 0.f ? num[e] / den : 0.f, den > 0.f ? num[e + 1] / den : 0.f);
}

}  // namespace attn
}  // namespace fpd

// fewtok_common.cuh — device building blocks of the few-token path (at most 16 block positions per call) used by
// the weight-streaming kernels of k_stream.cu.  Internal to libfpd.
//
// Conventions of that path: the 16 token rows are the N = 16 operand of tcgen05.mma and the weight tile is the
// M = 128 operand, so an accumulator holds 128 output features (TMEM lanes) x 16 tokens (columns); warps 2..5
// (128 threads, "epilogue threads") own TMEM lane quarters (warp & 3) and synchronise with named barrier 1.
#pragma once

#include "fpd_kernels.cuh"
#include <cuda_fp8.h>

#include "tc_primitives.cuh"

namespace fpd {
namespace fewtok {

constexpr int SBM = 128, SBK = 64, SBN = 16, SUK = 16;
constexpr int W_ATOM = SBM * SBK * 2;   // 16 KB: 128 weight rows x 64 K, 128-byte swizzle
constexpr int X_ATOM = SBN * SBK * 2;   // 2 KB: 16 tokens x 64 K
constexpr int G_ATOM = SBK * 2;         // 128 B of RMSNorm gain per K atom
constexpr int kEpiScratch = SBN * SBM * 4;   // 8 KB: one fp32 output tile, token-major [16][128]

__device__ __forceinline__ float bf(const bf16 v) { return __bfloat162float(v); }

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// the value half of pack_argmax
__device__ __forceinline__ float unpack_argmax_val(unsigned long long p) {
  uint32_t u = (uint32_t)(p >> 32);
  u = (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u;
  return __uint_as_float(u);
}

// (a1, a2) := the two largest of {a1, a2, b1, b2}, given a1 >= a2 and b1 >= b2 (packed words are distinct)
__device__ __forceinline__ void top2_merge(unsigned long long& a1, unsigned long long& a2, unsigned long long b1,
                                           unsigned long long b2) {
  const unsigned long long hi = a1 > b1 ? a1 : b1, lo = a1 > b1 ? b1 : a1;
  const unsigned long long s = a2 > b2 ? a2 : b2;
  a1 = hi;
  a2 = lo > s ? lo : s;
}

// 1/rms per token from per-(part, token) sums of squares left by the residual epilogues ([n_ss][16], fixed
// summation order), staged through `stage` (n_ss * 16 floats).  Result in s_inv[16] after the next epi_bar.
__device__ __forceinline__ void inv_from_partials(const float* ss_in, int n_ss, int d, float eps, float* stage,
                                                  float* s_inv, int et) {
  for (int i = et; i < n_ss * SBN; i += 128) stage[i] = __ldcg(ss_in + i);
  epi_bar();
  if (et < SBN) {
    float ss = 0.f;
    for (int t = 0; t < n_ss; t++) ss += stage[t * SBN + et];
    s_inv[et] = rsqrtf(ss / (float)d + eps);
  }
}

// 1/rms per token over whole rows already in the activation region (LM head: all K atoms resident).  Thread et
// sums the squares of row j = et / 8, physical 16-byte chunk et % 8 of every atom (the swizzle permutes chunks
// within a row, so the row sum is unaffected), then the 8 threads of a row combine in a fixed xor tree.
__device__ __forceinline__ void inv_from_rows(const uint8_t* act, int nkb, int d, float eps, float* s_inv, int et) {
  const int j = et >> 3, pc = et & 7;
  float ss = 0.f;
#pragma unroll 8
  for (int a = 0; a < nkb; a++) {
    const uint4 u = *reinterpret_cast<const uint4*>(act + a * X_ATOM + j * 128 + (pc << 4));
    const __nv_bfloat162* e = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int k = 0; k < 4; k++) {
      const float2 f = __bfloat1622float2(e[k]);
      ss += f.x * f.x + f.y * f.y;
    }
  }
  ss += __shfl_xor_sync(0xffffffffu, ss, 1);
  ss += __shfl_xor_sync(0xffffffffu, ss, 2);
  ss += __shfl_xor_sync(0xffffffffu, ss, 4);
  if (pc == 0) s_inv[j] = rsqrtf(ss / (float)d + eps);
}

// xn = bf16(x * inv[j] * g[k]) in place over the TMA-loaded atoms [a0, a0 + na) (na <= 4, 16 rows each): thread et
// takes row j = et / 8 and physical 16-byte chunk pc = et % 8 of every atom, which holds logical chunk pc ^ (j & 7)
// (128-byte swizzle).  gbuf: the gain slice, 128 bytes per atom.  Rows past the call's tokens are zero and stay so.
__device__ __forceinline__ void norm_atoms(uint8_t* act, const uint8_t* gbuf, const float* s_inv, int a0, int na,
                                           int et) {
  const int j = et >> 3, pc = et & 7, q = pc ^ (j & 7);
  const float inv = s_inv[j];
#pragma unroll
  for (int i = 0; i < 4; i++) {
    if (i < na) {
      uint4* xp = reinterpret_cast<uint4*>(act + (a0 + i) * X_ATOM + j * 128 + (pc << 4));
      const uint4 gu = *reinterpret_cast<const uint4*>(gbuf + (a0 + i) * G_ATOM + q * 16);
      uint4 u = *xp;
      __nv_bfloat162* e = reinterpret_cast<__nv_bfloat162*>(&u);
      const __nv_bfloat162* gg = reinterpret_cast<const __nv_bfloat162*>(&gu);
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const float2 xf = __bfloat1622float2(e[k]), gf = __bfloat1622float2(gg[k]);
        e[k] = __floats2bfloat162_rn(xf.x * inv * gf.x, xf.y * inv * gf.y);
      }
      *xp = u;
    }
  }
}

// ---- 8-bit operands (E4M3, OCP OFP8) with one power-of-two scale per 128 elements of a row ----------------------
// The exponent k of a group: the smallest integer with amax 2^-k <= 448 (the largest finite E4M3), clamped to
// [-126, 127]; 0 for an all-zero group.  From the bits of amax = (1 + m 2^-23) 2^(e - 127): 448 = 1.75 2^8, so
// k = e - 127 - 8 + (m > 0.75 2^23).  A subnormal amax gives the clamp.
__device__ __forceinline__ int fp8_group_exponent(float amax) {
  const uint32_t u = __float_as_uint(amax);
  const int e = (int)(u >> 23), m = (int)(u & 0x7FFFFFu);
  if (amax == 0.f) return 0;
  if (e == 0) return -126;
  const int k = e - 135 + (m > 0x600000 ? 1 : 0);
  return k < -126 ? -126 : (k > 127 ? 127 : k);
}
__device__ __forceinline__ float exp2_int(int k) { return __uint_as_float((uint32_t)(127 + k) << 23); }   // |k| <= 126

// Two E4M3 codes (round to nearest even, saturating) of x0, x1: x0 in the low byte.  A zero result is the +0 code.
__device__ __forceinline__ uint32_t e4m3x2(float x0, float x1) {
  uint32_t c = __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
  if ((c & 0x7Fu) == 0) c &= 0xFF00u;
  if ((c & 0x7F00u) == 0) c &= 0x00FFu;
  return c;
}

// The activation slice in 8-bit form, in place: bf16 atoms [a0, a0 + na) (na even, <= 4: 64 K each, 16 token rows,
// 128-byte swizzle), RMSNorm-ed on the way when `norm` (y = bf16(x * inv[t] * g[k]), the bf16 storage point of the
// projection input), become E4M3 blocks [a0/2, a0/2 + na/2) (128 K each, same row and swizzle layout, written over
// the bytes of atoms a0/2 ..), with s_xs[t * xs_ld + block] = 2^k of token t's group.  Thread et: pair = et / 4
// (token t = pair % 16, block pair / 16), quarter q = et % 4 covers the block's K elements [32q, 32q + 32).  Rows
// t >= M are zero.  Only the first group (a0 = 0) writes over bytes it reads: `first` puts a CTA barrier between
// its reads and writes.  Each thread fences its writes for the tensor core; the caller then arrives.
__device__ __forceinline__ void norm_quant_atoms(uint8_t* act, const uint8_t* gbuf, const float* s_inv, float* s_xs,
                                                 int xs_ld, int a0, int na, int M, int et, bool norm, bool first) {
  const int pair = et >> 2, q = et & 3, t = pair & 15, blk = pair >> 4;
  const bool on = blk < (na >> 1);
  const int atom = a0 + 2 * blk + (q >> 1);
  float x[32];
#pragma unroll
  for (int i = 0; i < 32; i++) x[i] = 0.f;
  if (on && t < M) {
    const uint8_t* src = act + atom * X_ATOM + t * 128;
    const float inv = norm ? s_inv[t] : 1.f;
#pragma unroll
    for (int c = 0; c < 4; c++) {
      const int lc = (q & 1) * 4 + c;
      const uint4 u = *reinterpret_cast<const uint4*>(src + ((lc ^ (t & 7)) << 4));
      const __nv_bfloat162* e = reinterpret_cast<const __nv_bfloat162*>(&u);
      if (norm) {
        const uint4 gu = *reinterpret_cast<const uint4*>(gbuf + atom * G_ATOM + lc * 16);
        const __nv_bfloat162* gg = reinterpret_cast<const __nv_bfloat162*>(&gu);
#pragma unroll
        for (int k = 0; k < 4; k++) {
          const float2 xf = __bfloat1622float2(e[k]), gf = __bfloat1622float2(gg[k]);
          const float2 y = __bfloat1622float2(__floats2bfloat162_rn(xf.x * inv * gf.x, xf.y * inv * gf.y));
          x[c * 8 + 2 * k] = y.x;
          x[c * 8 + 2 * k + 1] = y.y;
        }
      } else {
#pragma unroll
        for (int k = 0; k < 4; k++) {
          const float2 f = __bfloat1622float2(e[k]);
          x[c * 8 + 2 * k] = f.x;
          x[c * 8 + 2 * k + 1] = f.y;
        }
      }
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; i++) amax = fmaxf(amax, fabsf(x[i]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  const int k = fp8_group_exponent(amax);
  const float sc = exp2_int(-k);
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; i++)
    w[i] = e4m3x2(x[4 * i] * sc, x[4 * i + 1] * sc) | (e4m3x2(x[4 * i + 2] * sc, x[4 * i + 3] * sc) << 16);
  if (first) epi_bar();   // every thread has read its source chunks
  if (on) {
    uint8_t* dst = act + (a0 / 2 + blk) * X_ATOM + t * 128;
    *reinterpret_cast<uint4*>(dst + (((2 * q) ^ (t & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4*>(dst + (((2 * q + 1) ^ (t & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
    if (q == 0) s_xs[t * xs_ld + a0 / 2 + blk] = exp2_int(k);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic writes -> tensor-core reads
}

// Split-K without a reduce kernel: every CTA stores its fp32 partial tile ([splits][tiles][128 rows][16 tokens],
// 64 contiguous bytes per row); the last CTA of the tile to arrive (atomic counter, no waiting) sums all partials in
// split order into v — bit-reproducible — and resets the counter.  Returns true in that CTA.  All 128 epilogue
// threads call it.  Ordering: the stores of all threads precede thread 0's acquire-release counter update through
// the CTA barrier (the release is cumulative), and the winner's reads follow its acquire through the second
// barrier.  The winner loads up to eight splits at once: the reduction is one round trip to L2 per eight splits.
__device__ __forceinline__ bool splitk_last(float (&v)[16], float* part, int* counters, int split, int splits,
                                            int tile, int tiles, int row_in_tile, int et, int* s_flag) {
  if (splits <= 1) return true;
  float4* mine = reinterpret_cast<float4*>(part + (((size_t)split * tiles + tile) * SBM + row_in_tile) * SBN);
#pragma unroll
  for (int q = 0; q < 4; q++) __stcg(mine + q, make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
  epi_bar();
  if (et == 0) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(counters + tile) : "memory");
    *s_flag = old == splits - 1;
  }
  epi_bar();
  if (!*s_flag) return false;
#pragma unroll
  for (int j = 0; j < 16; j++) v[j] = 0.f;
  for (int s0 = 0; s0 < splits; s0 += 8) {
    float4 pv[8][4];
#pragma unroll
    for (int u = 0; u < 8; u++) {
      const float4* ps =
          reinterpret_cast<const float4*>(part + (((size_t)(s0 + u) * tiles + tile) * SBM + row_in_tile) * SBN);
#pragma unroll
      for (int q = 0; q < 4; q++) pv[u][q] = s0 + u < splits ? __ldcg(ps + q) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 8; u++)
#pragma unroll
      for (int q = 0; q < 4; q++) {
        v[4 * q] += pv[u][q].x;
        v[4 * q + 1] += pv[u][q].y;
        v[4 * q + 2] += pv[u][q].z;
        v[4 * q + 3] += pv[u][q].w;
      }
  }
  if (et == 0) counters[tile] = 0;
  return true;
}

// Sums each of 16 per-lane values over the 32 lanes of a warp in 16 shuffles (each round halves the values a lane
// keeps and trades the other half with its partner); returns the sum of value (lane >> 1) & 15, held by lanes 2t
// and 2t + 1 for token t.  Fixed order, so bit-reproducible.
__device__ __forceinline__ float warp_sum16(const float (&x)[16], int lane) {
  float a[8], b[4], c[2];
  const bool h16 = lane & 16, h8 = lane & 8, h4 = lane & 4, h2 = lane & 2;
#pragma unroll
  for (int i = 0; i < 8; i++) {
    const float send = h16 ? x[i] : x[i + 8];
    a[i] = (h16 ? x[i + 8] : x[i]) + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const float send = h8 ? a[i] : a[i + 4];
    b[i] = (h8 ? a[i + 4] : a[i]) + __shfl_xor_sync(0xffffffffu, send, 8);
  }
#pragma unroll
  for (int i = 0; i < 2; i++) {
    const float send = h4 ? b[i] : b[i + 2];
    c[i] = (h4 ? b[i + 2] : b[i]) + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  const float d = (h2 ? c[1] : c[0]) + __shfl_xor_sync(0xffffffffu, h2 ? c[0] : c[1], 2);
  return d + __shfl_xor_sync(0xffffffffu, d, 1);
}

// The residual-stream values of one 128-column tile that resid_epilogue adds to (loaded early, while the MMAs run:
// only the tile's own epilogue writes these columns).
__device__ __forceinline__ void resid_preload(float (&xv)[16], const bf16* x, int N, int tile, int M, int row_in_tile) {
  const int n = tile * SBM + row_in_tile;
#pragma unroll
  for (int j = 0; j < 16; j++) xv[j] = j < M ? bf(x[(size_t)j * N + n]) : 0.f;
}

// Residual epilogue of one 128-column tile: x[j][n] = bf16(xv + v) (and a copy in layer_out when given), and the
// tile's share of sum(x^2) per token into ss_out[tile][16].  All 128 epilogue threads call it.
__device__ __forceinline__ void resid_epilogue(const float (&v)[16], const float (&xv)[16], bf16* x, int N, int tile,
                                               int M, float* ss_out, bf16* layer_out, float* scratch, int quarter,
                                               int lane, int et) {
  const int n = tile * SBM + quarter * 32 + lane;
  float* red = scratch;   // [4 warps][16]
  float sq[16];
#pragma unroll
  for (int j = 0; j < 16; j++) {
    sq[j] = 0.f;
    if (j < M) {
      const bf16 nb = __float2bfloat16_rn(xv[j] + v[j]);
      x[(size_t)j * N + n] = nb;
      if (layer_out) layer_out[(size_t)j * N + n] = nb;
      sq[j] = bf(nb) * bf(nb);
    }
  }
  const float st = warp_sum16(sq, lane);
  if ((lane & 1) == 0) red[quarter * SBN + (lane >> 1)] = st;
  epi_bar();
  if (et < SBN) ss_out[tile * SBN + et] = red[et] + red[SBN + et] + red[2 * SBN + et] + red[3 * SBN + et];
  epi_bar();
}

// SwiGLU epilogue of one 64-feature tile: TMEM lanes 0..63 hold the gate of features f0 + lane, lanes 64..127 the
// up projection of the same features; hmid[j][f] = bf16(silu(gate) * up).
__device__ __forceinline__ void swiglu_epilogue(const float (&v)[16], bf16* hmid, int F, int tile, int M,
                                                float* scratch, int row_in_tile) {
  float* xch = scratch;   // [64][16]
  const bool up_half = row_in_tile >= 64;
  const int fr = up_half ? row_in_tile - 64 : row_in_tile;
  if (up_half) {
#pragma unroll
    for (int j = 0; j < 16; j++) xch[fr * SBN + j] = v[j];
  }
  epi_bar();
  if (!up_half) {
    const int f = tile * 64 + fr;
#pragma unroll
    for (int j = 0; j < 16; j++)
      if (j < M) {
        const float gv = v[j], uv = xch[fr * SBN + j];
        hmid[(size_t)j * F + f] = __float2bfloat16_rn(gv / (1.0f + expf(-gv)) * uv);
      }
  }
  epi_bar();
}

struct QkvOut {
  bf16 *q, *kblk, *vblk;           // q [M][nq][h], block keys / values [B][nkv][L][h]
  const bf16 *q_norm, *k_norm;
  const float2* rope;              // [positions][h/2] (cos, sin)
  int M, L, nq, nkv;
  float eps;
};

// q/k RMSNorm + rotate-half RoPE at position ctx_len + j (or plain v) of the heads of one 128-feature QKV tile.
// vals: the tile's fp32 sums in shared memory, token-major [16][128]; s_ctx: context length per request.  Every
// head of a tile has the same kind (q, k or v) because the q, k and v row blocks are multiples of 128 rows.  One
// warp per (token, head); the gain and the RoPE rows are loaded before any arithmetic so the loads overlap.
template <int H>
__device__ __forceinline__ void qkv_tile_epilogue(const QkvOut& p, const float* vals, int tile, const int* s_ctx,
                                                  int quarter, int lane) {
  constexpr int NV = H / 32, HPT = SBM / H, NU = SBN * HPT / 4;
  const int head0 = tile * HPT;
  const int kind = head0 < p.nq ? 0 : (head0 < p.nq + p.nkv ? 1 : 2);
  float g[NV];
  if (kind < 2) {
    const bf16* gp = kind == 0 ? p.q_norm : p.k_norm;
#pragma unroll
    for (int k = 0; k < NV; k++) g[k] = bf(gp[lane + 32 * k]);
  }
  float2 cs[NU][NV / 2];
#pragma unroll
  for (int i = 0; i < NU; i++) {
    const int u = quarter + 4 * i, j = u / HPT;
    if (kind < 2 && j < p.M) {
      const int pos = s_ctx[j / p.L] + j % p.L;
#pragma unroll
      for (int k = 0; k < NV / 2; k++) cs[i][k] = p.rope[(size_t)pos * (H / 2) + lane + 32 * k];
    }
  }
#pragma unroll
  for (int i = 0; i < NU; i++) {
    const int u = quarter + 4 * i, j = u / HPT, hh = u % HPT;
    if (j >= p.M) continue;
    const int b = j / p.L, jj = j % p.L, head = head0 + hh;
    float v[NV];
#pragma unroll
    for (int k = 0; k < NV; k++) v[k] = vals[j * SBM + hh * H + lane + 32 * k];
    bf16* dst;
    if (kind < 2) {
      float ss = 0.f;
#pragma unroll
      for (int k = 0; k < NV; k++) ss += v[k] * v[k];
      const float inv = rsqrtf(warp_sum(ss) / (float)H + p.eps);
#pragma unroll
      for (int k = 0; k < NV; k++) v[k] = v[k] * inv * g[k];
#pragma unroll
      for (int k = 0; k < NV / 2; k++) {
        const float x1 = v[k], x2 = v[k + NV / 2];
        v[k] = x1 * cs[i][k].x - x2 * cs[i][k].y;
        v[k + NV / 2] = x2 * cs[i][k].x + x1 * cs[i][k].y;
      }
      dst = kind == 0 ? p.q + ((size_t)j * p.nq + head) * H
                      : p.kblk + (((size_t)b * p.nkv + head - p.nq) * p.L + jj) * H;
    } else {
      dst = p.vblk + (((size_t)b * p.nkv + head - p.nq - p.nkv) * p.L + jj) * H;
    }
#pragma unroll
    for (int k = 0; k < NV; k++) dst[lane + 32 * k] = __float2bfloat16_rn(v[k]);
  }
}

}  // namespace fewtok
}  // namespace fpd

// k_gemm_tc.cu — persistent, warp-specialised tcgen05 GEMM for sm_103a, and the LM-head + argmax variant.
//
//   D[m][n] = sum_k X[m][k] * W[n][k]      X = activations [M, K] (K-major, bf16, may be K-segmented),
//                                          W = weights     [N, K] (K-major, bf16, [out, in])
//
// Two operand placements share one kernel:
//   SWAP  (few tokens, M <= 64): the 128-row MMA operand is a tile of W (output features) and the BN-row
//          operand holds the tokens.  Weight streaming is the whole cost at batch 1, so every SM pulls weight
//          tiles through a deep TMA ring; split-K over the grid supplies enough CTAs.
//   !SWAP (many tokens): the 128-row operand is a token tile and the BN-row (128/256) operand a weight tile.
//
// Roles (6 warps): warp 0 issues TMA loads into a STAGES-deep shared-memory ring (128-byte swizzled K-major
// tiles, one mbarrier pair per stage); warp 1 owns TMEM and one lane issues tcgen05.mma (M = 128, N = BN,
// K = 16 per instruction, fp32 accumulators in TMEM, two accumulator buffers so the epilogue of one tile
// overlaps the main loop of the next); warps 2-5 read the accumulators back with tcgen05.ld (each warp sees
// its 32-lane quarter of TMEM) and run the epilogue.  Every wait is bounded (tc::mbar_wait).
//
// Epilogues:  EPI_STORE  — fp32 partial sums to C[split][M][ldc] (split-K partials are reduced by the
//                          consumer row kernel, in fixed order).
//             EPI_ARGMAX — LM head (VFlash paper (zh) §2.5: constraints act on computed logits): the MMA rows
//                          are vocabulary ids of one legal range, the columns positions of that range's class;
//                          per position the (logit, id) maximum is folded into a 64-bit word by atomicMax
//                          (lowest id on ties, order independent).
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "fpd_kernels.cuh"
#include "tc_primitives.cuh"

namespace fpd {

namespace {

constexpr int BM = 128, BK = 64, UMMA_K = 16;
constexpr int kThreads = 192;
enum { EPI_STORE = 0, EPI_ARGMAX = 1, EPI_SWIGLU = 2, EPI_QKV_TOK = 3, EPI_RESID_TOK = 4, EPI_KV_CTX = 5 };

struct TcParams {
  CUtensorMap tm_x[8];   // activation K-segments (box rows: BN if swap else 128)
  CUtensorMap tm_w;      // weights (box rows: 128 if swap else BN)
  int n_seg, seg_k;
  int M, N, K;
  // EPI_STORE
  float* c;
  int ldc;
  size_t c_split_stride;
  int pt, qt, splits, k_split;   // tiles along the 128-row operand, the BN-row operand, and K splits
  // EPI_ARGMAX
  const int4* items;             // (range, first id, first sorted row, row count)
  const int* n_items;
  int implicit_rowtiles;         // > 0: unconstrained vocabulary, item t = (id tile t / rowtiles, row tile t % rowtiles)
  int implicit_total;
  int hi_tab[FPD_MAX_RANGES];    // end (exclusive) of every legal id range
  unsigned long long* packed;    // [sorted rows]
  unsigned long long* packed2;   // [sorted rows] second-best word (top-2 margin) or null
  const int* rows_sorted;        // sorted row -> original row (logits only)
  float* logits;                 // [n_rows, V] or null
  int V;
  // EPI_SWIGLU: W = [gate; up] rows [2F, K]; output hmid[M][F] = bf16(silu(gate) * up)
  bf16* hmid;
  int F;
  // EPI_QKV_TOK (token tiles): per head q/k RMSNorm + RoPE at position ctx_len[b] + j, bf16 q / block k / block v
  bf16 *q, *kblk, *vblk;
  const bf16 *q_norm, *k_norm;
  const float2* rope;
  const int32_t* ctx_len;
  int t_cap, L, nq, nkv, hd;
  float eps;
  // EPI_RESID_TOK (token tiles): x[m][n] = bf16(x + acc); ss_part[column tile][m] = that tile's sum of x^2
  bf16* xres;
  float* ss_part;
  // EPI_KV_CTX (token tiles of context rows): the B operand is [Wk; Wv] of every layer side by side, layer l's
  // kv_cols rows starting at row kv_row_base of wqkv[l] (tm_wl[l]); each context row row0 + m goes to its request's
  // position in the KV store [layer][b][K|V][g][t_cap][hd], K heads RMS-normed (k_norm_l[l]) and rotated
  CUtensorMap tm_wl[FPD_MAX_LAYERS];
  int kv_cols, kv_row_base, n_layers;
  bf16* store;
  const bf16* k_norm_l[FPD_MAX_LAYERS];
  const int32_t *row_off, *row_cnt, *pos_start;
  int batch, row0;
};

// A pipeline stage holds KS consecutive 64-element K atoms of both operands: [A atoms][B atoms].  Several
// atoms per stage make the TMA unit request KS adjacent 128-byte pieces of every weight row back to back.
template <int BN, int KS>
struct Cfg {
  static constexpr int A_ATOM = BM * BK * 2;   // 128 rows x 128 B
  static constexpr int B_ATOM = BN * BK * 2;
  static constexpr int A_BYTES = KS * A_ATOM;
  static constexpr int STAGE_BYTES = KS * (A_ATOM + B_ATOM);
  static constexpr int TMEM_COLS = (2 * BN < 32) ? 32 : 2 * BN;   // two accumulator buffers
};
// shared memory the SwiGLU epilogue uses to hand the up-projection values from the warps holding TMEM lanes
// 64..127 to the warps holding the gate values of the same features (lanes 0..63), weight-tile placement only
template <int BN, bool SWAP, int EPI>
constexpr int xch_bytes() {
  return (EPI == EPI_SWIGLU && SWAP) ? 64 * BN * 4 : 0;
}

struct Work {
  int a_row0, b_row0;   // first row of the 128-row (A) and BN-row (B) operand tiles
  int k0, k1, nkb;      // K range [k0, k1) and number of pipeline stages it takes
  int split;
  int range;            // EPI_ARGMAX: range index; rows valid below `b_cnt`
  int b_cnt;
};

template <bool SWAP, int BN, int EPI, int KS>
__device__ __forceinline__ bool get_work(const TcParams& p, int t, int total, Work& w) {
  if (t >= total) return false;
  if (EPI != EPI_ARGMAX) {
    const int pi = t % p.pt, qi = (t / p.pt) % p.qt, s = t / (p.pt * p.qt);
    w.a_row0 = pi * ((EPI == EPI_SWIGLU && SWAP) ? BM / 2 : BM);    // SwiGLU: first feature of the tile
    w.b_row0 = qi * ((EPI == EPI_SWIGLU && !SWAP) ? BN / 2 : BN);
    w.split = s;
    w.k0 = s * p.k_split;
    w.k1 = min(p.K, w.k0 + p.k_split);
    w.nkb = (w.k1 - w.k0 + KS * BK - 1) / (KS * BK);
    w.range = 0;
    w.b_cnt = BN;
  } else {
    if (p.implicit_rowtiles > 0) {
      const int ct = t / p.implicit_rowtiles, rt = t % p.implicit_rowtiles;
      w.range = 0;
      w.a_row0 = ct * BM;
      w.b_row0 = rt * BN;
      w.b_cnt = min(BN, p.M - rt * BN);
    } else {
      const int4 it = p.items[t];
      w.range = it.x;
      w.a_row0 = it.y;
      w.b_row0 = it.z;
      w.b_cnt = it.w;
    }
    w.split = 0;
    w.k0 = 0;
    w.k1 = p.K;
    w.nkb = (p.K + KS * BK - 1) / (KS * BK);
  }
  return true;
}

template <int BN, int STAGES, bool SWAP, int EPI, int KS>
__global__ void __launch_bounds__(kThreads, 1) tc_gemm_kernel(const __grid_constant__ TcParams p) {
  using C = Cfg<BN, KS>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* xch = reinterpret_cast<float*>(smem + STAGES * C::STAGE_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES + xch_bytes<BN, SWAP, EPI>());
  // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t full0 = tc::smem_u32(bars), empty0 = full0 + 8 * STAGES, tfull0 = empty0 + 8 * STAGES,
                 tempty0 = tfull0 + 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  pdl_trigger();
  // weight tiles never depend on earlier kernels, so the producer may fetch the first ring of them before
  // waiting for the predecessor grid; everything else (activations, item lists, outputs) comes after pdl_wait
  const bool explicit_items = EPI == EPI_ARGMAX && p.implicit_rowtiles == 0;
  if (explicit_items) pdl_wait();
  const int total = EPI != EPI_ARGMAX ? p.pt * p.qt * p.splits : (explicit_items ? *p.n_items : p.implicit_total);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; s++) {
      tc::mbar_init(full0 + 8 * s, 1);
      tc::mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; a++) {
      tc::mbar_init(tfull0 + 8 * a, 1);
      tc::mbar_init(tempty0 + 8 * a, 4);   // one arrival per epilogue warp
    }
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tc::smem_u32(tmem_slot), C::TMEM_COLS);
    tc::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    if (EPI == EPI_KV_CTX)
      for (int l = 0; l < p.n_layers; l++) tc::tma_prefetch(&p.tm_wl[l]);
    else
      tc::tma_prefetch(&p.tm_w);
    for (int s = 0; s < p.n_seg; s++) tc::tma_prefetch(&p.tm_x[s]);
  }
  // The single-lane roles reconverge with their warps first: a CTA barrier reached by part of a diverged
  // warp counts the whole warp, and the lagging lane would then pass it without waiting.
  __syncwarp();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      // weight / activation atoms of one stage; the stage's bytes are expected on its full barrier first
      auto load_w = [&](uint32_t sa, const Work& w, int k, int natoms, uint32_t fb) {
        for (int a = 0; a < natoms; a++) {
          const int ka = k + a * BK;
          if (EPI == EPI_SWIGLU) {   // weight atom = [gate rows f0.. ; up rows F+f0..], two half boxes
            const uint32_t dst = SWAP ? sa + a * C::A_ATOM : sa + C::A_BYTES + a * C::B_ATOM;
            const int half = SWAP ? C::A_ATOM / 2 : C::B_ATOM / 2;
            const int f0 = SWAP ? w.a_row0 : w.b_row0;
            tc::tma_load_2d(dst, &p.tm_w, ka, f0, fb);
            tc::tma_load_2d(dst + half, &p.tm_w, ka, p.F + f0, fb);
          } else if (SWAP) {
            tc::tma_load_2d(sa + a * C::A_ATOM, &p.tm_w, ka, w.a_row0, fb);
          } else if (EPI == EPI_KV_CTX) {   // column b_row0 of the side-by-side layers
            const int layer = w.b_row0 / p.kv_cols;
            tc::tma_load_2d(sa + C::A_BYTES + a * C::B_ATOM, &p.tm_wl[layer], ka,
                            w.b_row0 - layer * p.kv_cols + p.kv_row_base, fb);
          } else {
            tc::tma_load_2d(sa + C::A_BYTES + a * C::B_ATOM, &p.tm_w, ka, w.b_row0, fb);
          }
        }
      };
      auto load_x = [&](uint32_t sa, const Work& w, int k, int natoms, uint32_t fb) {
        for (int a = 0; a < natoms; a++) {
          const int ka = k + a * BK;
          const int seg = ka / p.seg_k, kx = ka - seg * p.seg_k;
          if (SWAP)
            tc::tma_load_2d(sa + C::A_BYTES + a * C::B_ATOM, &p.tm_x[seg], kx, w.b_row0, fb);
          else
            tc::tma_load_2d(sa + a * C::A_ATOM, &p.tm_x[seg], kx, w.a_row0, fb);
        }
      };
      auto atoms = [&](const Work& w, int kb) { return min(KS, (w.k1 - (w.k0 + kb * KS * BK)) / BK); };
      int pre = 0;
      Work w0;
      if (!explicit_items && get_work<SWAP, BN, EPI, KS>(p, blockIdx.x, total, w0)) {
        pre = min(STAGES, w0.nkb);
        for (int kb = 0; kb < pre; kb++) {   // fresh ring: the empty barriers need no wait
          const uint32_t fb = full0 + 8 * kb;
          const int na = atoms(w0, kb);
          tc::mbar_arrive_expect_tx(fb, na * (C::A_ATOM + C::B_ATOM));
          load_w(tc::smem_u32(smem + kb * C::STAGE_BYTES), w0, w0.k0 + kb * KS * BK, na, fb);
        }
      }
      if (!explicit_items) pdl_wait();
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool first = true;
      Work w;
      for (int t = blockIdx.x; get_work<SWAP, BN, EPI, KS>(p, t, total, w) && !*abort_flag; t += gridDim.x) {
        for (int kb = 0; kb < w.nkb; kb++) {
          const uint32_t fb = full0 + 8 * stage;
          const uint32_t sa = tc::smem_u32(smem + stage * C::STAGE_BYTES);
          const int k = w.k0 + kb * KS * BK;
          const int na = atoms(w, kb);
          if (!(first && kb < pre)) {
            if (!tc::mbar_wait(empty0 + 8 * stage, phase ^ 1)) { *abort_flag = 1; break; }
            tc::mbar_arrive_expect_tx(fb, na * (C::A_ATOM + C::B_ATOM));
            load_w(sa, w, k, na, fb);
          }
          load_x(sa, w, k, na, fb);
          issued++;
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        first = false;
      }
      if (*abort_flag) {
        // let the copies already issued land before the CTA can exit (bounded)
        for (int s = 0; s < STAGES && s < issued; s++) {
          if (--stage < 0) { stage = STAGES - 1; phase ^= 1; }
          tc::mbar_wait(full0 + 8 * stage, phase);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      Work w;
      for (int t = blockIdx.x; get_work<SWAP, BN, EPI, KS>(p, t, total, w); t += gridDim.x, it++) {
        const int acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        const uint32_t d_tmem = tmem_base + acc * BN;
        if (!*abort_flag && !tc::mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1)) *abort_flag = 1;
        tc::tc_fence_after();
        for (int kb = 0; kb < w.nkb && !*abort_flag; kb++) {
          if (!tc::mbar_wait(full0 + 8 * stage, phase)) { *abort_flag = 1; break; }
          tc::tc_fence_after();
          const uint32_t sa = tc::smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t sb = sa + C::A_BYTES;
          const int na = min(KS, (w.k1 - (w.k0 + kb * KS * BK)) / BK);
          for (int a = 0; a < na; a++) {
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; kk++) {
              const uint64_t da = tc::sw128_kmajor_desc(sa + a * C::A_ATOM + kk * UMMA_K * 2);
              const uint64_t db = tc::sw128_kmajor_desc(sb + a * C::B_ATOM + kk * UMMA_K * 2);
              tc::umma_bf16(d_tmem, da, db, idesc, (kb > 0 || a > 0 || kk > 0) ? 1u : 0u);
            }
          }
          tc::umma_commit(empty0 + 8 * stage);   // frees the stage once these MMAs have read it
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        tc::umma_commit(tfull0 + 8 * acc);       // accumulator ready (also on abort: never leave waiters)
      }
    }
  } else {
    // ---------------- epilogue: warps 2..5 ----------------
    if (!explicit_items) pdl_wait();            // outputs may still be read by the predecessor until it completes
    const int quarter = warp & 3;               // TMEM lanes [32*quarter, 32*quarter + 32)
    const int row_in_tile = quarter * 32 + lane;
    int it = 0;
    Work w;
    for (int t = blockIdx.x; get_work<SWAP, BN, EPI, KS>(p, t, total, w); t += gridDim.x, it++) {
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      if (!tc::mbar_wait(tfull0 + 8 * acc, acc_phase)) *abort_flag = 1;
      tc::tc_fence_after();
      const uint32_t t_acc = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
      if (EPI == EPI_STORE) {
        float* Cs = p.c + (size_t)w.split * p.c_split_stride;
        const bool empty_k = w.nkb == 0;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 16) {
          float v[16];
          tc::tmem_ld16(t_acc + c0, v);
          if (empty_k) {
#pragma unroll
            for (int j = 0; j < 16; j++) v[j] = 0.f;
          }
          if (SWAP) {
            const int n = w.a_row0 + row_in_tile;
            if (n < p.N) {
#pragma unroll
              for (int j = 0; j < 16; j++) {
                const int m = w.b_row0 + c0 + j;
                if (m < p.M) Cs[(size_t)m * p.ldc + n] = v[j];
              }
            }
          } else {
            const int m = w.a_row0 + row_in_tile;
            const int n0 = w.b_row0 + c0;
            if (m < p.M) {
              float* dst = Cs + (size_t)m * p.ldc + n0;
              if (n0 + 16 <= p.N && (p.ldc & 3) == 0) {
#pragma unroll
                for (int j = 0; j < 16; j += 4)
                  *reinterpret_cast<float4*>(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
              } else {
#pragma unroll
                for (int j = 0; j < 16; j++)
                  if (n0 + j < p.N) dst[j] = v[j];
              }
            }
          }
        }
      } else if (EPI == EPI_QKV_TOK) {
        // token m = a_row0 + row_in_tile holds the tile's BN features: whole heads, so the per-head RMSNorm and the
        // rotate-half pairs (i, i + hd/2) are in this thread's registers.  tcgen05.ld is warp-wide: every lane
        // loads, only rows below M store.
        const int m = w.a_row0 + row_in_tile;
        const bool mok = m < p.M;
        const int b = mok ? m / p.L : 0, j = mok ? m % p.L : 0;
        int cl = mok ? p.ctx_len[b] : 0;
        cl = clamp_ctx(cl, p.t_cap);
        const int hh = p.hd / 2;
        const float2* rope_row = p.rope + (size_t)(cl + j) * hh;
#pragma unroll 1
        for (int h0 = 0; h0 < BN && w.b_row0 + h0 < p.N; h0 += p.hd) {
          const int head = (w.b_row0 + h0) / p.hd;
          const int kind = head < p.nq ? 0 : (head < p.nq + p.nkv ? 1 : 2);
          bf16* dst = kind == 0 ? p.q + ((size_t)m * p.nq + head) * p.hd
                    : kind == 1 ? p.kblk + (((size_t)b * p.nkv + head - p.nq) * p.L + j) * p.hd
                                : p.vblk + (((size_t)b * p.nkv + head - p.nq - p.nkv) * p.L + j) * p.hd;
          if (kind == 2) {
#pragma unroll 1
            for (int c = 0; c < p.hd; c += 16) {
              float v[16];
              tc::tmem_ld16(t_acc + h0 + c, v);
              uint4 pk[2];
              bf16* pe = reinterpret_cast<bf16*>(pk);
#pragma unroll
              for (int e = 0; e < 16; e++) pe[e] = __float2bfloat16_rn(v[e]);
              if (mok) {
                reinterpret_cast<uint4*>(dst + c)[0] = pk[0];
                reinterpret_cast<uint4*>(dst + c)[1] = pk[1];
              }
            }
            continue;
          }
          float ss = 0.f;
#pragma unroll 1
          for (int c = 0; c < p.hd; c += 16) {
            float v[16];
            tc::tmem_ld16(t_acc + h0 + c, v);
#pragma unroll
            for (int e = 0; e < 16; e++) ss += v[e] * v[e];
          }
          const float inv = rsqrtf(ss / (float)p.hd + p.eps);
          const bf16* gain = kind == 0 ? p.q_norm : p.k_norm;
#pragma unroll 1
          for (int c = 0; c < hh; c += 16) {
            float a[16], bb[16];
            tc::tmem_ld16(t_acc + h0 + c, a);
            tc::tmem_ld16(t_acc + h0 + c + hh, bb);
            uint4 g1u[2], g2u[2], o1[2], o2[2];
            g1u[0] = reinterpret_cast<const uint4*>(gain + c)[0];
            g1u[1] = reinterpret_cast<const uint4*>(gain + c)[1];
            g2u[0] = reinterpret_cast<const uint4*>(gain + c + hh)[0];
            g2u[1] = reinterpret_cast<const uint4*>(gain + c + hh)[1];
            const bf16* g1 = reinterpret_cast<const bf16*>(g1u);
            const bf16* g2 = reinterpret_cast<const bf16*>(g2u);
            bf16* e1 = reinterpret_cast<bf16*>(o1);
            bf16* e2 = reinterpret_cast<bf16*>(o2);
#pragma unroll
            for (int e = 0; e < 16; e++) {
              const float2 cs = rope_row[c + e];
              const float x1 = a[e] * inv * __bfloat162float(g1[e]), x2 = bb[e] * inv * __bfloat162float(g2[e]);
              e1[e] = __float2bfloat16_rn(x1 * cs.x - x2 * cs.y);
              e2[e] = __float2bfloat16_rn(x2 * cs.x + x1 * cs.y);
            }
            if (mok) {
              reinterpret_cast<uint4*>(dst + c)[0] = o1[0];
              reinterpret_cast<uint4*>(dst + c)[1] = o1[1];
              reinterpret_cast<uint4*>(dst + c + hh)[0] = o2[0];
              reinterpret_cast<uint4*>(dst + c + hh)[1] = o2[1];
            }
          }
        }
      } else if (EPI == EPI_KV_CTX) {
        // context row row0 + m (m = a_row0 + row_in_tile): its request b (row_off[b] <= row < row_off[b + 1]) and
        // position pos_start[b] + row - row_off[b]; rows past the request's count are skipped, positions outside
        // [0, t_cap) are recorded and skipped.  tcgen05.ld is warp-wide: every lane loads, valid rows store.
        const int m = w.a_row0 + row_in_tile;
        const int grow = p.row0 + m;
        bool ok = m < p.M;
        int b = 0, pos = 0;
        if (ok) {
          int lo = 0, hi = p.batch;
          while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (p.row_off[mid] <= grow) lo = mid; else hi = mid;
          }
          b = lo;
          if (grow >= p.row_off[p.batch] || (p.row_cnt && grow - p.row_off[b] >= p.row_cnt[b])) {
            ok = false;
          } else {
            pos = (p.pos_start ? p.pos_start[b] : 0) + grow - p.row_off[b];
            if (pos < 0 || pos >= p.t_cap) {
              record_check(kCheckBadPosition);
              ok = false;
            }
          }
        }
        const int layer = w.b_row0 / p.kv_cols;
        const int hh = p.hd / 2;
        const float2* rope_row = p.rope + (size_t)(ok ? pos : 0) * hh;
        const bf16* gain = p.k_norm_l[layer];
#pragma unroll 1
        for (int h0 = 0; h0 < BN; h0 += p.hd) {
          const int hk = (w.b_row0 - layer * p.kv_cols + h0) / p.hd;   // [K heads | V heads] of the layer
          const int is_v = hk >= p.nkv, g = is_v ? hk - p.nkv : hk;
          bf16* dst = p.store + (((((size_t)layer * p.batch + b) * 2 + is_v) * p.nkv + g) * (size_t)p.t_cap + pos) * p.hd;
          if (is_v) {
#pragma unroll 1
            for (int c = 0; c < p.hd; c += 16) {
              float v[16];
              tc::tmem_ld16(t_acc + h0 + c, v);
              uint4 pk[2];
              bf16* pe = reinterpret_cast<bf16*>(pk);
#pragma unroll
              for (int e = 0; e < 16; e++) pe[e] = __float2bfloat16_rn(v[e]);
              if (ok) {
                reinterpret_cast<uint4*>(dst + c)[0] = pk[0];
                reinterpret_cast<uint4*>(dst + c)[1] = pk[1];
              }
            }
            continue;
          }
          float ss = 0.f;
#pragma unroll 1
          for (int c = 0; c < p.hd; c += 16) {
            float v[16];
            tc::tmem_ld16(t_acc + h0 + c, v);
#pragma unroll
            for (int e = 0; e < 16; e++) ss += v[e] * v[e];
          }
          const float inv = rsqrtf(ss / (float)p.hd + p.eps);
#pragma unroll 1
          for (int c = 0; c < hh; c += 16) {
            float a[16], bb[16];
            tc::tmem_ld16(t_acc + h0 + c, a);
            tc::tmem_ld16(t_acc + h0 + c + hh, bb);
            uint4 g1u[2], g2u[2], o1[2], o2[2];
            g1u[0] = reinterpret_cast<const uint4*>(gain + c)[0];
            g1u[1] = reinterpret_cast<const uint4*>(gain + c)[1];
            g2u[0] = reinterpret_cast<const uint4*>(gain + c + hh)[0];
            g2u[1] = reinterpret_cast<const uint4*>(gain + c + hh)[1];
            const bf16* g1 = reinterpret_cast<const bf16*>(g1u);
            const bf16* g2 = reinterpret_cast<const bf16*>(g2u);
            bf16* e1 = reinterpret_cast<bf16*>(o1);
            bf16* e2 = reinterpret_cast<bf16*>(o2);
#pragma unroll
            for (int e = 0; e < 16; e++) {
              const float2 cs = rope_row[c + e];
              const float x1 = a[e] * inv * __bfloat162float(g1[e]), x2 = bb[e] * inv * __bfloat162float(g2[e]);
              e1[e] = __float2bfloat16_rn(x1 * cs.x - x2 * cs.y);
              e2[e] = __float2bfloat16_rn(x2 * cs.x + x1 * cs.y);
            }
            if (ok) {
              reinterpret_cast<uint4*>(dst + c)[0] = o1[0];
              reinterpret_cast<uint4*>(dst + c)[1] = o1[1];
              reinterpret_cast<uint4*>(dst + c + hh)[0] = o2[0];
              reinterpret_cast<uint4*>(dst + c + hh)[1] = o2[1];
            }
          }
        }
      } else if (EPI == EPI_RESID_TOK) {
        // token m: x[m][n] = bf16(x + acc) over the tile's columns, and this column tile's share of sum(x^2)
        const int m = w.a_row0 + row_in_tile;
        const bool mok = m < p.M;
        float ss = 0.f;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 16) {
          float v[16];
          tc::tmem_ld16(t_acc + c0, v);
          const int n0 = w.b_row0 + c0;
          if (mok && n0 + 16 <= p.N) {
            uint4* xp = reinterpret_cast<uint4*>(p.xres + (size_t)m * p.N + n0);
            uint4 xu[2] = {xp[0], xp[1]};
            bf16* xe = reinterpret_cast<bf16*>(xu);
#pragma unroll
            for (int e = 0; e < 16; e++) {
              xe[e] = __float2bfloat16_rn(__bfloat162float(xe[e]) + v[e]);
              const float f = __bfloat162float(xe[e]);
              ss += f * f;
            }
            xp[0] = xu[0];
            xp[1] = xu[1];
          }
        }
        if (mok) p.ss_part[(size_t)(w.b_row0 / BN) * p.M + m] = ss;
      } else if (EPI == EPI_SWIGLU) {
        if (SWAP) {
          // lanes 0..63: gate of feature f0 + lane; lanes 64..127: up of feature f0 + lane - 64
          const bool up_half = row_in_tile >= 64;
          const int fr = up_half ? row_in_tile - 64 : row_in_tile;
          const int f = w.a_row0 + fr;
#pragma unroll 1
          for (int c0 = 0; c0 < BN; c0 += 16) {
            float v[16];
            tc::tmem_ld16(t_acc + c0, v);
            if (up_half) {
#pragma unroll
              for (int j = 0; j < 16; j++) xch[fr * BN + c0 + j] = v[j];
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (!up_half && f < p.F) {
#pragma unroll
              for (int j = 0; j < 16; j++) {
                const int m = w.b_row0 + c0 + j;
                if (m < p.M) {
                  const float gv = v[j], uv = xch[fr * BN + c0 + j];
                  p.hmid[(size_t)m * p.F + f] = __float2bfloat16_rn(gv / (1.0f + expf(-gv)) * uv);
                }
              }
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
          }
        } else {
          // columns 0..BN/2-1: gate of features f0.., columns BN/2..BN-1: up of the same features
          const int m = w.a_row0 + row_in_tile;
#pragma unroll 1
          for (int c0 = 0; c0 < BN / 2; c0 += 16) {
            float gv[16], uv[16];
            tc::tmem_ld16(t_acc + c0, gv);
            tc::tmem_ld16(t_acc + BN / 2 + c0, uv);
            const int f0 = w.b_row0 + c0;
            if (m < p.M) {
              bf16* dst = p.hmid + (size_t)m * p.F + f0;
              if (f0 + 16 <= p.F && (p.F & 7) == 0) {
                uint4 pk[2];
                bf16* pe = reinterpret_cast<bf16*>(pk);
#pragma unroll
                for (int j = 0; j < 16; j++) pe[j] = __float2bfloat16_rn(gv[j] / (1.0f + expf(-gv[j])) * uv[j]);
                reinterpret_cast<uint4*>(dst)[0] = pk[0];
                reinterpret_cast<uint4*>(dst)[1] = pk[1];
              } else {
#pragma unroll
                for (int j = 0; j < 16; j++)
                  if (f0 + j < p.F) dst[j] = __float2bfloat16_rn(gv[j] / (1.0f + expf(-gv[j])) * uv[j]);
              }
            }
          }
        }
      } else {
        // LM head: rows = vocabulary ids, columns = sorted positions of one class
        const int vid = w.a_row0 + row_in_tile;
        const bool vok = vid < p.hi_tab[w.range];
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 16) {
          float v[16];
          tc::tmem_ld16(t_acc + c0, v);
#pragma unroll
          for (int j = 0; j < 16; j++) {
            const int col = c0 + j;
            const bool ok = vok && col < w.b_cnt;
            unsigned long long best = ok ? pack_argmax(v[j], vid) : 0ull;
            if (!p.packed2) {
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) best = max(best, __shfl_xor_sync(0xffffffffu, best, o));
              if (lane == 0 && best) atomicMax(p.packed + w.b_row0 + col, best);
            } else {
              // top-2: the value an atomicMax displaces (or the candidate it rejects) is a candidate for the
              // second place, so every word but the final maximum reaches packed2
              unsigned long long second = 0ull;
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long b1 = __shfl_xor_sync(0xffffffffu, best, o);
                const unsigned long long b2 = __shfl_xor_sync(0xffffffffu, second, o);
                const unsigned long long lo = min(best, b1);
                best = max(best, b1);
                second = max(lo, max(second, b2));
              }
              if (lane == 0 && best) {
                const unsigned long long old = atomicMax(p.packed + w.b_row0 + col, best);
                atomicMax(p.packed2 + w.b_row0 + col, max(min(old, best), second));
              }
            }
            if (p.logits && ok) p.logits[(size_t)p.rows_sorted[w.b_row0 + col] * p.V + vid] = v[j];
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(tempty0 + 8 * acc);
    }
  }

  __syncwarp();
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ---- host side ------------------------------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

template <int BN, int STAGES, bool SWAP, int EPI, int KS>
constexpr size_t smem_bytes() {
  return (size_t)STAGES * Cfg<BN, KS>::STAGE_BYTES + xch_bytes<BN, SWAP, EPI>() + 1024 + 256;
}

template <int BN, int STAGES, bool SWAP, int EPI, int KS = 1>
cudaError_t set_attr() {
  static_assert(smem_bytes<BN, STAGES, SWAP, EPI, KS>() <= 227 * 1024, "shared memory");
  return cudaFuncSetAttribute(tc_gemm_kernel<BN, STAGES, SWAP, EPI, KS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)smem_bytes<BN, STAGES, SWAP, EPI, KS>());
}

template <int BN, int STAGES, bool SWAP, int EPI, int KS = 1>
cudaError_t launch_kernel(const TcParams& p, int grid, cudaStream_t st) {
  return launch_k(tc_gemm_kernel<BN, STAGES, SWAP, EPI, KS>, grid, kThreads, smem_bytes<BN, STAGES, SWAP, EPI, KS>(),
                  st, p);
}

// Few-token (weight-tile) kernels with 16-token tiles: one 64-element K atom per stage, 6 stages, 2 CTAs per SM.
constexpr int kSwap16CtasPerSm = 2;
}  // namespace

// Row-major bf16 matrix [rows, cols] with row stride ld (elements), boxes of 64 columns x box_rows rows,
// 128-byte swizzle (matches sw128_kmajor_desc).  Out-of-range boxes read zeros.
cudaError_t make_tmap(CUtensorMap* tm, const void* ptr, int rows, int cols, int ld, int box_rows) {
  if (rows < 1 || cols < BK) return cudaErrorInvalidValue;
  const uint64_t dims[2] = {(uint64_t)cols, (uint64_t)rows};
  const uint64_t strides[1] = {(uint64_t)ld * 2};
  const uint32_t box[2] = {(uint32_t)BK, (uint32_t)box_rows};
  return make_tmap_nd(tm, ptr, 2, dims, strides, box);
}

static cudaError_t make_tmap_typed(CUtensorMap* tm, CUtensorMapDataType dt, const void* ptr, int rank,
                                   const uint64_t* dims, const uint64_t* strides, const uint32_t* box);

cudaError_t make_tmap_nd(CUtensorMap* tm, const void* ptr, int rank, const uint64_t* dims, const uint64_t* strides,
                         const uint32_t* box) {
  return make_tmap_typed(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ptr, rank, dims, strides, box);
}

cudaError_t make_tmap_u8(CUtensorMap* tm, const void* ptr, int rows, int cols, int ld, int box_rows) {
  if (rows < 1 || cols < 128) return cudaErrorInvalidValue;
  const uint64_t dims[2] = {(uint64_t)cols, (uint64_t)rows};
  const uint64_t strides[1] = {(uint64_t)ld};
  const uint32_t box[2] = {128u, (uint32_t)box_rows};
  return make_tmap_typed(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, ptr, 2, dims, strides, box);
}

static cudaError_t make_tmap_typed(CUtensorMap* tm, CUtensorMapDataType dt, const void* ptr, int rank,
                                   const uint64_t* dims, const uint64_t* strides, const uint32_t* box) {
  auto enc = get_encode();
  if (!enc) return cudaErrorNotSupported;
  if (((uintptr_t)ptr & 15) || rank < 2 || rank > 3) return cudaErrorInvalidValue;
  cuuint64_t d[3], st[2];
  cuuint32_t b[3], estr[3] = {1, 1, 1};
  for (int i = 0; i < rank; i++) {
    d[i] = dims[i];
    b[i] = box[i];
  }
  for (int i = 0; i < rank - 1; i++) {
    if (strides[i] % 16) return cudaErrorInvalidValue;
    st[i] = strides[i];
  }
  CUresult r = enc(tm, dt, rank, const_cast<void*>(ptr), d, st, b, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Opt every instantiation into its shared-memory size once, outside any stream capture (fpd_model_create).
cudaError_t tc_init_attributes() {
  cudaError_t e = cudaSuccess;
  if (e == cudaSuccess) e = set_attr<16, 6, true, EPI_STORE>();
  if (e == cudaSuccess) e = set_attr<32, 5, true, EPI_STORE>();
  if (e == cudaSuccess) e = set_attr<64, 4, true, EPI_STORE>();
  if (e == cudaSuccess) e = set_attr<128, 6, false, EPI_STORE>();
  if (e == cudaSuccess) e = set_attr<256, 4, false, EPI_STORE>();
  if (e == cudaSuccess) e = set_attr<16, 6, true, EPI_ARGMAX>();
  if (e == cudaSuccess) e = set_attr<32, 5, true, EPI_ARGMAX>();
  if (e == cudaSuccess) e = set_attr<64, 4, true, EPI_ARGMAX>();
  if (e == cudaSuccess) e = set_attr<16, 10, true, EPI_SWIGLU>();
  if (e == cudaSuccess) e = set_attr<32, 8, true, EPI_SWIGLU>();
  if (e == cudaSuccess) e = set_attr<64, 6, true, EPI_SWIGLU>();
  if (e == cudaSuccess) e = set_attr<256, 4, false, EPI_SWIGLU>();
  if (e == cudaSuccess) e = set_attr<128, 6, false, EPI_QKV_TOK>();
  if (e == cudaSuccess) e = set_attr<256, 4, false, EPI_QKV_TOK>();
  if (e == cudaSuccess) e = set_attr<128, 6, false, EPI_RESID_TOK>();
  if (e == cudaSuccess) e = set_attr<256, 4, false, EPI_RESID_TOK>();
  if (e == cudaSuccess) e = set_attr<256, 4, false, EPI_KV_CTX>();
  if (e == cudaSuccess) e = set_attr<128, 6, false, EPI_KV_CTX>();
  return e;
}

// Token-tile plan for the fused epilogues (no split-K: the epilogue needs complete sums).  A CTA streams its
// operands at a rate set by the SM, not by the tile shape, so a tile costs about its operand bytes, (128 + bn) K,
// and the GEMM about waves x that: the weight-tile width (256 or 128) with the smaller product wins, 256 on ties.
TcPlan tc_plan_tok(int M, int N, int K, int num_sms) {
  TcPlan pl{};
  pl.swap = false;
  pl.pt = ceil_div(M, BM);
  const long w256 = ceil_div(pl.pt * ceil_div(N, 256), num_sms), w128 = ceil_div(pl.pt * ceil_div(N, 128), num_sms);
  pl.bn = w256 * (BM + 256) <= w128 * (BM + 128) ? 256 : 128;
  pl.qt = ceil_div(N, pl.bn);
  pl.splits = 1;
  pl.k_split = K;
  pl.grid = std::min(pl.pt * pl.qt, num_sms);
  return pl;
}

cudaError_t launch_tc_tok(const TokGemm& g, const TcPlan& pl, cudaStream_t st) {
  if (g.M <= 0) return cudaSuccess;
  if (g.K % BK || pl.swap || pl.splits != 1) return cudaErrorInvalidValue;
  TcParams p;
  memset(&p, 0, sizeof(p));
  cudaError_t e = make_tmap(&p.tm_x[0], g.x, g.M, g.K, g.K, BM);
  if (e != cudaSuccess) return e;
  e = make_tmap(&p.tm_w, g.w, g.N, g.K, g.K, pl.bn);
  if (e != cudaSuccess) return e;
  p.n_seg = 1;
  p.seg_k = g.K;
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.pt = pl.pt;
  p.qt = pl.qt;
  p.splits = 1;
  p.k_split = g.K;
  p.q = g.q;
  p.kblk = g.kblk;
  p.vblk = g.vblk;
  p.q_norm = g.q_norm;
  p.k_norm = g.k_norm;
  p.rope = g.rope;
  p.ctx_len = g.ctx_len;
  p.t_cap = g.t_cap;
  p.L = g.L;
  p.nq = g.nq;
  p.nkv = g.nkv;
  p.hd = g.hd;
  p.eps = g.eps;
  p.xres = g.xres;
  p.ss_part = g.ss_part;
  if (g.qkv) {
    if (pl.bn == 128) return launch_kernel<128, 6, false, EPI_QKV_TOK>(p, pl.grid, st);
    return launch_kernel<256, 4, false, EPI_QKV_TOK>(p, pl.grid, st);
  }
  if (pl.bn == 128) return launch_kernel<128, 6, false, EPI_RESID_TOK>(p, pl.grid, st);
  return launch_kernel<256, 4, false, EPI_RESID_TOK>(p, pl.grid, st);
}

// Width of the weight tile of the context K/V GEMM: whole heads per tile and whole tiles per layer; 0 if none fits.
static int kvctx_bn(const fpd_model_desc& d) {
  const int kv_cols = 2 * d.n_kv_heads * d.head_dim;
  for (int bn : {256, 128})
    if (kv_cols % bn == 0 && bn % d.head_dim == 0) return bn;
  return 0;
}

bool kvctx_supported(const fpd_model_desc& d) {
  return kvctx_bn(d) > 0 && (d.head_dim == 128 || d.head_dim == 64) && d.d_model % BK == 0 &&
         d.n_layers <= FPD_MAX_LAYERS;
}

cudaError_t launch_tc_kvctx(const KvCtxGemm& g, int num_sms, cudaStream_t st) {
  if (g.R <= 0) return cudaSuccess;
  const fpd_model_desc& d = *g.d;
  const int bn = kvctx_bn(d);
  if (!kvctx_supported(d)) return cudaErrorInvalidValue;
  TcParams p;
  memset(&p, 0, sizeof(p));
  const int h = d.head_dim, kv_cols = 2 * d.n_kv_heads * h, nqkv = (d.n_q_heads + 2 * d.n_kv_heads) * h;
  cudaError_t e = make_tmap(&p.tm_x[0], g.ctx, g.R, d.d_model, d.d_model, BM);
  for (int l = 0; l < d.n_layers && e == cudaSuccess; l++) {
    e = make_tmap(&p.tm_wl[l], g.wqkv[l], nqkv, d.d_model, d.d_model, bn);
    p.k_norm_l[l] = g.k_norm[l];
  }
  if (e != cudaSuccess) return e;
  p.n_seg = 1;
  p.seg_k = d.d_model;
  p.M = g.R;
  p.N = d.n_layers * kv_cols;
  p.K = d.d_model;
  p.pt = ceil_div(g.R, BM);
  p.qt = p.N / bn;
  p.splits = 1;
  p.k_split = d.d_model;
  p.kv_cols = kv_cols;
  p.kv_row_base = d.n_q_heads * h;
  p.n_layers = d.n_layers;
  p.store = g.store;
  p.rope = g.rope;
  p.row_off = g.row_off;
  p.row_cnt = g.row_cnt;
  p.pos_start = g.pos_start;
  p.batch = g.batch;
  p.row0 = g.row0;
  p.t_cap = g.t_cap;
  p.nkv = d.n_kv_heads;
  p.hd = h;
  p.eps = d.rms_eps;
  const int grid = std::min(p.pt * p.qt, num_sms);
  if (bn == 256) return launch_kernel<256, 4, false, EPI_KV_CTX>(p, grid, st);
  return launch_kernel<128, 6, false, EPI_KV_CTX>(p, grid, st);
}

TcPlan tc_plan_gemm(int M, int N, int K, int num_sms) {
  TcPlan pl{};
  const int nkb = K / BK;
  int ctas_per_sm;
  if (M <= 64) {
    pl.swap = true;
    pl.bn = M <= 16 ? 16 : (M <= 32 ? 32 : 64);
    pl.pt = ceil_div(N, BM);
    pl.qt = ceil_div(M, pl.bn);
    ctas_per_sm = pl.bn == 16 ? kSwap16CtasPerSm : 2;
  } else {
    pl.swap = false;
    pl.bn = N >= 1024 ? 256 : 128;
    pl.pt = ceil_div(M, BM);
    pl.qt = ceil_div(N, pl.bn);
    ctas_per_sm = 1;
  }
  const int tiles = pl.pt * pl.qt;
  const int slots = num_sms * ctas_per_sm;
  int splits = 1;
  if (2 * tiles <= slots || pl.swap) {
    if (tiles < slots) splits = std::max(1, std::min(slots / tiles, nkb / 4));
  } else {
    // More than half a wave of tiles: split K when the last wave is short.  A split of s costs ceil(tiles s / slots) waves
    // of K/s each, plus its extra fp32 partial (M N 4 bytes written and read back) spread over the SMs, counted in
    // the same unit (K elements a tile streams: (128 + bn) 2 bytes each).
    const double part_k = (double)M * N * 8 / slots / ((BM + pl.bn) * 2);
    double best = 0.0;
    for (int s = 1; s <= 4 && (s == 1 || nkb / s >= 8); s++) {
      const int kb = ceil_div(nkb, s);
      const double cost = (double)ceil_div(tiles * s, slots) * kb * BK + (s - 1) * part_k;
      if (s == 1 || cost < best) {
        best = cost;
        splits = s;
      }
    }
  }
  const int kb_per = ceil_div(nkb, splits);
  pl.k_split = kb_per * BK;
  pl.splits = ceil_div(nkb, kb_per);
  pl.grid = std::min(tiles * pl.splits, slots);
  return pl;
}

TcPlan tc_plan_force(int M, int N, int K, int num_sms, int placement) {
  TcPlan pl = tc_plan_gemm(M, N, K, num_sms);
  if (placement < 0 || (placement == 1) == pl.swap) return pl;
  const int nkb = K / BK;
  pl.swap = placement == 1;
  if (pl.swap) {
    pl.bn = M <= 16 ? 16 : (M <= 32 ? 32 : 64);
    pl.pt = ceil_div(N, BM);
    pl.qt = ceil_div(M, pl.bn);
  } else {
    pl.bn = N >= 1024 ? 256 : 128;
    pl.pt = ceil_div(M, BM);
    pl.qt = ceil_div(N, pl.bn);
  }
  const int slots = num_sms * (pl.swap ? 2 : 1);
  const int tiles = pl.pt * pl.qt;
  int splits = 1;
  if (tiles < slots) splits = std::max(1, std::min(slots / tiles, nkb / 4));
  const int kb_per = ceil_div(nkb, splits);
  pl.k_split = kb_per * BK;
  pl.splits = ceil_div(nkb, kb_per);
  pl.grid = std::min(tiles * pl.splits, slots);
  return pl;
}

namespace {
__global__ void sum_splits_kernel(float* __restrict__ out, const float* __restrict__ part, int splits, size_t n) {
  pdl_trigger();
  pdl_wait();
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    float a = 0.f;
    for (int s = 0; s < splits; s++) a += part[s * n + i];
    out[i] = a;
  }
}
}  // namespace

cudaError_t launch_sum_splits(float* out, const float* part, int splits, size_t n, cudaStream_t st) {
  return launch_k(sum_splits_kernel, (int)std::min<size_t>((n + 255) / 256, 4096), 256, 0, st, out, part, splits, n);
}

cudaError_t launch_tc_gemm(const GemmArgs& g, const TcPlan& pl, cudaStream_t st) {
  if (g.M <= 0 || g.N <= 0) return cudaSuccess;
  if (g.K % BK || g.seg_k % BK || g.k_split != pl.k_split) return cudaErrorInvalidValue;
  TcParams p;
  memset(&p, 0, sizeof(p));
  const int x_box = pl.swap ? pl.bn : BM, w_box = pl.swap ? BM : pl.bn;
  p.n_seg = g.K / g.seg_k;
  if (p.n_seg < 1 || p.n_seg > 8) return cudaErrorInvalidValue;
  for (int s = 0; s < p.n_seg; s++) {
    cudaError_t e = make_tmap(&p.tm_x[s], g.a[s], g.M, g.seg_k, g.lda, x_box);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = make_tmap(&p.tm_w, g.b, g.N, g.K, g.ldb, w_box);
  if (e != cudaSuccess) return e;
  p.seg_k = g.seg_k;
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.c = g.c;
  p.ldc = g.ldc;
  p.c_split_stride = g.c_split_stride;
  p.pt = pl.pt;
  p.qt = pl.qt;
  p.splits = pl.splits;
  p.k_split = pl.k_split;
  if (pl.swap) {
    if (pl.bn == 16) return launch_kernel<16, 6, true, EPI_STORE>(p, pl.grid, st);
    if (pl.bn == 32) return launch_kernel<32, 5, true, EPI_STORE>(p, pl.grid, st);
    return launch_kernel<64, 4, true, EPI_STORE>(p, pl.grid, st);
  }
  if (pl.bn == 128) return launch_kernel<128, 6, false, EPI_STORE>(p, pl.grid, st);
  return launch_kernel<256, 4, false, EPI_STORE>(p, pl.grid, st);
}

// Gate/up projection with the SwiGLU epilogue: one pass over [gate; up] (no split-K: the nonlinearity needs
// complete sums), tiles of 64 features (weight-tile placement) or 128 features (token-tile placement).
TcPlan tc_plan_swiglu(int M, int F, int K, int num_sms) {
  TcPlan pl{};
  pl.splits = 1;
  pl.k_split = K;
  if (M <= 64) {
    pl.swap = true;
    pl.bn = M <= 16 ? 16 : (M <= 32 ? 32 : 64);
    pl.pt = ceil_div(F, BM / 2);
    pl.qt = ceil_div(M, pl.bn);
  } else {
    pl.swap = false;
    pl.bn = 256;
    pl.pt = ceil_div(M, BM);
    pl.qt = ceil_div(F, 128);
  }
  pl.grid = std::min(pl.pt * pl.qt, num_sms);
  return pl;
}

cudaError_t launch_tc_swiglu(const bf16* x, int M, int K, const bf16* w_gate_up, int F, bf16* hmid, const TcPlan& pl,
                             cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  if (K % BK) return cudaErrorInvalidValue;
  TcParams p;
  memset(&p, 0, sizeof(p));
  const int x_box = pl.swap ? pl.bn : BM, w_box = pl.swap ? BM / 2 : pl.bn / 2;
  cudaError_t e = make_tmap(&p.tm_x[0], x, M, K, K, x_box);
  if (e != cudaSuccess) return e;
  e = make_tmap(&p.tm_w, w_gate_up, 2 * F, K, K, w_box);
  if (e != cudaSuccess) return e;
  p.n_seg = 1;
  p.seg_k = K;
  p.M = M;
  p.N = 2 * F;
  p.K = K;
  p.pt = pl.pt;
  p.qt = pl.qt;
  p.splits = 1;
  p.k_split = K;
  p.hmid = hmid;
  p.F = F;
  if (pl.swap) {
    if (pl.bn == 16) return launch_kernel<16, 10, true, EPI_SWIGLU>(p, pl.grid, st);
    if (pl.bn == 32) return launch_kernel<32, 8, true, EPI_SWIGLU>(p, pl.grid, st);
    return launch_kernel<64, 6, true, EPI_SWIGLU>(p, pl.grid, st);
  }
  return launch_kernel<256, 4, false, EPI_SWIGLU>(p, pl.grid, st);
}

int tc_lm_row_tile(int n_rows) { return n_rows <= 16 ? 16 : (n_rows <= 32 ? 32 : 64); }

cudaError_t launch_tc_lmhead(const LmPlan& lp, const bf16* z_sorted, int n_rows, const bf16* W, int d, int V,
                             const int4* items, const int* n_items, int max_items, unsigned long long* packed,
                             unsigned long long* packed2, const int* rows_sorted, float* logits, int num_sms,
                             bool unconstrained, cudaStream_t st) {
  if (d % BK) return cudaErrorInvalidValue;
  const int bn = lp.rt;
  TcParams p;
  memset(&p, 0, sizeof(p));
  cudaError_t e = make_tmap(&p.tm_x[0], z_sorted, n_rows, d, d, bn);
  if (e != cudaSuccess) return e;
  e = make_tmap(&p.tm_w, W, V, d, d, BM);
  if (e != cudaSuccess) return e;
  p.n_seg = 1;
  p.seg_k = d;
  p.M = n_rows;
  p.N = V;
  p.K = d;
  p.items = items;
  p.n_items = n_items;
  if (lp.n_class == 1 && lp.n_range == 1 && lp.range_lo[0] == 0 && lp.range_hi[0] == V && unconstrained) {
    p.implicit_rowtiles = ceil_div(n_rows, bn);
    p.implicit_total = p.implicit_rowtiles * ceil_div(V, BM);
  }
  for (int q = 0; q < lp.n_range; q++) p.hi_tab[q] = lp.range_hi[q];
  p.packed = packed;
  p.packed2 = packed2;
  p.rows_sorted = rows_sorted;
  p.logits = logits;
  p.V = V;
  const int n_work = p.implicit_rowtiles > 0 ? p.implicit_total : max_items;
  const int per_sm = 2;
  const int grid = std::max(1, std::min(n_work, per_sm * num_sms));
  if (bn == 16) return launch_kernel<16, 6, true, EPI_ARGMAX>(p, grid, st);
  if (bn == 32) return launch_kernel<32, 5, true, EPI_ARGMAX>(p, grid, st);
  return launch_kernel<64, 4, true, EPI_ARGMAX>(p, grid, st);
}

}  // namespace fpd

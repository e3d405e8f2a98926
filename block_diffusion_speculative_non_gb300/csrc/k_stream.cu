// k_stream.cu — the few-token path (at most 16 block positions in a call, e.g. one request's 16-position text
// block): weight-streaming tcgen05 GEMMs with the preceding RMSNorm applied while the activations are loaded,
// split-K reduced inside the GEMM, and the per-tile epilogues of the drafter layer fused in.
//
// At batch 1 the drafter pass is a stream of 1.8 GB of weights through 16 tokens (VFlash blog, "Key claims": the
// five-layer drafter runs one forward per block; FlashDrive §3.4: decoding is bandwidth-bound), so the design
// goal is to keep HBM busy and to spend as little time as possible between weight streams:
//
//   - One CTA per SM (grid = output tiles x K splits, each CTA one work item; the LM head is persistent over
//     its id tiles).  Warp 0 streams 128-row weight atoms (K = 64, 16 KB, 128-byte swizzle) through an 8-deep
//     TMA ring, starting before the predecessor kernel has finished (weights never depend on it).  Warp 1
//     issues tcgen05.mma (M = 128 weight rows, N = 16 tokens, K = 16, fp32 in TMEM).  Warps 2-5 build the
//     16-token activation slice ONCE in shared memory — applying RMSNorm on the way in when the GEMM consumes a
//     normed residual stream — and later run the epilogue from TMEM.
//   - RMSNorm on load: the residual kernels leave per-(tile, token) sums of squares of the bf16 residual; the
//     consumer adds them in a fixed order, so xn = bf16(x * rsqrt(mean(x^2) + eps) * g) equals what a separate
//     norm kernel would store (the bf16 storage point of the normed projection input).
//   - Split-K without a reduce kernel: every CTA writes its fp32 partial tile; the LAST CTA of a tile to arrive
//     (an atomic counter, no waiting) sums all partials in split order — bit-reproducible — and runs the
//     epilogue: q/k RMSNorm + RoPE for the QKV projection, residual add + sum of squares for O and down.
//   - LM head (no vocabulary constraint): every CTA keeps a running top-2 (logit, id) per position over its id
//     tiles and writes it to its own slot; a one-warp-per-position decode merges the slots (argmax with
//     lowest-id ties, and the top-2 margin).
#include <cstring>

#include "fewtok_common.cuh"

namespace fpd {

namespace {
using namespace fewtok;

constexpr int kSThreads = 192;
constexpr int kMinStages = 8;                 // weight ring depth: 8 atoms (128 KB) in flight per CTA; deeper rings
constexpr int kMaxStages = 8;                 // (10-14 atoms) measured slower on the 4B shape at batch 1
constexpr int kTmemCols = 32;                 // two 16-column accumulators
constexpr int kAccSlots = 8;                  // 8-bit weights: one 16-column accumulator per weight atom, 8 in flight
constexpr int kTmemCols8 = kAccSlots * SBN;
constexpr int kXRing = kMaxStages + kAccSlots;   // 8-bit: weight-row exponents of the last 16 weight atoms (128 B each)
constexpr int kActGroup = 4;                  // activation atoms per readiness barrier
constexpr int kMaxActGroups = 12;             // activation slices of up to 48 atoms (K <= 3072)
constexpr int kXsLd = 2 * kMaxActGroups;      // 8-bit activation scales per token: one per 128-element block
// misc region: mbarriers full[S], empty[S], act_tma[G], act_ready[G], tfull[8], tempty[8], xfull[16] | TMEM slot,
// abort, last-CTA flag | inverse RMS per token [16] | context length per request [16] | running top-2 per token
// [16][2] | 8-bit activation scales [16][kXsLd] | 8-bit weight-exponent ring [16][128]
constexpr int kMiscFlags = 8 * (2 * kMaxStages + 2 * kMaxActGroups + 2 * kAccSlots + kXRing);
constexpr int kMiscInv = kMiscFlags + 16;
constexpr int kMiscCtx = kMiscInv + SBN * 4;
constexpr int kMiscRun = kMiscCtx + SBN * 4;
constexpr int kMiscXs = kMiscRun + SBN * 16;
constexpr int kMiscXe = kMiscXs + SBN * kXsLd * 4;
constexpr int kMiscBytes = kMiscXe + kXRing * SBM;

struct StreamParams {
  CUtensorMap tm_w;            // weights [rows, K] bf16, box 64 x (128, SwiGLU: 64); 8-bit: E4M3 bytes, box 128 x ..
  CUtensorMap tm_x;            // activation source: 2-D [M rows, K] (box 64 x 16) or, for the LM head, 3-D
                               // [B][L-1 rows starting at block position 1][K] (box 64 x (L-1) x B)
  int x_rank;                  // 2 or 3
  uint32_t x_atom_bytes;       // bytes one activation atom load delivers
  int M;                       // tokens (<= 16)
  int N;                       // output features (SwiGLU: F; LM head: V)
  int K;
  int tiles, splits, k_split;  // output tiles, K splits, K elements per split (multiple of 64)
  int xform;                   // XF_*
  const float* ss_in;          // XF_NORM: sums of squares [n_ss][16]
  int n_ss;
  const bf16* gain;            // XF_NORM / XF_NORM_FULL: RMSNorm gain [K]
  float eps;
  // split-K reduction
  float* part;                 // [splits][tiles][128][16]
  int* counters;               // [tiles], zero on entry, left zero
  // SEPI_QKV
  bf16 *q, *kblk, *vblk;
  const bf16 *q_norm, *k_norm;
  const float2* rope;
  const int32_t* ctx_len;
  int t_cap, L, nq, nkv, h;
  // SEPI_RESID
  bf16* xres;                  // [M][N], updated in place
  float* ss_out;               // [tiles][16]
  // SEPI_SWIGLU
  bf16* hmid;                  // [M][N]
  // SEPI_ARGMAX
  unsigned long long* slots;   // [gridDim][16][2]
  float* logits;               // [M][N] or null
  const int8_t* w_exp;         // 8-bit weights: exponents, block-major: (row r, block b) at w_exp[b * exp_ld + r]
  int exp_ld;                  // a multiple of 128 (>= rows): every atom's 128 (SwiGLU: 2 x 64) rows are one copy
  int w_rows;                  // rows of the weight matrix
  int stages;                  // weight ring depth, kMinStages..kMaxStages
  uint32_t test_extra_tx;      // 0; a test makes the first stage's wait run out with it (bounded-wait check)
};

// FP8: E4M3 weight atoms of 128 rows x 128 K (16 KB, the same bytes as a bf16 atom), the activation slice
// quantised in place to E4M3 blocks of 128 K with one scale per (token, block), tcgen05.mma kind::f8f6f4 into one
// accumulator slot per weight atom, and the epilogue threads adding each atom's product times
// 2^(k_activation + k_weight) in fp32 registers.
template <int EPI, bool FP8>
__global__ void __launch_bounds__(kSThreads, 1) stream_gemm_kernel(const __grid_constant__ StreamParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int KA = FP8 ? 2 : 1;                             // 64-K activation atoms per weight atom
  constexpr int n_slots = FP8 ? kAccSlots : 2;
  constexpr uint32_t tmem_cols = FP8 ? kTmemCols8 : kTmemCols;
  const int n_act = p.k_split / SBK;                          // activation atoms of one split (LM head: all K)
  uint8_t* ring = smem;
  const int n_stages = p.stages;
  uint8_t* act = smem + n_stages * W_ATOM;
  uint8_t* gbuf = act + n_act * X_ATOM;
  float* scratch = reinterpret_cast<float*>(gbuf + n_act * G_ATOM);
  uint8_t* misc = reinterpret_cast<uint8_t*>(scratch) + kEpiScratch;
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + kMiscFlags);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_flag = reinterpret_cast<int*>(tmem_slot + 2);
  float* s_inv = reinterpret_cast<float*>(misc + kMiscInv);
  int* s_ctx = reinterpret_cast<int*>(misc + kMiscCtx);
  unsigned long long* s_run = reinterpret_cast<unsigned long long*>(misc + kMiscRun);
  float* s_xs = reinterpret_cast<float*>(misc + kMiscXs);
  const int8_t* s_xe = reinterpret_cast<const int8_t*>(misc + kMiscXe);
  const uint32_t full0 = tc::smem_u32(bars), empty0 = full0 + 8 * kMaxStages, actt0 = empty0 + 8 * kMaxStages,
                 actr0 = actt0 + 8 * kMaxActGroups, tfull0 = actr0 + 8 * kMaxActGroups,
                 tempty0 = tfull0 + 8 * kAccSlots, xfull0 = tempty0 + 8 * kAccSlots;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  pdl_trigger();
  const bool persistent = EPI == SEPI_ARGMAX;
  const int total = persistent ? p.tiles : p.tiles * p.splits;
  const int stride = persistent ? gridDim.x : total;   // one work item per CTA otherwise

  if (threadIdx.x == 0) {
    for (int s = 0; s < n_stages; s++) {
      tc::mbar_init(full0 + 8 * s, 1);
      tc::mbar_init(empty0 + 8 * s, 1);
    }
    for (int g = 0; g < kMaxActGroups; g++) {
      tc::mbar_init(actt0 + 8 * g, 1);
      tc::mbar_init(actr0 + 8 * g, 1);
    }
    for (int a = 0; a < n_slots; a++) {
      tc::mbar_init(tfull0 + 8 * a, 1);
      tc::mbar_init(tempty0 + 8 * a, 4);
    }
    if (FP8)
      for (int a = 0; a < kXRing; a++) tc::mbar_init(xfull0 + 8 * a, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tc::smem_u32(tmem_slot), tmem_cols);
    tc::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch(&p.tm_w);
    tc::tma_prefetch(&p.tm_x);
  }
  // The single-lane roles reconverge with their warps first: a CTA barrier reached by part of a diverged
  // warp counts the whole warp, and the lagging lane would then pass it without waiting.
  __syncwarp();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // work item t -> output tile, K range, weight atoms
  auto item = [&](int t, int& tile, int& split, int& k0, int& nkb) {
    tile = persistent ? t : t % p.tiles;
    split = persistent ? 0 : t / p.tiles;
    k0 = split * p.k_split;
    nkb = (min(p.K, k0 + p.k_split) - k0) / (SBK * KA);
  };
  int tile0, split0, k00, nkb0;   // the CTA's first item: its K slice is the activation slice
  item(blockIdx.x < total ? blockIdx.x : 0, tile0, split0, k00, nkb0);
  const int nxa0 = nkb0 * KA;     // its 64-K activation atoms

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int stage = 0, issued = 0, t = blockIdx.x, kb = 0, tile, split, k0, nkb;
      uint32_t phase = 0;
      if (t < total) item(t, tile, split, k0, nkb);
      auto issue_w = [&]() {
        const uint32_t fb = full0 + 8 * stage, dst = tc::smem_u32(ring + stage * W_ATOM);
        tc::mbar_arrive_expect_tx(fb, W_ATOM + (issued == 0 ? p.test_extra_tx : 0u));
        const int kx = k0 + kb * SBK * KA;   // element (= byte, 8-bit) column of the atom
        if (EPI == SEPI_SWIGLU) {   // atom = [gate rows f0..f0+63 ; up rows F+f0..F+f0+63]
          tc::tma_load_2d(dst, &p.tm_w, kx, tile * 64, fb);
          tc::tma_load_2d(dst + W_ATOM / 2, &p.tm_w, kx, p.N + tile * 64, fb);
        } else {
          tc::tma_load_2d(dst, &p.tm_w, kx, tile * SBM, fb);
        }
        if (FP8) {   // the atom's 128 row exponents into exponent slot issued % kXRing (read by the epilogue)
          const int xs = issued % kXRing;
          const uint32_t xb = xfull0 + 8 * xs, xd = tc::smem_u32(s_xe + xs * SBM);
          const int8_t* src = p.w_exp + (size_t)(kx / 128) * p.exp_ld;
          tc::mbar_arrive_expect_tx(xb, SBM);
          if (EPI == SEPI_SWIGLU) {
            tc::bulk_load(xd, src + tile * 64, 64, xb);
            tc::bulk_load(xd + 64, src + p.N + tile * 64, 64, xb);
          } else {
            tc::bulk_load(xd, src + tile * SBM, SBM, xb);
          }
        }
        issued++;
        if (++stage == n_stages) { stage = 0; phase ^= 1; }
        if (++kb == nkb) {
          kb = 0;
          t += stride;
          if (t < total) item(t, tile, split, k0, nkb);
        }
      };
      // the first ring of weights: weights never depend on earlier kernels, so no griddepcontrol.wait yet
      while (t < total && issued < n_stages) issue_w();
      // the activation slice (and the norm gain slice) once the predecessor kernel has completed, in groups of
      // kActGroup atoms so that the transform and the products start on the first group
      pdl_wait();
      if (blockIdx.x < total) {
        const bool gains = p.xform != XF_COPY;
        for (int g = 0; g * kActGroup < nxa0; g++) {
          const int a0 = g * kActGroup, na = min(kActGroup, nxa0 - a0);
          const uint32_t bar = actt0 + 8 * g;
          tc::mbar_arrive_expect_tx(bar, na * p.x_atom_bytes + (gains ? na * G_ATOM : 0));
          for (int a = a0; a < a0 + na; a++) {
            if (p.x_rank == 3)
              tc::tma_load_3d(tc::smem_u32(act + a * X_ATOM), &p.tm_x, k00 + a * SBK, 0, 0, bar);
            else
              tc::tma_load_2d(tc::smem_u32(act + a * X_ATOM), &p.tm_x, k00 + a * SBK, 0, bar);
          }
          if (gains) tc::bulk_load(tc::smem_u32(gbuf + a0 * G_ATOM), p.gain + k00 + a0 * SBK, na * G_ATOM, bar);
        }
      }
      while (t < total && !*abort_flag) {
        if (!tc::mbar_wait(empty0 + 8 * stage, phase ^ 1)) {
          *abort_flag = 1;
          break;
        }
        issue_w();
      }
      if (*abort_flag) {   // let the copies already issued land before the CTA may exit (bounded)
        for (int s = 0; s < n_stages && s < issued; s++) {
          if (--stage < 0) { stage = n_stages - 1; phase ^= 1; }
          tc::mbar_wait(full0 + 8 * stage, phase);
        }
        if (FP8)
          for (int c = issued - 1; c >= 0 && c >= issued - kXRing; c--)
            tc::mbar_wait(xfull0 + 8 * (c % kXRing), (c / kXRing) & 1);
        if (blockIdx.x < total)
          for (int g = 0; g * kActGroup < nxa0; g++) tc::mbar_wait(actt0 + 8 * g, 0);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0 && FP8) {
      // one accumulator slot per weight atom; the epilogue threads free a slot once they have read it
      constexpr uint32_t idesc = tc::idesc_e4m3_f32(SBM, SBN);
      int stage = 0, c = 0;
      uint32_t phase = 0;
      const uint32_t xs = tc::smem_u32(act);
      for (int t = blockIdx.x; t < total && !*abort_flag; t += stride) {
        int tile, split, k0, nkb;
        item(t, tile, split, k0, nkb);
        for (int kb = 0; kb < nkb && !*abort_flag; kb++, c++) {
          // 8-bit block kb is ready once its activation group has been quantised
          if ((kb * KA) % kActGroup == 0 && !tc::mbar_wait(actr0 + 8 * (kb * KA / kActGroup), 0)) { *abort_flag = 1; break; }
          const int slot = c % kAccSlots;
          if (c >= kAccSlots && !tc::mbar_wait(tempty0 + 8 * slot, ((c / kAccSlots) & 1) ^ 1)) { *abort_flag = 1; break; }
          if (!tc::mbar_wait(full0 + 8 * stage, phase)) { *abort_flag = 1; break; }
          tc::tc_fence_after();
          const uint32_t ws = tc::smem_u32(ring + stage * W_ATOM), d_tmem = tmem_base + slot * SBN;
#pragma unroll
          for (int kk = 0; kk < 4; kk++) {   // K = 32 bytes per instruction
            const uint64_t da = tc::sw128_kmajor_desc(ws + kk * 32);
            const uint64_t db = tc::sw128_kmajor_desc(xs + kb * X_ATOM + kk * 32);
            tc::umma_f8(d_tmem, da, db, idesc, kk > 0 ? 1u : 0u);
          }
          tc::umma_commit(empty0 + 8 * stage);
          tc::umma_commit(tfull0 + 8 * slot);
          if (++stage == n_stages) { stage = 0; phase ^= 1; }
        }
      }
    } else if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(SBM, SBN);
      // activation atoms are ready group by group: straight from TMA, or after the norm transform
      const uint32_t rdy0 = p.xform == XF_COPY ? actt0 : actr0;
      int stage = 0, it = 0;
      uint32_t phase = 0;
      const uint32_t xs = tc::smem_u32(act);
      for (int t = blockIdx.x; t < total; t += stride, it++) {
        int tile, split, k0, nkb;
        item(t, tile, split, k0, nkb);
        const int acc = it & 1;
        if (it >= 2 && !*abort_flag && !tc::mbar_wait(tempty0 + 8 * acc, ((it >> 1) & 1) ^ 1)) *abort_flag = 1;
        tc::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * SBN;
        for (int kb = 0; kb < nkb && !*abort_flag; kb++) {
          if (kb % kActGroup == 0 && !tc::mbar_wait(rdy0 + 8 * (kb / kActGroup), 0)) { *abort_flag = 1; break; }
          if (!tc::mbar_wait(full0 + 8 * stage, phase)) { *abort_flag = 1; break; }
          tc::tc_fence_after();
          const uint32_t ws = tc::smem_u32(ring + stage * W_ATOM);
#pragma unroll
          for (int kk = 0; kk < SBK / SUK; kk++) {
            const uint64_t da = tc::sw128_kmajor_desc(ws + kk * SUK * 2);
            const uint64_t db = tc::sw128_kmajor_desc(xs + kb * X_ATOM + kk * SUK * 2);
            tc::umma_bf16(d_tmem, da, db, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          tc::umma_commit(empty0 + 8 * stage);
          if (++stage == n_stages) { stage = 0; phase ^= 1; }
        }
        tc::umma_commit(tfull0 + 8 * acc);
      }
    }
  } else {
    // ---------------- activation transform + epilogue: warps 2..5 ----------------
    const int et = threadIdx.x - 64;          // 0..127
    const int quarter = warp & 3;             // TMEM lanes [32*quarter, 32*quarter + 32)
    const int row_in_tile = quarter * 32 + lane;
    pdl_wait();                               // inputs and outputs belong to earlier kernels
    if (p.xform == XF_NORM) inv_from_partials(p.ss_in, p.n_ss, p.K, p.eps, scratch, s_inv, et);
    if (EPI == SEPI_QKV && et < SBN) {
      int cl = et * p.L < p.M ? p.ctx_len[et] : 0;
      s_ctx[et] = clamp_ctx(cl, p.t_cap);
    }
    if (EPI == SEPI_ARGMAX && et < SBN) s_run[2 * et] = s_run[2 * et + 1] = 0ull;
    if (FP8) {
      // 8-bit: every activation group normed (when the GEMM consumes a normed stream) and quantised in one pass
      if (blockIdx.x < total) {
        const int n_groups = (nxa0 + kActGroup - 1) / kActGroup;
        if (p.xform == XF_NORM_FULL) {   // 1/rms from the whole rows: every group first
          for (int g = 0; g < n_groups; g++)
            if (!tc::mbar_wait(actt0 + 8 * g, 0)) *abort_flag = 1;
          inv_from_rows(act, nxa0, p.K, p.eps, s_inv, et);
        }
        epi_bar();   // s_inv complete
        for (int g = 0; g < n_groups; g++) {
          const int a0 = g * kActGroup, na = min(kActGroup, nxa0 - a0);
          if (p.xform != XF_NORM_FULL && !tc::mbar_wait(actt0 + 8 * g, 0)) *abort_flag = 1;
          norm_quant_atoms(act, gbuf, s_inv, s_xs, kXsLd, a0, na, p.M, et, p.xform != XF_COPY, g == 0);
          epi_bar();
          if (et == 0) tc::mbar_arrive(actr0 + 8 * g);
        }
      }
    } else if (blockIdx.x < total && p.xform != XF_COPY) {
      if (p.xform == XF_NORM_FULL) {   // 1/rms from the whole rows: every group first
        for (int g = 0; g * kActGroup < nxa0; g++)
          if (!tc::mbar_wait(actt0 + 8 * g, 0)) *abort_flag = 1;
        inv_from_rows(act, nxa0, p.K, p.eps, s_inv, et);
      }
      epi_bar();   // s_inv complete
      for (int g = 0; g * kActGroup < nxa0; g++) {
        if (p.xform == XF_NORM && !tc::mbar_wait(actt0 + 8 * g, 0)) *abort_flag = 1;
        norm_atoms(act, gbuf, s_inv, g * kActGroup, min(kActGroup, nxa0 - g * kActGroup), et);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic writes -> tensor-core reads
        epi_bar();
        if (et == 0) tc::mbar_arrive(actr0 + 8 * g);
      }
    }

    int it = 0, c8 = 0;
    for (int t = blockIdx.x; t < total; t += stride, it++) {
      int tile, split, k0, nkb;
      item(t, tile, split, k0, nkb);
      float xv[16];
      if (EPI == SEPI_RESID) resid_preload(xv, p.xres, p.N, tile, p.M, row_in_tile);
      float v[16];
      if (FP8) {
        // v = sum over the item's weight atoms of (block product) 2^(k_token + k_row); this thread's weight row
#pragma unroll
        for (int j = 0; j < 16; j++) v[j] = 0.f;
        for (int kb = 0; kb < nkb; kb++, c8++) {
          const int slot = c8 % kAccSlots, xs = c8 % kXRing;
          if (!*abort_flag && !tc::mbar_wait(tfull0 + 8 * slot, (c8 / kAccSlots) & 1)) *abort_flag = 1;
          // this atom's row exponent: its slot is rewritten only after this thread's warp frees the accumulator
          if (!*abort_flag && !tc::mbar_wait(xfull0 + 8 * xs, (c8 / kXRing) & 1)) *abort_flag = 1;
          const int ew = s_xe[xs * SBM + row_in_tile];
          tc::tc_fence_after();
          float u[16];
          tc::tmem_ld16(tmem_base + ((uint32_t)(quarter * 32) << 16) + slot * SBN, u);
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(tempty0 + 8 * slot);
          const float sw = exp2_int(ew);
#pragma unroll
          for (int j = 0; j < 16; j++) v[j] = fmaf(u[j], s_xs[j * kXsLd + kb] * sw, v[j]);
        }
        if (*abort_flag) {
#pragma unroll
          for (int j = 0; j < 16; j++) v[j] = 0.f;
        }
      } else {
        const int acc = it & 1;
        if (!tc::mbar_wait(tfull0 + 8 * acc, (it >> 1) & 1)) *abort_flag = 1;
        tc::tc_fence_after();
        tc::tmem_ld16(tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * SBN, v);
        if (*abort_flag) {
#pragma unroll
          for (int j = 0; j < 16; j++) v[j] = 0.f;
        }
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tempty0 + 8 * acc);
      }

      if (EPI == SEPI_QKV || EPI == SEPI_RESID) {
        if (splitk_last(v, p.part, p.counters, split, p.splits, tile, p.tiles, row_in_tile, et, s_flag)) {
          if (EPI == SEPI_RESID) {
            resid_epilogue(v, xv, p.xres, p.N, tile, p.M, p.ss_out, nullptr, scratch, quarter, lane, et);
          } else {
#pragma unroll
            for (int j = 0; j < 16; j++) scratch[j * SBM + row_in_tile] = v[j];
            epi_bar();
            QkvOut qo;
            qo.q = p.q;
            qo.kblk = p.kblk;
            qo.vblk = p.vblk;
            qo.q_norm = p.q_norm;
            qo.k_norm = p.k_norm;
            qo.rope = p.rope;
            qo.M = p.M;
            qo.L = p.L;
            qo.nq = p.nq;
            qo.nkv = p.nkv;
            qo.eps = p.eps;
            if (p.h == 128)
              qkv_tile_epilogue<128>(qo, scratch, tile, s_ctx, quarter, lane);
            else
              qkv_tile_epilogue<64>(qo, scratch, tile, s_ctx, quarter, lane);
            epi_bar();
          }
        }
      } else if (EPI == SEPI_SWIGLU) {   // split K when the feature tiles alone leave SMs idle
        if (splitk_last(v, p.part, p.counters, split, p.splits, tile, p.tiles, row_in_tile, et, s_flag))
          swiglu_epilogue(v, p.hmid, p.N, tile, p.M, scratch, row_in_tile);
      } else {
        // LM head: ids tile*128 + row, running top-2 per token
        const int vid = tile * SBM + row_in_tile;
        const bool ok = vid < p.N;
        unsigned long long* w2 = reinterpret_cast<unsigned long long*>(scratch);   // [4 warps][16][2]
#pragma unroll
        for (int j = 0; j < 16; j++) {
          unsigned long long a1 = (ok && j < p.M) ? pack_argmax(v[j], vid) : 0ull, a2 = 0ull;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long b1 = __shfl_xor_sync(0xffffffffu, a1, o);
            const unsigned long long b2 = __shfl_xor_sync(0xffffffffu, a2, o);
            top2_merge(a1, a2, b1, b2);
          }
          if (lane == 0) {
            w2[(quarter * SBN + j) * 2] = a1;
            w2[(quarter * SBN + j) * 2 + 1] = a2;
          }
          if (p.logits && ok && j < p.M) p.logits[(size_t)j * p.N + vid] = v[j];
        }
        epi_bar();
        if (et < SBN) {
          unsigned long long r1 = s_run[2 * et], r2 = s_run[2 * et + 1];
#pragma unroll
          for (int w = 0; w < 4; w++) top2_merge(r1, r2, w2[(w * SBN + et) * 2], w2[(w * SBN + et) * 2 + 1]);
          s_run[2 * et] = r1;
          s_run[2 * et + 1] = r2;
        }
        epi_bar();
      }
    }
    if (EPI == SEPI_ARGMAX && et < SBN) {
      p.slots[((size_t)blockIdx.x * SBN + et) * 2] = s_run[2 * et];
      p.slots[((size_t)blockIdx.x * SBN + et) * 2 + 1] = s_run[2 * et + 1];
    }
  }

  __syncwarp();
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem_base, tmem_cols);
  }
}

size_t stream_smem_bytes(int act_atoms, int stages) {
  return 1024 + (size_t)stages * W_ATOM + (size_t)act_atoms * (X_ATOM + G_ATOM) + kEpiScratch + kMiscBytes;
}

size_t stream_smem_bytes(int act_atoms) { return stream_smem_bytes(act_atoms, kMinStages); }

// The deepest ring that fits next to the activation slice: the more weight atoms a CTA holds, the more of its
// stream arrives while the preceding kernel is still finishing.
int stream_stages(int act_atoms) {
  int st = kMaxStages;
  while (st > kMinStages && stream_smem_bytes(act_atoms, st) > 227 * 1024) st--;
  return st;
}

template <int EPI>
cudaError_t launch_stream(const StreamParams& p, int grid, bool fp8, cudaStream_t st) {
  const size_t smem = stream_smem_bytes(p.k_split / SBK, p.stages);
  if (fp8) return launch_k(stream_gemm_kernel<EPI, true>, grid, kSThreads, smem, st, p);
  return launch_k(stream_gemm_kernel<EPI, false>, grid, kSThreads, smem, st, p);
}

template <int EPI>
cudaError_t stream_attr() {
  cudaError_t e = cudaFuncSetAttribute(stream_gemm_kernel<EPI, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       227 * 1024);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(stream_gemm_kernel<EPI, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  return e;
}

// ---- embedding gather for the few-token path: x rows + their sums of squares; clears the split-K counters ---------
__global__ void embed_ss_kernel(bf16* __restrict__ x, float* __restrict__ ss, int* __restrict__ counters, int n_cnt,
                                const bf16* __restrict__ embed, const int32_t* __restrict__ anchor, int32_t mask_id,
                                int L, int d, int V) {
  // wait first, trigger second: the kernels after this one may then read anything written before the call
  // (the context store, ctx_len) ahead of their own griddepcontrol.wait
  pdl_wait();
  pdl_trigger();
  __shared__ float red[32];
  const int r = blockIdx.x, b = r / L, j = r % L;
  if (r == 0)
    for (int i = threadIdx.x; i < n_cnt; i += blockDim.x) counters[i] = 0;
  int id = j == 0 ? anchor[b] : mask_id;
  const bool bad = id < 0 || id >= V;
  if (bad) {
    if (threadIdx.x == 0) record_check(kCheckBadToken);
    id = 0;
  }
  const uint4* src = reinterpret_cast<const uint4*>(embed + (size_t)id * d);
  uint4* dx = reinterpret_cast<uint4*>(x + (size_t)r * d);
  float s = 0.f;
  for (int i = threadIdx.x; i < d / 8; i += blockDim.x) {
    const uint4 u = bad ? make_uint4(0, 0, 0, 0) : src[i];
    dx[i] = u;
    const bf16* e = reinterpret_cast<const bf16*>(&u);
#pragma unroll
    for (int k = 0; k < 8; k++) s += bf(e[k]) * bf(e[k]);
  }
  s = warp_sum(s);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); w++) t += red[w];
    ss[r] = t;   // one partial per token: ss[0][r]
  }
}

// ---- argmax decode of the LM-head slots: one warp per position -------------------------------------------------
__global__ void stream_decode_kernel(int32_t* __restrict__ tokens, float* __restrict__ margin,
                                     const unsigned long long* __restrict__ slots, int n_slots, int n_rows) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (r >= n_rows) return;
  unsigned long long a1 = 0ull, a2 = 0ull;
  for (int g = lane; g < n_slots; g += 32)
    top2_merge(a1, a2, __ldcg(slots + ((size_t)g * SBN + r) * 2), __ldcg(slots + ((size_t)g * SBN + r) * 2 + 1));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long b1 = __shfl_xor_sync(0xffffffffu, a1, o);
    const unsigned long long b2 = __shfl_xor_sync(0xffffffffu, a2, o);
    top2_merge(a1, a2, b1, b2);
  }
  if (lane == 0) {
    if (!a1) record_check(kCheckNoLegalId);
    tokens[r] = a1 ? unpack_argmax_id(a1) : -1;
    if (margin)
      margin[r] = !a1 ? 0.f : (a2 ? (float)((double)unpack_argmax_val(a1) - (double)unpack_argmax_val(a2)) : INFINITY);
  }
}

}  // namespace

bool stream_shape_ok(const fpd_model_desc& d) {
  return d.d_model % SBM == 0 && (d.n_q_heads * d.head_dim) % SBM == 0 && (d.n_kv_heads * d.head_dim) % SBM == 0 &&
         d.d_ff % 64 == 0 && d.d_model % SBK == 0 && stream_smem_bytes(d.d_model / SBK) <= 227 * 1024 &&
         d.d_model / SBK <= kActGroup * kMaxActGroups;
}

StreamPlan stream_plan(int tiles, int K, int num_sms, bool split_ok, bool fp8) {
  StreamPlan pl{};
  pl.tiles = tiles;
  const int gran = fp8 ? 2 : 1;   // 64-K atoms per weight atom (8-bit atoms hold 128 K)
  const int nu = K / (SBK * gran);
  int splits = 1;
  if (split_ok && tiles < num_sms) splits = std::max(1, std::min(num_sms / tiles, nu / 2));
  int u_per = ceil_div(nu, splits);
  // the activation slice must fit next to the ring
  while (u_per > 1 && stream_smem_bytes(u_per * gran) > 227 * 1024) u_per = ceil_div(u_per, 2);
  const int kb_per = u_per * gran;
  pl.k_split = kb_per * SBK;
  pl.splits = ceil_div(nu, u_per);
  pl.grid = tiles * pl.splits;
  return pl;
}

size_t stream_part_floats(const StreamPlan& pl) { return pl.splits > 1 ? (size_t)pl.splits * pl.tiles * SBN * SBM : 0; }

cudaError_t launch_stream_gemm(const StreamGemm& g, cudaStream_t st) {
  StreamParams p;
  memset(&p, 0, sizeof(p));
  const int box_rows = g.epi == SEPI_SWIGLU ? 64 : SBM;
  const int w_rows = g.epi == SEPI_SWIGLU ? 2 * g.N : g.N;
  if (g.M < 1 || g.M > SBN || g.K % SBK || g.plan.k_split / SBK > kActGroup * kMaxActGroups)
    return cudaErrorInvalidValue;
  if (g.fp8 && (g.K % 128 || g.plan.k_split % 128 || !g.w8 || !g.w_exp || g.exp_ld % 128 || g.exp_ld < w_rows ||
                ((uintptr_t)g.w_exp & 15)))
    return cudaErrorInvalidValue;
  cudaError_t e = g.fp8 ? make_tmap_u8(&p.tm_w, g.w8, w_rows, g.K, g.K, box_rows)
                        : make_tmap(&p.tm_w, g.w, w_rows, g.K, g.K, box_rows);
  p.w_exp = g.w_exp;
  p.exp_ld = g.exp_ld;
  p.w_rows = w_rows;
  if (e != cudaSuccess) return e;
  if (g.xform == XF_NORM_FULL) {
    // rows of the LM head are block positions 1..L-1 of every request: a 3-D view [B][L-1][K] of hidden
    const int nb = g.M / (g.lm_block - 1);
    if (nb * (g.lm_block - 1) != g.M) return cudaErrorInvalidValue;
    const uint64_t dims[3] = {(uint64_t)g.K, (uint64_t)(g.lm_block - 1), (uint64_t)nb};
    const uint64_t strides[2] = {(uint64_t)g.ldx * 2, (uint64_t)g.lm_block * g.ldx * 2};
    const uint32_t box[3] = {(uint32_t)SBK, (uint32_t)(g.lm_block - 1), (uint32_t)nb};
    e = make_tmap_nd(&p.tm_x, g.x + g.ldx, 3, dims, strides, box);
    p.x_rank = 3;
    p.x_atom_bytes = (uint32_t)g.M * SBK * 2;
  } else {
    e = make_tmap(&p.tm_x, g.x, g.M, g.K, g.ldx, SBN);
    p.x_rank = 2;
    p.x_atom_bytes = X_ATOM;
  }
  if (e != cudaSuccess) return e;
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.tiles = g.plan.tiles;
  p.splits = g.plan.splits;
  p.k_split = g.plan.k_split;
  p.stages = stream_stages(g.plan.k_split / SBK);
  p.test_extra_tx = g.test_extra_tx;
  p.xform = g.xform;
  p.ss_in = g.ss_in;
  p.n_ss = g.n_ss;
  p.gain = g.gain;
  p.eps = g.eps;
  p.part = g.part;
  p.counters = g.counters;
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
  p.h = g.h;
  p.xres = g.xres;
  p.ss_out = g.ss_out;
  p.hmid = g.hmid;
  p.slots = g.slots;
  p.logits = g.logits;
  switch (g.epi) {
    case SEPI_QKV: return launch_stream<SEPI_QKV>(p, g.plan.grid, g.fp8, st);
    case SEPI_RESID: return launch_stream<SEPI_RESID>(p, g.plan.grid, g.fp8, st);
    case SEPI_SWIGLU: return launch_stream<SEPI_SWIGLU>(p, g.plan.grid, g.fp8, st);
    default: return launch_stream<SEPI_ARGMAX>(p, g.plan.grid, g.fp8, st);
  }
}

cudaError_t stream_init_attributes() {
  cudaError_t e = stream_attr<SEPI_QKV>();
  if (e == cudaSuccess) e = stream_attr<SEPI_RESID>();
  if (e == cudaSuccess) e = stream_attr<SEPI_SWIGLU>();
  if (e == cudaSuccess) e = stream_attr<SEPI_ARGMAX>();
  return e;
}

cudaError_t launch_embed_ss(bf16* x, float* ss, int* counters, int n_cnt, const bf16* embed, const int32_t* anchor,
                            int32_t mask_id, int B, int L, int d, int V, cudaStream_t st) {
  return launch_k(embed_ss_kernel, B * L, 256, 0, st, x, ss, counters, n_cnt, embed, anchor, mask_id, L, d, V);
}

cudaError_t launch_stream_decode(int32_t* tokens, float* margin, const unsigned long long* slots, int n_slots,
                                 int n_rows, cudaStream_t st) {
  return launch_k(stream_decode_kernel, 1, SBN * 32, 0, st, tokens, margin, slots, n_slots, n_rows);
}

}  // namespace fpd

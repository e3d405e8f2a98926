// k_attention_tc.cu — a5 for long blocks on the 5th-generation tensor cores: bidirectional grouped-query attention
// of query tiles of one (request, kv head) over [context K/V ; block K/V], head dim 128.
//
// VFlash paper (zh) §2.1: the fused target features enter every drafter layer as keys and values and the block is
// predicted in one bidirectional pass, so there is no mask inside a request.  At primitive lengths (L = 381, 385)
// the attention is a dense contraction: 4 (T + L) L h flops per head, about a quarter of the block's flops, so it
// runs on tcgen05 with the accumulators in tensor memory.
//
// One CTA = two query tiles of 128 rows (row r of a tile = position * group + head within the kv head's rows) x
// one KV split; both tiles share every K/V tile.  Warps:
//   0      TMA producer: K and V tiles of 128 keys (two 64-dim boxes each, 128-byte swizzle) into 2-slot rings;
//   1      MMA issuer: S_t = Q_t K_i^T for tile t = 0, 1 (M = 128 rows, N = 128 keys, fp32 into t's TMEM buffer),
//          and O_t += (P_hi + P_lo)_t V_i with P read from tensor memory and V as an MN-major shared-memory operand;
//          it issues S_t for the next key tile right after O_t's product, so each warpgroup waits only for its
//          own tile's MMAs;
//   2..5   softmax of tile 0, 6..9 softmax of tile 1, one thread per query row (= TMEM lane): the row maximum from
//          a first pass over S, then p = 2^(s log2e/sqrt(h) - m) written back over S 32 keys at a time as two bf16
//          terms (split_bf16x2; hi at columns [32c, 32c + 16), lo at [32c + 16, 32c + 32) for keys 32c..32c + 31,
//          so each chunk overwrites only the S columns it has just read); O in TMEM is rescaled only when the row
//          maximum rises by more than 2^8 over the reference (p then stays below 2^8), so O / l is exact;
//   10     clears the V rows past the last valid key of a partial tile (p = 0 there, and 0 x a stale non-finite
//          value would still be NaN).
// Two softmax warps share each SM sub-partition, so one hides the other's load and exponent latency, and each
// K/V tile is loaded once for 256 query rows.  The tensor core runs one thread's products in issue order, so
// S_t for key tile i + 1 may overwrite P_t of tile i as soon as that product has been issued.
// With one split the CTA writes O / l as bf16; with several it writes the unnormalised partial (o, m, l) that the
// merge kernel of k_attention.cu combines in split order.  Every mbarrier wait is bounded (tc::mbar_wait).
#include <cstring>

#include "fpd_kernels.cuh"
#include "tc_primitives.cuh"

namespace fpd {

namespace {

constexpr int AQ = 128, AKT = 128, AH = 128;
constexpr int NQT = 2;                     // query tiles per CTA, one softmax warpgroup each
constexpr int kAThreads = 11 * 32;
constexpr int NSTAGE = 2;
constexpr int TILE_BYTES = AKT * AH * 2;   // 32 KB: 128 rows x 128 dims, two 64-dim swizzle atoms
constexpr int ATOM_BYTES = TILE_BYTES / 2;
// shared memory: Q[2] | K[2] | V[2] | barriers
constexpr int SM_Q = 0, SM_K = NQT * TILE_BYTES, SM_V = SM_K + NSTAGE * TILE_BYTES, SM_BAR = SM_V + NSTAGE * TILE_BYTES;
// barriers: q_ready[tile], k_full[slot], k_empty[slot], v_full[slot], v_empty[slot], v_ready[slot] (stale rows
// cleared), s_full[tile], p_full[tile], pv_done[tile]
enum {
  B_Q = 0,
  B_KF = B_Q + NQT,
  B_KE = B_KF + NSTAGE,
  B_VF = B_KE + NSTAGE,
  B_VE = B_VF + NSTAGE,
  B_VR = B_VE + NSTAGE,
  B_SF = B_VR + NSTAGE,
  B_PF = B_SF + NQT,
  B_PV = B_PF + NQT,
  B_N = B_PV + NQT
};
constexpr size_t kASmem = 1024 + (size_t)SM_BAR + 8 * B_N + 16;
static_assert(kASmem <= 232448, "attention tile set exceeds the shared memory of one CTA");
constexpr int kTmemCols = 512;   // S/P of tile t at 128 t, O of tile t at 256 + 128 t
constexpr uint32_t kTmemO = 256;
constexpr float kRescaleLog2 = 8.f;

struct AttnTcParams {
  CUtensorMap tm_store;   // context KV store viewed as [rows][h]
  CUtensorMap tm_kblk;    // block keys [B * nkv * L][h]
  CUtensorMap tm_vblk;    // block values [B * nkv * L][h]
  const bf16* q;          // [B * L][nq][h]
  bf16* out;              // [B * L][nq][h]
  float* o_part;          // [splits][B * L][nq][h]
  float2* ml;             // [splits][B * L][nq]
  const int32_t* ctx_len;
  int batch, L, nq, nkv, t_cap, layer, rows, splits, chunk;
};

// Instruction descriptor of kind::f16 with fp32 accumulation and bf16 A and B; b_mn: B is MN-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
// Shared-memory descriptor of an MN-major operand stored as 128-byte-swizzled rows of 64 MN elements: successive
// 8-row groups along K are 1024 bytes apart (SBO), successive 64-element blocks along MN are `lbo` bytes apart.
__device__ __forceinline__ uint64_t sw128_mn_desc(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// D (TMEM) += A (TMEM: lane = row, 32-bit column = two consecutive K elements) x B (shared memory descriptor).
__device__ __forceinline__ void umma_ts_bf16(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  uint32_t u[16];
#pragma unroll
  for (int e = 0; e < 16; e++) u[e] = __float_as_uint(v[e]);
  tmem_st16(taddr, u);
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// 32 TMEM lanes x 32 consecutive columns -> 32 registers, without waiting (tmem_wait_ld completes a batch).
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 2^x on the special-function unit (ex2.approx, flush-to-zero): relative error near 2^-22 over the range used
// here (x <= 8), and 2^-inf = 0 for masked keys.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void named_bar(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

// The key tiles of a split: context tiles over [kb, min(ke, T)) from the store, then block tiles over
// [max(kb, T), ke) from kblk / vblk; each tile holds up to 128 keys.
struct TileList {
  int T, kb, ke, n_ctx, n_blk;
  __device__ void init(int T_, int kb_, int ke_) {
    T = T_;
    kb = kb_;
    ke = ke_;
    const int ce = min(ke, T), bb = max(kb, T);
    n_ctx = ce > kb ? (ce - kb + AKT - 1) / AKT : 0;
    n_blk = ke > bb ? (ke - bb + AKT - 1) / AKT : 0;
  }
  __device__ int count() const { return n_ctx + n_blk; }
  // first key (absolute) and number of valid keys of tile i
  __device__ void tile(int i, int& first, int& valid, bool& ctx) const {
    if (i < n_ctx) {
      first = kb + i * AKT;
      valid = min(AKT, min(ke, T) - first);
      ctx = true;
    } else {
      first = max(kb, T) + (i - n_ctx) * AKT;
      valid = min(AKT, ke - first);
      ctx = false;
    }
  }
};

__global__ void __launch_bounds__(kAThreads, 1) attn_tc_kernel(const __grid_constant__ AttnTcParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + B_N);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = tc::smem_u32(bars);
  auto bar = [&](int i) { return bar0 + 8 * i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qp = blockIdx.x, bg = blockIdx.y, split = blockIdx.z;
  const int b = bg / p.nkv, g = bg % p.nkv, grp = p.nq / p.nkv, nrows = p.L * grp;

  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int t = 0; t < NQT; t++) {
      tc::mbar_init(bar(B_Q + t), 1);
      tc::mbar_init(bar(B_SF + t), 1);
      tc::mbar_init(bar(B_PF + t), 4);
      tc::mbar_init(bar(B_PV + t), 1);
    }
    for (int s = 0; s < NSTAGE; s++) {
      tc::mbar_init(bar(B_KF + s), 1);
      tc::mbar_init(bar(B_KE + s), 1);
      tc::mbar_init(bar(B_VF + s), 1);
      tc::mbar_init(bar(B_VE + s), 1);
      tc::mbar_init(bar(B_VR + s), 1);
    }
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tc::smem_u32(tmem_slot), kTmemCols);
    tc::tmem_relinquish();
  }
  // The single-lane roles reconverge with their warps first: a CTA barrier reached by part of a diverged
  // warp counts the whole warp, and the lagging lane would then pass it without waiting.
  __syncwarp();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();   // q, block K/V and the context store come from earlier kernels

  const int T = clamp_ctx(p.ctx_len[b], p.t_cap);
  const int n_keys = T + p.L;
  TileList tl;
  tl.init(T, min(n_keys, split * p.chunk), min(n_keys, (split + 1) * p.chunk));
  const int n_tiles = tl.count();

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tc::tma_prefetch(&p.tm_store);
      tc::tma_prefetch(&p.tm_kblk);
      tc::tma_prefetch(&p.tm_vblk);
      const int kv_row0 = (((p.layer * p.batch + b) * 2 + 0) * p.nkv + g) * p.t_cap;
      const int vv_row0 = (((p.layer * p.batch + b) * 2 + 1) * p.nkv + g) * p.t_cap;
      const int blk_row0 = (b * p.nkv + g) * p.L;
      for (int i = 0; i < n_tiles && !*abort_flag; i++) {
        const int s = i % NSTAGE;
        const uint32_t ph = ((i / NSTAGE) & 1) ^ 1;
        int first, valid;
        bool ctx;
        tl.tile(i, first, valid, ctx);
        const uint32_t kd = tc::smem_u32(smem + SM_K + s * TILE_BYTES), vd = tc::smem_u32(smem + SM_V + s * TILE_BYTES);
        if (i >= NSTAGE && !tc::mbar_wait(bar(B_KE + s), ph)) { *abort_flag = 1; break; }
        tc::mbar_arrive_expect_tx(bar(B_KF + s), TILE_BYTES);
        for (int a = 0; a < 2; a++) {
          if (ctx) tc::tma_load_2d(kd + a * ATOM_BYTES, &p.tm_store, a * 64, kv_row0 + first, bar(B_KF + s));
          else tc::tma_load_2d(kd + a * ATOM_BYTES, &p.tm_kblk, a * 64, blk_row0 + first - T, bar(B_KF + s));
        }
        if (i >= NSTAGE && !tc::mbar_wait(bar(B_VE + s), ph)) { *abort_flag = 1; break; }
        tc::mbar_arrive_expect_tx(bar(B_VF + s), TILE_BYTES);
        for (int a = 0; a < 2; a++) {
          if (ctx) tc::tma_load_2d(vd + a * ATOM_BYTES, &p.tm_store, a * 64, vv_row0 + first, bar(B_VF + s));
          else tc::tma_load_2d(vd + a * ATOM_BYTES, &p.tm_vblk, a * 64, blk_row0 + first - T, bar(B_VF + s));
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(AQ, AKT, 0);   // Q x K, both K-major in shared memory
      constexpr uint32_t id_o = idesc_bf16(AQ, AH, 1);    // P (TMEM) x V (MN-major in shared memory)
      for (int t = 0; t < NQT; t++)
        if (!tc::mbar_wait(bar(B_Q + t), 0)) *abort_flag = 1;
      tc::tc_fence_after();
      auto issue_s = [&](int t, int i) {   // S_t = Q_t K_i^T into tile t's buffer
        const uint32_t qs = tc::smem_u32(smem + SM_Q + t * TILE_BYTES);
        const uint32_t ks = tc::smem_u32(smem + SM_K + (i % NSTAGE) * TILE_BYTES);
#pragma unroll
        for (int kk = 0; kk < AH / 16; kk++) {
          const uint64_t da = tc::sw128_kmajor_desc(qs + (kk >> 2) * ATOM_BYTES + (kk & 3) * 32);
          const uint64_t db = tc::sw128_kmajor_desc(ks + (kk >> 2) * ATOM_BYTES + (kk & 3) * 32);
          tc::umma_bf16(tmem + t * AKT, da, db, id_s, kk > 0 ? 1u : 0u);
        }
        tc::umma_commit(bar(B_SF + t));
      };
      auto wait_k = [&](int i) {
        if (!tc::mbar_wait(bar(B_KF + i % NSTAGE), (i / NSTAGE) & 1)) { *abort_flag = 1; return false; }
        tc::tc_fence_after();
        return true;
      };
      auto issue_pv = [&](int t, int i) {   // O_t += (P_hi + P_lo)_t V_i
        const int s = i % NSTAGE;
        const uint32_t ph = (i / NSTAGE) & 1;
        if (!tc::mbar_wait(bar(B_PF + t), i & 1) || !tc::mbar_wait(bar(B_VF + s), ph) ||
            !tc::mbar_wait(bar(B_VR + s), ph)) {
          *abort_flag = 1;
          return false;
        }
        tc::tc_fence_after();
        const uint32_t vs = tc::smem_u32(smem + SM_V + s * TILE_BYTES);
        const uint32_t pt = tmem + t * AKT;
#pragma unroll
        for (int kk = 0; kk < AKT / 16; kk++) {
          // keys 16 kk .. 16 kk + 15: chunk kk / 2, half kk % 2 -> hi at 32 c + 8 h, lo at 32 c + 16 + 8 h
          const uint32_t col = 32 * (kk >> 1) + 8 * (kk & 1);
          const uint64_t db = sw128_mn_desc(vs + kk * 16 * 128, ATOM_BYTES);
          umma_ts_bf16(tmem + kTmemO + t * AH, pt + col, db, id_o, (i > 0 || kk > 0) ? 1u : 0u);
          umma_ts_bf16(tmem + kTmemO + t * AH, pt + col + 16, db, id_o, 1u);
        }
        tc::umma_commit(bar(B_PV + t));
        if (t == NQT - 1) tc::umma_commit(bar(B_VE + s));
        return true;
      };
      if (n_tiles > 0 && wait_k(0)) {
        for (int t = 0; t < NQT; t++) issue_s(t, 0);
        tc::umma_commit(bar(B_KE + 0));
      }
      // each tile's next S follows its own product, so one warpgroup never waits for the other's softmax
      for (int i = 0; i < n_tiles && !*abort_flag; i++) {
        const bool more = i + 1 < n_tiles;
        if (!issue_pv(0, i)) break;
        if (more && !wait_k(i + 1)) break;
        if (more) issue_s(0, i + 1);
        if (!issue_pv(1, i)) break;
        if (more) {
          issue_s(1, i + 1);
          tc::umma_commit(bar(B_KE + (i + 1) % NSTAGE));
        }
      }
    }
  } else if (warp < 2 + 4 * NQT) {
    // ---------------- softmax of tile t: thread = query row = TMEM lane ----------------
    const int t = (warp - 2) >> 2, quarter = warp & 3, r = quarter * 32 + lane;
    const int qi = (qp * NQT + t) * AQ + r;
    const bool row_ok = qi < nrows;
    const int j = row_ok ? qi / grp : 0, head = g * grp + (row_ok ? qi % grp : 0);
    // Q row r -> shared memory (K-major, 128-byte swizzle: chunk c of row r at c ^ (r & 7))
    {
      uint8_t* qs = smem + SM_Q + t * TILE_BYTES;
      const uint4* src = reinterpret_cast<const uint4*>(p.q + (((size_t)b * p.L + j) * p.nq + head) * AH);
      uint4 u[16];
#pragma unroll
      for (int c = 0; c < 16; c++) u[c] = row_ok ? src[c] : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int c = 0; c < 16; c++)
        *reinterpret_cast<uint4*>(qs + (c >> 3) * ATOM_BYTES + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = u[c];
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      named_bar(1 + t, 128);
      if (r == 0) tc::mbar_arrive(bar(B_Q + t));
    }
    const float sl2 = rsqrtf((float)AH) * 1.4426950408889634f;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t st = tmem + lane_off + t * AKT, ot = tmem + lane_off + kTmemO + t * AH;
    float m_ref = -INFINITY, l = 0.f;
    for (int i = 0; i < n_tiles && !*abort_flag; i++) {
      int first, valid;
      bool ctx;
      tl.tile(i, first, valid, ctx);
      if (!tc::mbar_wait(bar(B_SF + t), i & 1)) *abort_flag = 1;
      tc::tc_fence_after();
      // pass 1: the row maximum of the raw scores (keys past `valid` excluded), scaled once (sl2 > 0)
      float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int h = 0; h < AKT; h += 64) {
        float sv[64];
        tmem_ld32_nowait(st + h, sv);
        tmem_ld32_nowait(st + h + 32, sv + 32);
        tmem_wait_ld();
        if (valid < AKT) {   // a partial tile (warp-uniform)
#pragma unroll
          for (int e = 0; e < 64; e++)
            if (h + e >= valid) sv[e] = -INFINITY;
        }
#pragma unroll
        for (int e = 0; e < 64; e++) mq[e & 3] = fmaxf(mq[e & 3], sv[e]);
      }
      const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * sl2;
      const bool need = mx > m_ref + kRescaleLog2;
      if (__any_sync(0xffffffffu, need)) {   // tcgen05.ld/st are warp-wide: every lane takes part
        // O_t may only be rescaled once every product into it (up to key tile i - 1) has finished
        if (i >= 1 && !tc::mbar_wait(bar(B_PV + t), (i - 1) & 1)) *abort_flag = 1;
        tc::tc_fence_after();
        const float m_new = need ? mx : m_ref;
        const float cf = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - m_new);
        if (i >= 1) {
#pragma unroll 1
          for (int c0 = 0; c0 < AH; c0 += 16) {
            float o[16];
            tc::tmem_ld16(ot + c0, o);
#pragma unroll
            for (int e = 0; e < 16; e++) o[e] *= cf;
            tmem_st16(ot + c0, o);
          }
        }
        l *= cf;
        m_ref = m_new;
      }
      // pass 2, 32 keys at a time: p = 2^(s sl2 - m_ref) (0 past `valid`) as hi + lo bf16 terms over the columns
      // just read: hi at [32c, 32c + 16), lo at [32c + 16, 32c + 32), two keys per 32-bit column
      const float nm = -m_ref;
      float lq[2] = {0.f, 0.f};   // two chains of the running sum, combined in a fixed order
#pragma unroll
      for (int c0 = 0; c0 < AKT; c0 += 32) {
        float sv[32];
        tmem_ld32_nowait(st + c0, sv);
        tmem_wait_ld();
        if (valid < c0 + 32) {
#pragma unroll
          for (int e = 0; e < 32; e++)
            if (c0 + e >= valid) sv[e] = -INFINITY;
        }
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float p0 = ex2(fmaf(sv[e], sl2, nm)), p1 = ex2(fmaf(sv[e + 1], sl2, nm));
          lq[0] += p0;
          lq[1] += p1;
          split_bf16x2(p0, p1, hi[e / 2], lo[e / 2]);
        }
        tmem_st16(st + c0, hi);
        tmem_st16(st + c0 + 16, lo);
      }
      l += lq[0] + lq[1];
      tmem_wait_st();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(bar(B_PF + t));
    }
    // epilogue: O_t / l (one split) or the partial (o, m, l)
    if (n_tiles > 0 && !tc::mbar_wait(bar(B_PV + t), (n_tiles - 1) & 1)) *abort_flag = 1;
    tc::tc_fence_after();
    const size_t orow = ((size_t)b * p.L + j) * p.nq + head;
#pragma unroll 1
    for (int c0 = 0; c0 < AH; c0 += 16) {
      float o[16];
      if (n_tiles > 0) {
        tc::tmem_ld16(ot + c0, o);
      } else {
#pragma unroll
        for (int e = 0; e < 16; e++) o[e] = 0.f;
      }
      if (!row_ok) continue;
      if (p.splits == 1) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        uint4 pk[2];
        bf16* pe = reinterpret_cast<bf16*>(pk);
#pragma unroll
        for (int e = 0; e < 16; e++) pe[e] = __float2bfloat16_rn(o[e] * inv);
        uint4* dst = reinterpret_cast<uint4*>(p.out + orow * AH + c0);
        dst[0] = pk[0];
        dst[1] = pk[1];
      } else {
        float4* dst = reinterpret_cast<float4*>(p.o_part + ((size_t)split * p.rows * p.nq + orow) * AH + c0);
#pragma unroll
        for (int e = 0; e < 16; e += 4) dst[e / 4] = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
      }
    }
    if (row_ok && p.splits > 1) p.ml[(size_t)split * p.rows * p.nq + orow] = make_float2(m_ref, l);
  } else {
    // ---------------- V rows past the last valid key -> 0 ----------------
    for (int i = 0; i < n_tiles && !*abort_flag; i++) {
      const int s = i % NSTAGE;
      int first, valid;
      bool ctx;
      tl.tile(i, first, valid, ctx);
      if (!tc::mbar_wait(bar(B_VF + s), (i / NSTAGE) & 1)) *abort_flag = 1;
      if (valid < AKT) {
        // row k of the tile: 128 bytes at k * 128 in each of the two 64-dim atoms (the swizzle permutes within a row)
        uint8_t* tile = smem + SM_V + s * TILE_BYTES;
        for (int c = lane; c < (AKT - valid) * 16; c += 32) {
          const int k = valid + (c >> 4), a = (c >> 3) & 1, q = c & 7;
          *reinterpret_cast<uint4*>(tile + a * ATOM_BYTES + k * 128 + q * 16) = make_uint4(0, 0, 0, 0);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(bar(B_VR + s));
    }
  }

  __syncwarp();
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool attn_tc_supported(int head_dim, int L, int nq, int nkv) { return head_dim == AH && L * (nq / nkv) >= AQ; }

// One CTA per SM (the shared memory allows no second): the split count s minimises the waves times the key tiles a
// CTA walks, ceil(base s / SMs) * ceil(keys / (s AKT)), plus the split's own cost;
// ties go to fewer splits.  A split adds about two key tiles of work to each CTA: its fp32 partial row out, and the
// merge pass that reads it back.
void attn_tc_plan(int batch, int L, int nq, int nkv, int t_cap, int num_sms, int* splits, int* chunk) {
  const int q_pairs = ceil_div(ceil_div(L * (nq / nkv), AQ), NQT);
  const long base = (long)q_pairs * batch * nkv;
  const int max_keys = t_cap + L;
  const int key_tiles = ceil_div(max_keys, AKT);
  const int s_max = std::max(1, std::min(key_tiles, 128));
  int best_s = 1;
  double best = 0.0;
  for (int s = 1; s <= s_max; s++) {
    const long waves = (base * s + num_sms - 1) / num_sms;
    const double cost = (double)waves * (ceil_div(key_tiles, s) + (s > 1 ? 2 : 0));
    if (s == 1 || cost < best) {
      best = cost;
      best_s = s;
    }
  }
  const int ch = ceil_div(key_tiles, best_s) * AKT;
  *chunk = ch;
  *splits = ceil_div(max_keys, ch);
}

cudaError_t attn_tc_init_attributes() {
  return cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kASmem);
}

cudaError_t launch_attention_tc(const AttnArgs& a, bf16* out, cudaStream_t st) {
  if (a.head_dim != AH) return cudaErrorInvalidValue;
  AttnTcParams p;
  memset(&p, 0, sizeof(p));
  const uint64_t store_rows = a.layer >= 0 ? (uint64_t)(a.layer + 1) * a.batch * 2 * a.nkv * a.t_cap : 0;
  const uint64_t dims_s[2] = {(uint64_t)AH, store_rows};
  const uint64_t str[1] = {(uint64_t)AH * 2};
  const uint32_t box[2] = {64u, (uint32_t)AKT};
  cudaError_t e = make_tmap_nd(&p.tm_store, a.store, 2, dims_s, str, box);
  const uint64_t dims_b[2] = {(uint64_t)AH, (uint64_t)a.batch * a.nkv * a.L};
  if (e == cudaSuccess) e = make_tmap_nd(&p.tm_kblk, a.kblk, 2, dims_b, str, box);
  if (e == cudaSuccess) e = make_tmap_nd(&p.tm_vblk, a.vblk, 2, dims_b, str, box);
  if (e != cudaSuccess) return e;
  p.q = a.q;
  p.out = out;
  p.o_part = a.o_part;
  p.ml = a.ml;
  p.ctx_len = a.ctx_len;
  p.batch = a.batch;
  p.L = a.L;
  p.nq = a.nq;
  p.nkv = a.nkv;
  p.t_cap = a.t_cap;
  p.layer = a.layer;
  p.rows = a.rows;
  p.splits = a.splits;
  p.chunk = a.chunk;
  const int grp = a.nq / a.nkv;
  dim3 grid(ceil_div(ceil_div(a.L * grp, AQ), NQT), a.batch * a.nkv, a.splits);
  cudaError_t err = launch_k(attn_tc_kernel, grid, kAThreads, kASmem, st, p);
  if (err != cudaSuccess || a.splits == 1) return err;
  return launch_attn_merge(a, out, st);
}

}  // namespace fpd

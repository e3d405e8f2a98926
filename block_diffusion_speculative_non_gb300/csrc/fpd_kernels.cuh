// fpd_kernels.cuh — launch interfaces of the kernels behind the C ABI (internal).
#pragma once

#include <algorithm>

#include "fpd_internal.cuh"

namespace fpd {

// ---- GEMM:  C[split][m][n] = sum_{k in split} A[m][k] * B[n][k]   (fp32 partials) ------------------------------
struct GemmArgs {
  const bf16* a[8];     // K-segments of A; segment s covers k in [s*seg_k, (s+1)*seg_k)
  int seg_k;
  int lda;              // row stride of every A segment (elements)
  const bf16* b;        // B [N, K] row-major (weights, [out, in])
  int ldb;
  float* c;             // C [splits][M][ldc]
  int ldc;
  size_t c_split_stride;
  int M, N, K;
  int k_split;          // K elements per split (multiple of 64)
};

// tcgen05 GEMM: the plan fixes operand placement, tile width, split-K and grid for a shape.
struct TcPlan {
  bool swap;      // weights on the 128-row MMA operand (few tokens)
  int bn;         // width of the other operand's tile
  int pt, qt;     // tiles along the 128-row and the bn-row operand
  int splits, k_split;
  int grid;       // persistent CTAs
};
TcPlan tc_plan_gemm(int M, int N, int K, int num_sms);
TcPlan tc_plan_force(int M, int N, int K, int num_sms, int placement);   // placement 0: tokens on 128 rows, 1: weights
cudaError_t launch_tc_gemm(const GemmArgs& g, const TcPlan& plan, cudaStream_t st);
TcPlan tc_plan_swiglu(int M, int F, int K, int num_sms);
// Context K/V of every layer in one token-tile GEMM (a2): rows [row0, row0 + R) of the fused, normed context ctx
// [R][d] against [Wk; Wv] of all layers, with the K-norm + RoPE and the store writes in the epilogue.
struct KvCtxGemm {
  const fpd_model_desc* d;
  const bf16* ctx;
  int R;
  const void* const* wqkv;          // [layers] weights [(H_q + 2 H_kv) h, d]
  const bf16* const* k_norm;        // [layers] gains [h]
  const float2* rope;
  bf16* store;                      // [layers][batch][K|V][H_kv][t_cap][h]
  int batch, t_cap, row0;
  const int32_t *row_off, *row_cnt, *pos_start;
};
bool kvctx_supported(const fpd_model_desc& d);
cudaError_t launch_tc_kvctx(const KvCtxGemm& g, int num_sms, cudaStream_t st);

// hmid[M][F] = bf16(silu(x . Wg^T) * (x . Wu^T)) with W = [Wg; Wu] ([2F, K]), one tcgen05 pass
cudaError_t launch_tc_swiglu(const bf16* x, int M, int K, const bf16* w_gate_up, int F, bf16* hmid, const TcPlan& pl,
                             cudaStream_t st);
// Token-tile GEMMs (many tokens) with the layer epilogue fused: qkv = true — q/k RMSNorm + RoPE, bf16 q / block
// k / block v; qkv = false — residual add into xres and per-(column tile, token) sums of squares into ss_part
// [N / plan.bn][M].  W [N, K] weights, x [M, K] activations; no split-K.
struct TokGemm {
  bool qkv;
  const bf16* x;
  const bf16* w;
  int M, N, K;
  bf16 *q, *kblk, *vblk;
  const bf16 *q_norm, *k_norm;
  const float2* rope;
  const int32_t* ctx_len;
  int t_cap, L, nq, nkv, hd;
  float eps;
  bf16* xres;
  float* ss_part;
};
TcPlan tc_plan_tok(int M, int N, int K, int num_sms);
cudaError_t launch_tc_tok(const TokGemm& g, const TcPlan& pl, cudaStream_t st);
// xn[m][k] = bf16(x[m][k] * rsqrt(sum_t ss_part[t][m] / d + eps) * g[k]), one block per row
cudaError_t launch_norm_rows(bf16* xn, const bf16* x, const float* ss_part, int n_part, const bf16* g, int M, int d,
                             float eps, cudaStream_t st);
cudaError_t tc_init_attributes();     // once per process, before any stream capture
cudaError_t attn_init_attributes();
cudaError_t launch_sum_splits(float* out, const float* part, int splits, size_t n, cudaStream_t st);

// ---- few-token path (k_stream.cu): weight-streaming GEMMs with fused norm-on-load and epilogues ---------------
enum { SEPI_QKV = 0, SEPI_RESID = 1, SEPI_SWIGLU = 2, SEPI_ARGMAX = 3 };
enum { XF_COPY = 0, XF_NORM = 1, XF_NORM_FULL = 2 };
constexpr int kStreamMaxTokens = 16;
struct StreamPlan {
  int tiles, splits, k_split, grid;
};
struct StreamGemm {
  int epi;                        // SEPI_*
  StreamPlan plan;
  const bf16* w;                  // weights [N, K] ([2F, K] for SwiGLU), K-major
  int M, N, K;
  const bf16* x;                  // activation source rows, row stride ldx
  int ldx, xform, lm_block;
  const float* ss_in;             // sums of squares [n_ss][16] (XF_NORM)
  int n_ss;
  const bf16* gain;
  float eps;
  float* part;                    // split-K partials [splits][tiles][16][128]
  int* counters;                  // [tiles], zero on entry
  bf16 *q, *kblk, *vblk;          // SEPI_QKV outputs
  const bf16 *q_norm, *k_norm;
  const float2* rope;
  const int32_t* ctx_len;
  int t_cap, L, nq, nkv, h;
  bf16* xres;                     // SEPI_RESID: residual stream [M][N]
  float* ss_out;                  // SEPI_RESID: sums of squares [tiles][16]
  bf16* hmid;                     // SEPI_SWIGLU output [M][N]
  unsigned long long* slots;      // SEPI_ARGMAX: [grid][16][2]
  float* logits;                  // SEPI_ARGMAX: [M][N] or null
  uint32_t test_extra_tx = 0;     // test hook only: bytes the first weight stage expects beyond what arrives
  // 8-bit weights (E4M3 codes [rows, K] and exponents [rows, K/128], K a multiple of 128) instead of w
  bool fp8 = false;
  const uint8_t* w8 = nullptr;
  const int8_t* w_exp = nullptr;
  int exp_ld = 0;                 // exponents block-major: (row r, 128-block b) at w_exp[b * exp_ld + r];
                                  // exp_ld a multiple of 128, >= rows; w_exp 16-byte aligned
};
bool stream_shape_ok(const fpd_model_desc& d);
StreamPlan stream_plan(int tiles, int K, int num_sms, bool split_ok, bool fp8);
size_t stream_part_floats(const StreamPlan& pl);
cudaError_t launch_stream_gemm(const StreamGemm& g, cudaStream_t st);
cudaError_t stream_init_attributes();
cudaError_t launch_embed_ss(bf16* x, float* ss, int* counters, int n_cnt, const bf16* embed, const int32_t* anchor,
                            int32_t mask_id, int B, int L, int d, int V, cudaStream_t st);
cudaError_t launch_quantize_fp8(const bf16* w, int N, int K, int ld, uint8_t* codes, int8_t* exps, int exp_rs,
                                int exp_cs, int num_sms, cudaStream_t st);
cudaError_t launch_stream_decode(int32_t* tokens, float* margin, const unsigned long long* slots, int n_slots,
                                 int n_rows, cudaStream_t st);

// ---- row ops -------------------------------------------------------------------------------------------------
cudaError_t launch_rmsnorm_partials(bf16* out, const float* part, int nsplit, size_t split_stride, const bf16* g,
                                    int rows, int d, float eps, cudaStream_t st);
cudaError_t launch_qkv_post(bf16* q, bf16* kblk, bf16* vblk, const float* part, int nsplit, size_t split_stride,
                            const bf16* q_norm, const bf16* k_norm, const float2* rope, const int32_t* ctx_len,
                            int t_cap, int B, int L, int nq, int nkv, int h, float eps, cudaStream_t st);
cudaError_t launch_kv_post(bf16* store, const float* part, int nsplit, size_t split_stride, const bf16* k_norm,
                           const float2* rope, const int32_t* row_off, const int32_t* row_cnt, const int32_t* pos_start,
                           int batch, int layer, int t_cap, int row0, int rows, int nkv, int h, float eps,
                           cudaStream_t st);
cudaError_t launch_residual_norm(bf16* x, bf16* xn, const float* part, int nsplit, size_t split_stride, const bf16* g,
                                 int rows, int d, float eps, cudaStream_t st);
cudaError_t launch_embed_norm(bf16* x, bf16* xn, const bf16* embed, const int32_t* anchor, int32_t mask_id,
                              const bf16* g, int B, int L, int d, int V, float eps, cudaStream_t st);

// ---- attention ---------------------------------------------------------------------------------------------
struct AttnArgs {
  const bf16* q;        // [B*L, nq, h]
  const bf16* store;    // context KV store [layer][b][K|V][g][t_cap][h]
  const bf16* kblk;     // [B, nkv, L, h]
  const bf16* vblk;
  const int32_t* ctx_len;
  float* o_part;        // [splits][B*L][nq][h]
  float2* ml;           // [splits][B*L][nq]  (running max, running sum)
  int batch, L, nq, nkv, head_dim, t_cap, layer;
  int rows;             // B*L
  int splits, chunk;    // KV splits and keys per split
};
void attn_plan(int batch, int L, int nq, int nkv, int t_cap, int num_sms, int* splits, int* chunk);
cudaError_t launch_attention(const AttnArgs& a, bf16* out, cudaStream_t st);          // mma.sync tiles of 64 rows
cudaError_t launch_attn_merge(const AttnArgs& a, bf16* out, cudaStream_t st);         // split merge, fixed order
// few-token attention (k_attention_short.cu): at most 64 query rows per (request, kv head); the KV splits of one
// (request, kv head) form a thread-block cluster and merge through distributed shared memory (no partials, no merge
// kernel).  The call's first kernel must trigger its successors only after its own griddepcontrol.wait: the
// kernel reads the context store before waiting.
bool attn_short_supported(int head_dim, int L, int nq, int nkv);
cudaError_t attn_short_init_attributes();
cudaError_t launch_attention_short(const AttnArgs& a, bf16* out, cudaStream_t st);
// tcgen05 attention (k_attention_tc.cu): 128-row query tiles, head_dim 128; same partial layout and merge
bool attn_tc_supported(int head_dim, int L, int nq, int nkv);
void attn_tc_plan(int batch, int L, int nq, int nkv, int t_cap, int num_sms, int* splits, int* chunk);
cudaError_t attn_tc_init_attributes();
cudaError_t launch_attention_tc(const AttnArgs& a, bf16* out, cudaStream_t st);

// ---- LM head + constrained argmax ------------------------------------------------------------------------------
struct LmPlan {
  int n_class, n_range, n_rows, L;
  int ct, rt;           // column (id) tile and row (position) tile of one work item
  int range_lo[FPD_MAX_RANGES], range_hi[FPD_MAX_RANGES], range_class[FPD_MAX_RANGES];
};
// rows_sorted: sorted slot -> original row (-1 past the last placed row); inv_sorted: original row -> slot.
cudaError_t launch_lm_plan(const LmPlan& p, const int16_t* pos_class, int* rows_sorted, int* inv_sorted,
                           int* class_row_off, int4* items, int* n_items, unsigned long long* packed,
                           unsigned long long* packed2, int max_items, cudaStream_t st);
int tc_lm_row_tile(int n_rows);
cudaError_t launch_tc_lmhead(const LmPlan& lp, const bf16* z_sorted, int n_rows, const bf16* W, int d, int V,
                             const int4* items, const int* n_items, int max_items, unsigned long long* packed,
                             unsigned long long* packed2, const int* rows_sorted, float* logits, int num_sms,
                             bool unconstrained, cudaStream_t st);
// tokens[r] = argmax id; margin[r] (optional) = top-1 minus top-2 fp32 logit (+inf with one legal id)
struct PairTable {
  int n, off_id;
  int16_t p[FPD_MAX_PAIRS], q[FPD_MAX_PAIRS];
};
cudaError_t launch_pair_offscreen(int32_t* tokens, float* margin, const unsigned long long* packed,
                                  const unsigned long long* packed2, const int* inv_sorted, const bf16* z,
                                  const bf16* w_lm, int d, int L, int B, const PairTable& pt, cudaStream_t st);
cudaError_t launch_lm_decode(int32_t* tokens, float* margin, const unsigned long long* packed,
                             const unsigned long long* packed2, const int* inv_sorted, int n, cudaStream_t st);
// RMSNorm of block rows into sorted order: out[i] = norm(hidden[map(rows_sorted[i])]), map drops anchors.
cudaError_t launch_rmsnorm_gather(bf16* out, const bf16* in, const bf16* g, const int* rows_sorted, int rows, int d,
                                  float eps, int L, cudaStream_t st);

// ---- verify -----------------------------------------------------------------------------------------------------
struct VerifyTables {
  int n_class;
  int class_off[FPD_MAX_CLASSES + 1];
  int lo[FPD_MAX_RANGES], hi[FPD_MAX_RANGES];
};
cudaError_t launch_verify(int mode, int B, int L, const int32_t* draft, const int32_t* target, const VerifyTables& tb,
                          const int16_t* pos_class, const int8_t* rule, int32_t pad_id, int32_t* accept,
                          int32_t* committed, int32_t* valid, const float* margin, float tau, cudaStream_t st);
cudaError_t launch_sd_advance(int B, int L, int t_cap, int32_t* accept, const int32_t* committed, int32_t* ctx_len,
                              int32_t* pos_start, int32_t* anchor, cudaStream_t st);

}  // namespace fpd

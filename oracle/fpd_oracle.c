/*
 * fpd_oracle.c — plain, slow, CPU reference of the block-drafter hot path.  TEST INFRASTRUCTURE ONLY:
 * only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may load it.  It shares no code,
 * header, table or helper with the CUDA library.
 *
 * Every dot product and every reduction is accumulated in double.  Values are rounded to bf16 (round to
 * nearest, ties to even) exactly where the product stores a bf16 tensor:
 *   fused context ctx; context K and V; the normed inputs of every projection (attention-norm and
 *   MLP-norm outputs); q, k, v of the block after q/k-norm and RoPE; the attention output o; the residual
 *   stream after each sub-layer; the MLP hidden silu(g)*u; the final normed z.
 * Logits stay double; the argmax decision is taken on the logits rounded to fp32 (the precision the GPU
 * kernel decides in), lowest id first on ties.
 *
 * Method sources (page title, section):
 *   - VFlash paper (Chinese translation), §2.1 "Preliminaries": fused selected-layer target features are
 *     injected as keys and values into every drafter layer; one bidirectional pass predicts the masked
 *     positions; greedy verification accepts up to the first disagreement.
 *   - VFlash paper (zh), §2.2: a block is one observed start token followed by L-1 mask tokens.
 *   - VFlash paper (zh), §2.3: dedicated coordinate tokens (1001 ids) or fixed-width numerals (sign + five
 *     digit slots, unused high digits padded with the mask token).
 *   - VFlash paper (zh), §2.5 "Inference": per-position legal vocabulary applied on computed logits;
 *     schema acceptance keeps the first k positions.
 *   - VFlash blog, "Method": 16-position text blocks, longest matching prefix plus the target's own token.
 *   - VFlash blog, "Key claims": five-layer non-causal transformer drafter.
 * Readings where the pages are silent (layer form, norm and RoPE constants, fusion form, acceptance
 * conventions) are the ones listed with the design notes of this repository: pre-norm layer with per-head
 * q/k RMSNorm and rotate-half RoPE, RMSNorm y = x / sqrt(mean(x^2) + eps) * g, attention scale 1/sqrt(h),
 * fusion = concatenation -> linear -> RMSNorm shared by all layers.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_MAX_LAYERS 8

typedef struct oracle_model {
  int32_t n_layers, d, nq, nkv, h, F, V, nf;
  double eps, theta;
  const uint16_t *embed, *w_fc, *hidden_norm, *final_norm, *lm_head;
  const uint16_t *attn_norm[OR_MAX_LAYERS], *wqkv[OR_MAX_LAYERS], *q_norm[OR_MAX_LAYERS],
      *k_norm[OR_MAX_LAYERS], *wo[OR_MAX_LAYERS], *mlp_norm[OR_MAX_LAYERS], *w_gate_up[OR_MAX_LAYERS],
      *w_down[OR_MAX_LAYERS];
  /* FP8 copies (E4M3 codes + one power-of-two exponent per 128 elements of a row), or NULL: see the f2 section */
  const uint8_t *q_wqkv[OR_MAX_LAYERS], *q_wo[OR_MAX_LAYERS], *q_gate_up[OR_MAX_LAYERS], *q_down[OR_MAX_LAYERS],
      *q_lm_head;
  const int8_t *e_wqkv[OR_MAX_LAYERS], *e_wo[OR_MAX_LAYERS], *e_gate_up[OR_MAX_LAYERS], *e_down[OR_MAX_LAYERS],
      *e_lm_head;
} oracle_model;

/* ------------------------------------------------------------------------------------------------------ */
/* bf16 <-> double                                                                                         */

double oracle_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a double to the nearest bf16 (8 significant bits, float's exponent range), ties to even.  Done in
 * one step from the double value, so there is no double rounding through float. */
uint16_t oracle_round_bf16(double x) {
  if (isnan(x)) return 0x7FC0;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (a == 0.0) return sign;
  if (isinf(a)) return sign | 0x7F80;
  int e;
  double m = frexp(a, &e);             /* a = m * 2^e, m in [0.5, 1) */
  int bits = 8;                        /* significant bits of a normal bf16 */
  if (e < -125) bits = 8 - (-125 - e); /* below float's smallest normal (2^-126): fewer bits */
  double r;
  if (bits <= 0) {
    r = (bits == 0 && m > 0.5) ? 1.0 : 0.0; /* rounds to the smallest subnormal or to zero */
    if (bits < 0) r = 0.0;
    bits = 0;
  } else {
    r = nearbyint(ldexp(m, bits));     /* current rounding mode: to nearest, ties to even */
  }
  double v = ldexp(r, e - bits);
  float f = (float)v;                  /* exact: v has at most 8 significant bits, or overflows to inf */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16) | sign;
}

static inline double bf(uint16_t b) { return oracle_bf16_to_double(b); }
static inline double rbf(double x) { return bf(oracle_round_bf16(x)); } /* value after bf16 storage */

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* ------------------------------------------------------------------------------------------------------ */
/* Building blocks                                                                                         */

/* RMSNorm: y_i = x_i / sqrt(mean_j x_j^2 + eps) * g_i. */
void oracle_rmsnorm(int n, const double* x, const uint16_t* g, double eps, double* y) {
  double ss = 0.0;
  for (int i = 0; i < n; i++) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss / n + eps);
  for (int i = 0; i < n; i++) y[i] = x[i] * inv * bf(g[i]);
}

/* Rotate-half RoPE at position pos: the pair (x_i, x_{i+h/2}) turns by angle pos * theta^(-2i/h). */
void oracle_rope(int h, double* x, double pos, double theta) {
  int half = h / 2;
  for (int i = 0; i < half; i++) {
    double ang = pos * pow(theta, -2.0 * (double)i / (double)h);
    double c = cos(ang), s = sin(ang);
    double x1 = x[i], x2 = x[i + half];
    x[i] = x1 * c - x2 * s;
    x[i + half] = x2 * c + x1 * s;
  }
}

double oracle_silu(double v) { return v / (1.0 + exp(-v)); }

/* Y[m][n] = sum_k X[m][k] * W[n][k] for W row-major [N, K] in bf16 (a linear layer without bias).
 * Output rows are taken in groups of 32 so a group of X stays in cache while W streams; every output is
 * one plain double sum over k. */
void oracle_linear(int M, int N, int K, const double* X, const uint16_t* W, double* Y) {
  const int G = 32;
  for (int m0 = 0; m0 < M; m0 += G) {
    int m1 = m0 + G < M ? m0 + G : M;
#pragma omp parallel
    {
      double* w = (double*)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(static)
      for (int n = 0; n < N; n++) {
        const uint16_t* wr = W + (size_t)n * K;
        for (int k = 0; k < K; k++) w[k] = bf(wr[k]);
        for (int m = m0; m < m1; m++) {
          const double* xr = X + (size_t)m * K;
          double acc = 0.0;
          for (int k = 0; k < K; k++) acc += xr[k] * w[k];
          Y[(size_t)m * N + n] = acc;
        }
      }
      free(w);
    }
  }
}

/* ------------------------------------------------------------------------------------------------------ */
/* f2: 8-bit weights and activations.  FlashDrive §3.4 "Quantization": low-bit weights shrink the bytes a
 * memory-bound decoding step has to load, and 8-bit activations let the products run on 8-bit matrix units.
 * The 8-bit type here is E4M3 of the OCP 8-bit floating-point format (OFP8): 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits; code (e, m) is (1 + m/8) 2^(e-7) for e >= 1 and (m/8) 2^-6 for e = 0; the code with
 * e = 15, m = 7 is NaN, so the largest finite magnitude is 448 (e = 15, m = 6).
 *
 * Quantisation group: 128 consecutive elements of one row (a weight row, or one token's activation row), with a
 * power-of-two scale 2^k: k is the smallest integer with amax * 2^-k <= 448 (amax = the group's largest
 * magnitude), clamped to [-126, 127], and k = 0 for an all-zero group.  Each element becomes the E4M3 code
 * nearest to x * 2^-k, ties to the even code (mantissa bit 0 clear); a zero result is the +0 code.  The value
 * the group stands for is decode(code) * 2^k.                                                               */

double oracle_e4m3_decode(uint8_t c) {
  const int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

/* nearest code, ties to even; magnitudes above 448 saturate to 448 */
uint8_t oracle_e4m3_encode(double x) {
  const int neg = x < 0;
  double a = fabs(x);
  if (a > 448.0) a = 448.0;
  int code;
  if (a < ldexp(1.0, -6)) {
    code = (int)rint(a * 512.0);                /* subnormal steps of 2^-9; 8 steps = the smallest normal */
  } else {
    int E;
    const double f = frexp(a, &E);             /* a = f 2^E, f in [0.5, 1): exponent e - 7 = E - 1 */
    const int mant = (int)rint((2.0 * f - 1.0) * 8.0);   /* 0..8; 8 carries into the next exponent */
    code = ((E - 1 + 7) << 3) + mant;
  }
  if (code == 0) return 0;
  return (uint8_t)(code | (neg ? 0x80 : 0));
}

int oracle_block_exponent(double amax) {
  if (!(amax > 0.0)) return 0;
  int E;
  const double f = frexp(amax, &E);            /* amax = f 2^E; 448 = 0.875 2^9 */
  int k = E - 9 + (f > 0.875 ? 1 : 0);
  if (k < -126) k = -126;
  if (k > 127) k = 127;
  return k;
}

/* one group of 128 values: its exponent, and its codes */
static int8_t quantize_group(const double* x, uint8_t* codes) {
  double amax = 0.0;
  for (int i = 0; i < 128; i++)
    if (fabs(x[i]) > amax) amax = fabs(x[i]);
  const int k = oracle_block_exponent(amax);
  for (int i = 0; i < 128; i++) codes[i] = oracle_e4m3_encode(ldexp(x[i], -k));
  return (int8_t)k;
}

/* codes [N, K] and exponents [N, K/128] of the rows of X (K a multiple of 128) */
void oracle_quantize_fp8(int N, int K, const double* X, uint8_t* codes, int8_t* exps) {
#pragma omp parallel for schedule(static)
  for (int n = 0; n < N; n++)
    for (int g = 0; g < K / 128; g++)
      exps[(size_t)n * (K / 128) + g] = quantize_group(X + (size_t)n * K + (size_t)g * 128, codes + (size_t)n * K + (size_t)g * 128);
}

/* the same for a bf16 matrix (weights) */
void oracle_quantize_fp8_bf16(int N, int K, const uint16_t* W, uint8_t* codes, int8_t* exps) {
#pragma omp parallel for schedule(static)
  for (int n = 0; n < N; n++) {
    double x[128];
    for (int g = 0; g < K / 128; g++) {
      for (int i = 0; i < 128; i++) x[i] = bf(W[(size_t)n * K + (size_t)g * 128 + i]);
      exps[(size_t)n * (K / 128) + g] = quantize_group(x, codes + (size_t)n * K + (size_t)g * 128);
    }
  }
}

static void dequant_row(int K, const uint8_t* q, const int8_t* e, double* out) {
  for (int k = 0; k < K; k++) out[k] = ldexp(oracle_e4m3_decode(q[k]), e[k / 128]);
}

/* Y[m][n] = sum_k Xq[m][k] Wq[n][k] with both operands in the quantised form above: the activation rows X are
 * quantised here (the same rule as the weights), the weights come as codes + exponents. */
void oracle_linear_fp8(int M, int N, int K, const double* X, const uint8_t* Wq, const int8_t* We, double* Y) {
  uint8_t* xq = (uint8_t*)malloc((size_t)M * K);
  int8_t* xe = (int8_t*)malloc((size_t)M * (K / 128));
  double* xd = (double*)malloc(sizeof(double) * (size_t)M * K);
  oracle_quantize_fp8(M, K, X, xq, xe);
  for (int m = 0; m < M; m++) dequant_row(K, xq + (size_t)m * K, xe + (size_t)m * (K / 128), xd + (size_t)m * K);
#pragma omp parallel
  {
    double* w = (double*)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(static)
    for (int n = 0; n < N; n++) {
      dequant_row(K, Wq + (size_t)n * K, We + (size_t)n * (K / 128), w);
      for (int m = 0; m < M; m++) {
        const double* xr = xd + (size_t)m * K;
        double acc = 0.0;
        for (int k = 0; k < K; k++) acc += xr[k] * w[k];
        Y[(size_t)m * N + n] = acc;
      }
    }
    free(w);
  }
  free(xq);
  free(xe);
  free(xd);
}

/* the linear layers of the drafter pass: bf16 weights, or the FP8 copies when fp8 is set */
static void linear_of(int fp8, int M, int N, int K, const double* X, const uint16_t* W, const uint8_t* Wq,
                      const int8_t* We, double* Y) {
  if (fp8)
    oracle_linear_fp8(M, N, K, X, Wq, We, Y);
  else
    oracle_linear(M, N, K, X, W, Y);
}

/* Softmax attention of nq_rows query rows (each h values) over n_keys keys/values (bf16 rows of h):
 *   o_r = sum_t softmax_t(q_r . k_t * scale) v_t
 * Keys/values are given as two row lists (context rows then block rows) so callers need not copy.
 * No mask: every query sees every key (the drafter is bidirectional, VFlash (zh) §2.1). */
void oracle_attention(int h, int nq_rows, const double* q, int n_ctx, const uint16_t* kc, const uint16_t* vc,
                      int n_blk, const double* kb, const double* vb, double scale, double* o) {
  int n = n_ctx + n_blk;
  double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  for (int r = 0; r < nq_rows; r++) {
    const double* qr = q + (size_t)r * h;
    double mx = -INFINITY;
    for (int t = 0; t < n_ctx; t++) {
      double acc = 0.0;
      for (int i = 0; i < h; i++) acc += qr[i] * bf(kc[(size_t)t * h + i]);
      s[t] = acc * scale;
      if (s[t] > mx) mx = s[t];
    }
    for (int t = 0; t < n_blk; t++) {
      double acc = 0.0;
      for (int i = 0; i < h; i++) acc += qr[i] * kb[(size_t)t * h + i];
      s[n_ctx + t] = acc * scale;
      if (s[n_ctx + t] > mx) mx = s[n_ctx + t];
    }
    double den = 0.0;
    for (int t = 0; t < n; t++) {
      s[t] = exp(s[t] - mx);
      den += s[t];
    }
    double* orow = o + (size_t)r * h;
    for (int i = 0; i < h; i++) orow[i] = 0.0;
    for (int t = 0; t < n_ctx; t++) {
      double p = s[t] / den;
      for (int i = 0; i < h; i++) orow[i] += p * bf(vc[(size_t)t * h + i]);
    }
    for (int t = 0; t < n_blk; t++) {
      double p = s[n_ctx + t] / den;
      for (int i = 0; i < h; i++) orow[i] += p * vb[(size_t)t * h + i];
    }
  }
  free(s);
}

/* ------------------------------------------------------------------------------------------------------ */
/* KV store addressing: [layer][request][K|V][kv_head][t_cap][h]                                             */

static size_t kv_index(const oracle_model* m, int batch, int t_cap, int l, int b, int kv, int g, int t) {
  return ((((((size_t)l * batch + b) * 2 + kv) * m->nkv + g) * (size_t)t_cap + t) * m->h);
}

/* a1 + a2: context fusion and per-layer context K/V (VFlash (zh) §2.1; FlashDrive §3.2).
 *   ctx = bf16(RMSNorm_hidden_norm(concat_s F_s . w_fc^T))
 *   K^l = bf16(RoPE_pos(RMSNorm_k_norm^l(ctx . Wk^l^T))) per kv head,  V^l = bf16(ctx . Wv^l^T)
 * pos = pos_start[b] (0 when NULL) + row index within the request.  Returns 0, or -1 on bad sizes. */
int oracle_prepare_context(const oracle_model* m, int batch, int total_rows, const int32_t* row_off,
                           const int32_t* pos_start, const uint16_t* const* feats, uint16_t* kv_store,
                           int t_cap) {
  const int d = m->d, nf = m->nf, h = m->h;
  if (row_off[0] != 0 || row_off[batch] != total_rows) return -1;
  for (int b = 0; b < batch; b++) {
    int p0 = pos_start ? pos_start[b] : 0;
    if (row_off[b + 1] < row_off[b] || p0 < 0 || p0 + row_off[b + 1] - row_off[b] > t_cap) return -1;
  }
  const int chunk = 256;
  double* cat = (double*)malloc(sizeof(double) * (size_t)chunk * nf * d);
  double* y = (double*)malloc(sizeof(double) * (size_t)chunk * d);
  double* ctx = (double*)malloc(sizeof(double) * (size_t)chunk * d);
  double* kv = (double*)malloc(sizeof(double) * (size_t)chunk * 2 * m->nkv * h);
  double* tmp = (double*)malloc(sizeof(double) * (size_t)(d > h ? d : h));
  for (int r0 = 0; r0 < total_rows; r0 += chunk) {
    int nr = total_rows - r0 < chunk ? total_rows - r0 : chunk;
    /* concatenation of the n_f target-layer features, in the given order */
    for (int r = 0; r < nr; r++)
      for (int s = 0; s < nf; s++)
        for (int k = 0; k < d; k++) cat[((size_t)r * nf + s) * d + k] = bf(feats[s][(size_t)(r0 + r) * d + k]);
    oracle_linear(nr, d, nf * d, cat, m->w_fc, y);
    for (int r = 0; r < nr; r++) {
      oracle_rmsnorm(d, y + (size_t)r * d, m->hidden_norm, m->eps, tmp);
      for (int k = 0; k < d; k++) ctx[(size_t)r * d + k] = rbf(tmp[k]);
    }
    for (int l = 0; l < m->n_layers; l++) {
      /* rows nq*h .. (nq+2nkv)*h of wqkv are this layer's k heads then v heads */
      oracle_linear(nr, 2 * m->nkv * h, d, ctx, m->wqkv[l] + (size_t)m->nq * h * d, kv);
      for (int r = 0; r < nr; r++) {
        int row = r0 + r, b = 0;
        while (row >= row_off[b + 1]) b++;
        int pos = (pos_start ? pos_start[b] : 0) + row - row_off[b];
        for (int g = 0; g < m->nkv; g++) {
          double* kr = kv + ((size_t)r * 2 * m->nkv + g) * h;
          double* vr = kv + ((size_t)r * 2 * m->nkv + m->nkv + g) * h;
          oracle_rmsnorm(h, kr, m->k_norm[l], m->eps, tmp);
          oracle_rope(h, tmp, (double)pos, m->theta);
          uint16_t* kd = kv_store + kv_index(m, batch, t_cap, l, b, 0, g, pos);
          uint16_t* vd = kv_store + kv_index(m, batch, t_cap, l, b, 1, g, pos);
          for (int i = 0; i < h; i++) {
            kd[i] = oracle_round_bf16(tmp[i]);
            vd[i] = oracle_round_bf16(vr[i]);
          }
        }
      }
    }
  }
  free(cat); free(y); free(ctx); free(kv); free(tmp);
  return 0;
}

/* a3..a7: one bidirectional drafter pass (VFlash (zh) §2.1, §2.2; VFlash blog "Key claims").
 * Block of request b: position 0 = anchor[b], positions 1..L-1 = mask_id; block position j has RoPE
 * position ctx_len[b] + j.  Per layer (pre-norm):
 *   xn = bf16(RMSNorm_attn(x)); [q|k|v] = xn . Wqkv^T;
 *   q, k per head: bf16(RoPE(RMSNorm_{q,k}(.))); v: bf16(v)
 *   o = bf16(softmax(q [Kctx; Kblk]^T / sqrt(h)) [Vctx; Vblk])    (GQA: q head i uses kv head i/(nq/nkv))
 *   x = bf16(x + o . Wo^T)
 *   xn = bf16(RMSNorm_mlp(x)); u = bf16(silu(xn . Wg^T) * (xn . Wu^T)); x = bf16(x + u . Wdown^T)
 * hidden_out [B*L, d] = x after the last layer; layer_hidden (optional) [n_layers, B*L, d].
 * fp8 != 0: the four projections take the FP8 form of the f2 section (weights from the q_ and e_ copies, the
 * bf16 activations xn, o, xn, u quantised per 128-element group of each row).
 * Layers [l0, l1) only, starting from the residual x_in [B*L, d] (bf16) when given, else from the embedding rows
 * (a stage of the pass fed another implementation's residual stream). */
int oracle_draft_block(const oracle_model* m, int batch, int L, const uint16_t* kv_store, int t_cap,
                       const int32_t* ctx_len, const int32_t* anchor, int32_t mask_id, uint16_t* hidden_out,
                       uint16_t* layer_hidden, int fp8, int l0, int l1, const uint16_t* x_in) {
  const int d = m->d, h = m->h, nq = m->nq, nkv = m->nkv, F = m->F;
  const int M = batch * L, nqkv = (nq + 2 * nkv) * h, grp = nq / nkv;
  if (L < 1 || batch < 1 || nq % nkv || l0 < 0 || l1 > m->n_layers || l0 >= l1) return -1;
  for (int b = 0; b < batch; b++) {
    if (ctx_len[b] < 0 || ctx_len[b] > t_cap) return -1;
    if (anchor[b] < 0 || anchor[b] >= m->V) return -1;
  }
  if (mask_id < 0 || mask_id >= m->V) return -1;
  double* x = (double*)malloc(sizeof(double) * (size_t)M * d);
  double* xn = (double*)malloc(sizeof(double) * (size_t)M * d);
  double* qkv = (double*)malloc(sizeof(double) * (size_t)M * nqkv);
  double* q = (double*)malloc(sizeof(double) * (size_t)M * nq * h);
  double* kb = (double*)malloc(sizeof(double) * (size_t)M * nkv * h);  /* [b][g][j][h] */
  double* vb = (double*)malloc(sizeof(double) * (size_t)M * nkv * h);
  double* o = (double*)malloc(sizeof(double) * (size_t)M * nq * h);
  double* dx = (double*)malloc(sizeof(double) * (size_t)M * (d > 2 * F ? d : 2 * F));
  double* hm = (double*)malloc(sizeof(double) * (size_t)M * F);
  const double scale = 1.0 / sqrt((double)h);

  for (int b = 0; b < batch; b++)
    for (int j = 0; j < L; j++) {
      int id = j == 0 ? anchor[b] : mask_id;
      size_t r = (size_t)b * L + j;
      for (int k = 0; k < d; k++) x[r * d + k] = x_in ? bf(x_in[r * d + k]) : bf(m->embed[(size_t)id * d + k]);
    }

  for (int l = l0; l < l1; l++) {
    for (int r = 0; r < M; r++) {
      oracle_rmsnorm(d, x + (size_t)r * d, m->attn_norm[l], m->eps, xn + (size_t)r * d);
      for (int k = 0; k < d; k++) xn[(size_t)r * d + k] = rbf(xn[(size_t)r * d + k]);
    }
    linear_of(fp8, M, nqkv, d, xn, m->wqkv[l], m->q_wqkv[l], m->e_wqkv[l], qkv);
#pragma omp parallel
    {
      double* t = (double*)malloc(sizeof(double) * (size_t)h);
#pragma omp for schedule(static)
      for (int r = 0; r < M; r++) {
        int b = r / L, j = r % L;
        double pos = (double)(ctx_len[b] + j);
        const double* row = qkv + (size_t)r * nqkv;
        for (int i = 0; i < nq; i++) {
          oracle_rmsnorm(h, row + (size_t)i * h, m->q_norm[l], m->eps, t);
          oracle_rope(h, t, pos, m->theta);
          for (int e = 0; e < h; e++) q[((size_t)r * nq + i) * h + e] = rbf(t[e]);
        }
        for (int g = 0; g < nkv; g++) {
          oracle_rmsnorm(h, row + (size_t)(nq + g) * h, m->k_norm[l], m->eps, t);
          oracle_rope(h, t, pos, m->theta);
          size_t dst = (((size_t)b * nkv + g) * L + j) * h;
          for (int e = 0; e < h; e++) {
            kb[dst + e] = rbf(t[e]);
            vb[dst + e] = rbf(row[(size_t)(nq + nkv + g) * h + e]);
          }
        }
      }
      free(t);
    }
    /* attention: one call per (request, q head) over that request's context and block keys */
#pragma omp parallel
    {
      double* qh = (double*)malloc(sizeof(double) * (size_t)L * h);
      double* oh = (double*)malloc(sizeof(double) * (size_t)L * h);
#pragma omp for schedule(dynamic) collapse(2)
      for (int b = 0; b < batch; b++)
        for (int i = 0; i < nq; i++) {
          int g = i / grp;
          for (int j = 0; j < L; j++)
            for (int e = 0; e < h; e++) qh[(size_t)j * h + e] = q[(((size_t)b * L + j) * nq + i) * h + e];
          const uint16_t* kc = kv_store + kv_index(m, batch, t_cap, l, b, 0, g, 0);
          const uint16_t* vc = kv_store + kv_index(m, batch, t_cap, l, b, 1, g, 0);
          oracle_attention(h, L, qh, ctx_len[b], kc, vc, L, kb + ((size_t)b * nkv + g) * L * h,
                           vb + ((size_t)b * nkv + g) * L * h, scale, oh);
          for (int j = 0; j < L; j++)
            for (int e = 0; e < h; e++) o[(((size_t)b * L + j) * nq + i) * h + e] = rbf(oh[(size_t)j * h + e]);
        }
      free(qh);
      free(oh);
    }
    linear_of(fp8, M, d, nq * h, o, m->wo[l], m->q_wo[l], m->e_wo[l], dx);
    for (size_t e = 0; e < (size_t)M * d; e++) x[e] = rbf(x[e] + dx[e]);
    for (int r = 0; r < M; r++) {
      oracle_rmsnorm(d, x + (size_t)r * d, m->mlp_norm[l], m->eps, xn + (size_t)r * d);
      for (int k = 0; k < d; k++) xn[(size_t)r * d + k] = rbf(xn[(size_t)r * d + k]);
    }
    linear_of(fp8, M, 2 * F, d, xn, m->w_gate_up[l], m->q_gate_up[l], m->e_gate_up[l], dx); /* gate | up */
    for (int r = 0; r < M; r++)
      for (int f = 0; f < F; f++) {
        double gv = dx[(size_t)r * 2 * F + f], uv = dx[(size_t)r * 2 * F + F + f];
        hm[(size_t)r * F + f] = rbf(oracle_silu(gv) * uv);
      }
    linear_of(fp8, M, d, F, hm, m->w_down[l], m->q_down[l], m->e_down[l], dx);
    for (size_t e = 0; e < (size_t)M * d; e++) x[e] = rbf(x[e] + dx[e]);
    if (layer_hidden)
      for (size_t e = 0; e < (size_t)M * d; e++)
        layer_hidden[(size_t)l * M * d + e] = oracle_round_bf16(x[e]);
  }
  for (size_t e = 0; e < (size_t)M * d; e++) hidden_out[e] = oracle_round_bf16(x[e]);
  free(x); free(xn); free(qkv); free(q); free(kb); free(vb); free(o); free(dx); free(hm);
  return 0;
}

/* a8: final RMSNorm, LM head restricted to the position's legal ids, argmax (VFlash (zh) §2.5).
 * For block positions j = 1..L-1: z = bf16(RMSNorm_final(hidden)); logit_v = z . W_lm[v] for legal v only;
 * token = argmax over legal v of float(logit_v), lowest id first on ties.
 *   pos_class NULL: every id in [0, V) is legal.  Otherwise class c's ids are the union of ranges
 *   class_ranges[2*class_off[c] ..].
 * Outputs: tokens [B, L-1]; logits (optional) [B*(L-1), V] double, only legal columns written;
 * margin (optional) [B*(L-1)] = top-1 minus top-2 fp32 logit (INFINITY when one id is legal).
 * fp8 != 0: logits from the FP8 LM-head copy and the quantised z (f2 section). */
int oracle_constrain_argmax(const oracle_model* m, int batch, int L, const uint16_t* hidden, int n_class,
                            const int32_t* class_off, const int32_t* class_ranges, const int16_t* pos_class,
                            int32_t* tokens, double* logits, double* margin, int fp8) {
  const int d = m->d, V = m->V, P = L - 1;
  if (L < 2) return -1;
  const int all_off[2] = {0, 1};
  const int32_t all_rng[2] = {0, V};
  if (!pos_class) {
    n_class = 1;
    class_off = all_off;
    class_ranges = all_rng;
  }
  double* z = (double*)malloc(sizeof(double) * (size_t)batch * P * d);
  double* tmp = (double*)malloc(sizeof(double) * (size_t)d);
  for (int b = 0; b < batch; b++)
    for (int j = 1; j < L; j++) {
      int r = b * P + j - 1;
      for (int k = 0; k < d; k++) tmp[k] = bf(hidden[((size_t)b * L + j) * d + k]);
      oracle_rmsnorm(d, tmp, m->final_norm, m->eps, z + (size_t)r * d);
      for (int k = 0; k < d; k++) z[(size_t)r * d + k] = rbf(z[(size_t)r * d + k]);
    }
  free(tmp);
  int rc = 0;
  for (int c = 0; c < n_class && rc == 0; c++) {
    /* rows of this class */
    int nrow = 0;
    int* rows = (int*)malloc(sizeof(int) * (size_t)(batch * P > 0 ? batch * P : 1));
    for (int b = 0; b < batch; b++)
      for (int j = 1; j < L; j++) {
        int cls = pos_class ? pos_class[(size_t)b * L + j] : 0;
        if (cls < 0 || cls >= n_class) rc = -1;
        if (cls == c) rows[nrow++] = b * P + j - 1;
      }
    if (nrow == 0 || rc) { free(rows); continue; }
    double* zc = (double*)malloc(sizeof(double) * (size_t)nrow * d);
    for (int i = 0; i < nrow; i++) memcpy(zc + (size_t)i * d, z + (size_t)rows[i] * d, sizeof(double) * d);
    float* best = (float*)malloc(sizeof(float) * nrow);
    float* second = (float*)malloc(sizeof(float) * nrow);
    int* arg = (int*)malloc(sizeof(int) * nrow);
    for (int i = 0; i < nrow; i++) { best[i] = -INFINITY; second[i] = -INFINITY; arg[i] = -1; }
    for (int q = class_off[c]; q < class_off[c + 1]; q++) {
      int lo = class_ranges[2 * q], hi = class_ranges[2 * q + 1];
      if (lo < 0 || hi > V || lo >= hi) { rc = -1; break; }
      int n = hi - lo;
      double* lg = (double*)malloc(sizeof(double) * (size_t)nrow * n);
      linear_of(fp8, nrow, n, d, zc, m->lm_head + (size_t)lo * d, fp8 ? m->q_lm_head + (size_t)lo * d : NULL,
                fp8 ? m->e_lm_head + (size_t)lo * (d / 128) : NULL, lg);
      /* ids ascending within and across ranges (ranges are sorted), so strict '>' keeps the lowest id */
      for (int i = 0; i < nrow; i++)
        for (int v = 0; v < n; v++) {
          double lv = lg[(size_t)i * n + v];
          float f = (float)lv;
          if (logits) logits[(size_t)rows[i] * V + lo + v] = lv;
          if (f > best[i]) { second[i] = best[i]; best[i] = f; arg[i] = lo + v; }
          else if (f > second[i]) second[i] = f;
        }
      free(lg);
    }
    for (int i = 0; i < nrow; i++) {
      tokens[rows[i]] = arg[i];
      if (margin) margin[rows[i]] = isinf(second[i]) ? INFINITY : (double)best[i] - (double)second[i];
    }
    free(zc); free(best); free(second); free(arg); free(rows);
  }
  free(z);
  return rc;
}

/* ------------------------------------------------------------------------------------------------------ */
/* a9: acceptance                                                                                           */

static int in_class(int tok, int c, const int32_t* class_off, const int32_t* class_ranges) {
  for (int q = class_off[c]; q < class_off[c + 1]; q++)
    if (tok >= class_ranges[2 * q] && tok < class_ranges[2 * q + 1]) return 1;
  return 0;
}

/* Text mode (VFlash blog "Method"; VFlash (zh) §2.1): n = longest prefix with d_i == t_i (i <= L-1),
 * accept = n + 1, committed = d_1..d_n, t_{n+1}.
 * Schema mode (VFlash (zh) §2.5): p = first position 1..L-1 whose rule fails; accept = p - 1, or L - 1
 * when none fails; committed = d_1..d_accept.  Rules:
 *   1 member: token in its class;  2 digit: member, and pad allowed only while the previous slot is not a
 *   digit slot holding a real digit;  3 last digit: member and not pad (plus the same ordering rule).
 * Committed entries beyond accept are -1.  valid[b] = 1 when nothing failed. */
int oracle_verify(int mode, int batch, int L, const int32_t* draft, const int32_t* target, int n_class,
                  const int32_t* class_off, const int32_t* class_ranges, const int16_t* pos_class,
                  const int8_t* rule, int32_t pad_id, int32_t* accept_len, int32_t* committed, int32_t* valid) {
  if (L < 2) return -1;
  for (int b = 0; b < batch; b++) {
    const int32_t* dr = draft + (size_t)b * (L - 1);
    int32_t* cm = committed + (size_t)b * L;
    int acc, ok;
    if (mode == 0) {
      const int32_t* tg = target + (size_t)b * L;
      int n = 0;
      while (n < L - 1 && dr[n] == tg[n]) n++;
      for (int i = 0; i < n; i++) cm[i] = dr[i];
      cm[n] = tg[n];
      acc = n + 1;
      ok = n == L - 1;
    } else {
      int p = L; /* first failing position, L when none */
      for (int j = 1; j < L && p == L; j++) {
        int rl = rule[(size_t)b * L + j];
        int tok = dr[j - 1];
        int fail = 0;
        if (rl != 0) {
          int c = pos_class[(size_t)b * L + j];
          if (c < 0 || c >= n_class) return -1;
          if (!in_class(tok, c, class_off, class_ranges)) fail = 1;
        }
        if (rl == 2 || rl == 3) {
          int prev_rule = rule[(size_t)b * L + j - 1];
          int prev_real_digit = (j >= 2) && (prev_rule == 2 || prev_rule == 3) && dr[j - 2] != pad_id;
          if (tok == pad_id && (rl == 3 || prev_real_digit)) fail = 1;
        }
        if (fail) p = j;
      }
      acc = p - 1;
      for (int i = 0; i < acc; i++) cm[i] = dr[i];
      ok = p == L;
    }
    for (int i = acc; i < L; i++) cm[i] = -1;
    accept_len[b] = acc;
    if (valid) valid[b] = ok;
  }
  return 0;
}

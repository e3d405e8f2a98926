// fpd_api.cu — the C ABI declared in include/fpd.h: host-side validation, the model handle, workspace
// carving, and the order of kernel launches of each call.  Every entry point validates all of its arguments
// before it launches anything and returns an fpd_status; nothing here synchronises, allocates or copies
// between host and device except fpd_model_create / fpd_model_destroy / fpd_device_status.
#include <nvtx3/nvToolsExt.h>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "fpd_kernels.cuh"

namespace fpd {
std::atomic<uint64_t> g_launches{0};
}

using namespace fpd;

namespace {

thread_local std::string t_err;

fpd_status fail(fpd_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_err = buf;
  return s;
}

fpd_status cuda_fail(cudaError_t e, const char* where) {
  return fail(FPD_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

#define FPD_CUDA(call, where)                         \
  do {                                                \
    cudaError_t e_ = (call);                          \
    if (e_ != cudaSuccess) return cuda_fail(e_, where); \
  } while (0)

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// ---- workspace carving -------------------------------------------------------------------------------------------
struct Carver {
  size_t off = 0;
  char* base = nullptr;
  template <class T>
  T* take(size_t count) {
    off = align_up(off, 256);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += count * sizeof(T);
    return p;
  }
};

constexpr int kPrepChunk = 4096;   // context rows per fusion/projection pass (bounds the workspace)
constexpr int kLmColTile = 128;    // vocabulary ids per LM-head work item (the 128-row MMA operand)

// Largest split-K partial buffer (floats) any row count 1..R_max needs for an N x K GEMM.  The split count
// only changes where the tile counts change, so the row counts at tile boundaries cover the maximum.
size_t part_floats_bound(const Model& m, int R_max, int N, int K) {
  size_t best = 0;
  auto eval = [&](int R) {
    if (R < 1 || R > R_max) return;
    TcPlan pl = tc_plan_gemm(R, N, K, m.num_sms);
    best = std::max(best, (size_t)pl.splits * R * N);
  };
  eval(16); eval(32); eval(64); eval(R_max);
  for (int R = 128; R <= R_max; R += 128) eval(R);
  return best;
}

struct DraftWs {
  bf16 *xn, *q, *kblk, *vblk, *o, *hmid;
  float* part;
  float* o_part;
  float2* ml;
  int att_splits, att_chunk;
  TcPlan p_qkv, p_o, p_sw, p_down;
  // many-token path: token-tile GEMMs with fused epilogues; sums of squares [column tiles][M]
  bool tok, att_tc;
  float* ss_tok;
  // few-token path (k_stream.cu)
  bool stream;
  StreamPlan s_qkv, s_o, s_sw, s_down;
  float *ss_a, *ss_b;       // sums of squares of the residual stream [parts][16]
  int *cnt_qkv, *cnt_o, *cnt_down, *cnt_sw, n_cnt;
};

// The few-token path takes calls with at most 16 block positions in all.
bool use_stream(const Model& m, int B, int L) { return B * L <= kStreamMaxTokens && stream_shape_ok(m.d); }

// Shapes whose streamed matrices can take the 8-bit form: every K a multiple of the 128-element group.
bool fp8_shape_ok(const fpd_model_desc& d) {
  return stream_shape_ok(d) && d.d_model % 128 == 0 && (d.n_q_heads * d.head_dim) % 128 == 0 && d.d_ff % 128 == 0;
}

DraftWs carve_draft_stream(const Model& m, Carver& c, int B, int L, int t_cap, bool fp8) {
  const auto& d = m.d;
  DraftWs w{};
  w.stream = true;
  const int M = B * L, S = kStreamMaxTokens;
  const int nqkv = (d.n_q_heads + 2 * d.n_kv_heads) * d.head_dim, nqh = d.n_q_heads * d.head_dim;
  w.s_qkv = stream_plan(nqkv / 128, d.d_model, m.num_sms, true, fp8);
  w.s_o = stream_plan(d.d_model / 128, nqh, m.num_sms, true, fp8);
  w.s_sw = stream_plan(d.d_ff / 64, d.d_model, m.num_sms, true, fp8);
  w.s_down = stream_plan(d.d_model / 128, d.d_ff, m.num_sms, true, fp8);
  const size_t part = std::max(std::max(stream_part_floats(w.s_qkv), stream_part_floats(w.s_o)),
                               std::max(stream_part_floats(w.s_down), stream_part_floats(w.s_sw)));
  w.part = c.take<float>(std::max<size_t>(part, 1));
  w.q = c.take<bf16>((size_t)M * nqh);
  w.kblk = c.take<bf16>((size_t)M * d.n_kv_heads * d.head_dim);
  w.vblk = c.take<bf16>((size_t)M * d.n_kv_heads * d.head_dim);
  w.o = c.take<bf16>((size_t)M * nqh);
  w.hmid = c.take<bf16>((size_t)M * d.d_ff);
  w.ss_a = c.take<float>((size_t)(d.d_model / 128) * S);
  w.ss_b = c.take<float>((size_t)(d.d_model / 128) * S);
  w.n_cnt = w.s_qkv.tiles + 2 * w.s_o.tiles + w.s_sw.tiles;
  w.cnt_qkv = c.take<int>(w.n_cnt);
  w.cnt_o = w.cnt_qkv ? w.cnt_qkv + w.s_qkv.tiles : nullptr;
  w.cnt_down = w.cnt_o ? w.cnt_o + w.s_o.tiles : nullptr;
  w.cnt_sw = w.cnt_down ? w.cnt_down + w.s_o.tiles : nullptr;
  attn_plan(B, L, d.n_q_heads, d.n_kv_heads, t_cap, m.num_sms, &w.att_splits, &w.att_chunk);
  w.o_part = c.take<float>((size_t)w.att_splits * M * nqh);
  w.ml = c.take<float2>((size_t)w.att_splits * M * d.n_q_heads);
  return w;
}

// From 257 block positions: token tiles on the 128-row MMA operand, epilogues fused into the GEMMs.  A projection
// does about M flops per weight byte, so below the bf16 tensor rate / HBM rate (about 260) a block is HBM-bound,
// and the weight tiles on the 128-row operand with K split over all SMs (reduced by the row kernels) stream the
// weights faster than token tiles, which leave SMs idle on the narrow projections (256 rows, 16 x 16 positions:
// 1.29 -> 1.15 ms per step at context 512, 2.72 -> 2.08 ms at 8192).
constexpr int kTokMinRows = 257;
// Context preparation takes the one-GEMM K/V path (EPI_KV_CTX) from 65 rows.
constexpr int kKvCtxMinRows = 65;

DraftWs carve_draft_tok(const Model& m, Carver& c, int B, int L, int t_cap) {
  const auto& d = m.d;
  DraftWs w{};
  w.tok = true;
  const int M = B * L;
  const int nqkv = (d.n_q_heads + 2 * d.n_kv_heads) * d.head_dim, nqh = d.n_q_heads * d.head_dim;
  w.p_qkv = tc_plan_tok(M, nqkv, d.d_model, m.num_sms);
  w.p_o = tc_plan_tok(M, d.d_model, nqh, m.num_sms);
  w.p_sw = tc_plan_swiglu(M, d.d_ff, d.d_model, m.num_sms);
  w.p_down = tc_plan_tok(M, d.d_model, d.d_ff, m.num_sms);
  w.xn = c.take<bf16>((size_t)M * d.d_model);
  w.q = c.take<bf16>((size_t)M * nqh);
  w.kblk = c.take<bf16>((size_t)M * d.n_kv_heads * d.head_dim);
  w.vblk = c.take<bf16>((size_t)M * d.n_kv_heads * d.head_dim);
  w.o = c.take<bf16>((size_t)M * nqh);
  w.hmid = c.take<bf16>((size_t)M * d.d_ff);
  w.ss_tok = c.take<float>((size_t)ceil_div(d.d_model, 128) * M);
  w.att_tc = attn_tc_supported(d.head_dim, L, d.n_q_heads, d.n_kv_heads);
  if (w.att_tc)
    attn_tc_plan(B, L, d.n_q_heads, d.n_kv_heads, t_cap, m.num_sms, &w.att_splits, &w.att_chunk);
  else
    attn_plan(B, L, d.n_q_heads, d.n_kv_heads, t_cap, m.num_sms, &w.att_splits, &w.att_chunk);
  w.o_part = c.take<float>((size_t)w.att_splits * M * nqh);
  w.ml = c.take<float2>((size_t)w.att_splits * M * d.n_q_heads);
  return w;
}

DraftWs carve_draft(const Model& m, Carver& c, int B, int L, int t_cap, bool fp8) {
  if (use_stream(m, B, L)) return carve_draft_stream(m, c, B, L, t_cap, fp8);
  if (B * L >= kTokMinRows) return carve_draft_tok(m, c, B, L, t_cap);
  const auto& d = m.d;
  DraftWs w{};
  const int M = B * L;
  const int nqkv = (d.n_q_heads + 2 * d.n_kv_heads) * d.head_dim, nqh = d.n_q_heads * d.head_dim;
  w.p_qkv = tc_plan_gemm(M, nqkv, d.d_model, m.num_sms);
  w.p_o = tc_plan_gemm(M, d.d_model, nqh, m.num_sms);
  w.p_sw = tc_plan_swiglu(M, d.d_ff, d.d_model, m.num_sms);
  w.p_down = tc_plan_gemm(M, d.d_model, d.d_ff, m.num_sms);
  size_t part = 0;
  part = std::max(part, (size_t)w.p_qkv.splits * M * nqkv);
  part = std::max(part, (size_t)w.p_o.splits * M * d.d_model);
  part = std::max(part, (size_t)w.p_down.splits * M * d.d_model);
  w.xn = c.take<bf16>((size_t)M * d.d_model);
  w.part = c.take<float>(part);
  w.q = c.take<bf16>((size_t)M * nqh);
  w.kblk = c.take<bf16>((size_t)M * d.n_kv_heads * d.head_dim);
  w.vblk = c.take<bf16>((size_t)M * d.n_kv_heads * d.head_dim);
  w.o = c.take<bf16>((size_t)M * nqh);
  w.hmid = c.take<bf16>((size_t)M * d.d_ff);
  attn_plan(B, L, d.n_q_heads, d.n_kv_heads, t_cap, m.num_sms, &w.att_splits, &w.att_chunk);
  w.o_part = c.take<float>((size_t)w.att_splits * M * nqh);
  w.ml = c.take<float2>((size_t)w.att_splits * M * d.n_q_heads);
  return w;
}

struct ArgmaxWs {
  bf16* z;   // final-normed rows in class-sorted order
  int *rows_sorted, *inv_sorted, *class_row_off, *n_items;
  unsigned long long *packed, *packed2;
  int4* items;
  int max_items, row_tile;
  // few-token unconstrained path: per-CTA top-2 slots
  bool stream;
  StreamPlan s_lm;
  unsigned long long* slots;
};

ArgmaxWs carve_argmax(const Model& m, Carver& c, int B, int L, bool constrained) {
  ArgmaxWs w{};
  const int n_rows = B * (L - 1);
  if (!constrained && n_rows <= kStreamMaxTokens && stream_shape_ok(m.d)) {
    w.stream = true;
    w.s_lm.tiles = ceil_div(m.d.vocab, 128);
    w.s_lm.splits = 1;
    w.s_lm.k_split = m.d.d_model;
    w.s_lm.grid = std::min(w.s_lm.tiles, m.num_sms);
    w.slots = c.take<unsigned long long>((size_t)w.s_lm.grid * kStreamMaxTokens * 2);
    return w;
  }
  w.row_tile = tc_lm_row_tile(n_rows);
  w.z = c.take<bf16>((size_t)n_rows * m.d.d_model);
  w.rows_sorted = c.take<int>(n_rows);
  w.inv_sorted = c.take<int>(n_rows);
  w.class_row_off = c.take<int>(FPD_MAX_CLASSES + 1);
  w.n_items = c.take<int>(1);
  w.packed = c.take<unsigned long long>(n_rows);
  w.packed2 = c.take<unsigned long long>(n_rows);
  w.max_items = (ceil_div(m.d.vocab, kLmColTile) + 1 + FPD_MAX_RANGES) * (ceil_div(n_rows, w.row_tile) + FPD_MAX_CLASSES);
  w.items = c.take<int4>(w.max_items);
  return w;
}

struct PrepWs {
  float* part;
  bf16* ctx;
  int chunk;
};

PrepWs carve_prep(const Model& m, Carver& c, int rows_max) {
  PrepWs w{};
  const auto& d = m.d;
  w.chunk = std::max(1, std::min(kPrepChunk, rows_max));
  const size_t a = part_floats_bound(m, w.chunk, d.d_model, d.n_feat * d.d_model);
  const size_t b = part_floats_bound(m, w.chunk, 2 * d.n_kv_heads * d.head_dim, d.d_model);
  w.part = c.take<float>(std::max(a, b));
  w.ctx = c.take<bf16>((size_t)w.chunk * d.d_model);
  return w;
}

// Either weight form: the model may switch to 8-bit weights after the caller sized its workspace.
size_t ws_draft_bytes(const Model& m, int B, int L, int t_cap) {
  Carver c0, c1;
  carve_draft(m, c0, B, L, t_cap, false);
  if (fp8_shape_ok(m.d)) carve_draft(m, c1, B, L, t_cap, true);
  return std::max(c0.off, c1.off);
}
size_t ws_argmax_bytes(const Model& m, int B, int L) {
  Carver c0, c1;
  carve_argmax(m, c0, B, L, false);
  carve_argmax(m, c1, B, L, true);
  return std::max(c0.off, c1.off);
}
size_t ws_prep_bytes(const Model& m, int rows) {
  Carver c;
  carve_prep(m, c, rows);
  return c.off;
}

fpd_status check_device(const Model& m) {
  int cur = -1;
  cudaError_t e = cudaGetDevice(&cur);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (cur != m.device) return fail(FPD_ERR_INVALID_ARG, "current device %d is not the model's device %d", cur, m.device);
  return FPD_OK;
}

// ---- layout validation --------------------------------------------------------------------------------------
fpd_status check_layout(const fpd_vocab_layout* lay, int V) {
  if (!lay->class_off || !lay->class_ranges || !lay->pos_class)
    return fail(FPD_ERR_INVALID_ARG, "layout: class_off, class_ranges and pos_class must be non-null");
  if (lay->n_class < 1 || lay->n_class > FPD_MAX_CLASSES)
    return fail(FPD_ERR_CAPACITY, "layout: n_class %d outside [1, %d]", lay->n_class, FPD_MAX_CLASSES);
  if (lay->class_off[0] != 0) return fail(FPD_ERR_SHAPE, "layout: class_off[0] must be 0");
  for (int c = 0; c < lay->n_class; c++) {
    const int q0 = lay->class_off[c], q1 = lay->class_off[c + 1];
    if (q1 <= q0) return fail(FPD_ERR_SHAPE, "layout: class %d has no id range", c);
    if (q1 > FPD_MAX_RANGES) return fail(FPD_ERR_CAPACITY, "layout: more than %d id ranges", FPD_MAX_RANGES);
    for (int q = q0; q < q1; q++) {
      const int lo = lay->class_ranges[2 * q], hi = lay->class_ranges[2 * q + 1];
      if (lo < 0 || hi > V || lo >= hi) return fail(FPD_ERR_SHAPE, "layout: range %d = [%d, %d) invalid for V = %d", q, lo, hi, V);
      if (q > q0 && lo < lay->class_ranges[2 * q - 1])
        return fail(FPD_ERR_SHAPE, "layout: ranges of class %d must be sorted and disjoint", c);
    }
  }
  return FPD_OK;
}

}  // namespace

// ============================================================================================================
extern "C" {

struct fpd_model : public Model {};

}  // extern "C"

namespace fpd {
// Services of this file for entry points defined in other translation units of the library.
fpd_status set_last_error(fpd_status s, const char* msg) {
  t_err = msg;
  return s;
}
size_t argmax_scratch_bytes(const fpd_model* m, int batch, int block_len) { return ws_argmax_bytes(*m, batch, block_len); }

// NVTX range over one entry point; with FPD_DEBUG the call's kernels are also waited for and checked.
struct ApiScope {
  const char* name;
  cudaStream_t st;
  ApiScope(const char* n, void* s) : name(n), st((cudaStream_t)s) { nvtxRangePushA(n); }
  ~ApiScope() { nvtxRangePop(); }
  fpd_status done(fpd_status r) const {
#ifdef FPD_DEBUG
    if (r != FPD_OK) return r;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return r;
    cudaError_t e = cudaStreamSynchronize(st);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return set_last_error(FPD_ERR_CUDA, (std::string(name) + ": " + cudaGetErrorString(e)).c_str());
    int32_t code = 0;
    if (cudaMemcpyFromSymbol(&code, g_device_check, sizeof(code)) == cudaSuccess && code != 0)
      return set_last_error(FPD_ERR_DEVICE_CHECK, (std::string(name) + ": device check " + std::to_string(code)).c_str());
#endif
    return r;
  }
};
}  // namespace fpd

extern "C" {

const char* fpd_last_error(void) { return t_err.c_str(); }

uint64_t fpd_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

fpd_status fpd_device_status(void* stream, int32_t* code) {
  if (!code) return fail(FPD_ERR_INVALID_ARG, "code must be non-null");
  cudaStream_t st = (cudaStream_t)stream;
  int32_t h = 0, zero = 0;
  FPD_CUDA(cudaMemcpyFromSymbolAsync(&h, g_device_check, sizeof(h), 0, cudaMemcpyDeviceToHost, st), "read check word");
  FPD_CUDA(cudaStreamSynchronize(st), "cudaStreamSynchronize");
  FPD_CUDA(cudaMemcpyToSymbolAsync(g_device_check, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st), "clear check word");
  FPD_CUDA(cudaStreamSynchronize(st), "cudaStreamSynchronize");
  *code = h;
  return h ? fail(FPD_ERR_DEVICE_CHECK, "device check %d", h) : FPD_OK;
}

fpd_status fpd_model_create(const fpd_model_desc* desc, const fpd_weights* w, fpd_model** out) {
  if (!desc || !w || !out) return fail(FPD_ERR_INVALID_ARG, "desc, weights and out must be non-null");
  *out = nullptr;
  const fpd_model_desc& d = *desc;
  if (d.n_layers < 1 || d.n_layers > FPD_MAX_LAYERS) return fail(FPD_ERR_UNSUPPORTED, "n_layers %d", d.n_layers);
  if (d.head_dim != 64 && d.head_dim != 128) return fail(FPD_ERR_UNSUPPORTED, "head_dim %d (64 or 128)", d.head_dim);
  if (d.d_model < 64 || d.d_model % 64 || d.d_ff < 64 || d.d_ff % 64)
    return fail(FPD_ERR_UNSUPPORTED, "d_model %d / d_ff %d must be positive multiples of 64", d.d_model, d.d_ff);
  if (d.d_model > 16384)   // the row kernels hold one row per CTA of at most 1024 threads x 16 values
    return fail(FPD_ERR_UNSUPPORTED, "d_model %d exceeds 16384", d.d_model);
  if (d.n_kv_heads < 1 || d.n_q_heads < d.n_kv_heads || d.n_q_heads % d.n_kv_heads)
    return fail(FPD_ERR_UNSUPPORTED, "n_q_heads %d must be a multiple of n_kv_heads %d", d.n_q_heads, d.n_kv_heads);
  if ((d.n_q_heads * d.head_dim) % 64) return fail(FPD_ERR_UNSUPPORTED, "n_q_heads * head_dim must be a multiple of 64");
  if (d.vocab < 2) return fail(FPD_ERR_SHAPE, "vocab %d", d.vocab);
  if (d.n_feat < 1 || d.n_feat > 8) return fail(FPD_ERR_UNSUPPORTED, "n_feat %d (1..8)", d.n_feat);
  if (d.max_pos < 2) return fail(FPD_ERR_SHAPE, "max_pos %d", d.max_pos);
  if (!(d.rms_eps > 0.f) || !(d.rope_theta > 1.f)) return fail(FPD_ERR_SHAPE, "rms_eps must be > 0 and rope_theta > 1");
  const void* glob[] = {w->embed, w->w_fc, w->hidden_norm, w->final_norm, w->lm_head};
  for (const void* p : glob)
    if (!p || !aligned16(p)) return fail(FPD_ERR_INVALID_ARG, "a global weight pointer is null or not 16-byte aligned");
  for (int l = 0; l < d.n_layers; l++) {
    const void* lp[] = {w->attn_norm[l], w->wqkv[l], w->q_norm[l], w->k_norm[l],
                        w->wo[l],        w->mlp_norm[l], w->w_gate_up[l], w->w_down[l]};
    for (const void* p : lp)
      if (!p || !aligned16(p)) return fail(FPD_ERR_INVALID_ARG, "layer %d: a weight pointer is null or not 16-byte aligned", l);
  }
  {
    static std::once_flag once;
    static cudaError_t init_err = cudaSuccess;
    std::call_once(once, [] {
      init_err = tc_init_attributes();
      if (init_err == cudaSuccess) init_err = attn_init_attributes();
      if (init_err == cudaSuccess) init_err = stream_init_attributes();
      if (init_err == cudaSuccess) init_err = attn_tc_init_attributes();
      if (init_err == cudaSuccess) init_err = attn_short_init_attributes();
    });
    if (init_err != cudaSuccess) return cuda_fail(init_err, "kernel attributes");
  }
  fpd_model* m = new fpd_model();
  m->d = d;
  m->w = *w;
  cudaError_t e = cudaGetDevice(&m->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, m->device);
  if (e != cudaSuccess) {
    delete m;
    return cuda_fail(e, "device query");
  }
  // RoPE table: angle(pos, i) = pos * theta^(-2i/h), evaluated in double, stored as fp32 (cos, sin).
  const int half = d.head_dim / 2;
  std::vector<float2> tab((size_t)d.max_pos * half);
  for (int i = 0; i < half; i++) {
    const double f = std::pow((double)d.rope_theta, -2.0 * i / d.head_dim);
    for (int p = 0; p < d.max_pos; p++) {
      const double a = (double)p * f;
      tab[(size_t)p * half + i] = make_float2((float)std::cos(a), (float)std::sin(a));
    }
  }
  e = cudaMalloc(&m->rope, tab.size() * sizeof(float2));
  if (e == cudaSuccess) e = cudaMemcpy(m->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    if (m->rope) cudaFree(m->rope);
    delete m;
    return cuda_fail(e, "RoPE table");
  }
  *out = m;
  return FPD_OK;
}

void fpd_model_destroy(fpd_model* m) {
  if (!m) return;
  if (m->rope) cudaFree(m->rope);
  if (m->fp8_buf) cudaFree(m->fp8_buf);
  delete m;
}

fpd_status fpd_model_enable_fp8(fpd_model* m, void* stream) {
  ApiScope scope("fpd_model_enable_fp8", stream);
  if (!m) return fail(FPD_ERR_INVALID_ARG, "model must be non-null");
  if (m->fp8) return FPD_OK;
  const fpd_model_desc& d = m->d;
  if (!fp8_shape_ok(d))
    return fail(FPD_ERR_UNSUPPORTED, "8-bit weights need the few-token path's shapes and d_model, n_q_heads * head_dim "
                                     "and d_ff multiples of 128");
  fpd_status ds = check_device(*m);
  if (ds) return ds;
  const int nqkv = (d.n_q_heads + 2 * d.n_kv_heads) * d.head_dim, nqh = d.n_q_heads * d.head_dim;
  struct Job {
    const void* w;
    int N, K;
    Model::F8* dst;
  };
  std::vector<Job> jobs;
  for (int l = 0; l < d.n_layers; l++) {
    jobs.push_back({m->w.wqkv[l], nqkv, d.d_model, &m->f8_qkv[l]});
    jobs.push_back({m->w.wo[l], d.d_model, nqh, &m->f8_o[l]});
    jobs.push_back({m->w.w_gate_up[l], 2 * d.d_ff, d.d_model, &m->f8_gu[l]});
    jobs.push_back({m->w.w_down[l], d.d_model, d.d_ff, &m->f8_down[l]});
  }
  jobs.push_back({m->w.lm_head, d.vocab, d.d_model, &m->f8_lm});
  // exponents block-major [K/128][align_up(N, 128)]: one 128-byte copy brings a weight atom's 128 row exponents
  size_t bytes = 0;
  for (const Job& j : jobs)
    bytes = align_up(align_up(bytes, 256) + (size_t)j.N * j.K, 256) + align_up((size_t)j.N, 128) * (j.K / 128);
  void* buf = nullptr;
  cudaError_t e = cudaMalloc(&buf, bytes + 256);
  if (e != cudaSuccess) return cuda_fail(e, "8-bit weight copies");
  cudaStream_t st = (cudaStream_t)stream;
  size_t off = 0;
  for (const Job& j : jobs) {
    off = align_up(off, 256);
    uint8_t* q = (uint8_t*)buf + off;
    off = align_up(off + (size_t)j.N * j.K, 256);
    int8_t* ex = (int8_t*)buf + off;
    const int ld = (int)align_up((size_t)j.N, 128);
    off += (size_t)ld * (j.K / 128);
    if (e == cudaSuccess) e = cudaMemsetAsync(ex, 0, (size_t)ld * (j.K / 128), st);
    if (e == cudaSuccess) e = launch_quantize_fp8((const bf16*)j.w, j.N, j.K, j.K, q, ex, 1, ld, m->num_sms, st);
    j.dst->ld = ld;
    j.dst->q = q;
    j.dst->e = ex;
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    cudaFree(buf);
    for (const Job& j : jobs) *j.dst = Model::F8{};
    return cuda_fail(e, "8-bit weight quantisation");
  }
  m->fp8_buf = buf;
  m->fp8 = true;
  return scope.done(FPD_OK);
}

fpd_status fpd_quantize_fp8(const void* w, int rows, int cols, int ld, void* codes, void* exps, void* stream) {
  ApiScope scope("fpd_quantize_fp8", stream);
  if (!w || !codes || !exps) return fail(FPD_ERR_INVALID_ARG, "w, codes and exps must be non-null");
  if (rows < 1 || cols < 128 || cols % 128 || ld < cols || ld % 8)
    return fail(FPD_ERR_SHAPE, "rows %d, cols %d (a positive multiple of 128), ld %d (>= cols, a multiple of 8)", rows,
                cols, ld);
  if (!aligned16(w) || !aligned16(codes)) return fail(FPD_ERR_INVALID_ARG, "w and codes must be 16-byte aligned");
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = launch_quantize_fp8((const bf16*)w, rows, cols, ld, (uint8_t*)codes, (int8_t*)exps, cols / 128, 1, sms,
                            (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "fpd_quantize_fp8");
  return scope.done(FPD_OK);
}

int32_t fpd_model_fp8_enabled(const fpd_model* m) { return m && m->fp8 ? 1 : 0; }

size_t fpd_kv_store_bytes(const fpd_model* m, int batch, int t_cap) {
  if (!m || batch < 1 || t_cap < 1) return 0;
  return (size_t)m->d.n_layers * batch * 2 * m->d.n_kv_heads * (size_t)t_cap * m->d.head_dim * sizeof(bf16);
}

size_t fpd_workspace_bytes(const fpd_model* m, int batch, int max_block_len, int t_cap) {
  if (!m || batch < 1 || max_block_len < 2 || t_cap < 1) return 0;
  // Calls may use any smaller batch and block length; the carve is not monotone in them (the attention
  // split count grows as the batch shrinks), so take the maximum over all of them.
  size_t a = 0, b = 0;
  for (int bb = 1; bb <= batch; bb++)
    for (int ll = 2; ll <= max_block_len; ll++) {
      a = std::max(a, ws_draft_bytes(*m, bb, ll, t_cap));
      b = std::max(b, ws_argmax_bytes(*m, bb, ll));
    }
  size_t c = ws_prep_bytes(*m, (int)std::min<long long>((long long)batch * t_cap, 1 << 30));
  return std::max(a, std::max(b, c)) + 256;
}

// ---- a1 + a2 ------------------------------------------------------------------------------------------------
fpd_status fpd_prepare_context(fpd_model* m, int batch, int total_rows, const int32_t* row_off,
                               const int32_t* pos_start, const void* const* feats, void* kv_store, int t_cap,
                               void* workspace, size_t ws_bytes, void* stream) {
  return fpd_prepare_context_rows(m, batch, total_rows, row_off, nullptr, pos_start, feats, kv_store, t_cap, workspace,
                                  ws_bytes, stream);
}

static fpd_status prepare_rows_impl(fpd_model* m, int batch, int total_rows, const int32_t* row_off,
                                    const int32_t* row_cnt, const int32_t* pos_start, const void* const* feats,
                                    void* kv_store, int t_cap, void* workspace, size_t ws_bytes, void* stream) {
  if (!m) return fail(FPD_ERR_INVALID_ARG, "model is null");
  const auto& d = m->d;
  if (batch < 1 || total_rows < 0 || t_cap < 1) return fail(FPD_ERR_SHAPE, "batch %d, total_rows %d, t_cap %d", batch, total_rows, t_cap);
  if (t_cap > d.max_pos) return fail(FPD_ERR_CAPACITY, "t_cap %d exceeds max_pos %d", t_cap, d.max_pos);
  if ((long long)total_rows > (long long)batch * t_cap) return fail(FPD_ERR_CAPACITY, "total_rows %d exceeds batch * t_cap", total_rows);
  if (!row_off || !feats || !kv_store || !workspace) return fail(FPD_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(kv_store) || !aligned16(workspace)) return fail(FPD_ERR_INVALID_ARG, "kv_store/workspace not 16-byte aligned");
  for (int s = 0; s < d.n_feat && total_rows > 0; s++)
    if (!feats[s] || !aligned16(feats[s])) return fail(FPD_ERR_INVALID_ARG, "feats[%d] null or not 16-byte aligned", s);
  fpd_status ds = check_device(*m);
  if (ds) return ds;
  Carver c;
  c.base = (char*)workspace;
  PrepWs w = carve_prep(*m, c, total_rows);
  if (c.off > ws_bytes) return fail(FPD_ERR_CAPACITY, "workspace %zu < %zu bytes", ws_bytes, c.off);
  if (total_rows == 0) return FPD_OK;
  cudaStream_t st = (cudaStream_t)stream;
  const int h = d.head_dim, nkv = d.n_kv_heads;
  for (int r0 = 0; r0 < total_rows; r0 += w.chunk) {
    const int R = std::min(w.chunk, total_rows - r0);
    GemmArgs g{};
    for (int s = 0; s < d.n_feat; s++) g.a[s] = (const bf16*)feats[s] + (size_t)r0 * d.d_model;
    g.seg_k = d.d_model;
    g.lda = d.d_model;
    g.b = (const bf16*)m->w.w_fc;
    g.ldb = d.n_feat * d.d_model;
    g.c = w.part;
    g.ldc = d.d_model;
    g.M = R;
    g.N = d.d_model;
    g.K = d.n_feat * d.d_model;
    g.c_split_stride = (size_t)R * g.N;
    const TcPlan pf = tc_plan_gemm(R, g.N, g.K, m->num_sms);
    g.k_split = pf.k_split;
    FPD_CUDA(launch_tc_gemm(g, pf, st), "fusion GEMM");
    FPD_CUDA(launch_rmsnorm_partials(w.ctx, w.part, pf.splits, g.c_split_stride, (const bf16*)m->w.hidden_norm, R,
                                     d.d_model, d.rms_eps, st),
             "fusion RMSNorm");
    if (R >= kKvCtxMinRows && !row_cnt && kvctx_supported(d)) {
      // every layer's K/V in one token-tile GEMM whose epilogue norms, rotates and stores (no fp32 round trip);
      // appends with device-side row counts (the accepted rows of a speculative step) keep the per-layer path
      const bf16* kn[FPD_MAX_LAYERS];
      for (int l = 0; l < d.n_layers; l++) kn[l] = (const bf16*)m->w.k_norm[l];
      KvCtxGemm kg{};
      kg.d = &d;
      kg.ctx = w.ctx;
      kg.R = R;
      kg.wqkv = m->w.wqkv;
      kg.k_norm = kn;
      kg.rope = m->rope;
      kg.store = (bf16*)kv_store;
      kg.batch = batch;
      kg.t_cap = t_cap;
      kg.row0 = r0;
      kg.row_off = row_off;
      kg.row_cnt = row_cnt;
      kg.pos_start = pos_start;
      FPD_CUDA(launch_tc_kvctx(kg, m->num_sms, st), "context K/V GEMM + store epilogue");
      continue;
    }
    for (int l = 0; l < d.n_layers; l++) {
      GemmArgs k{};
      k.a[0] = w.ctx;
      k.seg_k = d.d_model;
      k.lda = d.d_model;
      k.b = (const bf16*)m->w.wqkv[l] + (size_t)d.n_q_heads * h * d.d_model;  // k rows then v rows
      k.ldb = d.d_model;
      k.c = w.part;
      k.ldc = 2 * nkv * h;
      k.M = R;
      k.N = 2 * nkv * h;
      k.K = d.d_model;
      k.c_split_stride = (size_t)R * k.N;
      const TcPlan pk = tc_plan_gemm(R, k.N, k.K, m->num_sms);
      k.k_split = pk.k_split;
      FPD_CUDA(launch_tc_gemm(k, pk, st), "context K/V GEMM");
      FPD_CUDA(launch_kv_post((bf16*)kv_store, w.part, pk.splits, k.c_split_stride, (const bf16*)m->w.k_norm[l],
                              m->rope, row_off, row_cnt, pos_start, batch, l, t_cap, r0, R, nkv, h, d.rms_eps, st),
               "context K/V epilogue");
    }
  }
  return FPD_OK;
}

// ---- a3..a7 -------------------------------------------------------------------------------------------------
static fpd_status draft_block_impl(fpd_model* m, int batch, int L, const void* kv_store, int t_cap,
                                   const int32_t* ctx_len, const int32_t* anchor, int32_t mask_id, void* hidden_out,
                                   void* layer_hidden, void* workspace, size_t ws_bytes, void* stream) {
  if (!m) return fail(FPD_ERR_INVALID_ARG, "model is null");
  const auto& d = m->d;
  if (batch < 1 || L < 2 || t_cap < 1) return fail(FPD_ERR_SHAPE, "batch %d, block_len %d, t_cap %d", batch, L, t_cap);
  if ((long long)t_cap + L > d.max_pos) return fail(FPD_ERR_CAPACITY, "t_cap + block_len %d exceeds max_pos %d", t_cap + L, d.max_pos);
  if (mask_id < 0 || mask_id >= d.vocab) return fail(FPD_ERR_SHAPE, "mask_id %d outside [0, %d)", mask_id, d.vocab);
  if (!kv_store || !ctx_len || !anchor || !hidden_out || !workspace) return fail(FPD_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(kv_store) || !aligned16(hidden_out) || !aligned16(workspace) || (layer_hidden && !aligned16(layer_hidden)))
    return fail(FPD_ERR_INVALID_ARG, "kv_store/hidden_out/layer_hidden/workspace not 16-byte aligned");
  fpd_status ds = check_device(*m);
  if (ds) return ds;
  Carver c;
  c.base = (char*)workspace;
  DraftWs w = carve_draft(*m, c, batch, L, t_cap, m->fp8);
  if (c.off > ws_bytes) return fail(FPD_ERR_CAPACITY, "workspace %zu < %zu bytes", ws_bytes, c.off);
  cudaStream_t st = (cudaStream_t)stream;
  const int M = batch * L, dm = d.d_model, h = d.head_dim, nq = d.n_q_heads, nkv = d.n_kv_heads, F = d.d_ff;
  const int nqkv = (nq + 2 * nkv) * h;
  bf16* x = (bf16*)hidden_out;
  AttnArgs a{};
  a.q = w.q;
  a.store = (const bf16*)kv_store;
  a.kblk = w.kblk;
  a.vblk = w.vblk;
  a.ctx_len = ctx_len;
  a.o_part = w.o_part;
  a.ml = w.ml;
  a.batch = batch;
  a.L = L;
  a.nq = nq;
  a.nkv = nkv;
  a.head_dim = h;
  a.t_cap = t_cap;
  a.rows = M;
  a.splits = w.att_splits;
  a.chunk = w.att_chunk;
  if (w.stream) {
    // few-token path: 5 kernels per layer, norms applied on load, split-K reduced inside the GEMMs, attention
    // splits merged inside the attention kernel
    const bool short_attn = attn_short_supported(h, L, nq, nkv);
    FPD_CUDA(launch_embed_ss(x, w.ss_a, w.cnt_qkv, w.n_cnt, (const bf16*)m->w.embed, anchor, mask_id, batch, L, dm,
                             d.vocab, st),
             "embedding");
    int n_ss = 1;
    for (int l = 0; l < d.n_layers; l++) {
      StreamGemm g{};
      g.M = M;
      g.eps = d.rms_eps;
      g.part = w.part;
      // QKV projection of RMSNorm_attn(x), q/k norm + RoPE at ctx_len + j
      g.epi = SEPI_QKV;
      g.plan = w.s_qkv;
      g.w = (const bf16*)m->w.wqkv[l];
      g.fp8 = m->fp8;
      g.w8 = m->f8_qkv[l].q;
      g.w_exp = m->f8_qkv[l].e;
      g.exp_ld = m->f8_qkv[l].ld;
      g.N = nqkv;
      g.K = dm;
      g.x = x;
      g.ldx = dm;
      g.xform = XF_NORM;
      g.ss_in = w.ss_a;
      g.n_ss = n_ss;
      g.gain = (const bf16*)m->w.attn_norm[l];
      g.counters = w.cnt_qkv;
      g.q = w.q;
      g.kblk = w.kblk;
      g.vblk = w.vblk;
      g.q_norm = (const bf16*)m->w.q_norm[l];
      g.k_norm = (const bf16*)m->w.k_norm[l];
      g.rope = m->rope;
      g.ctx_len = ctx_len;
      g.t_cap = t_cap;
      g.L = L;
      g.nq = nq;
      g.nkv = nkv;
      g.h = h;
      FPD_CUDA(launch_stream_gemm(g, st), "QKV GEMM + q/k norm + RoPE");
      a.layer = l;
      FPD_CUDA(short_attn ? launch_attention_short(a, w.o, st) : launch_attention(a, w.o, st), "attention");
      // O projection + residual
      StreamGemm o = g;
      o.epi = SEPI_RESID;
      o.plan = w.s_o;
      o.w = (const bf16*)m->w.wo[l];
      o.w8 = m->f8_o[l].q;
      o.w_exp = m->f8_o[l].e;
      o.exp_ld = m->f8_o[l].ld;
      o.N = dm;
      o.K = nq * h;
      o.x = w.o;
      o.ldx = nq * h;
      o.xform = XF_COPY;
      o.counters = w.cnt_o;
      o.xres = x;
      o.ss_out = w.ss_b;
      FPD_CUDA(launch_stream_gemm(o, st), "O GEMM + residual");
      // gate/up of RMSNorm_mlp(x) with SwiGLU
      StreamGemm u = g;
      u.epi = SEPI_SWIGLU;
      u.plan = w.s_sw;
      u.w = (const bf16*)m->w.w_gate_up[l];
      u.w8 = m->f8_gu[l].q;
      u.w_exp = m->f8_gu[l].e;
      u.exp_ld = m->f8_gu[l].ld;
      u.N = F;
      u.K = dm;
      u.x = x;
      u.ldx = dm;
      u.xform = XF_NORM;
      u.ss_in = w.ss_b;
      u.n_ss = dm / 128;
      u.gain = (const bf16*)m->w.mlp_norm[l];
      u.hmid = w.hmid;
      u.counters = w.cnt_sw;
      FPD_CUDA(launch_stream_gemm(u, st), "gate/up + SwiGLU");
      // down projection + residual
      StreamGemm dn = o;
      dn.plan = w.s_down;
      dn.w = (const bf16*)m->w.w_down[l];
      dn.w8 = m->f8_down[l].q;
      dn.w_exp = m->f8_down[l].e;
      dn.exp_ld = m->f8_down[l].ld;
      dn.K = F;
      dn.x = w.hmid;
      dn.ldx = F;
      dn.counters = w.cnt_down;
      dn.ss_out = w.ss_a;
      FPD_CUDA(launch_stream_gemm(dn, st), "down GEMM + residual");
      n_ss = dm / 128;
      if (layer_hidden)
        FPD_CUDA(cudaMemcpyAsync((bf16*)layer_hidden + (size_t)l * M * dm, x, (size_t)M * dm * sizeof(bf16),
                                 cudaMemcpyDeviceToDevice, st),
                 "layer_hidden copy");
    }
    return FPD_OK;
  }
  FPD_CUDA(launch_embed_norm(x, w.xn, (const bf16*)m->w.embed, anchor, mask_id, (const bf16*)m->w.attn_norm[0], batch,
                             L, dm, d.vocab, d.rms_eps, st),
           "embed + attention norm");
  if (w.tok) {
    for (int l = 0; l < d.n_layers; l++) {
      TokGemm g{};
      g.qkv = true;
      g.x = w.xn;
      g.w = (const bf16*)m->w.wqkv[l];
      g.M = M;
      g.N = nqkv;
      g.K = dm;
      g.q = w.q;
      g.kblk = w.kblk;
      g.vblk = w.vblk;
      g.q_norm = (const bf16*)m->w.q_norm[l];
      g.k_norm = (const bf16*)m->w.k_norm[l];
      g.rope = m->rope;
      g.ctx_len = ctx_len;
      g.t_cap = t_cap;
      g.L = L;
      g.nq = nq;
      g.nkv = nkv;
      g.hd = h;
      g.eps = d.rms_eps;
      FPD_CUDA(launch_tc_tok(g, w.p_qkv, st), "QKV GEMM + q/k norm + RoPE");
      a.layer = l;
      FPD_CUDA(w.att_tc ? launch_attention_tc(a, w.o, st) : launch_attention(a, w.o, st), "attention");
      TokGemm r{};
      r.qkv = false;
      r.x = w.o;
      r.w = (const bf16*)m->w.wo[l];
      r.M = M;
      r.N = dm;
      r.K = nq * h;
      r.xres = x;
      r.ss_part = w.ss_tok;
      FPD_CUDA(launch_tc_tok(r, w.p_o, st), "O GEMM + residual");
      FPD_CUDA(launch_norm_rows(w.xn, x, w.ss_tok, w.p_o.qt, (const bf16*)m->w.mlp_norm[l], M, dm, d.rms_eps, st),
               "MLP norm");
      FPD_CUDA(launch_tc_swiglu(w.xn, M, dm, (const bf16*)m->w.w_gate_up[l], F, w.hmid, w.p_sw, st), "gate/up + SwiGLU");
      r.x = w.hmid;
      r.w = (const bf16*)m->w.w_down[l];
      r.K = F;
      FPD_CUDA(launch_tc_tok(r, w.p_down, st), "down GEMM + residual");
      if (l + 1 < d.n_layers)
        FPD_CUDA(launch_norm_rows(w.xn, x, w.ss_tok, w.p_down.qt, (const bf16*)m->w.attn_norm[l + 1], M, dm, d.rms_eps,
                                  st),
                 "attention norm");
      if (layer_hidden)
        FPD_CUDA(cudaMemcpyAsync((bf16*)layer_hidden + (size_t)l * M * dm, x, (size_t)M * dm * sizeof(bf16),
                                 cudaMemcpyDeviceToDevice, st),
                 "layer_hidden copy");
    }
    return FPD_OK;
  }
  auto gemm = [&](const bf16* A, int K, const void* W, int N, const TcPlan& pl) {
    GemmArgs g{};
    g.a[0] = A;
    g.seg_k = K;
    g.lda = K;
    g.b = (const bf16*)W;
    g.ldb = K;
    g.c = w.part;
    g.ldc = N;
    g.c_split_stride = (size_t)M * N;
    g.M = M;
    g.N = N;
    g.K = K;
    g.k_split = pl.k_split;
    return launch_tc_gemm(g, pl, st);
  };
  for (int l = 0; l < d.n_layers; l++) {
    // xn holds RMSNorm_attn(x) here (from the embedding or the previous layer's last residual kernel)
    FPD_CUDA(gemm(w.xn, dm, m->w.wqkv[l], nqkv, w.p_qkv), "QKV GEMM");
    FPD_CUDA(launch_qkv_post(w.q, w.kblk, w.vblk, w.part, w.p_qkv.splits, (size_t)M * nqkv,
                             (const bf16*)m->w.q_norm[l], (const bf16*)m->w.k_norm[l], m->rope, ctx_len, t_cap, batch,
                             L, nq, nkv, h, d.rms_eps, st),
             "q/k norm + RoPE");
    a.layer = l;
    FPD_CUDA(launch_attention(a, w.o, st), "attention");
    FPD_CUDA(gemm(w.o, nq * h, m->w.wo[l], dm, w.p_o), "O GEMM");
    FPD_CUDA(launch_residual_norm(x, w.xn, w.part, w.p_o.splits, (size_t)M * dm, (const bf16*)m->w.mlp_norm[l], M, dm,
                                  d.rms_eps, st),
             "residual + MLP norm");
    FPD_CUDA(launch_tc_swiglu(w.xn, M, dm, (const bf16*)m->w.w_gate_up[l], F, w.hmid, w.p_sw, st), "gate/up + SwiGLU");
    FPD_CUDA(gemm(w.hmid, F, m->w.w_down[l], dm, w.p_down), "down GEMM");
    const bf16* next_norm = l + 1 < d.n_layers ? (const bf16*)m->w.attn_norm[l + 1] : nullptr;
    FPD_CUDA(launch_residual_norm(x, w.xn, w.part, w.p_down.splits, (size_t)M * dm, next_norm, M, dm, d.rms_eps, st),
             "residual + next attention norm");
    if (layer_hidden)
      FPD_CUDA(cudaMemcpyAsync((bf16*)layer_hidden + (size_t)l * M * dm, x, (size_t)M * dm * sizeof(bf16),
                               cudaMemcpyDeviceToDevice, st),
               "layer_hidden copy");
  }
  return FPD_OK;
}

// ---- a8 -----------------------------------------------------------------------------------------------------
static fpd_status constrain_argmax_impl(fpd_model* m, int batch, int L, const void* hidden,
                                        const fpd_vocab_layout* layout, int32_t* tokens_out, float* logits_out,
                                        float* margin_out, void* workspace, size_t ws_bytes, void* stream) {
  if (!m) return fail(FPD_ERR_INVALID_ARG, "model is null");
  const auto& d = m->d;
  if (batch < 1 || L < 2) return fail(FPD_ERR_SHAPE, "batch %d, block_len %d", batch, L);
  if (!hidden || !tokens_out || !workspace) return fail(FPD_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(hidden) || !aligned16(workspace)) return fail(FPD_ERR_INVALID_ARG, "hidden/workspace not 16-byte aligned");
  PairTable pt{};
  if (layout) {
    fpd_status s = check_layout(layout, d.vocab);
    if (s) return s;
    if (layout->n_pairs < 0 || layout->n_pairs > FPD_MAX_PAIRS || (layout->n_pairs > 0 && !layout->pairs))
      return fail(FPD_ERR_INVALID_ARG, "n_pairs %d (0..%d) or null pairs", layout->n_pairs, FPD_MAX_PAIRS);
    if (layout->n_pairs > 0 && (layout->off_id < 0 || layout->off_id >= d.vocab))
      return fail(FPD_ERR_SHAPE, "off_id %d outside [0, %d)", layout->off_id, d.vocab);
    pt.n = layout->n_pairs;
    pt.off_id = layout->off_id;
    for (int k = 0; k < pt.n; k++) {
      const int pp = layout->pairs[2 * k], qq = layout->pairs[2 * k + 1];
      if (pp < 1 || pp >= L || qq < 1 || qq >= L || pp == qq)
        return fail(FPD_ERR_SHAPE, "pair %d = (%d, %d) outside block positions 1..%d", k, pp, qq, L - 1);
      pt.p[k] = (int16_t)pp;
      pt.q[k] = (int16_t)qq;
    }
  }
  fpd_status ds = check_device(*m);
  if (ds) return ds;
  Carver c;
  c.base = (char*)workspace;
  ArgmaxWs w = carve_argmax(*m, c, batch, L, layout != nullptr);
  if (c.off > ws_bytes) return fail(FPD_ERR_CAPACITY, "workspace %zu < %zu bytes", ws_bytes, c.off);
  cudaStream_t st = (cudaStream_t)stream;
  const int n_rows = batch * (L - 1);
  if (w.stream) {
    // few positions, whole vocabulary: final norm on load, per-CTA top-2 slots, one decode kernel
    StreamGemm g{};
    g.epi = SEPI_ARGMAX;
    g.plan = w.s_lm;
    g.w = (const bf16*)m->w.lm_head;
    g.fp8 = m->fp8;
    g.w8 = m->f8_lm.q;
    g.w_exp = m->f8_lm.e;
    g.exp_ld = m->f8_lm.ld;
    g.M = n_rows;
    g.N = d.vocab;
    g.K = d.d_model;
    g.x = (const bf16*)hidden;
    g.ldx = d.d_model;
    g.xform = XF_NORM_FULL;
    g.lm_block = L;
    g.gain = (const bf16*)m->w.final_norm;
    g.eps = d.rms_eps;
    g.slots = w.slots;
    g.logits = logits_out;
    FPD_CUDA(launch_stream_gemm(g, st), "LM head + argmax");
    FPD_CUDA(launch_stream_decode(tokens_out, margin_out, w.slots, w.s_lm.grid, n_rows, st), "argmax decode");
    return FPD_OK;
  }
  LmPlan p{};
  p.n_rows = n_rows;
  p.L = L;
  p.ct = kLmColTile;
  p.rt = w.row_tile;
  if (layout) {
    p.n_class = layout->n_class;
    p.n_range = layout->class_off[layout->n_class];
    for (int cl = 0; cl < layout->n_class; cl++)
      for (int q = layout->class_off[cl]; q < layout->class_off[cl + 1]; q++) {
        p.range_lo[q] = layout->class_ranges[2 * q];
        p.range_hi[q] = layout->class_ranges[2 * q + 1];
        p.range_class[q] = cl;
      }
  } else {
    p.n_class = 1;
    p.n_range = 1;
    p.range_lo[0] = 0;
    p.range_hi[0] = d.vocab;
    p.range_class[0] = 0;
  }
  FPD_CUDA(launch_lm_plan(p, layout ? layout->pos_class : nullptr, w.rows_sorted, w.inv_sorted, w.class_row_off,
                          w.items, w.n_items, w.packed, w.packed2, w.max_items, st),
           "LM-head plan");
  FPD_CUDA(launch_rmsnorm_gather(w.z, (const bf16*)hidden, (const bf16*)m->w.final_norm, w.rows_sorted, n_rows,
                                 d.d_model, d.rms_eps, L, st),
           "final norm");
  FPD_CUDA(launch_tc_lmhead(p, w.z, n_rows, (const bf16*)m->w.lm_head, d.d_model, d.vocab, w.items, w.n_items,
                            w.max_items, w.packed, (margin_out || pt.n) ? w.packed2 : nullptr, w.rows_sorted, logits_out,
                            m->num_sms, layout == nullptr, st),
           "LM head + argmax");
  FPD_CUDA(launch_lm_decode(tokens_out, margin_out, w.packed, w.packed2, w.inv_sorted, n_rows, st), "argmax decode");
  FPD_CUDA(launch_pair_offscreen(tokens_out, margin_out, w.packed, w.packed2, w.inv_sorted, w.z,
                                 (const bf16*)m->w.lm_head, d.d_model, L, batch, pt, st),
           "off-screen pairs");
  return FPD_OK;
}

// ---- a9 -----------------------------------------------------------------------------------------------------
static fpd_status verify_impl(int mode, int batch, int L, const int32_t* draft, const int32_t* target,
                              const fpd_vocab_layout* layout, const int8_t* rule, int32_t pad_id, int32_t* accept_len,
                              int32_t* committed, int32_t* valid_out, void* stream, const float* margin = nullptr,
                              float tau = 0.f) {
  if (mode != FPD_VERIFY_TEXT && mode != FPD_VERIFY_SCHEMA) return fail(FPD_ERR_INVALID_ARG, "mode %d", mode);
  if (batch < 1 || L < 2) return fail(FPD_ERR_SHAPE, "batch %d, block_len %d", batch, L);
  if (!draft || !accept_len || !committed) return fail(FPD_ERR_INVALID_ARG, "null pointer argument");
  VerifyTables tb{};
  if (mode == FPD_VERIFY_TEXT) {
    if (!target) return fail(FPD_ERR_INVALID_ARG, "text mode needs target");
  } else {
    if (!layout || !rule) return fail(FPD_ERR_INVALID_ARG, "schema mode needs layout and rule");
    fpd_status s = check_layout(layout, INT32_MAX);
    if (s) return s;
    tb.n_class = layout->n_class;
    for (int cl = 0; cl <= layout->n_class; cl++) tb.class_off[cl] = layout->class_off[cl];
    for (int q = 0; q < layout->class_off[layout->n_class]; q++) {
      tb.lo[q] = layout->class_ranges[2 * q];
      tb.hi[q] = layout->class_ranges[2 * q + 1];
    }
  }
  FPD_CUDA(launch_verify(mode, batch, L, draft, target, tb, layout ? layout->pos_class : nullptr, rule, pad_id,
                         accept_len, committed, valid_out, margin, tau, (cudaStream_t)stream),
           "verify");
  return FPD_OK;
}

static fpd_status sd_advance_impl(int batch, int L, int t_cap, int32_t* accept_len, const int32_t* committed,
                                  int32_t* ctx_len, int32_t* pos_start, int32_t* anchor, void* stream) {
  if (batch < 1 || L < 2 || t_cap < 1) return fail(FPD_ERR_SHAPE, "batch %d, block_len %d, t_cap %d", batch, L, t_cap);
  if (!accept_len || !committed || !ctx_len || !pos_start || !anchor) return fail(FPD_ERR_INVALID_ARG, "null pointer argument");
  FPD_CUDA(launch_sd_advance(batch, L, t_cap, accept_len, committed, ctx_len, pos_start, anchor, (cudaStream_t)stream),
           "speculative-step advance");
  return FPD_OK;
}

// ---- exported entry points: an NVTX range around each call; in a build with FPD_DEBUG defined, every call
// that is not being captured into a graph also synchronises its stream and returns the first CUDA error or
// device-side check of its kernels as its own status ---------------------------------------------------------
fpd_status fpd_prepare_context_rows(fpd_model* m, int batch, int total_rows, const int32_t* row_off,
                                    const int32_t* row_cnt, const int32_t* pos_start, const void* const* feats,
                                    void* kv_store, int t_cap, void* workspace, size_t ws_bytes, void* stream) {
  ApiScope scope("fpd_prepare_context", stream);
  return scope.done(prepare_rows_impl(m, batch, total_rows, row_off, row_cnt, pos_start, feats, kv_store, t_cap,
                                      workspace, ws_bytes, stream));
}

fpd_status fpd_draft_block(fpd_model* m, int batch, int L, const void* kv_store, int t_cap, const int32_t* ctx_len,
                           const int32_t* anchor, int32_t mask_id, void* hidden_out, void* layer_hidden,
                           void* workspace, size_t ws_bytes, void* stream) {
  ApiScope scope("fpd_draft_block", stream);
  return scope.done(draft_block_impl(m, batch, L, kv_store, t_cap, ctx_len, anchor, mask_id, hidden_out, layer_hidden,
                                     workspace, ws_bytes, stream));
}

fpd_status fpd_constrain_argmax(fpd_model* m, int batch, int L, const void* hidden, const fpd_vocab_layout* layout,
                                int32_t* tokens_out, float* logits_out, float* margin_out, void* workspace,
                                size_t ws_bytes, void* stream) {
  ApiScope scope("fpd_constrain_argmax", stream);
  return scope.done(constrain_argmax_impl(m, batch, L, hidden, layout, tokens_out, logits_out, margin_out, workspace,
                                          ws_bytes, stream));
}

fpd_status fpd_verify(int mode, int batch, int L, const int32_t* draft, const int32_t* target,
                      const fpd_vocab_layout* layout, const int8_t* rule, int32_t pad_id, int32_t* accept_len,
                      int32_t* committed, int32_t* valid_out, void* stream) {
  ApiScope scope("fpd_verify", stream);
  return scope.done(verify_impl(mode, batch, L, draft, target, layout, rule, pad_id, accept_len, committed, valid_out,
                                stream));
}

fpd_status fpd_verify_prefix(int batch, int L, const int32_t* draft, const float* margin, float tau,
                             const fpd_vocab_layout* layout, const int8_t* rule, int32_t pad_id, int32_t* accept_len,
                             int32_t* committed, int32_t* valid_out, void* stream) {
  ApiScope scope("fpd_verify_prefix", stream);
  if (!margin) return fail(FPD_ERR_INVALID_ARG, "prefix verification needs the margins");
  if (!(tau >= 0.f)) return fail(FPD_ERR_SHAPE, "tau must be a non-negative number");
  return scope.done(verify_impl(FPD_VERIFY_SCHEMA, batch, L, draft, nullptr, layout, rule, pad_id, accept_len,
                                committed, valid_out, stream, margin, tau));
}

fpd_status fpd_sd_advance(int batch, int L, int t_cap, int32_t* accept_len, const int32_t* committed,
                          int32_t* ctx_len, int32_t* pos_start, int32_t* anchor, void* stream) {
  ApiScope scope("fpd_sd_advance", stream);
  return scope.done(sd_advance_impl(batch, L, t_cap, accept_len, committed, ctx_len, pos_start, anchor, stream));
}

}  // extern "C"

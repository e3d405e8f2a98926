// fpd_testing.cu — diagnostic entry points declared in include/fpd_testing.h (single-kernel checks).
#include "../../include/fpd_testing.h"
#include "fpd_kernels.cuh"

using namespace fpd;

namespace {
int current_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return n;
}

bool attributes_ready() {
  static cudaError_t e = [] {
    cudaError_t r = tc_init_attributes();
    if (r == cudaSuccess) r = attn_init_attributes();
    if (r == cudaSuccess) r = attn_tc_init_attributes();
    if (r == cudaSuccess) r = attn_short_init_attributes();
    if (r == cudaSuccess) r = stream_init_attributes();
    return r;
  }();
  return e == cudaSuccess;
}

void attn_test_plan(int impl, int batch, int L, int nq, int nkv, int t_cap, int sms, int* splits, int* chunk) {
  if (impl == 1)
    attn_tc_plan(batch, L, nq, nkv, t_cap, sms, splits, chunk);
  else
    attn_plan(batch, L, nq, nkv, t_cap, sms, splits, chunk);
}
// The "lowbias32" integer hash (C. Wellons, "Prospecting for Hash Functions", 2018): a counter-based source of
// the synthetic target's pseudo-random ids.
__device__ __forceinline__ uint32_t lowbias32(uint32_t x) {
  x ^= x >> 16;
  x *= 0x7feb352du;
  x ^= x >> 15;
  x *= 0x846ca68bu;
  x ^= x >> 16;
  return x;
}

// target[b][i], i < L: the draft's id for i < g, at i = g (< L - 1) an id != draft (draft + 1 + u mod (V - 1)),
// past it (and at i = L - 1 when every draft id agrees) u mod V, u = lowbias32(salt * 0x9E3779B9 + b * L + i).
__global__ void synthetic_target_kernel(int B, int L, int V, const int32_t* __restrict__ draft,
                                        const int32_t* __restrict__ agree, uint32_t salt, int32_t* __restrict__ target) {
  const int b = blockIdx.x, i = threadIdx.x;
  if (i >= L) return;
  int g = agree[b];
  g = g < 0 ? 0 : (g > L - 1 ? L - 1 : g);
  const uint32_t u = lowbias32(salt * 0x9E3779B9u + (uint32_t)(b * L + i));
  int t;
  if (i < g) t = draft[(size_t)b * (L - 1) + i];
  else if (i == g && i < L - 1) t = (int)(((uint32_t)draft[(size_t)b * (L - 1) + i] + 1u + u % (uint32_t)(V - 1)) % (uint32_t)V);
  else t = (int)(u % (uint32_t)V);
  target[(size_t)b * L + i] = t;
}
}  // namespace

extern "C" {

fpd_status fpd_test_synthetic_target(int batch, int block_len, int vocab, const int32_t* draft, const int32_t* agree,
                                     uint32_t salt, int32_t* target, void* stream) {
  if (batch < 1 || block_len < 2 || block_len > 1024 || vocab < 2) return FPD_ERR_SHAPE;
  if (!draft || !agree || !target) return FPD_ERR_INVALID_ARG;
  synthetic_target_kernel<<<batch, ((block_len + 31) / 32) * 32, 0, (cudaStream_t)stream>>>(batch, block_len, vocab,
                                                                                           draft, agree, salt, target);
  return cudaGetLastError() == cudaSuccess ? FPD_OK : FPD_ERR_CUDA;
}

size_t fpd_test_stream_timeout_workspace_bytes(void) { return 64 * 1024; }

fpd_status fpd_test_stream_timeout(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace || workspace_bytes < fpd_test_stream_timeout_workspace_bytes()) return FPD_ERR_CAPACITY;
  const int sms = current_sms();
  if (!sms || !attributes_ready()) return FPD_ERR_CUDA;
  char* base = (char*)workspace;
  StreamGemm g{};
  g.epi = SEPI_RESID;
  g.M = 16;
  g.N = 128;
  g.K = 64;
  g.plan = stream_plan(1, g.K, sms, false, false);
  g.w = (const bf16*)base;                         // 128 x 64 weights: 16 KB
  g.x = (const bf16*)(base + 16384);               // 16 x 64 activations: 2 KB
  g.ldx = g.K;
  g.xform = XF_COPY;
  g.xres = (bf16*)(base + 20480);                  // 16 x 128 residual: 4 KB
  g.ss_out = (float*)(base + 24576);               // 1 x 16
  g.part = (float*)(base + 32768);
  g.counters = (int*)(base + 28672);
  g.test_extra_tx = 16;                            // the first weight stage waits for 16 bytes that never come
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(workspace, 0, fpd_test_stream_timeout_workspace_bytes(), st) != cudaSuccess) return FPD_ERR_CUDA;
  return launch_stream_gemm(g, st) == cudaSuccess ? FPD_OK : FPD_ERR_CUDA;
}

size_t fpd_test_stream_gemm_workspace_bytes(int N, int K, int fp8) {
  const int sms = current_sms();
  if (!sms || N < 128 || N % 128 || K < 128 || K % 128) return 0;
  const StreamPlan pl = stream_plan(N / 128, K, sms, true, fp8 != 0);
  return 4096 + align_up(stream_part_floats(pl) * sizeof(float), 256) + align_up((size_t)(N / 128) * 16 * 4, 256) +
         align_up((size_t)(N / 128) * 4, 256);
}

fpd_status fpd_test_stream_gemm(int fp8, int M, int N, int K, const void* X, const void* W, const void* W8,
                                const void* Wexp, void* y, void* workspace, size_t workspace_bytes, void* stream) {
  if (M < 1 || M > 16 || N < 128 || N % 128 || K < 128 || K % 128) return FPD_ERR_SHAPE;
  if (!X || !y || !workspace || (fp8 ? (!W8 || !Wexp) : !W)) return FPD_ERR_INVALID_ARG;
  const size_t need = fpd_test_stream_gemm_workspace_bytes(N, K, fp8);
  if (!need || workspace_bytes < need) return FPD_ERR_CAPACITY;
  const int sms = current_sms();
  if (!sms || !attributes_ready()) return FPD_ERR_CUDA;
  StreamGemm g{};
  g.epi = SEPI_RESID;
  g.M = M;
  g.N = N;
  g.K = K;
  g.plan = stream_plan(N / 128, K, sms, true, fp8 != 0);
  g.w = (const bf16*)W;
  g.fp8 = fp8 != 0;
  g.w8 = (const uint8_t*)W8;
  g.w_exp = (const int8_t*)Wexp;   // block-major [K/128][N]
  g.exp_ld = N;
  g.x = (const bf16*)X;
  g.ldx = K;
  g.xform = XF_COPY;
  g.xres = (bf16*)y;
  char* base = (char*)workspace;
  size_t off = 0;
  g.part = (float*)(base + off);
  off = align_up(off + stream_part_floats(g.plan) * sizeof(float), 256);
  g.ss_out = (float*)(base + off);
  off = align_up(off + (size_t)(N / 128) * 16 * 4, 256);
  g.counters = (int*)(base + off);
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(workspace, 0, need, st) != cudaSuccess) return FPD_ERR_CUDA;
  return launch_stream_gemm(g, st) == cudaSuccess ? FPD_OK : FPD_ERR_CUDA;
}

size_t fpd_test_gemm_workspace_bytes(int M, int N, int K) {
  if (M < 1 || N < 1 || K < 64) return 0;
  const int sms = current_sms();
  if (!sms) return 0;
  size_t best = (size_t)M * N;
  for (int pl = -1; pl <= 1; pl++) {
    TcPlan p = tc_plan_force(M, N, K, sms, pl);
    best = std::max(best, (size_t)p.splits * M * N);
  }
  return best * sizeof(float);
}

fpd_status fpd_test_gemm(int placement, int M, int N, int K, const void* A, const void* B, float* C, void* workspace,
                         size_t workspace_bytes, void* stream) {
  if (M < 1 || N < 1 || K < 64 || K % 64 || placement < -1 || placement > 1) return FPD_ERR_SHAPE;
  if (!A || !B || !C || !workspace) return FPD_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  const int sms = current_sms();
  if (!sms || !attributes_ready()) return FPD_ERR_CUDA;
  GemmArgs g{};
  g.a[0] = (const bf16*)A;
  g.seg_k = K;
  g.lda = K;
  g.b = (const bf16*)B;
  g.ldb = K;
  g.ldc = N;
  g.M = M;
  g.N = N;
  g.K = K;
  const TcPlan pl = tc_plan_force(M, N, K, sms, placement);
  if ((size_t)pl.splits * M * N * sizeof(float) > workspace_bytes) return FPD_ERR_CAPACITY;
  g.c = (float*)workspace;
  g.c_split_stride = (size_t)M * N;
  g.k_split = pl.k_split;
  if (launch_tc_gemm(g, pl, st) != cudaSuccess) return FPD_ERR_CUDA;
  return launch_sum_splits(C, (const float*)workspace, pl.splits, (size_t)M * N, st) == cudaSuccess ? FPD_OK : FPD_ERR_CUDA;
}

fpd_status fpd_test_swiglu(int M, int F, int K, const void* X, const void* W, void* hmid, void* stream) {
  if (M < 1 || F < 1 || K < 64 || K % 64) return FPD_ERR_SHAPE;
  if (!X || !W || !hmid) return FPD_ERR_INVALID_ARG;
  const int sms = current_sms();
  if (!sms || !attributes_ready()) return FPD_ERR_CUDA;
  const TcPlan pl = tc_plan_swiglu(M, F, K, sms);
  return launch_tc_swiglu((const bf16*)X, M, K, (const bf16*)W, F, (bf16*)hmid, pl, (cudaStream_t)stream) == cudaSuccess
             ? FPD_OK
             : FPD_ERR_CUDA;
}

size_t fpd_test_attention_workspace_bytes(int impl, int batch, int L, int nq, int nkv, int head_dim, int t_cap) {
  const int sms = current_sms();
  if (!sms || batch < 1 || L < 1 || nkv < 1 || nq % nkv) return 0;
  int splits = 1, chunk = 0;
  attn_test_plan(impl, batch, L, nq, nkv, t_cap, sms, &splits, &chunk);
  const size_t rows = (size_t)batch * L;
  return align_up((size_t)splits * rows * nq * head_dim * sizeof(float), 256) + (size_t)splits * rows * nq * sizeof(float2);
}

fpd_status fpd_test_attention(int impl, int batch, int L, int nq, int nkv, int head_dim, int t_cap, int layer,
                              const int32_t* ctx_len, const void* q, const void* kblk, const void* vblk,
                              const void* store, void* out, void* workspace, size_t workspace_bytes, void* stream) {
  if (impl < 0 || impl > 2 || batch < 1 || L < 1 || nkv < 1 || nq % nkv || t_cap < 1 || layer < 0) return FPD_ERR_SHAPE;
  if (head_dim != 64 && head_dim != 128) return FPD_ERR_UNSUPPORTED;
  if (impl == 1 && !attn_tc_supported(head_dim, L, nq, nkv)) return FPD_ERR_UNSUPPORTED;
  if (impl == 2 && !attn_short_supported(head_dim, L, nq, nkv)) return FPD_ERR_UNSUPPORTED;
  if (!ctx_len || !q || !kblk || !vblk || !store || !out || !workspace) return FPD_ERR_INVALID_ARG;
  const int sms = current_sms();
  if (!sms || !attributes_ready()) return FPD_ERR_CUDA;
  if (workspace_bytes < fpd_test_attention_workspace_bytes(impl, batch, L, nq, nkv, head_dim, t_cap))
    return FPD_ERR_CAPACITY;
  AttnArgs a{};
  a.q = (const bf16*)q;
  a.store = (const bf16*)store;
  a.kblk = (const bf16*)kblk;
  a.vblk = (const bf16*)vblk;
  a.ctx_len = ctx_len;
  a.batch = batch;
  a.L = L;
  a.nq = nq;
  a.nkv = nkv;
  a.head_dim = head_dim;
  a.t_cap = t_cap;
  a.layer = layer;
  a.rows = batch * L;
  attn_test_plan(impl, batch, L, nq, nkv, t_cap, sms, &a.splits, &a.chunk);
  const size_t rows = (size_t)batch * L;
  a.o_part = (float*)workspace;
  a.ml = (float2*)((char*)workspace + align_up((size_t)a.splits * rows * nq * head_dim * sizeof(float), 256));
  cudaStream_t st = (cudaStream_t)stream;
  const cudaError_t e = impl == 2   ? launch_attention_short(a, (bf16*)out, st)
                        : impl == 1 ? launch_attention_tc(a, (bf16*)out, st)
                                    : launch_attention(a, (bf16*)out, st);
  return e == cudaSuccess ? FPD_OK : FPD_ERR_CUDA;
}

}  // extern "C"

// ---- launch plans, host only ---------------------------------------------------------------------------------
extern "C" int fpd_test_plan(int kind, int M, int N, int K, int num_sms, int32_t* out) {
  if (!out || M < 1 || N < 1 || K < 64 || K % 64 || num_sms < 1) return FPD_ERR_SHAPE;
  fpd::TcPlan pl{};
  if (kind == 0) {
    pl = fpd::tc_plan_gemm(M, N, K, num_sms);
  } else if (kind == 1) {
    pl = fpd::tc_plan_tok(M, N, K, num_sms);
  } else if (kind == 2) {
    pl = fpd::tc_plan_swiglu(M, N, K, num_sms);
  } else if (kind == 3) {
    const fpd::StreamPlan sp = fpd::stream_plan(N, K, num_sms, true, false);
    pl.swap = true;
    pl.bn = 16;
    pl.pt = sp.tiles;
    pl.qt = 1;
    pl.splits = sp.splits;
    pl.k_split = sp.k_split;
    pl.grid = sp.grid;
  } else {
    return FPD_ERR_INVALID_ARG;
  }
  out[0] = pl.swap ? 1 : 0;
  out[1] = pl.bn;
  out[2] = pl.pt;
  out[3] = pl.qt;
  out[4] = pl.splits;
  out[5] = pl.k_split;
  out[6] = pl.grid;
  return FPD_OK;
}

extern "C" int fpd_test_attn_plan(int impl, int batch, int L, int nq, int nkv, int t_cap, int num_sms, int32_t* splits,
                                  int32_t* chunk) {
  if (!splits || !chunk || batch < 1 || L < 1 || nkv < 1 || nq % nkv || t_cap < 1 || num_sms < 1) return FPD_ERR_SHAPE;
  int s = 1, c = 0;
  attn_test_plan(impl, batch, L, nq, nkv, t_cap, num_sms, &s, &c);
  *splits = s;
  *chunk = c;
  return FPD_OK;
}

/*
 * fpd_testing.h — diagnostic entry points of libfpd used by the test-suite to check single kernels in
 * isolation against plain PyTorch fp32 references.  They are not part of the drafter hot path and no paper
 * passage defines them; the hot-path entry points are declared in fpd.h.
 */
#ifndef FPD_TESTING_H_
#define FPD_TESTING_H_

#include "fpd.h"

#ifdef __cplusplus
extern "C" {
#endif

/* C[M, N] (fp32, row-major) = A[M, K] . B[N, K]^T with A, B bf16 row-major device matrices, computed by the
 * library's tcgen05 GEMM kernel with the production plan for this shape (placement -1), or with the token tile on
 * the 128-row MMA operand (placement 0), or with the weight tile there (placement 1).  K must be a multiple of 64.
 * workspace holds the split-K partial sums: at least fpd_test_gemm_workspace_bytes(M, N, K) bytes.  Asynchronous. */
fpd_status fpd_test_gemm(int placement, int M, int N, int K, const void* A, const void* B, float* C, void* workspace,
                         size_t workspace_bytes, void* stream);
size_t fpd_test_gemm_workspace_bytes(int M, int N, int K);

/* hmid[M, F] (bf16) = silu(X . Wg^T) * (X . Wu^T) for X [M, K] and W = [Wg; Wu] ([2F, K]) bf16 row-major device
 * matrices, with the gate/up tcgen05 kernel and its SwiGLU epilogue.  Asynchronous on stream. */
fpd_status fpd_test_swiglu(int M, int F, int K, const void* X, const void* W, void* hmid, void* stream);

/* The drafter's block attention of one layer in isolation: out [batch * L, n_q_heads, head_dim] bf16 =
 * softmax(q . [K_ctx ; K_blk]^T / sqrt(h)) [V_ctx ; V_blk] per request and q head (kv head = q head / group), with
 * q [batch * L, nq, h], k_blk / v_blk [batch, nkv, L, h], the context of layer `layer` in store
 * ([n_layers >= layer + 1][batch][K|V][nkv][t_cap][h]) and ctx_len [batch] (all device).  impl 0: the mma.sync
 * kernel (64-row tiles); impl 1: the tcgen05 kernel (128-row tiles, head_dim 128 and L * group >= 128 only);
 * impl 2: the few-token cluster kernel (L * group <= 64; needs no workspace).
 * workspace: fpd_test_attention_workspace_bytes bytes.  Asynchronous on stream. */
fpd_status fpd_test_attention(int impl, int batch, int L, int nq, int nkv, int head_dim, int t_cap, int layer,
                              const int32_t* ctx_len, const void* q, const void* kblk, const void* vblk,
                              const void* store, void* out, void* workspace, size_t workspace_bytes, void* stream);
size_t fpd_test_attention_workspace_bytes(int impl, int batch, int L, int nq, int nkv, int head_dim, int t_cap);

/* The synthetic target row of a text speculative step (a stand-in for the target model's greedy ids, which the
 * pages' workloads would supply): target [batch, block_len] int32 from draft [batch, block_len - 1] and agree
 * [batch] (g, the number of leading positions on which the target agrees with the draft):
 *   target[b][i] = draft[b][i]                          for i < g
 *   target[b][g] = (draft[b][g] + 1 + u mod (V - 1)) mod V   when g < block_len - 1 (never the draft's id)
 *   target[b][i] = u mod V                              otherwise (past g, and the bonus position when g = L - 1)
 * with u = lowbias32(salt * 0x9E3779B9 + b * block_len + i) (C. Wellons' "lowbias32" integer hash, uint32
 * arithmetic).  Asynchronous on stream. */
fpd_status fpd_test_synthetic_target(int batch, int block_len, int vocab, const int32_t* draft, const int32_t* agree,
                                     uint32_t salt, int32_t* target, void* stream);

/* Failure detection without a fault: runs one 16 x 128 x 64 weight-streaming GEMM whose first weight stage is
 * declared 16 bytes larger than its copy, so the MMA warp's bounded mbarrier wait runs out after 1 s.  The kernel
 * records FPD_CHECK_WAIT_TIMEOUT, abandons its loops and returns normally (its TMEM freed); fpd_device_status then
 * reports the code and the context stays usable.  workspace: fpd_test_stream_timeout_workspace_bytes() bytes of
 * device memory (zeroed by the call).  Asynchronous on stream. */
fpd_status fpd_test_stream_timeout(void* workspace, size_t workspace_bytes, void* stream);
size_t fpd_test_stream_timeout_workspace_bytes(void);

/* One weight-streaming GEMM (the few-token path's kernel, residual epilogue) in isolation:
 *   y[M, N] (bf16, updated in place) = bf16(y + X . W^T)
 * X [M, K] bf16 (M <= 16), y [M, N] bf16, N a multiple of 128, with the production split-K plan for N x K.
 * fp8 = 0: W [N, K] bf16 (K a multiple of 64).  fp8 = 1: W8 [N, K] E4M3 codes and Wexp the exponents of the f2 form
 * of fpd.h, block-major [K/128, N] (16-byte aligned; K a multiple of 128); X is quantised per token and 128 elements
 * inside the kernel.
 * workspace: fpd_test_stream_gemm_workspace_bytes(N, K, fp8) bytes (zeroed by the call).  Asynchronous. */
fpd_status fpd_test_stream_gemm(int fp8, int M, int N, int K, const void* X, const void* W, const void* W8,
                                const void* Wexp, void* y, void* workspace, size_t workspace_bytes, void* stream);
size_t fpd_test_stream_gemm_workspace_bytes(int N, int K, int fp8);

/* Host only (no GPU, no CUDA call): the launch plan the library picks for a GEMM of M activation rows, N output
 * features and K reduction length on num_sms SMs.  kind 0: fp32-partial GEMM of the context fusion and the 17-256-row
 * blocks; 1: token-tile GEMM with a fused epilogue; 2: gate/up + SwiGLU (N = F features); 3: weight-streaming GEMM of
 * the few-token path (N = output tiles of 128 rows).  out[7] = {weights on the 128-row operand, width of the other
 * operand's tile, tiles along the 128-row operand, tiles along the other, K splits, K per split, grid}.
 * Returns FPD_OK, or FPD_ERR_SHAPE / FPD_ERR_INVALID_ARG for arguments outside those ranges. */
int fpd_test_plan(int kind, int M, int N, int K, int num_sms, int32_t* out);
/* Host only: the key splits and keys per split of the attention (impl 0: mma.sync tiles, 1: tensor-memory kernel). */
int fpd_test_attn_plan(int impl, int batch, int L, int nq, int nkv, int t_cap, int num_sms, int32_t* splits,
                       int32_t* chunk);

#ifdef __cplusplus
}
#endif
#endif /* FPD_TESTING_H_ */

// k_verify.cu — a9: block-wide acceptance-length scan, one warp per request.
//
// Text mode (VFlash blog, "Method"; VFlash paper (zh) §2.1): greedy verification keeps the longest prefix on
// which the draft agrees with the target's own greedy tokens, plus the target's next token.
// Schema mode (VFlash paper (zh) §2.5): the primitive is accepted whole when the schema validator passes;
// otherwise the positions before the first failing one are retained.  Fixed-width numeral rules follow
// §2.3 (unused HIGH digits hold the mask/pad token; the last digit slot holds a real digit).
// The first failing position is found 32 positions at a time with __ballot_sync + __ffs.
#include "fpd_kernels.cuh"

namespace fpd {

__device__ __forceinline__ bool in_class(int tok, int c, const VerifyTables& t) {
  for (int q = t.class_off[c]; q < t.class_off[c + 1]; q++)
    if (tok >= t.lo[q] && tok < t.hi[q]) return true;
  return false;
}

__global__ void verify_kernel(int mode, int B, int L, const int32_t* __restrict__ draft,
                              const int32_t* __restrict__ target, VerifyTables tb,
                              const int16_t* __restrict__ pos_class, const int8_t* __restrict__ rule, int32_t pad_id,
                              int32_t* __restrict__ accept, int32_t* __restrict__ committed,
                              int32_t* __restrict__ valid, const float* __restrict__ margin, float tau) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= B) return;
  const int32_t* dr = draft + (size_t)b * (L - 1);
  int32_t* cm = committed + (size_t)b * L;
  int acc, ok;
  if (mode == FPD_VERIFY_TEXT) {
    const int32_t* tg = target + (size_t)b * L;
    int n = L - 1;
    for (int base = 0; base < L - 1; base += 32) {
      const int i = base + lane;
      const unsigned m = __ballot_sync(0xffffffffu, i < L - 1 && dr[i] != tg[i]);
      if (m) { n = base + __ffs(m) - 1; break; }
    }
    for (int i = lane; i < L; i += 32) cm[i] = i < n ? dr[i] : (i == n ? tg[n] : -1);
    acc = n + 1;
    ok = n == L - 1;
  } else {
    const int16_t* pc = pos_class + (size_t)b * L;
    const int8_t* rl = rule + (size_t)b * L;
    int p = L;
    for (int base = 1; base < L; base += 32) {
      const int j = base + lane;
      bool fail = false;
      if (j < L) {
        const int r = rl[j], tok = dr[j - 1];
        if (r != FPD_RULE_NONE) {
          const int c = pc[j];
          if (c < 0 || c >= tb.n_class) {
            record_check(kCheckBadClass);
            fail = true;
          } else if (!in_class(tok, c, tb)) {
            fail = true;
          }
        }
        // f3 (VFlash paper (zh) §2.5): an uncertain coordinate ends the kept prefix like a failing rule
        if (r == FPD_RULE_CONFIDENT && margin && !(margin[(size_t)b * (L - 1) + j - 1] >= tau)) fail = true;
        if (r == FPD_RULE_DIGIT || r == FPD_RULE_DIGIT_LAST) {
          const int pr = rl[j - 1];
          const bool prev_real = j >= 2 && (pr == FPD_RULE_DIGIT || pr == FPD_RULE_DIGIT_LAST) && dr[j - 2] != pad_id;
          if (tok == pad_id && (r == FPD_RULE_DIGIT_LAST || prev_real)) fail = true;
        }
      }
      const unsigned m = __ballot_sync(0xffffffffu, fail);
      if (m) { p = base + __ffs(m) - 1; break; }
    }
    acc = p - 1;
    for (int i = lane; i < L; i += 32) cm[i] = i < acc ? dr[i] : -1;
    ok = p == L;
  }
  if (lane == 0) {
    accept[b] = acc;
    if (valid) valid[b] = ok;
  }
}

cudaError_t launch_verify(int mode, int B, int L, const int32_t* draft, const int32_t* target, const VerifyTables& tb,
                          const int16_t* pos_class, const int8_t* rule, int32_t pad_id, int32_t* accept,
                          int32_t* committed, int32_t* valid, const float* margin, float tau, cudaStream_t st) {
  return launch_k(verify_kernel, ceil_div(B, 4), 128, 0, st, mode, B, L, draft, target, tb, pos_class, rule, pad_id,
                  accept, committed, valid, margin, tau);
}

// ---- the step between a text verification and the next block (one thread per request) ------------------------
// VFlash blog, "Method": blocks follow one another; FlashDrive §3.2: the target's features at the accepted
// positions extend the context.  The anchor and the n accepted drafts (accept = n + 1 rows) join the context at
// ctx_len, and the last committed token (the target's token at the first mismatch) anchors the next block.
__global__ void sd_advance_kernel(int B, int L, int t_cap, int32_t* __restrict__ accept,
                                  const int32_t* __restrict__ committed, int32_t* __restrict__ ctx_len,
                                  int32_t* __restrict__ pos_start, int32_t* __restrict__ anchor) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int cl = clamp_ctx(ctx_len[b], t_cap);
  int a = accept[b];
  a = a < 0 ? 0 : (a > L ? L : a);
  if (cl + a > t_cap) {
    record_check(kCheckCtxOverflow);
    a = t_cap - cl;
  }
  pos_start[b] = cl;
  ctx_len[b] = cl + a;
  accept[b] = a;
  if (a > 0) anchor[b] = committed[(size_t)b * L + a - 1];
}

cudaError_t launch_sd_advance(int B, int L, int t_cap, int32_t* accept, const int32_t* committed, int32_t* ctx_len,
                              int32_t* pos_start, int32_t* anchor, cudaStream_t st) {
  return launch_k(sd_advance_kernel, ceil_div(B, 128), 128, 0, st, B, L, t_cap, accept, committed, ctx_len, pos_start,
                  anchor);
}

}  // namespace fpd

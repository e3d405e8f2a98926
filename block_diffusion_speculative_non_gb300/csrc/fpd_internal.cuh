// fpd_internal.cuh — shared internals of libfpd (kernels + C ABI).  Not part of the public ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "../../include/fpd.h"

namespace fpd {

using bf16 = __nv_bfloat16;

// ---- device-side check word (bounded waits that ran out, ids out of range) --------------------------------
// Kernels never trap: they record the first failure here and skip the offending access.
enum DeviceCheck : int32_t {
  kCheckOk = 0,
  kCheckBadToken = 1,        // an id outside [0, V) reached the embedding gather
  kCheckWaitTimeout = 2,     // an mbarrier / flag wait exceeded its limit
  kCheckNoLegalId = 3,       // a position's class had no legal id (empty argmax)
  kCheckBadClass = 4,        // pos_class outside [0, n_class)
  kCheckBadContext = 5,      // a ctx_len outside [0, t_cap] (clamped)
  kCheckBadPosition = 6,     // a context row's position outside [0, t_cap) (row skipped)
  kCheckCtxOverflow = 7,     // an accepted append would pass t_cap (count capped)
};
extern __device__ int32_t g_device_check;

__device__ __forceinline__ void record_check(int32_t code) { atomicCAS(&g_device_check, 0, code); }
// ctx_len of a request, clamped to [0, t_cap]; a value outside is the caller's contract broken: recorded.
__device__ __forceinline__ int clamp_ctx(int cl, int t_cap) {
  if (cl < 0 || cl > t_cap) {
    record_check(kCheckBadContext);
    cl = cl < 0 ? 0 : t_cap;
  }
  return cl;
}

// ---- host-side bookkeeping ---------------------------------------------------------------------------------
extern std::atomic<uint64_t> g_launches;
inline void count_launch(uint64_t n = 1) { g_launches.fetch_add(n, std::memory_order_relaxed); }

// ---- programmatic dependent launch ---------------------------------------------------------------------------
// Every kernel of the library is launched with programmatic stream serialisation: it may start while its
// predecessor in the stream is still running.  pdl_trigger() lets the next kernel launch; pdl_wait() blocks
// until every predecessor grid has completed and its memory is visible.  A kernel touches no buffer another
// kernel writes or reads before pdl_wait() (the GEMM producer only prefetches weight tiles, which nothing
// writes, into its own shared memory).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  count_launch();
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ---- model -------------------------------------------------------------------------------------------------
struct Model {
  fpd_model_desc d;
  fpd_weights w;
  int device = 0;
  int num_sms = 0;
  float2* rope = nullptr;   // [max_pos][head_dim/2] (cos, sin), built in double on the host
  // 8-bit copies of the weight-streamed matrices (fpd_model_enable_fp8), in one allocation the model owns
  struct F8 {
    const uint8_t* q = nullptr;   // E4M3 codes [rows, K]
    const int8_t* e = nullptr;    // exponents, block-major [K / 128][ld]
    int ld = 0;                   // rows rounded up to a multiple of 128
  };
  bool fp8 = false;
  void* fp8_buf = nullptr;
  F8 f8_qkv[FPD_MAX_LAYERS], f8_o[FPD_MAX_LAYERS], f8_gu[FPD_MAX_LAYERS], f8_down[FPD_MAX_LAYERS], f8_lm;
};

// ---- small helpers -----------------------------------------------------------------------------------------
__host__ __device__ constexpr inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ constexpr inline size_t align_up(size_t a, size_t b) { return (a + b - 1) / b * b; }

// Softmax weights as the operand of O += P V: (a, b) -> two packed bf16 pairs (a in the low half) with
// a = hi_a + lo_a and b = hi_b + lo_b to about 2^-17 relative (hi = bf16(x), lo = bf16(x - hi), round to nearest
// even).  Both pairs multiply the bf16 V tile with fp32 accumulation, so the product sees P nearly as exactly as
// fp32 arithmetic would while both operands stay bf16.
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(hi) : "f"(b), "f"(a));
  const float ha = __uint_as_float(hi << 16), hb = __uint_as_float(hi & 0xFFFF0000u);
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(lo) : "f"(b - hb), "f"(a - ha));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Orderable packing of (fp32 value, id) into 64 bits: a larger packed word means a larger value, and for
// equal values the SMALLER id.  atomicMax over packed words is therefore an argmax with lowest-id ties,
// independent of the order in which CTAs arrive.
__device__ __forceinline__ unsigned long long pack_argmax(float v, int id) {
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)id);
}
__device__ __forceinline__ int unpack_argmax_id(unsigned long long p) {
  return (int)(0xFFFFFFFFu - (uint32_t)(p & 0xFFFFFFFFull));
}

// ---- per-head RMSNorm + rotate-half RoPE on a warp's head ----------------------------------------------------------
// Lane `lane` holds elements e = lane + 32k (k < H/32) of one head (H = head_dim).  The RoPE pair of element i
// (< H/2) is i + H/2, held by the same lane.  rope[pos * H/2 + i] = (cos, sin) of angle pos * theta^(-2i/H).
template <int H>
__device__ __forceinline__ void head_norm_rope(float (&v)[H / 32], const bf16* __restrict__ gain, float eps,
                                               const float2* __restrict__ rope_row, bool do_norm, bool do_rope) {
  constexpr int NV = H / 32;
  const int lane = threadIdx.x & 31;
  if (do_norm) {
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < NV; k++) ss += v[k] * v[k];
    const float inv = rsqrtf(warp_sum(ss) / (float)H + eps);
#pragma unroll
    for (int k = 0; k < NV; k++) v[k] = v[k] * inv * __bfloat162float(gain[lane + 32 * k]);
  }
  if (do_rope) {
#pragma unroll
    for (int k = 0; k < NV / 2; k++) {
      const float2 cs = rope_row[lane + 32 * k];
      const float x1 = v[k], x2 = v[k + NV / 2];
      v[k] = x1 * cs.x - x2 * cs.y;
      v[k + NV / 2] = x2 * cs.x + x1 * cs.y;
    }
  }
}

}  // namespace fpd

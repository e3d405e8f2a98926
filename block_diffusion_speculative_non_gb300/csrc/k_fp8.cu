// k_fp8.cu — the 8-bit weight copies of the weight-streaming GEMMs (FlashDrive §3.4 "Quantization": low-bit
// weights cut the bytes a memory-bound decoding step loads).  A bf16 matrix [N, K] (K a multiple of 128) becomes
// E4M3 codes [N, K] plus one power-of-two exponent per 128 consecutive elements of a row (int8, at
// exps[n * exp_rs + block * exp_cs]: [N, K / 128] for the C ABI, block-major [K / 128, N] for the model's copies):
// k = the smallest integer with amax 2^-k <= 448, code = E4M3 nearest to w 2^-k (ties to even, +0 for zero).
// The value a code stands for, decode(code) 2^k, is what the 8-bit GEMMs multiply.
#include "fewtok_common.cuh"

namespace fpd {

namespace {
using namespace fewtok;

// One warp per 128-element group, grid-stride: lane l takes elements 4l .. 4l + 3 (8-byte loads, 4-byte stores).
__global__ void quantize_fp8_kernel(const bf16* __restrict__ w, int N, int K, int ld, uint8_t* __restrict__ codes,
                                    int8_t* __restrict__ exps, int exp_rs, int exp_cs) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const long groups = (long)N * (K / 128);
  const long warps = (long)gridDim.x * (blockDim.x >> 5);
  for (long gi = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); gi < groups; gi += warps) {
    const long n = gi / (K / 128), g = gi % (K / 128);
    const uint2 u = *reinterpret_cast<const uint2*>(w + n * ld + g * 128 + lane * 4);
    const __nv_bfloat162* e = reinterpret_cast<const __nv_bfloat162*>(&u);
    const float2 a = __bfloat1622float2(e[0]), b = __bfloat1622float2(e[1]);
    float amax = fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(b.x), fabsf(b.y)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const int k = fp8_group_exponent(amax);
    const float sc = exp2_int(-k);
    const uint32_t c = e4m3x2(a.x * sc, a.y * sc) | (e4m3x2(b.x * sc, b.y * sc) << 16);
    *reinterpret_cast<uint32_t*>(codes + n * K + g * 128 + lane * 4) = c;
    if (lane == 0) exps[n * exp_rs + g * exp_cs] = (int8_t)k;
  }
}

}  // namespace

cudaError_t launch_quantize_fp8(const bf16* w, int N, int K, int ld, uint8_t* codes, int8_t* exps, int exp_rs,
                                int exp_cs, int num_sms, cudaStream_t st) {
  if (N < 1 || K < 128 || K % 128 || ld < K || ld % 4) return cudaErrorInvalidValue;
  const long groups = (long)N * (K / 128);
  const int blocks = (int)std::min<long>((groups + 7) / 8, (long)num_sms * 16);
  return launch_k(quantize_fp8_kernel, blocks, 256, 0, st, w, N, K, ld, codes, exps, exp_rs, exp_cs);
}

}  // namespace fpd

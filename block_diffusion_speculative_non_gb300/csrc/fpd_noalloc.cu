// fpd_noalloc.cu — fpd_constrain_argmax_noalloc: the constrained LM-head argmax with its scratch memory in a
// fixed, file-scope device array instead of a caller-allocated workspace.
//
// Some callers cannot call cudaMalloc at all: a host framework that owns the whole device heap and forbids
// its plugins from allocating, or a latency-critical loop where cudaMalloc's implicit device synchronisation
// and unbounded run time are not allowed.  They still own their inputs and outputs, but they have no way to
// hand the library a workspace.  This entry point serves them: its scratch lives in g_noalloc_scratch below,
// which the CUDA runtime places on every device that loads the library and keeps until the process exits.
//
// Host code must never pass g_noalloc_scratch itself to a kernel: on the host that name is a stand-in
// object, not a device address (a kernel given it would fault, or on a system where the GPU can read host
// memory, silently use the wrong memory).  The device address is asked for once per device with
// cudaGetSymbolAddress, with that device current, and cached.
#include <cstdio>
#include <mutex>

#include "fpd_kernels.cuh"

namespace fpd {
fpd_status set_last_error(fpd_status s, const char* msg);
size_t argmax_scratch_bytes(const fpd_model* m, int batch, int block_len);
}  // namespace fpd

using namespace fpd;

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;   // 8 MiB on every device that loads the library
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up on the first call per device).
fpd_status scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_last_error(FPD_ERR_CUDA, "cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices) return set_last_error(FPD_ERR_UNSUPPORTED, "device ordinal above 63");
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return set_last_error(FPD_ERR_CUDA, "cudaGetSymbolAddress of the static scratch array failed");
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return FPD_OK;
}

}  // namespace

extern "C" {

fpd_status fpd_constrain_argmax_noalloc(fpd_model* model, int batch, int block_len, const void* hidden,
                                        const fpd_vocab_layout* layout, int32_t* tokens_out, float* logits_out,
                                        void* stream) {
  if (!model) return set_last_error(FPD_ERR_INVALID_ARG, "model is null");
  if (batch < 1 || block_len < 2) return set_last_error(FPD_ERR_SHAPE, "batch must be >= 1 and block_len >= 2");
  const size_t need = argmax_scratch_bytes(model, batch, block_len);
  if (need > kNoAllocScratchBytes) {
    char msg[200];
    snprintf(msg, sizeof(msg),
             "batch %d x block_len %d needs %zu bytes of scratch; the static scratch array holds %zu bytes",
             batch, block_len, need, kNoAllocScratchBytes);
    return set_last_error(FPD_ERR_CAPACITY, msg);
  }
  void* scratch = nullptr;
  fpd_status s = scratch_address(&scratch);
  if (s) return s;
  return fpd_constrain_argmax(model, batch, block_len, hidden, layout, tokens_out, logits_out, nullptr, scratch,
                              kNoAllocScratchBytes, stream);
}

}  // extern "C"

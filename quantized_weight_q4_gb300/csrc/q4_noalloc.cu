// Routed experts with built-in scratch: an entry point that allocates nothing.
//
// q4_moe_experts_ex needs a workspace for its intermediate rows (SiLU(g)*u and
// the per-slot down outputs).  Some callers cannot provide one or let the
// library allocate it: code that runs while a CUDA graph is being captured in
// global mode (cudaMalloc is illegal there), real-time or embedded loops that
// must not allocate after start-up, and hosts whose memory manager owns all
// device memory and forbids foreign cudaMalloc calls.  For them this file
// keeps the scratch in a fixed, file-scope device array that every GPU loading
// the library holds until the process exits.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "q4.h"
#include "q4_kernels.h"

namespace {

// 8 MiB of scratch per device: enough for T * topk * (H + I) * 4 bytes of
// intermediate rows, e.g. 52 tokens of a DeepSeek-V2-sized layer (top-6 of
// 160 experts, H = 5120, I = 1536).
constexpr size_t kStaticScratchBytes = size_t(8) << 20;
__device__ __align__(256) unsigned char g_q4_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device.  The first call on a
// device looks the address up; host code must never use the array's name as
// a device pointer.
int static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return Q4_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_q4_static_scratch) != cudaSuccess || !p) return Q4_ERR_CUDA;
    g_static_ptr[dev] = p;
  }
  *out = g_static_ptr[dev];
  return Q4_OK;
}

}  // namespace

extern "C" {

size_t q4_moe_static_scratch_bytes(void) { return kStaticScratchBytes; }

int q4_moe_experts_noalloc(float* out, const void* x, int x_dtype, const void* W_gate,
                           const void* W_up, const void* W_down, const int32_t* topk_idx,
                           const float* topk_w, int64_t T, int64_t topk, int64_t E, int64_t H,
                           int64_t I, void* stream) {
  if (T <= 0 || topk <= 0 || E <= 0 || H <= 0 || I <= 0) return Q4_ERR_ARG;
  // the least the call takes; with the 8 MiB it may not take the persistent form
  const size_t need = q4::moe_min_workspace_bytes(T, topk, H, I);
  if (need > kStaticScratchBytes) return Q4_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int rc = static_scratch(&scratch);
  if (rc != Q4_OK) return rc;
  return q4_moe_experts_ex(out, x, x_dtype, W_gate, W_up, W_down, topk_idx, topk_w, T, topk, E,
                           H, I, scratch, kStaticScratchBytes, stream);
}

}  // extern "C"

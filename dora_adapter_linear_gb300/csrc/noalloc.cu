// LoRA linear forward for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc (or any allocator) once they are running: inference
// runtimes that plan every byte of device memory up front, plugin hosts that forbid
// allocation after start-up, or code that must not touch the allocator on its hot path.
// lora_linear_fwd_noalloc() runs the same kernels as lora_linear_fwd() but takes its scratch
// from one fixed array that lives in this library's device image, so the caller only
// passes inputs and outputs.
#include <mutex>

#include "../../include/lora_gb300.h"
#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = LORA_NOALLOC_SCRATCH_BYTES;

// The scratch itself.  Every GPU that loads this library holds it until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_dev[64] = {nullptr};  // device address of g_noalloc_scratch, per device

// Host code cannot use &g_noalloc_scratch (that is a host-side shadow, not a device address):
// look the device address up once per device, with that device current.
lora_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return LORA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_dev[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return LORA_ERR_CUDA;
    g_scratch_dev[dev] = p;
  }
  *out = g_scratch_dev[dev];
  return LORA_OK;
}

}  // namespace

extern "C" lora_status lora_linear_fwd_noalloc(const lora_shape* sh, const void* X, const void* W0, const void* A,
                                               const void* B, const void* bias, float s, void* Y, void* Z_save,
                                               void* stream) {
  const size_t need = lora_workspace_bytes(LORA_OP_LINEAR_FWD, sh);
  if (need == 0) return sh == nullptr ? LORA_ERR_INVALID_ARG : LORA_ERR_UNSUPPORTED;
  if (need > kNoAllocScratchBytes) return LORA_ERR_WORKSPACE;  // problem larger than the fixed scratch
  void* scratch = nullptr;
  lora_status e = scratch_for_current_device(&scratch);
  if (e != LORA_OK) return e;
  // the error word at the head of the scratch must start clear for this call
  if (cudaMemsetAsync(scratch, 0, 256, static_cast<cudaStream_t>(stream)) != cudaSuccess) return LORA_ERR_CUDA;
  return lora_linear_fwd(sh, X, W0, A, B, bias, s, Y, Z_save, scratch, kNoAllocScratchBytes, stream);
}

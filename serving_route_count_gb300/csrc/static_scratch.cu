// static_scratch.cu - moe_run for callers that cannot allocate device memory.
//
// Some callers cannot hand the library a scratch buffer: code running under another framework's
// memory pool that exposes no allocator to plug-ins, sandboxed or embedded runtimes where
// cudaMalloc is unavailable or forbidden after start-up, and hot paths that must never allocate.
// For them this entry point runs the layer with its scratch in a fixed-size array that lives in
// the library's own device image: the caller passes only the weights, inputs and output.
//
// The array is a file-scope __device__ variable, so every GPU that loads the library holds its
// kStaticScratchBytes until the process exits, and every call on a device shares it: calls whose
// executions overlap on the GPU (different streams, or different host threads) race on it and
// must be serialised by the caller.  Each call overwrites what it needs (the layer's kernels do
// not rely on any previous contents: the routing launch clears the error word, the quantiser
// launch clears the accumulation buffers), and the array keeps the last call's contents.
#include <mutex>

#include "moe_common.cuh"
#include "../../include/moe_gb300.h"

namespace {

constexpr size_t kStaticScratchBytes = 16u << 20;   // 16 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the array on the current device, resolved once per device and cached for
// the life of the process (the cache assumes the device's primary context lives that long: after
// cudaDeviceReset the cached address would be stale).  Host code must not use the symbol itself:
// on the host it is a stand-in, not a device address.
moe_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    (void)cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_run_static_scratch(const moe_plan_t* plan, const moe_prepared* weights,
                                  const void* x, const int32_t* topk_ids,
                                  const float* topk_weights, void* out, int M, void* stream) {
  if (plan == nullptr || weights == nullptr) return MOE_ERR_ARG;
  size_t need = 0;
  moe_status st = moe_scratch_bytes(plan, &need);
  if (st != MOE_OK) return st;
  if (need > kStaticScratchBytes) return MOE_ERR_CAPACITY;
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != MOE_OK) return st;
  return moe_run(plan, weights, scratch, kStaticScratchBytes, x, topk_ids, topk_weights, out, M,
                 stream);
}

moe_status moe_get_device_error_static(const moe_plan_t* plan, void* stream, int* code) {
  if (plan == nullptr || code == nullptr) return MOE_ERR_ARG;
  size_t need = 0;
  moe_status st = moe_scratch_bytes(plan, &need);
  if (st != MOE_OK) return st;
  if (need > kStaticScratchBytes) return MOE_ERR_CAPACITY;
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != MOE_OK) return st;
  return moe_get_device_error(plan, scratch, stream, code);
}

}  // extern "C"

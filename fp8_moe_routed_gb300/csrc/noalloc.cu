// noalloc.cu -- a forward wi GMM entry point for callers that cannot allocate
// device memory.
//
// fp8moe_gmm_silu_fp8_fwd needs a caller-provided workspace for the quantized
// activation (one e4m3 code per input element plus one f32 scale per row). Some
// callers have no way to provide one: a plugin running inside a host framework
// whose caching allocator already owns nearly all device memory (a cudaMalloc of
// its own would fail, and cudaMalloc/cudaFree can also synchronize the device
// and stall the framework's streams), or a runtime with a fixed memory budget
// that forbids allocations after start-up. This entry point gives them the same
// operation with the workspace taken from a fixed, file-scope device array.
//
// The array is kNoAllocScratchBytes (32 MiB) per GPU, reserved on every device
// that loads this library for as long as the process lives. Calls whose
// workspace would exceed it are rejected with FP8MOE_EWORKSPACE before anything
// is launched. All calls share the one array: two calls that overlap on the GPU
// (different streams, no ordering between them) race on it. Every call fully
// rewrites what it later reads (codes and scales of the rows it covers), so no
// contents need clearing between calls.
//
// The array's device address is looked up once per device and kept. A
// cudaDeviceReset (or anything else that tears down and re-creates the
// device's primary context) reloads the module, possibly elsewhere, and leaves
// the kept address dangling: do not call this entry point again in a process
// after resetting the device.
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "fp8moe.h"
#include "kernels.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

// In host code this name is only a stand-in for the device array, not its
// address: the address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

}  // namespace

extern "C" int fp8moe_gmm_silu_fp8_fwd_noalloc(const void* lhs, int64_t M, int64_t K,
                                                const uint8_t* codes, const float* scale,
                                                int32_t E, int64_t N,
                                                const int32_t* group_sizes, void* out,
                                                fp8moe_stream_t stream) {
  // the regular entry point's argument checks first, so that a bad argument
  // gets the same code here as there, whatever the size
  int empty = 0;
  int rc = fp8moe_internal_check_fwd_args(lhs, M, K, codes, scale, E, N, group_sizes, out, 1,
                                          &empty);
  if (rc != FP8MOE_OK || empty) return rc;
  const size_t need = fp8moe_workspace_size(FP8MOE_OP_GMM_SILU_FP8_FWD, M, K, N, E);
  if (need > kNoAllocScratchBytes) return FP8MOE_EWORKSPACE;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    fp8moe_internal_set_cuda_error((int)e);
    return FP8MOE_ECUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return FP8MOE_EUNSUPPORTED;
  void* scratch = nullptr;
  {
    // Set-up, once per device, with that device current (the first call on a
    // device does it, so that call should come before any stream capture).
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || p == nullptr) {
        fp8moe_internal_set_cuda_error((int)(e != cudaSuccess ? e : cudaErrorInvalidSymbol));
        (void)cudaGetLastError();
        return FP8MOE_ECUDA;
      }
      g_scratch_ptr[dev] = p;
    }
    scratch = g_scratch_ptr[dev];
  }
  return fp8moe_gmm_silu_fp8_fwd(lhs, M, K, codes, scale, E, N, group_sizes, out, scratch,
                                 kNoAllocScratchBytes, stream);
}

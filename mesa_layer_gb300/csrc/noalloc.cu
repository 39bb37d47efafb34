// noalloc.cu -- mesa_forward_chunked for callers that cannot allocate device memory.
//
// Some callers have no way to obtain device memory at the point where they run the layer:
// a host program that hands all GPU memory to its own pool and forbids cudaMalloc, a plugin
// inside a framework that only passes it input and output buffers, or code that records
// work into a CUDA graph, where cudaMalloc is not allowed while the stream is captured.
// This entry point needs nothing from them beyond inputs and outputs: its scratch memory is
// a fixed array in the library's device image (kNoAllocScratchBytes, 32 MiB), which every
// GPU that loads the library keeps until the process exits.
//
// The array's name in host code is only a host-side handle, not a device address, so the
// device address is looked up once per device with cudaGetSymbolAddress, on the first call
// made while that device is current, and cached.  Every call shares the same array: calls
// that overlap on the GPU (on different streams, or from different host threads without
// ordering) race on it.  Nothing in the array needs to start at zero except the status
// word, which mesa_forward_chunked clears itself on every call.
#include <mutex>

#include "../../include/mesa.h"

namespace {

constexpr size_t kNoAllocScratchBytes = MESA_NOALLOC_MAX_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (nullptr on failure).
void *scratch_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int mesa_forward_chunked_noalloc(int B, int H, int T, int dk, int dv, int dtype,
                                            const void *q, const void *k, const void *v,
                                            const float *gamma, const float *lambda_diag,
                                            int cg_iters, float cg_tol, int chunk, void *out,
                                            int32_t *iters_used, cudaStream_t stream) {
  const size_t need = mesa_forward_workspace_size(B, H, T, dk, dv, chunk);
  if (need == 0) return (B < 0 || H < 0 || T < 0) ? MESA_ERR_INVALID_ARG : MESA_ERR_UNSUPPORTED;
  if (need > kNoAllocScratchBytes) return MESA_ERR_WORKSPACE;
  void *scratch = scratch_for_current_device();
  if (!scratch) return MESA_ERR_CUDA;
  return mesa_forward_chunked(B, H, T, dk, dv, dtype, q, k, v, gamma, lambda_diag, cg_iters,
                              cg_tol, chunk, out, iters_used, nullptr, nullptr, nullptr, nullptr,
                              scratch, kNoAllocScratchBytes, stream);
}

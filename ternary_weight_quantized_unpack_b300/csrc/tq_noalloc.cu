// tq_gemv_noalloc: tq_gemv for callers that cannot provide a workspace.
//
// Some callers cannot hand the library device memory: code that must not call into an allocator at
// the point of use (cudaMalloc can synchronise the device and block, which a latency-critical or
// real-time decode loop may not afford), or plain C callers without an allocator of their own.  For
// them this entry point keeps the GEMV's scratch (the transformed activations and per-group sums the
// prep kernel writes) in one fixed array of this library, in device memory, of kScratchBytes bytes.
// It allocates nothing.
//
// Set-up: the first call made with a given device current looks up that device's copy of the array
// (cudaGetSymbolAddress) and remembers it; make that first call before any stream capture.
// Nothing in the array has to start at zero: every call writes the scratch before it reads it.
// The array is shared by all calls on a device, so two calls whose kernels overlap in time (on
// different streams, or from different host threads without ordering) race on it: serialise them.
#include <mutex>

#include "tq_internal.cuh"
#include "tq_kernels.cuh"

namespace tq {
namespace {

constexpr size_t kScratchBytes = static_cast<size_t>(1) << 20;  // 1 MiB
static __device__ __align__(256) uint8_t g_gemv_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// This device's scratch array (looked up once per device, with that device current).
cudaError_t scratch_ptr(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_gemv_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace tq

using namespace tq;

extern "C" tq_status tq_gemv_noalloc(const tq_desc* d, const uint32_t* codes, const uint16_t* scales,
                                     const uint16_t* x, int batch, float* y, void* stream) {
  tq_status st = check_gemv_desc(d);
  if (st != TQ_OK) return st;
  if (batch < 1 || batch > kMaxBatch) return TQ_ERR_INVALID_ARG;
  if (!codes || !scales || !x || !y) return TQ_ERR_INVALID_ARG;
  if (!aligned(codes, 16) || !aligned(scales, 16) || !aligned(x, 16) || !aligned(y, 16)) return TQ_ERR_MISALIGNED;
  const size_t need = gemv_workspace_bytes(d, batch);
  if (need == 0) return TQ_ERR_UNSUPPORTED;
  if (need > kScratchBytes) return TQ_ERR_WORKSPACE;  // the shape needs more scratch than the fixed array
  if (!status_ptr()) return TQ_ERR_CUDA;
  void* scratch = nullptr;
  if (const cudaError_t e = scratch_ptr(&scratch); e != cudaSuccess) return cuda_fail(e);
  const cudaError_t e = launch_gemv(d, codes, scales, x, batch, y, scratch, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return TQ_OK;
}

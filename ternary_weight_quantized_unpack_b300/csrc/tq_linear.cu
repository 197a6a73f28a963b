// Entry points of the dense ternary contraction: tq_gemv (decode) and tq_gemm (prefill).
#include "tq_internal.cuh"
#include "tq_kernels.cuh"

namespace tq {
namespace {

tq_status check_ptrs(const uint32_t* codes, const uint16_t* scales, const uint16_t* x, const void* y,
                     const void* ws) {
  if (!codes || !scales || !x || !y || !ws) return TQ_ERR_INVALID_ARG;
  if (!aligned(codes, 16) || !aligned(scales, 16) || !aligned(x, 16) || !aligned(y, 16)) return TQ_ERR_MISALIGNED;
  if (!aligned(ws, 256)) return TQ_ERR_MISALIGNED;
  return TQ_OK;
}

}  // namespace
}  // namespace tq

using namespace tq;

extern "C" size_t tq_gemv_workspace_bytes(const tq_desc* d, int batch) {
  if (check_gemv_desc(d) != TQ_OK || batch < 1 || batch > kMaxBatch) return 0;
  return gemv_workspace_bytes(d, batch);
}

extern "C" tq_status tq_gemv(const tq_desc* d, const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                             int batch, float* y, void* workspace, size_t workspace_bytes, void* stream) {
  tq_status st = check_gemv_desc(d);
  if (st != TQ_OK) return st;
  if (batch < 1 || batch > kMaxBatch) return TQ_ERR_INVALID_ARG;
  if ((st = check_ptrs(codes, scales, x, y, workspace)) != TQ_OK) return st;
  const size_t need = tq_gemv_workspace_bytes(d, batch);
  if (need == 0) return TQ_ERR_UNSUPPORTED;  // the activations of a CTA's K-range do not fit shared memory
  if (workspace_bytes < need) return TQ_ERR_WORKSPACE;
  if (!status_ptr()) return TQ_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = launch_gemv(d, codes, scales, x, batch, y, workspace, s);
  if (e != cudaSuccess) return cuda_fail(e);
  return TQ_OK;
}

extern "C" int tq_gemv_kernel_count(const tq_desc* d, int batch) {
  if (check_gemv_desc(d) != TQ_OK || batch < 1 || batch > kMaxBatch) return -1;
  return gemv_kernel_count(d, batch);
}

extern "C" size_t tq_gemm_workspace_bytes(const tq_desc* d, int M) {
  if (check_linear_desc(d) != TQ_OK || M < 1) return 0;
  return gemm_workspace_bytes(d, M);
}

extern "C" tq_status tq_gemm(const tq_desc* d, const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                             int M, uint16_t* y, void* workspace, size_t workspace_bytes, void* stream) {
  tq_status st = check_linear_desc(d);
  if (st != TQ_OK) return st;
  if (M < 1) return TQ_ERR_INVALID_ARG;
  if ((st = check_ptrs(codes, scales, x, y, workspace)) != TQ_OK) return st;
  if (workspace_bytes < tq_gemm_workspace_bytes(d, M)) return TQ_ERR_WORKSPACE;
  if (!status_ptr()) return TQ_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (const cudaError_t e = launch_gemm(d, codes, scales, x, M, y, workspace, s); e != cudaSuccess) return cuda_fail(e);
  return TQ_OK;
}

extern "C" size_t tq_gemm_fp8_workspace_bytes(const tq_desc* d, int M) {
  if (check_linear_desc(d) != TQ_OK || M < 1) return 0;
  return gemm_fp8_workspace_bytes(d, M);
}

extern "C" tq_status tq_gemm_fp8(const tq_desc* d, const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                                 int M, uint16_t* y, void* workspace, size_t workspace_bytes, void* stream) {
  tq_status st = check_linear_desc(d);
  if (st != TQ_OK) return st;
  if (M < 1) return TQ_ERR_INVALID_ARG;
  if (static_cast<long long>(d->N) * (d->K / 16) >= (1ll << 31)) return TQ_ERR_UNSUPPORTED;  // decode index range
  if ((st = check_ptrs(codes, scales, x, y, workspace)) != TQ_OK) return st;
  if (workspace_bytes < tq_gemm_fp8_workspace_bytes(d, M)) return TQ_ERR_WORKSPACE;
  if (!status_ptr()) return TQ_ERR_CUDA;
  if (const cudaError_t e = launch_gemm_fp8(d, codes, scales, x, M, y, workspace, static_cast<cudaStream_t>(stream));
      e != cudaSuccess)
    return cuda_fail(e);
  return TQ_OK;
}

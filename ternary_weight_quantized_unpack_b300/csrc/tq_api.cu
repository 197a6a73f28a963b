// libtq host entry points that do not launch compute: sizes, status, version.
#include <cstring>

#include "tq_internal.cuh"
#include "tq_kernels.cuh"

namespace tq {

__device__ int g_status = 0;

namespace {
constexpr int kMaxDevices = 64;
int* g_status_addr[kMaxDevices] = {nullptr};
thread_local int g_last_cuda = 0;
}  // namespace

tq_status cuda_fail(cudaError_t e) {
  g_last_cuda = static_cast<int>(e);
  (void)cudaGetLastError();
  return TQ_ERR_CUDA;
}

// Address of this device's status word; looked up once per device (current device at call time).
int* status_ptr() {
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidDevice);
    return nullptr;
  }
  if (!g_status_addr[dev]) {
    void* p = nullptr;
    const cudaError_t es = cudaGetSymbolAddress(&p, g_status);
    if (es != cudaSuccess) {
      cuda_fail(es);
      return nullptr;
    }
    g_status_addr[dev] = static_cast<int*>(p);
  }
  return g_status_addr[dev];
}

namespace {
tq_status check_desc_rules(const tq_desc* d, bool allow_3bit) {
  if (!d || d->N < 1 || d->K < 1) return TQ_ERR_INVALID_ARG;
  if (d->packing == TQ_PACK_3BIT && !allow_3bit) return TQ_ERR_UNSUPPORTED;
  if (d->packing != TQ_PACK_B3 && d->packing != TQ_PACK_2BIT && d->packing != TQ_PACK_3BIT) return TQ_ERR_INVALID_ARG;
  if (d->group != 64 && d->group != 128) return TQ_ERR_UNSUPPORTED;
  if (d->fwht_block != 0 && d->fwht_block != kFwhtBlock) return TQ_ERR_UNSUPPORTED;
  if (d->K % kFwhtBlock != 0) return TQ_ERR_UNSUPPORTED;
  if (d->flags & ~TQ_STATIC_WEIGHTS) return TQ_ERR_INVALID_ARG;
  return TQ_OK;
}
}  // namespace

tq_status check_linear_desc(const tq_desc* d) { return check_desc_rules(d, false); }
tq_status check_gemv_desc(const tq_desc* d) { return check_desc_rules(d, true); }

}  // namespace tq

using namespace tq;

static bool desc_ok(const tq_desc* d) {
  return d && d->N >= 1 && d->K >= 1 &&
         (d->packing == TQ_PACK_B3 || d->packing == TQ_PACK_2BIT || d->packing == TQ_PACK_3BIT);
}

extern "C" size_t tq_row_pitch_words(const tq_desc* d) {
  return desc_ok(d) ? static_cast<size_t>(pitch_words(d->K, d->packing)) : 0;
}

extern "C" size_t tq_packed_bytes(const tq_desc* d) {
  return desc_ok(d) ? static_cast<size_t>(d->N) * pitch_words(d->K, d->packing) * 4 : 0;
}

extern "C" size_t tq_scale_bytes(const tq_desc* d) {
  if (!desc_ok(d) || d->group < 1) return 0;
  return static_cast<size_t>(d->N) * groups_of(d->K, d->group) * 2;
}

extern "C" tq_status tq_device_status(int32_t* out) {
  if (!out) return TQ_ERR_INVALID_ARG;
  int* p = status_ptr();
  if (!p) return TQ_ERR_CUDA;
  int v = 0;
  if (const cudaError_t e = cudaDeviceSynchronize(); e != cudaSuccess) return cuda_fail(e);
  if (const cudaError_t e = cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost); e != cudaSuccess) return cuda_fail(e);
  const int zero = 0;
  if (const cudaError_t e = cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice); e != cudaSuccess) return cuda_fail(e);
  *out = v;
  return TQ_OK;
}

extern "C" const char* tq_status_str(tq_status s) {
  switch (s) {
    case TQ_OK: return "ok";
    case TQ_ERR_INVALID_ARG: return "invalid argument";
    case TQ_ERR_UNSUPPORTED: return "unsupported shape or option";
    case TQ_ERR_MISALIGNED: return "misaligned pointer";
    case TQ_ERR_INVALID_CODE: return "invalid packed code or trit";
    case TQ_ERR_CUDA: return "CUDA error";
    case TQ_ERR_TIMEOUT: return "bounded device wait timed out";
    case TQ_ERR_WORKSPACE: return "workspace too small";
    case TQ_ERR_RANGE: return "transformed activation outside FP16 range";
  }
  return "unknown status";
}

extern "C" int tq_version(void) { return 1; }

extern "C" int tq_last_cuda_error(void) {
  const int e = g_last_cuda;
  g_last_cuda = 0;
  return e;
}

// Block Walsh-Hadamard transform of activations.
//
// The weights were rotated by a Hadamard transform before ternarisation; inference applies the
// matching fast transform to the activations, O(n log n) per block ("27B 大模型塞进 5.9GB：三值量化，
// 凭什么「不崩」？", section 二 ①).  Sylvester (natural) order, orthonormal scaling 1/sqrt(128), block
// 128 along K.
//
// A warp takes kBlocksPerWarp consecutive 128-blocks of the flattened [rows][K] array (rows are
// contiguous), all its loads issued first: each lane loads 4 consecutive values of a block (one
// 8-byte load of bf16), two butterfly stages run in registers and five across lanes with shuffles;
// no shared memory.
#include "tq_internal.cuh"
#include "tq_kernels.cuh"

namespace tq {

constexpr float kInvSqrt128 = 0.08838834764831845f;

template <typename In>
__device__ __forceinline__ void load4(const In* p, float (&v)[4]);

template <>
__device__ __forceinline__ void load4<uint16_t>(const uint16_t* p, float (&v)[4]) {
  const uint2 raw = *reinterpret_cast<const uint2*>(p);
  v[0] = bf16_bits_to_float(static_cast<uint16_t>(raw.x & 0xffffu));
  v[1] = bf16_bits_to_float(static_cast<uint16_t>(raw.x >> 16));
  v[2] = bf16_bits_to_float(static_cast<uint16_t>(raw.y & 0xffffu));
  v[3] = bf16_bits_to_float(static_cast<uint16_t>(raw.y >> 16));
}

template <>
__device__ __forceinline__ void load4<float>(const float* p, float (&v)[4]) {
  const float4 raw = *reinterpret_cast<const float4*>(p);
  v[0] = raw.x; v[1] = raw.y; v[2] = raw.z; v[3] = raw.w;
}

constexpr int kBlocksPerWarp = 4;

template <typename In>
__global__ void fwht_kernel(const In* __restrict__ x, void* __restrict__ out, int out_fp16, int rows, int K,
                            int apply, int* status) {
  const int warps_per_block = blockDim.x >> 5;
  const long long wid = static_cast<long long>(blockIdx.x) * warps_per_block + (threadIdx.x >> 5);
  const long long nblk = static_cast<long long>(rows) * (K / kFwhtBlock);
  const long long b0 = wid * kBlocksPerWarp;
  if (b0 >= nblk) return;  // whole warp exits together
  const int lane = threadIdx.x & 31;
  float v[kBlocksPerWarp][4];
#pragma unroll
  for (int i = 0; i < kBlocksPerWarp; ++i)
    if (b0 + i < nblk) load4<In>(x + static_cast<size_t>(b0 + i) * kFwhtBlock + 4 * lane, v[i]);
#pragma unroll
  for (int i = 0; i < kBlocksPerWarp; ++i) {
    if (b0 + i >= nblk) break;
    const size_t base = static_cast<size_t>(b0 + i) * kFwhtBlock + 4 * lane;
    if (apply) {
      fwht128_warp(v[i]);
#pragma unroll
      for (int j = 0; j < 4; ++j) v[i][j] *= kInvSqrt128;
    }
    if (out_fp16) {
      __half h[4];
      bool overflow = false;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        h[j] = __float2half_rn(v[i][j]);
        overflow |= __hisinf(h[j]) != 0;
      }
      if (overflow) record_error(status, TQ_ERR_RANGE);
      uint2 packed;
      packed.x = static_cast<uint32_t>(__half_as_ushort(h[0])) | (static_cast<uint32_t>(__half_as_ushort(h[1])) << 16);
      packed.y = static_cast<uint32_t>(__half_as_ushort(h[2])) | (static_cast<uint32_t>(__half_as_ushort(h[3])) << 16);
      *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + base) = packed;
    } else {
      *reinterpret_cast<float4*>(static_cast<float*>(out) + base) =
          make_float4(v[i][0], v[i][1], v[i][2], v[i][3]);
    }
  }
}

cudaError_t launch_fwht_bf16(const uint16_t* x, void* out, int out_fp16, int rows, int K, int apply,
                             cudaStream_t s) {
  const long long warps = (static_cast<long long>(rows) * (K / kFwhtBlock) + kBlocksPerWarp - 1) / kBlocksPerWarp;
  const int threads = 256;
  const unsigned blocks = static_cast<unsigned>((warps * 32 + threads - 1) / threads);
  fwht_kernel<uint16_t><<<blocks, threads, 0, s>>>(x, out, out_fp16, rows, K, apply, status_ptr());
  return cudaPeekAtLastError();
}

cudaError_t launch_fwht_f32(const float* x, float* out, int rows, int K, cudaStream_t s) {
  const long long warps = (static_cast<long long>(rows) * (K / kFwhtBlock) + kBlocksPerWarp - 1) / kBlocksPerWarp;
  const int threads = 256;
  const unsigned blocks = static_cast<unsigned>((warps * 32 + threads - 1) / threads);
  fwht_kernel<float><<<blocks, threads, 0, s>>>(x, out, 0, rows, K, 1, status_ptr());
  return cudaPeekAtLastError();
}

}  // namespace tq

using namespace tq;

extern "C" tq_status tq_fwht(const uint16_t* x, void* out, int out_fp16, int rows, int K, int block, void* stream) {
  if (!x || !out || rows < 1 || K < 1) return TQ_ERR_INVALID_ARG;
  if (block != kFwhtBlock || K % kFwhtBlock != 0) return TQ_ERR_UNSUPPORTED;
  if (!aligned(x, 16) || !aligned(out, 16)) return TQ_ERR_MISALIGNED;
  if (!status_ptr()) return TQ_ERR_CUDA;
  const cudaError_t e = launch_fwht_bf16(x, out, out_fp16 ? 1 : 0, rows, K, 1, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return TQ_OK;
}

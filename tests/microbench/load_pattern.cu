// Code-load patterns of the decode kernels, in isolation: one launch reads a 17408 x 256-word matrix
// (the 17408 x 5120 base-3 gate projection, 17.8 MB) with no decode work; 24 copies (> L2) are
// cycled so every launch reads from HBM.  Time per launch includes the launch itself.
//   coalesced     : grid-stride 16-byte loads over the flat array
//   column 16 B   : base-3 decode layout, a lane reads 16 bytes of each of its 2 rows per step
//   column 32 B   : the same with 32-byte loads (two steps per load)
//   row lines     : 8 lanes read one row's 128 bytes per load
//   TMA tile      : one 64-row x 128-byte tile per warp by cp.async.bulk.tensor (128-byte swizzle)
//   2-bit 32/64   : 2-bit decode layout (16-row slab, lanes of a quad on adjacent words), 4- or 8-byte loads
// Build and run (one GPU; needs libcuda for the tensor map):
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 -o /tmp/load_pattern load_pattern.cu -lcuda && /tmp/load_pattern
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <cstdio>

#define CK(x)                                                                  \
  do {                                                                         \
    cudaError_t e_ = (x);                                                      \
    if (e_ != cudaSuccess) {                                                   \
      printf("CUDA error %s at line %d\n", cudaGetErrorString(e_), __LINE__); \
      return 1;                                                                \
    }                                                                          \
  } while (0)

constexpr int N = 17408, P = 256, kCopies = 24;

__global__ void coalesced(const uint4* __restrict__ p, size_t n16, uint32_t* out) {
  uint32_t acc = 0;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n16;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const uint4 v = __ldg(p + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  if (acc == 0x9e3779b9u) out[threadIdx.x] = acc;
}
// warp -> (64-row slab, unit of 32 words); lane -> rows lane, lane + 32
template <bool V8>
__global__ void column(const uint32_t* __restrict__ codes, uint32_t* out) {
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int nw = (gridDim.x * blockDim.x) >> 5, nunit = P / 32;
  uint32_t acc = 0;
  for (int wu = gw; wu < (N / 64) * nunit; wu += nw) {
    const int slab = wu / nunit, u = wu % nunit;
    const uint32_t* r0 = codes + static_cast<size_t>(slab * 64 + lane) * P + u * 32;
    const uint32_t* r1 = r0 + static_cast<size_t>(32) * P;
    if (V8) {
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        uint32_t a[8], b[8];
        asm volatile("ld.global.nc.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7])
                     : "l"(r0 + 8 * s));
        asm volatile("ld.global.nc.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7])
                     : "l"(r1 + 8 * s));
#pragma unroll
        for (int i = 0; i < 8; ++i) acc ^= a[i] ^ b[i];
      }
    } else {
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint4 a = __ldg(reinterpret_cast<const uint4*>(r0) + s), b = __ldg(reinterpret_cast<const uint4*>(r1) + s);
        acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w;
      }
    }
  }
  if (acc == 0x9e3779b9u) out[threadIdx.x] = acc;
}
__global__ void row_lines(const uint32_t* __restrict__ codes, uint32_t* out) {
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int nw = (gridDim.x * blockDim.x) >> 5, nunit = P / 32;
  uint32_t acc = 0;
  for (int wu = gw; wu < (N / 64) * nunit; wu += nw) {
    const int slab = wu / nunit, u = wu % nunit;
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const int row = slab * 64 + r * 4 + (lane >> 3);
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(codes + static_cast<size_t>(row) * P + u * 32) + (lane & 7));
      acc ^= a.x ^ a.y ^ a.z ^ a.w;
    }
  }
  if (acc == 0x9e3779b9u) out[threadIdx.x] = acc;
}
// 2-bit layout over the same bytes viewed as rows of 320 words: warp = 16-row slab x 32 words
template <int W>
__global__ void two_bit(const uint32_t* __restrict__ codes, int rows, uint32_t* out) {
  constexpr int P2 = 320;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const int nw = (gridDim.x * blockDim.x) >> 5, nunit = P2 / 32;
  uint32_t acc = 0;
  for (int wu = gw; wu < (rows / 16) * nunit; wu += nw) {
    const int slab = wu / nunit, u = wu % nunit;
    const uint32_t* r0 = codes + static_cast<size_t>(slab * 16 + g) * P2 + u * 32 + 2 * q;
    const uint32_t* r8 = r0 + static_cast<size_t>(8) * P2;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (W == 1) {
        acc ^= __ldg(r0 + 8 * j) ^ __ldg(r0 + 8 * j + 1) ^ __ldg(r8 + 8 * j) ^ __ldg(r8 + 8 * j + 1);
      } else {
        const uint2 a = __ldg(reinterpret_cast<const uint2*>(r0 + 8 * j)), b = __ldg(reinterpret_cast<const uint2*>(r8 + 8 * j));
        acc ^= a.x ^ a.y ^ b.x ^ b.y;
      }
    }
  }
  if (acc == 0x9e3779b9u) out[threadIdx.x] = acc;
}

__device__ __forceinline__ uint32_t sa(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }
__global__ void __launch_bounds__(512) tma_tile(const __grid_constant__ CUtensorMap tm, uint32_t* out, int* err) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint64_t bar[16];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gw = blockIdx.x * (blockDim.x >> 5) + w, nw = (gridDim.x * blockDim.x) >> 5, nunit = P / 32;
  uint8_t* tile = sm + w * 8192;
  if (lane == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sa(&bar[w])));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  uint32_t acc = 0, ph = 0;
  for (int wu = gw; wu < (N / 64) * nunit; wu += nw) {
    const int slab = wu / nunit, u = wu % nunit;
    if (lane == 0) {
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], 8192;" ::"r"(sa(&bar[w])) : "memory");
      asm volatile(
          "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
              sa(tile)),
          "l"(&tm), "r"(u * 32), "r"(slab * 64), "r"(sa(&bar[w]))
          : "memory");
    }
    bool ok = false;
    for (int i = 0; i < (1 << 22) && !ok; ++i) {
      uint32_t r;
      asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                   : "=r"(r)
                   : "r"(sa(&bar[w])), "r"(ph)
                   : "memory");
      ok = r != 0;
    }
    if (!ok) {
      if (lane == 0) atomicAdd(err, 1);
      return;
    }
    ph ^= 1;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const uint4 a = reinterpret_cast<const uint4*>(tile + lane * 128)[s ^ (lane & 7)];
      const uint4 b = reinterpret_cast<const uint4*>(tile + (lane + 32) * 128)[s ^ (lane & 7)];
      acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w;
    }
    __syncwarp();
  }
  if (acc == 0x9e3779b9u) out[threadIdx.x] = acc;
}

int main() {
  const size_t bytes = static_cast<size_t>(N) * P * 4;
  uint32_t* buf;
  uint32_t* out;
  int* err;
  CK(cudaMalloc(&buf, bytes * kCopies));
  CK(cudaMalloc(&out, 4096));
  CK(cudaMalloc(&err, 4));
  CK(cudaMemset(buf, 0x5a, bytes * kCopies));
  CK(cudaMemset(err, 0, 4));
  static CUtensorMap tms[kCopies];
  for (int c = 0; c < kCopies; ++c) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(P), static_cast<cuuint64_t>(N)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(P) * 4};
    cuuint32_t box[2] = {32, 64}, es[2] = {1, 1};
    if (cuTensorMapEncodeTiled(&tms[c], CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, buf + static_cast<size_t>(c) * N * P, dims,
                               strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      printf("tensor map encoding failed\n");
      return 1;
    }
  }
  CK(cudaFuncSetAttribute(tma_tile, cudaFuncAttributeMaxDynamicSharedMemorySize, 16 * 8192));
  cudaEvent_t e0, e1;
  CK(cudaEventCreate(&e0));
  CK(cudaEventCreate(&e1));
  auto run = [&](const char* name, auto launch) -> int {
    for (int c = 0; c < kCopies; ++c) launch(c);
    CK(cudaEventRecord(e0));
    for (int it = 0; it < 3; ++it)
      for (int c = 0; c < kCopies; ++c) launch(c);
    CK(cudaEventRecord(e1));
    CK(cudaEventSynchronize(e1));
    float ms = 0.f;
    CK(cudaEventElapsedTime(&ms, e0, e1));
    const double us = ms * 1e3 / (3 * kCopies);
    printf("%-26s %7.2f us per launch  %7.0f GB/s\n", name, us, bytes / us / 1e3);
    return 0;
  };
  auto at = [&](int c) { return buf + static_cast<size_t>(c) * N * P; };
  const int rows2 = static_cast<int>(bytes / 4 / 320) / 16 * 16;
  if (run("coalesced, 592 x 512", [&](int c) { coalesced<<<592, 512>>>(reinterpret_cast<const uint4*>(at(c)), bytes / 16, out); }) ||
      run("column 16 B, 136 x 512", [&](int c) { column<false><<<136, 512>>>(at(c), out); }) ||
      run("column 32 B, 136 x 512", [&](int c) { column<true><<<136, 512>>>(at(c), out); }) ||
      run("row lines, 136 x 512", [&](int c) { row_lines<<<136, 512>>>(at(c), out); }) ||
      run("TMA tile, 136 x 512", [&](int c) { tma_tile<<<136, 512, 16 * 8192>>>(tms[c], out, err); }) ||
      run("2-bit 4 B, 136 x 512", [&](int c) { two_bit<1><<<136, 512>>>(at(c), rows2, out); }) ||
      run("2-bit 8 B, 136 x 512", [&](int c) { two_bit<2><<<136, 512>>>(at(c), rows2, out); }))
    return 1;
  CK(cudaGetLastError());
  CK(cudaDeviceSynchronize());
  int e = 0;
  CK(cudaMemcpy(&e, err, 4, cudaMemcpyDeviceToHost));
  if (e) {
    printf("TMA waits that timed out: %d\n", e);
    return 1;
  }
  return 0;
}

// Tensor-core instruction options for the 2-bit decode GEMV, in isolation:
//   accuracy of mma.sync m16n8k32 e4m3 x e4m3 -> f32 with A = trit digits d * 2^-9 (e4m3 subnormals)
//   against an exact fp64 sum (worst |D - exact| / (|C| + sum |A B|));
//   issue rate of mma.sync m16n8k32 e4m3 (512 weights per instruction) and m16n8k16 f16 (256) with
//   8 independent accumulators per warp, in weights per cycle per SM.
// Build and run (one GPU):
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 -o /tmp/mma_fp8_vs_f16 mma_fp8_vs_f16.cu && /tmp/mma_fp8_vs_f16
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cstdio>
#include <cstdint>
#include <cstdlib>
#include <cmath>
#include <vector>
#define CK(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { printf("CUDA %s line %d\n", cudaGetErrorString(e_), __LINE__); return 1; } } while (0)

__device__ __forceinline__ void mma_f8(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
               : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3]) : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
               : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3]) : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// one MMA per warp on given fragments: A [16][32] bytes, B [32][8] bytes (col), C [16][8] f32 -> D
__global__ void one_f8(const uint8_t* A, const uint8_t* B, const float* C, float* D, int chain) {
  const int lane = threadIdx.x, g = lane >> 2, q = lane & 3;
  auto a4 = [&](int r, int k0) { uint32_t v = 0; for (int i = 0; i < 4; ++i) v |= uint32_t(A[r * 32 + k0 + i]) << (8 * i); return v; };
  auto b4 = [&](int k0, int n) { uint32_t v = 0; for (int i = 0; i < 4; ++i) v |= uint32_t(B[n * 32 + k0 + i]) << (8 * i); return v; };
  uint32_t a0 = a4(g, 4 * q), a1 = a4(g + 8, 4 * q), a2 = a4(g, 16 + 4 * q), a3 = a4(g + 8, 16 + 4 * q);
  uint32_t b0 = b4(4 * q, g), b1 = b4(16 + 4 * q, g);
  float c[4] = {C[g * 8 + 2 * q], C[g * 8 + 2 * q + 1], C[(g + 8) * 8 + 2 * q], C[(g + 8) * 8 + 2 * q + 1]};
  for (int i = 0; i < chain; ++i) mma_f8(c, a0, a1, a2, a3, b0, b1);
  D[g * 8 + 2 * q] = c[0]; D[g * 8 + 2 * q + 1] = c[1]; D[(g + 8) * 8 + 2 * q] = c[2]; D[(g + 8) * 8 + 2 * q + 1] = c[3];
}

template <int KIND>
__global__ void __launch_bounds__(512) thr(int iters, float* out, unsigned long long* cyc) {
  const int lane = threadIdx.x & 31;
  uint32_t a0 = lane * 0x01010101u & 0x03030303u, a1 = a0 ^ 0x01000100u, a2 = a0 ^ 0x00010001u, a3 = a0 ^ 0x02000200u;
  uint32_t b0 = 0x38383838u ^ lane, b1 = 0x30303030u ^ lane;
  if (KIND == 1) { a0 &= 0x03ff03ffu; a1 &= 0x03ff03ffu; a2 &= 0x03ff03ffu; a3 &= 0x03ff03ffu; b0 = 0x3c003c00u ^ lane; b1 = 0x38003800u ^ lane; }
  float c[8][4] = {};
  __syncwarp();
  const long long t0 = clock64();
#pragma unroll 1
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (KIND == 0) mma_f8(c[j], a0 ^ j, a1, a2, a3, b0, b1); else mma_f16(c[j], a0 ^ j, a1, a2, a3, b0, b1);
    }
  }
  const long long t1 = clock64();
  float s = 0; for (int j = 0; j < 8; ++j) s += c[j][0] + c[j][1] + c[j][2] + c[j][3];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if (lane == 0) atomicAdd(cyc, (unsigned long long)(t1 - t0));
}

static double e4m3_val(uint8_t b) {
  int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
  double v = e == 0 ? m * std::ldexp(1.0, -9) : (1 + m / 8.0) * std::ldexp(1.0, e - 7);
  if (e == 15 && m == 7) v = NAN;
  return s ? -v : v;
}

int main() {
  // accuracy
  std::vector<uint8_t> A(16 * 32), B(8 * 32);
  std::vector<float> C(128), D(128);
  uint8_t *dA, *dB; float *dC, *dD;
  CK(cudaMalloc(&dA, 512)); CK(cudaMalloc(&dB, 256)); CK(cudaMalloc(&dC, 512)); CK(cudaMalloc(&dD, 512));
  srand(1);
  double worst = 0;
  for (int trial = 0; trial < 2000; ++trial) {
    for (auto& a : A) a = rand() % 3;  // d * 2^-9
    for (auto& b : B) { int e = 1 + rand() % 14, m = rand() % 8, s = rand() & 1; b = uint8_t((s << 7) | (e << 3) | m); }
    const int mode = trial % 4;
    for (int i = 0; i < 128; ++i) C[i] = mode == 0 ? 0.f : (float)((rand() / (double)RAND_MAX - 0.5) * std::ldexp(1.0, (mode == 1 ? -6 : mode == 2 ? 0 : 4)));
    CK(cudaMemcpy(dA, A.data(), 512, cudaMemcpyHostToDevice)); CK(cudaMemcpy(dB, B.data(), 256, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dC, C.data(), 512, cudaMemcpyHostToDevice));
    one_f8<<<1, 32>>>(dA, dB, dC, dD, 1);
    CK(cudaMemcpy(D.data(), dD, 512, cudaMemcpyDeviceToHost));
    for (int m = 0; m < 16; ++m) for (int n = 0; n < 8; ++n) {
      double ex = C[m * 8 + n], ab = std::fabs(C[m * 8 + n]);
      for (int k = 0; k < 32; ++k) { double p = A[m * 32 + k] * std::ldexp(1.0, -9) * e4m3_val(B[n * 32 + k]); ex += p; ab += std::fabs(p); }
      const double err = std::fabs(D[m * 8 + n] - ex) / ab;
      if (err > worst) worst = err;
    }
  }
  printf("e4m3 m16n8k32 accuracy: worst |D-exact| / (|C| + sum|AB|) = %.3e (= %.2f x 2^-23)\n", worst, worst / std::ldexp(1.0, -23));
  // throughput
  int sms = 0; CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
  float* out; unsigned long long* cyc;
  CK(cudaMalloc(&out, sms * 1024 * 4)); CK(cudaMalloc(&cyc, 8));
  for (int kind = 0; kind < 2; ++kind) for (int w : {4, 8, 16}) {
    const int iters = 1024;
    auto k = kind == 0 ? thr<0> : thr<1>;
    k<<<sms, 32 * w>>>(iters, out, cyc);
    CK(cudaMemset(cyc, 0, 8));
    k<<<sms, 32 * w>>>(iters, out, cyc);
    CK(cudaDeviceSynchronize());
    unsigned long long c = 0; CK(cudaMemcpy(&c, cyc, 8, cudaMemcpyDeviceToHost));
    const double per_warp = double(c) / (double(sms) * w);  // cycles for iters*8 MMAs
    const double mma_per_clk_sm = iters * 8.0 * w / per_warp;
    printf("%s warps/SM %2d: %.3f MMA/clk/SM -> %.1f weights/clk/SM\n", kind == 0 ? "e4m3 m16n8k32" : "f16 m16n8k16 ", w,
           mma_per_clk_sm, mma_per_clk_sm * (kind == 0 ? 512 : 256));
  }
  return 0;
}

// Decode inner loops in isolation: the code words, the base-3 chunk table and x^ sit in shared memory,
// so the loop's own cost is timed (clock64), without global memory, prologue or reduction.
//   base-3 "column" step: 4 words of 2 rows per thread -> 4 table words each -> 20 MMA operands ->
//           5 mma.sync m16n8k16 per word pair;
//   2-bit "shared-row" group: 2 words of 2 rows per thread -> 16 operands -> 8 mma.sync.
// Variants separate the cost of the tensor-core instruction from the decode around it.
// Build and run (one GPU):
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 -o /tmp/decode_loop decode_loop.cu && /tmp/decode_loop
#include <cuda_fp16.h>
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

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// base-3 word -> four chunk-table words (two exact reciprocal multiplies, then base 243)
template <bool TABLE>
__device__ __forceinline__ void chunks(uint32_t w, const uint32_t* lutA, const uint32_t* lutB, uint32_t (&L)[4]) {
  const uint32_t v = min(w, 3486784400u);
  const uint32_t hi = __umulhi(v + 1u, 2383401723u) >> 15;
  const uint32_t lo = v - hi * 59049u;
  const uint32_t bl = __umulhi(lo, 17675008u), al = lo - bl * 243u;
  const uint32_t bh = __umulhi(hi, 17675008u), ah = hi - bh * 243u;
  if (!TABLE) {
    L[0] = al * 0x10001u, L[1] = bl * 0x10001u, L[2] = ah * 0x10001u, L[3] = bh * 0x10001u;
    return;
  }
  L[0] = lutA[al * 32], L[1] = lutB[bl * 32], L[2] = lutA[ah * 32], L[3] = lutB[bh * 32];
}
__device__ __forceinline__ uint32_t operand(const uint32_t (&L)[4], int j) {
  const uint32_t a = j < 5 ? L[0] : L[2], b = j < 5 ? L[1] : L[3];
  const int f = j % 5;
  const uint32_t m = 0x00030003u << (2 * f);
  return f < 2 ? (a & m) : f == 2 ? ((a | b) & m) : (b & m);
}

constexpr int kWords = 2 * 243 * 32 + 8192 + 4096 + 1024;  // table, codes, x^, group data

// mode 0: full step, 4 accumulator chains; 1: full step, 1 chain; 2: chunk split without the table;
// 3: the 5 MMAs per word pair alone (fixed operands)
template <int MODE>
__global__ void b3_step(int iters, float* out, unsigned long long* cyc) {
  extern __shared__ uint32_t sm[];
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  for (int i = threadIdx.x; i < kWords; i += blockDim.x) sm[i] = (i * 2654435761u) & 0x0fff0fffu;
  __syncthreads();
  const uint32_t* lutA = sm + lane;
  const uint32_t* lutB = lutA + 243 * 32;
  const uint32_t* codes = sm + 2 * 243 * 32 + ((threadIdx.x >> 5) & 15) * 512;
  const uint32_t* xh = sm + 2 * 243 * 32 + 8192;
  const bool bsup = (g & 3) == q;
  constexpr int C = MODE == 1 ? 1 : 4;
  float cc[C][4] = {};
  uint4 bp = make_uint4(0, 0, 0, 0);
  __syncwarp();
  const long long t0 = clock64();
#pragma unroll 1
  for (int it = 0; it < iters; ++it) {
    const int st = it & 3;
    const uint4 c1 = reinterpret_cast<const uint4*>(codes)[st * 32 + lane];  // consecutive lanes, no conflict
    const uint4 c2 = reinterpret_cast<const uint4*>(codes)[(st ^ 2) * 32 + lane];
    const uint32_t wa[4] = {c1.x, c1.y, c1.z, c1.w}, wb[4] = {c2.x, c2.y, c2.z, c2.w};
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      uint32_t La[4], Lb[4];
      if (MODE == 3) {
        La[0] = La[1] = La[2] = La[3] = wa[wi] & 0x03ff03ffu;
        Lb[0] = Lb[1] = Lb[2] = Lb[3] = wb[wi] & 0x03ff03ffu;
      } else {
        chunks<MODE != 2>(wa[wi], lutA, lutB, La);
        chunks<MODE != 2>(wb[wi], lutA, lutB, Lb);
      }
#pragma unroll
      for (int mj = 0; mj < 5; ++mj) {
        const int mm = wi * 5 + mj;
        if ((mm & 1) == 0 && bsup) bp = reinterpret_cast<const uint4*>(xh)[(it * 10 + (mm >> 1)) & 1023];
        uint32_t a0, a1, a2, a3;
        if (MODE == 3) {
          a0 = La[0], a1 = Lb[0], a2 = La[1], a3 = Lb[1];
        } else {
          a0 = operand(La, 2 * mj), a2 = operand(La, 2 * mj + 1), a1 = operand(Lb, 2 * mj), a3 = operand(Lb, 2 * mj + 1);
        }
        mma16816(cc[mm % C], a0, a1, a2, a3, (mm & 1) ? bp.z : bp.x, (mm & 1) ? bp.w : bp.y);
      }
    }
  }
  const long long t1 = clock64();
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < C; ++c) s += cc[c][0] + cc[c][1] + cc[c][2] + cc[c][3];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if (lane == 0) atomicAdd(cyc, static_cast<unsigned long long>(t1 - t0));
}

// mode 0: full group, 1 chain; 1: full group, 4 chains; 2: the 8 MMAs per group alone (fixed operands)
template <int MODE>
__global__ void b2_group(int iters, float* out, unsigned long long* cyc) {
  extern __shared__ uint32_t sm[];
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  for (int i = threadIdx.x; i < kWords; i += blockDim.x) sm[i] = (i * 2654435761u) & 0x0fff0fffu;
  __syncthreads();
  const uint32_t* codes = sm + ((threadIdx.x >> 5) & 15) * 512;  // 16 rows x 32 words, 128-byte swizzle
  const uint32_t* xh = sm + 8192;
  const float* V = reinterpret_cast<const float*>(sm + 8192 + 4096);
  constexpr int C = MODE == 0 ? 1 : 4;
  float acc[4] = {}, cc[C][4];
  __syncwarp();
  const long long t0 = clock64();
#pragma unroll 1
  for (int it = 0; it < iters; ++it) {
    const int j = it & 3;
    const uint32_t w0 = codes[g * 32 + (((2 * j) ^ g) & 7) * 4 + q];
    const uint32_t w1 = codes[g * 32 + (((2 * j + 1) ^ g) & 7) * 4 + q];
    const uint32_t w80 = codes[(g + 8) * 32 + (((2 * j) ^ g) & 7) * 4 + q];
    const uint32_t w81 = codes[(g + 8) * 32 + (((2 * j + 1) ^ g) & 7) * 4 + q];
    const float2 v = *reinterpret_cast<const float2*>(V + ((j * 8 + 2 * q) & 1023));
#pragma unroll
    for (int c = 0; c < C; ++c) {
      cc[c][0] = c ? 0.f : v.x, cc[c][1] = c ? 0.f : v.y, cc[c][2] = c ? 0.f : v.x, cc[c][3] = c ? 0.f : v.y;
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint32_t w = u ? w1 : w0, w8 = u ? w81 : w80, w2 = w >> 10, w82 = w8 >> 10;
      uint32_t pr[8], pr8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        pr[k] = k < 5 ? (w & (0x00030003u << (2 * k))) : (w2 & (0x00030003u << (2 * (k - 5))));
        pr8[k] = k < 5 ? (w8 & (0x00030003u << (2 * k))) : (w82 & (0x00030003u << (2 * (k - 5))));
      }
      uint4 bp;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        if ((jj & 1) == 0) bp = reinterpret_cast<const uint4*>(xh)[((j * 4 + u * 2 + (jj >> 1)) * 32 + lane) & 1023];
        const uint32_t b0 = (jj & 1) ? bp.z : bp.x, b1 = (jj & 1) ? bp.w : bp.y;
        if (MODE == 2)
          mma16816(cc[(u * 4 + jj) % C], w & 0x03ff03ffu, w8 & 0x03ff03ffu, w2 & 0x03ff03ffu, w82 & 0x03ff03ffu, b0, b1);
        else
          mma16816(cc[(u * 4 + jj) % C], pr[2 * jj], pr8[2 * jj], pr[2 * jj + 1], pr8[2 * jj + 1], b0, b1);
      }
    }
    const float m = __half2float(*reinterpret_cast<const __half*>(V + ((j * 8 + g) & 1023)));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float s = cc[0][i];
#pragma unroll
      for (int c = 1; c < C; ++c) s += cc[c][i];
      acc[i] = fmaf(m, s, acc[i]);
    }
  }
  const long long t1 = clock64();
  out[blockIdx.x * blockDim.x + threadIdx.x] = acc[0] + acc[1] + acc[2] + acc[3];
  if (lane == 0) atomicAdd(cyc, static_cast<unsigned long long>(t1 - t0));
}

int main() {
  int sms = 0;
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
  float* out;
  unsigned long long* cyc;
  CK(cudaMalloc(&out, static_cast<size_t>(sms) * 1024 * 4));
  CK(cudaMalloc(&cyc, 8));
  const int smem = kWords * 4;
  // trits per unit of work: base-3 step = 32 lanes x 2 rows x 4 words x 20; 2-bit group = 16 rows x 128
  auto run = [&](auto kern, const char* name, int warps, double trits, const char* unit) -> int {
    CK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    const int iters = 512;
    kern<<<sms, 32 * warps, smem>>>(iters, out, cyc);
    CK(cudaMemset(cyc, 0, 8));
    kern<<<sms, 32 * warps, smem>>>(iters, out, cyc);
    CK(cudaDeviceSynchronize());
    unsigned long long c = 0;
    CK(cudaMemcpy(&c, cyc, 8, cudaMemcpyDeviceToHost));
    const double per = static_cast<double>(c) / (static_cast<double>(sms) * warps * iters);
    printf("%-34s warps/SM %2d: %7.1f cycles per %s per warp, %6.1f trits/cycle/SM\n", name, warps, per, unit,
           trits * warps / per);
    return 0;
  };
  for (int w : {1, 4, 16}) {
    if (run(b3_step<0>, "base-3 step, 4 chains", w, 5120, "step") ||
        run(b3_step<1>, "base-3 step, 1 chain", w, 5120, "step") ||
        run(b3_step<2>, "base-3 step, no table", w, 5120, "step") ||
        run(b3_step<3>, "base-3 step, MMAs only", w, 5120, "step"))
      return 1;
  }
  for (int w : {1, 4, 16, 32}) {
    if (run(b2_group<0>, "2-bit group, 1 chain", w, 2048, "group") ||
        run(b2_group<1>, "2-bit group, 4 chains", w, 2048, "group") ||
        run(b2_group<2>, "2-bit group, MMAs only", w, 2048, "group"))
      return 1;
  }
  return 0;
}

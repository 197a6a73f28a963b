// Straightforward CUDA-core kernels for the ternary contraction: a warp-per-row GEMV and a
// shared-memory tiled GEMM.  They decode the packed codes in registers (never writing decoded
// weights to global memory, cosmocat.dev "27B 大模型塞进 5.9GB", section 二 ③) and apply the group
// scale per trit.  They are the small-shape path and the baseline for the tensor-core kernels.
#include "tq_internal.cuh"
#include "tq_kernels.cuh"
#include "tq_simple.cuh"

namespace tq {

__constant__ uint32_t c_pow3[20] = {1u, 3u, 9u, 27u, 81u, 243u, 729u, 2187u, 6561u, 19683u, 59049u, 177147u,
                                    531441u, 1594323u, 4782969u, 14348907u, 43046721u, 129140163u, 387420489u,
                                    1162261467u};

namespace {

template <int PACKING, int MAXB>
__global__ void __launch_bounds__(256) gemv_simple_kernel(const uint32_t* __restrict__ codes,
                                                          const uint16_t* __restrict__ scales,
                                                          const float* __restrict__ xt, int N, int K, int P, int G,
                                                          int batch, float* __restrict__ y) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * (blockDim.x >> 5) + warp;
  if (n >= N) return;
  float acc[MAXB];
#pragma unroll
  for (int b = 0; b < MAXB; ++b) acc[b] = 0.f;
  row_dot_accumulate<PACKING, MAXB>(codes + static_cast<size_t>(n) * P, scales + static_cast<size_t>(n) * groups_of(K, G),
                                    xt, K, K, G, batch, lane, acc);
#pragma unroll
  for (int b = 0; b < MAXB; ++b) {
    const float v = warp_sum(acc[b]);
    if (lane == 0 && b < batch) y[static_cast<size_t>(b) * N + n] = v;
  }
}

template <int PACKING>
__global__ void __launch_bounds__(256) gemm_simple_kernel(const uint32_t* __restrict__ codes,
                                                          const uint16_t* __restrict__ scales,
                                                          const float* __restrict__ xt, int M, int N, int K, int P,
                                                          int G, uint16_t* __restrict__ y) {
  constexpr int PER = PACKING == TQ_PACK_B3 ? kB3Trits : kB2Trits;
  __shared__ float Ws[32][65];  // decoded s*t, [k][row]
  __shared__ float Xs[32][65];  // x~, [k][token]
  const int n0 = blockIdx.x * 64, m0 = blockIdx.y * 64;
  const int tid = threadIdx.x;
  const int tr = tid >> 4, tc = tid & 15;
  const int ng = groups_of(K, G);
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int k0 = 0; k0 < K; k0 += 32) {
    for (int e = tid; e < 64 * 32; e += 256) {
      const int r = e >> 5, kk = e & 31;
      const int n = n0 + r, k = k0 + kk;
      float w = 0.f;
      if (n < N && k < K) {
        const uint32_t v = codes[static_cast<size_t>(n) * P + k / PER];
        const int q = k % PER;
        int dgt = PACKING == TQ_PACK_B3 ? static_cast<int>((v / c_pow3[q]) % 3u) : static_cast<int>((v >> (2 * q)) & 3u);
        if (dgt == 3) dgt = 1;
        w = static_cast<float>(dgt - 1) * half_bits_to_float(scales[static_cast<size_t>(n) * ng + k / G]);
      }
      Ws[kk][r] = w;
    }
    for (int e = tid; e < 64 * 32; e += 256) {
      const int m = e >> 5, kk = e & 31;
      Xs[kk][m] = (m0 + m < M && k0 + kk < K) ? xt[static_cast<size_t>(m0 + m) * K + k0 + kk] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < 32; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = Ws[kk][tr * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Xs[kk][tc * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tr * 4 + i, m = m0 + tc * 4 + j;
      if (n < N && m < M) y[static_cast<size_t>(m) * N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[i][j]));
    }
}

}  // namespace

cudaError_t launch_gemv_simple(const tq_desc* d, const uint32_t* codes, const uint16_t* scales, const float* xt,
                               int batch, float* y, cudaStream_t s) {
  const int P = pitch_words(d->K, d->packing);
  const unsigned blocks = static_cast<unsigned>((d->N + 7) / 8);
#define TQ_GEMV_CASE(PK, MB)                                                                                  \
  gemv_simple_kernel<PK, MB><<<blocks, 256, 0, s>>>(codes, scales, xt, d->N, d->K, P, d->group, batch, y)
  if (d->packing == TQ_PACK_B3) {
    if (batch <= 1) TQ_GEMV_CASE(TQ_PACK_B3, 1);
    else if (batch <= 4) TQ_GEMV_CASE(TQ_PACK_B3, 4);
    else TQ_GEMV_CASE(TQ_PACK_B3, 16);
  } else {
    if (batch <= 1) TQ_GEMV_CASE(TQ_PACK_2BIT, 1);
    else if (batch <= 4) TQ_GEMV_CASE(TQ_PACK_2BIT, 4);
    else TQ_GEMV_CASE(TQ_PACK_2BIT, 16);
  }
#undef TQ_GEMV_CASE
  return cudaPeekAtLastError();
}

cudaError_t launch_gemm_simple(const tq_desc* d, const uint32_t* codes, const uint16_t* scales, const float* xt,
                               int M, uint16_t* y, cudaStream_t s) {
  const int P = pitch_words(d->K, d->packing);
  dim3 grid((d->N + 63) / 64, (M + 63) / 64);
  if (d->packing == TQ_PACK_B3)
    gemm_simple_kernel<TQ_PACK_B3><<<grid, 256, 0, s>>>(codes, scales, xt, M, d->N, d->K, P, d->group, y);
  else
    gemm_simple_kernel<TQ_PACK_2BIT><<<grid, 256, 0, s>>>(codes, scales, xt, M, d->N, d->K, P, d->group, y);
  return cudaPeekAtLastError();
}

}  // namespace tq

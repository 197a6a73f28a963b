// Offline quantizer: dense bf16 W [N][K] -> packed ternary codes + FP16 group scales.
//
// The steps are the ones "27B 大模型塞进 5.9GB：三值量化，凭什么「不崩」？" puts before the kernels:
// section 二 ① rotate the weights by a Hadamard transform before compressing them, section 二 ② give
// each group of 128 weights its own FP16 scale, section 一 keep three levels -1, 0, +1 of it.  The
// rounding rule is not on the pages; this library uses the absmean rule of BitNet b1.58: the scale is
// the mean |w'| of the group, and t is the level of {-1, 0, +1} nearest to w' / scale, a value exactly
// halfway between 0 and the scale going to 0.
//
// Arithmetic, chosen so that the result does not depend on the order of any sum:
//   u = H_128 w per 128-block (unnormalised Sylvester), in fp64: every u is a signed sum of 128 bf16
//       values, exact in fp64 when the magnitudes in the block span less than 2^38;
//   m = sum_{group} |u| / group, exact when they span less than 2^31;
//   S = fp16_rn(m * c) with c = 2^-3.5 rounded to fp64 (c = 1 without the transform);
//   t = sign(u) if |u| * c > S / 2 (each product rounded once in fp64), else 0.
// So any exact evaluation of these definitions - in particular a plain fp64 CPU one - gives the same
// trits and scales bit for bit.
//
// One CTA per row: its warps rotate and ternarize the row's 128-blocks (one block per warp at a time,
// 4 values per lane), keep the trits in shared memory, and then pack the row into code words
// (base-3: 20 trits per uint32; 2-bit: 16) written with coalesced stores.  Offline work: one pass over
// W (2 bytes per weight) plus the codes and scales written.
#include "tq_internal.cuh"

namespace tq {
namespace quant {

constexpr int kThreads = 256;
constexpr double kInvSqrt128 = 0.08838834764831845;  // 2^-3.5, rounded to fp64
constexpr int kMaxK = 196608;                         // the row's trits must fit in shared memory

template <int G>
__global__ void __launch_bounds__(kThreads) quantize_kernel(const uint16_t* __restrict__ w, uint32_t* __restrict__ codes,
                                                          uint16_t* __restrict__ scales, int K, int P, int packing,
                                                          int fwht, int* status) {
  extern __shared__ int8_t trit_row[];
  const int n = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nb = K / kFwhtBlock, ng = K / G;
  const uint16_t* wr = w + static_cast<size_t>(n) * K;
  const double c = fwht ? kInvSqrt128 : 1.0;
  bool bad = false;
  for (int b = warp; b < nb; b += kThreads / 32) {
    const int k0 = b * kFwhtBlock + 4 * lane;
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(wr + k0));
    double v[4] = {static_cast<double>(bf16_bits_to_float(static_cast<uint16_t>(raw.x & 0xffffu))),
                   static_cast<double>(bf16_bits_to_float(static_cast<uint16_t>(raw.x >> 16))),
                   static_cast<double>(bf16_bits_to_float(static_cast<uint16_t>(raw.y & 0xffffu))),
                   static_cast<double>(bf16_bits_to_float(static_cast<uint16_t>(raw.y >> 16)))};
    if (fwht) fwht128_warp(v);
    double a = (fabs(v[0]) + fabs(v[1])) + (fabs(v[2]) + fabs(v[3]));
    // sum over the lanes of the group: 32 lanes for G = 128, 16 for G = 64 (exact in fp64)
#pragma unroll
    for (int o = G / 8; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    const __half S = __double2half(a * (1.0 / G) * c);
    const float Sf = __half2float(S);
    if (!isfinite(a) || isinf(Sf)) bad = true;
    const double lim = static_cast<double>(Sf) * 0.5;
    char4 t;
    t.x = static_cast<signed char>(fabs(v[0]) * c > lim ? (v[0] > 0.0 ? 1 : -1) : 0);
    t.y = static_cast<signed char>(fabs(v[1]) * c > lim ? (v[1] > 0.0 ? 1 : -1) : 0);
    t.z = static_cast<signed char>(fabs(v[2]) * c > lim ? (v[2] > 0.0 ? 1 : -1) : 0);
    t.w = static_cast<signed char>(fabs(v[3]) * c > lim ? (v[3] > 0.0 ? 1 : -1) : 0);
    *reinterpret_cast<char4*>(trit_row + k0) = t;
    if ((lane & (G / 4 - 1)) == 0) scales[static_cast<size_t>(n) * ng + k0 / G] = __half_as_ushort(S);
  }
  if (bad) record_error(status, TQ_ERR_RANGE);
  __syncthreads();
  // pack: word j holds trits j * per .. j * per + per - 1 (t = 0 past K and in padding words)
  const int per = packing == TQ_PACK_B3 ? kB3Trits : kB2Trits;
  uint32_t* cr = codes + static_cast<size_t>(n) * P;
  for (int j = threadIdx.x; j < P; j += kThreads) {
    uint32_t v = 0;
    for (int i = per - 1; i >= 0; --i) {
      const int k = j * per + i;
      const uint32_t d = static_cast<uint32_t>((k < K ? trit_row[k] : 0) + 1);
      v = packing == TQ_PACK_B3 ? v * 3u + d : (v << 2) | d;
    }
    cr[j] = v;
  }
}

}  // namespace quant
}  // namespace tq

using namespace tq;

extern "C" tq_status tq_quantize(const tq_desc* d, const uint16_t* w, uint32_t* codes, uint16_t* scales,
                                 void* stream) {
  if (!d || !w || !codes || !scales) return TQ_ERR_INVALID_ARG;
  if (d->N < 1 || d->K < 1 || d->flags != 0) return TQ_ERR_INVALID_ARG;
  if (d->packing != TQ_PACK_B3 && d->packing != TQ_PACK_2BIT) return TQ_ERR_INVALID_ARG;
  if (d->group != 64 && d->group != 128) return TQ_ERR_UNSUPPORTED;
  if (d->fwht_block != 0 && d->fwht_block != kFwhtBlock) return TQ_ERR_UNSUPPORTED;
  if (d->K % kFwhtBlock != 0 || d->K > quant::kMaxK) return TQ_ERR_UNSUPPORTED;
  if (!aligned(w, 16) || !aligned(codes, 16) || !aligned(scales, 2)) return TQ_ERR_MISALIGNED;
  int* status = status_ptr();
  if (!status) return TQ_ERR_CUDA;
  const int P = pitch_words(d->K, d->packing);
  const size_t smem = static_cast<size_t>(d->K);
  auto kern = d->group == 128 ? quant::quantize_kernel<128> : quant::quantize_kernel<64>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_fail(e);
  kern<<<d->N, quant::kThreads, smem, static_cast<cudaStream_t>(stream)>>>(w, codes, scales, d->K, P, d->packing,
                                                                          d->fwht_block != 0, status);
  TQ_CHECK_LAUNCH();
  return TQ_OK;
}

// Device helper of the CUDA-core MoE kernels (internal).
#pragma once

#include "tq_internal.cuh"

namespace tq {

// One warp accumulates acc[b] += sum_k s[g(k)] t[k] x[b][k] over one packed row (lane-strided
// words; the caller reduces across lanes).  x rows have leading dimension ldx.
template <int PACKING, int MAXB>
__device__ __forceinline__ void row_dot_accumulate(const uint32_t* __restrict__ row,
                                                   const uint16_t* __restrict__ srow,
                                                   const float* __restrict__ x, int K, int ldx, int G, int batch,
                                                   int lane, float (&acc)[MAXB]) {
  constexpr int PER = PACKING == TQ_PACK_B3 ? kB3Trits : kB2Trits;
  const int used = (K + PER - 1) / PER;
  for (int j = lane; j < used; j += 32) {
    uint32_t v = __ldg(row + j);
#pragma unroll
    for (int q = 0; q < PER; ++q) {
      int dgt;
      if (PACKING == TQ_PACK_B3) {
        dgt = static_cast<int>(v % 3u);
        v /= 3u;
      } else {
        dgt = static_cast<int>((v >> (2 * q)) & 3u);
        if (dgt == 3) dgt = 1;
      }
      const int k = j * PER + q;
      if (k < K && dgt != 1) {
        const float st = static_cast<float>(dgt - 1) * half_bits_to_float(__ldg(srow + k / G));
#pragma unroll
        for (int b = 0; b < MAXB; ++b)
          if (b < batch) acc[b] = fmaf(st, __ldg(x + static_cast<size_t>(b) * ldx + k), acc[b]);
      }
    }
  }
}

}  // namespace tq

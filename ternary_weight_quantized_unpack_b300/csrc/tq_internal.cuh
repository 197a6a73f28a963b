// Internal helpers shared by the libtq CUDA sources (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "tq.h"

namespace tq {

constexpr int kB3Trits = 20;             // trits per base-3 word
constexpr int kB2Trits = 16;             // trits per 2-bit word
constexpr uint32_t kB3Max = 3486784400u; // 3^20 - 1
constexpr uint32_t kB3Zero = 1743392200u;  // all digits 1 (t = 0)
constexpr uint32_t kB2Zero = 0x55555555u;  // all fields 1 (t = 0)
constexpr int kFwhtBlock = 128;
constexpr int kMaxBatch = 16;

// Device status word: the first error any kernel recorded since the last tq_device_status()
// (0 = none).  Defined once in tq_api.cu; kernels receive its address (status_ptr()).
int* status_ptr();

// Remembers a failed CUDA call for tq_last_cuda_error() (per host thread), clears CUDA's sticky-free
// last-error slot and returns TQ_ERR_CUDA.
tq_status cuda_fail(cudaError_t e);

__device__ __forceinline__ void record_error(int* status, int code) { atomicCAS(status, 0, code); }

// 3-bit codes: a word has ten 3-bit slots, five per 16-bit half (bits 15 and 31 zero), so that one
// mask takes a code from each half.  A block of 64 codes takes 7 words: word i < 6 holds codes
// 10i..10i+9 of the block in slots 0..9, word 6 holds codes 60, 61 in slots 0, 1 and 62, 63 in slots
// 5, 6 (its other slots hold digit 4, q = 0).  Digit = q + 4.
constexpr int kQ3PerWord = 10;
constexpr int kQ3Block = 64;
constexpr int kQ3WordsPerBlock = 7;
__host__ __device__ __forceinline__ int q3_slot_bit(int slot) { return slot < 5 ? 3 * slot : 3 * slot + 1; }
// code of slot `slot` of word i (0..6) of a block, or -1 for a padding slot
__host__ __device__ __forceinline__ int q3_slot_code(int i, int slot) {
  if (i < 6) return 10 * i + slot;
  return slot == 0 || slot == 1 ? 60 + slot : slot == 5 || slot == 6 ? 57 + slot : -1;
}

__host__ __device__ __forceinline__ int trits_per_word(int packing) {
  return packing == TQ_PACK_B3 ? kB3Trits : kB2Trits;
}
__host__ __device__ __forceinline__ int pitch_words(int K, int packing) {
  const int w = packing == TQ_PACK_3BIT ? (K + kQ3Block - 1) / kQ3Block * kQ3WordsPerBlock
                                        : (K + trits_per_word(packing) - 1) / trits_per_word(packing);
  return (w + 3) & ~3;
}
__host__ __device__ __forceinline__ int groups_of(int K, int group) { return (K + group - 1) / group; }

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
__device__ __forceinline__ float half_bits_to_float(uint16_t b) {
  return __half2float(__ushort_as_half(b));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// In-warp block Walsh-Hadamard transform of 128 values, 4 per lane (lane l holds elements
// 4l..4l+3), Sylvester order, unnormalised: v <- H_128 v.  Butterfly (a, b) -> (a + b, a - b)
// on pairs (i, i + h) for h = 1, 2 (in registers) and h = 4..64 (lane bit log2(h/4)).
template <typename T>
__device__ __forceinline__ void fwht128_warp(T (&v)[4]) {
  T a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
  v[0] = a0 + a2; v[2] = a0 - a2; v[1] = a1 + a3; v[3] = a1 - a3;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      T p = __shfl_xor_sync(0xffffffffu, v[j], m);
      v[j] = upper ? (p - v[j]) : (v[j] + p);
    }
  }
}

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace tq

#define TQ_CHECK_LAUNCH()                                   \
  do {                                                      \
    const cudaError_t e_ = cudaPeekAtLastError();           \
    if (e_ != cudaSuccess) return tq::cuda_fail(e_);        \
  } while (0)

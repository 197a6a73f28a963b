// Packing and unpacking of ternary weights.
//
// base-3: 20 trits per 32-bit word, word = sum_i (t_i + 1) 3^i (the TurboQuant-MLX 1.58-bit Qwen3.6-35B-A3B page, section
// "为什么 1.58bit 没变成乱码", point 3: base-3 code, 20 ternary indices per 32-bit integer, ~1.6 bpw).
// 2-bit : 16 trits per word, field (t + 1) at bits 2i; field 3 is not a valid code.
// 3-bit : codes q in -4..3 of the non-expert linears, digit q + 4 at bits 3j of a word, 10 per word,
// each block of 64 codes in 7 words (word 6 holds four codes and six q = 0 digits).
// Rows are padded to a multiple of 4 words (16 bytes) so every row starts 16-byte aligned; every
// padding trit (code) is 0.
#include "tq_internal.cuh"

namespace tq {
namespace {

__global__ void pack_kernel(const int8_t* __restrict__ trits, uint32_t* __restrict__ codes, int N, int K, int P,
                            int packing, int* status) {
  const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<size_t>(N) * P) return;
  const int n = static_cast<int>(i / P), j = static_cast<int>(i % P);
  const int8_t* row = trits + static_cast<size_t>(n) * K;
  bool bad = false;
  uint32_t w = 0;
  if (packing == TQ_PACK_3BIT) {
    const int b = j / kQ3WordsPerBlock, i = j - b * kQ3WordsPerBlock;
    for (int q = 0; q < kQ3PerWord; ++q) {
      const int c = q3_slot_code(i, q), k = kQ3Block * b + c;
      int v = c >= 0 && k < K ? row[k] : 0;
      if (v < -4 || v > 3) { bad = true; v = 0; }
      w |= static_cast<uint32_t>(v + 4) << q3_slot_bit(q);
    }
  } else if (packing == TQ_PACK_B3) {
    // Horner from the most significant digit: w = (((d19) 3 + d18) 3 + ...) 3 + d0
    for (int q = kB3Trits - 1; q >= 0; --q) {
      const int k = j * kB3Trits + q;
      int t = k < K ? row[k] : 0;
      if (t < -1 || t > 1) { bad = true; t = 0; }
      w = w * 3u + static_cast<uint32_t>(t + 1);
    }
  } else {
    for (int q = 0; q < kB2Trits; ++q) {
      const int k = j * kB2Trits + q;
      int t = k < K ? row[k] : 0;
      if (t < -1 || t > 1) { bad = true; t = 0; }
      w |= static_cast<uint32_t>(t + 1) << (2 * q);
    }
  }
  if (bad) record_error(status, TQ_ERR_INVALID_CODE);
  codes[i] = w;
}

__global__ void unpack_kernel(const uint32_t* __restrict__ codes, int8_t* __restrict__ trits, int N, int K, int P,
                              int packing, int* invalid_words, int* status) {
  const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<size_t>(N) * P) return;
  const int n = static_cast<int>(i / P), j = static_cast<int>(i % P);
  uint32_t v = codes[i];
  int8_t* row = trits + static_cast<size_t>(n) * K;
  bool bad;
  if (packing == TQ_PACK_3BIT) {
    bad = (v & 0x80008000u) != 0u;
    const int b = j / kQ3WordsPerBlock, i = j - b * kQ3WordsPerBlock;
    for (int q = 0; q < kQ3PerWord; ++q) {
      const int c = q3_slot_code(i, q), k = kQ3Block * b + c;
      if (c >= 0 && k < K) row[k] = static_cast<int8_t>(static_cast<int>((v >> q3_slot_bit(q)) & 7u) - 4);
    }
  } else if (packing == TQ_PACK_B3) {
    bad = v > kB3Max;
    for (int q = 0; q < kB3Trits; ++q) {
      const uint32_t d = v % 3u;
      v /= 3u;
      const int k = j * kB3Trits + q;
      if (k < K) row[k] = static_cast<int8_t>(static_cast<int>(d) - 1);
    }
  } else {
    bad = false;
    for (int q = 0; q < kB2Trits; ++q) {
      const uint32_t f = (v >> (2 * q)) & 3u;
      bad |= f == 3u;
      const int k = j * kB2Trits + q;
      if (k < K) row[k] = static_cast<int8_t>(f == 3u ? 0 : static_cast<int>(f) - 1);
    }
  }
  if (bad) {
    if (invalid_words) atomicAdd(invalid_words, 1);
    record_error(status, TQ_ERR_INVALID_CODE);
  }
}

tq_status check_desc_basic(const tq_desc* d) {
  if (!d || d->N < 1 || d->K < 1) return TQ_ERR_INVALID_ARG;
  if (d->packing != TQ_PACK_B3 && d->packing != TQ_PACK_2BIT && d->packing != TQ_PACK_3BIT) return TQ_ERR_INVALID_ARG;
  return TQ_OK;
}

}  // namespace
}  // namespace tq

using namespace tq;

extern "C" tq_status tq_pack(const tq_desc* d, const int8_t* trits, uint32_t* codes, void* stream) {
  tq_status st = check_desc_basic(d);
  if (st != TQ_OK) return st;
  if (!trits || !codes) return TQ_ERR_INVALID_ARG;
  if (!aligned(codes, 16)) return TQ_ERR_MISALIGNED;
  const int P = pitch_words(d->K, d->packing);
  const size_t words = static_cast<size_t>(d->N) * P;
  const int threads = 256;
  const unsigned blocks = static_cast<unsigned>((words + threads - 1) / threads);
  int* status = status_ptr();
  if (!status) return TQ_ERR_CUDA;
  pack_kernel<<<blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(trits, codes, d->N, d->K, P, d->packing,
                                                                          status);
  TQ_CHECK_LAUNCH();
  return TQ_OK;
}

extern "C" tq_status tq_unpack(const tq_desc* d, const uint32_t* codes, int8_t* trits, int32_t* invalid_words,
                               void* stream) {
  tq_status st = check_desc_basic(d);
  if (st != TQ_OK) return st;
  if (!trits || !codes) return TQ_ERR_INVALID_ARG;
  if (!aligned(codes, 16) || (invalid_words && !aligned(invalid_words, 4))) return TQ_ERR_MISALIGNED;
  const int P = pitch_words(d->K, d->packing);
  const size_t words = static_cast<size_t>(d->N) * P;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* status = status_ptr();
  if (!status) return TQ_ERR_CUDA;
  if (invalid_words) {
    const cudaError_t e = cudaMemsetAsync(invalid_words, 0, sizeof(int32_t), s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  const int threads = 256;
  const unsigned blocks = static_cast<unsigned>((words + threads - 1) / threads);
  unpack_kernel<<<blocks, threads, 0, s>>>(codes, trits, d->N, d->K, P, d->packing, invalid_words, status);
  TQ_CHECK_LAUNCH();
  return TQ_OK;
}

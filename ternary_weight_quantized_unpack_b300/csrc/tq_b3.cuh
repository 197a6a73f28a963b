// Base-3 decode pieces shared by the kernels that take base-3 words apart on the fly: the chunk
// lookup table and the split of a word into its four 5-trit chunks.
//
// A word holds 20 trits as the integer sum of (t_i + 1) * 3^i (20 trits per 32-bit integer, the
// TurboQuant-MLX page, "为什么 1.58bit 没变成乱码", point 3).  Two exact reciprocal multiplies split
// it into four chunks of 5 digits (3^5 = 243 values); a table turns a chunk into its digits placed
// in FP16 pair fields, so that one mask per pair yields an MMA operand register.
#pragma once

#include "tq_internal.cuh"

namespace tq {

// Chunk lookup table: for a 5-trit chunk c (digits d0..d4), entry "A" places the digits at FP16
// pair fields (lo0, hi0, lo1, hi1, lo2) and entry "B" at (hi2, lo3, hi3, lo4, hi4), where loI / hiI
// are bits 2I / 16 + 2I.  Each entry is stored REP times in a row (entry c, copy r at c * REP + r),
// so that lane l reading copy l % REP spreads a warp's reads over the banks.
template <int REP>
struct __align__(128) B3Lut {  // bulk-copied: 16-byte alignment required
  static constexpr uint32_t kWords = 2u * 243u * REP;
  static constexpr uint32_t kBytes = kWords * 4u;
  uint32_t v[kWords];
};

template <int REP>
constexpr B3Lut<REP> make_b3_lut() {
  B3Lut<REP> L{};
  for (int c = 0; c < 243; ++c) {
    int d[5] = {0, 0, 0, 0, 0};
    int x = c;
    for (int i = 0; i < 5; ++i) {
      d[i] = x % 3;
      x /= 3;
    }
    const uint32_t a = static_cast<uint32_t>(d[0] | (d[1] << 16) | (d[2] << 2) | (d[3] << 18) | (d[4] << 4));
    const uint32_t b = static_cast<uint32_t>((d[0] << 20) | (d[1] << 6) | (d[2] << 22) | (d[3] << 8) | (d[4] << 24));
    for (int l = 0; l < REP; ++l) {
      L.v[c * REP + l] = a;
      L.v[243 * REP + c * REP + l] = b;
    }
  }
  return L;
}

// Base-3 word -> the table words of its four chunks: L0 / L1 (trits 0..9), L2 / L3 (trits 10..19).
// lutA / lutB point at this lane's copy of the "A" and "B" halves of the table.  A word above
// 3^20 - 1 (not a valid code) is read as 3^20 - 1.
template <int REP>
__device__ __forceinline__ void b3_chunks(uint32_t w, const uint32_t* __restrict__ lutA,
                                          const uint32_t* __restrict__ lutB, uint32_t (&L)[4]) {
  const uint32_t v = min(w, kB3Max);
  const uint32_t hi = __umulhi(v + 1u, 2383401723u) >> 15;  // v / 3^10, exact for v < 3^20
  const uint32_t lo = v - hi * 59049u;
  const uint32_t bl = __umulhi(lo, 17675008u);                // lo / 243, exact for lo < 3^10
  const uint32_t al = lo - bl * 243u;
  const uint32_t bh = __umulhi(hi, 17675008u);
  const uint32_t ah = hi - bh * 243u;
  L[0] = lutA[al * REP];
  L[1] = lutB[bl * REP];
  L[2] = lutA[ah * REP];
  L[3] = lutB[bh * REP];
}

// Pair j (0..9) of a decoded word as an MMA operand register: (trit 2j, trit 2j+1) in the
// (lo, hi) halves at field j % 5.  Fields 0, 1 come from the "A" entry, 3, 4 from "B", 2 from both.
__device__ __forceinline__ uint32_t b3_pair(const uint32_t (&L)[4], int j) {
  const uint32_t a = j < 5 ? L[0] : L[2], b = j < 5 ? L[1] : L[3];
  const int f = j % 5;
  const uint32_t m = 0x00030003u << (2 * f);
  return f < 2 ? (a & m) : f == 2 ? ((a | b) & m) : (b & m);
}

}  // namespace tq

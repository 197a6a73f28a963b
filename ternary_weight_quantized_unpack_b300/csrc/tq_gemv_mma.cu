// Decode GEMV: y[b][n] = sum_g s[n][g] sum_{k in g} t[n][k] x~[b][k], batch 1..16.
//
// The weights stream from HBM once; everything else is arranged so the stream is the bottleneck:
//  * Decode is register-only.  A 2-bit digit d = t + 1 placed in mantissa bits 2i of an FP16 half
//    with a zero exponent is the subnormal d * 2^(2i-24), exactly, so one LOP3 turns a code word into
//    two FP16 tensor-core operands.  The position factor 2^(8-2i) and the offset t = d - 1 are folded
//    into the activations: x^ = x~ * 2^-e * 2^(8-2i) and, per group, the accumulator starts at
//    -2^-16 * sum(x~ 2^-e) (e: exponent of the 128-block, shared by the batch).
//  * Base-3 words (20 trits per uint32: tantan.ink/?p=490, "为什么 1.58bit 没变成乱码", point 3) are
//    split into four 5-trit chunks by two exact reciprocal multiplies; a 243-entry table (replicated
//    per lane, conflict-free) places the chunk's digits into those bit fields.
//  * The multiply-add runs on mma.sync m16n8k16 (FP16 x FP16 -> FP32).  On B300, tcgen05.mma costs
//    ~120 cycles per K=16 step whatever N is, so with N <= 16 it retires only ~17 trits/cycle/SM;
//    mma.sync m16n8k16 retires 126, above the ~80 the HBM rate requires.
//  * Each group of 64 or 128 weights has its own FP16 scale (cosmocat.dev "27B 大模型塞进 5.9GB",
//    section 二 ②): every MMA covers one group only, and the group's 16x8 result is folded into the
//    output with one FMA per element.
//  * The block Walsh-Hadamard transform of the activations (same page, section 二 ①) is computed by
//    each CTA for its own K-range in the prologue, into shared memory; no separate launch.
//
// Two register layouts:
//  2-bit ("shared-row"): a warp owns 16 rows; the four threads of a quad share a row and take words
//      2q, 2q+1 (group 128) or word q (group 64) of every group, so each MMA is group-pure.  N = 8
//      batch columns per MMA.
//  base-3 ("column"): a warp owns 64 rows and each thread decodes two whole rows (identical schedule,
//      natural trit order), because 20-trit words straddle groups.  The B operand is zero except where
//      the column matches the quad thread that supplied the K-slots, so one MMA yields four
//      independent row dot products per quad: N = 4 thread columns x 2 batch rows.
#include <algorithm>
#include <mutex>

#include "tq_internal.cuh"
#include "tq_kernels.cuh"
#include "tq_sm100.cuh"

namespace tq {
namespace gemv {

using namespace sm100;

constexpr int kMaxWarps = 16;
constexpr uint32_t kLutWords = 2u * 243u * 32u;

template <int PACK>
struct Unit {
  static constexpr int TRITS = PACK == TQ_PACK_B3 ? 640 : 512;  // 32 code words
  static constexpr int SLAB = PACK == TQ_PACK_B3 ? 64 : 16;     // rows per warp
};

// Chunk lookup table (base-3): for a 5-trit chunk c (digits d0..d4), entry "A" places the digits at
// FP16 pair fields (lo0, hi0, lo1, hi1, lo2) and entry "B" at (hi2, lo3, hi3, lo4, hi4), where
// loI / hiI are bits 2I / 16 + 2I.  Each entry is replicated 32 times so that lane l reads bank l.
struct LutTable {
  uint32_t v[kLutWords];
};
constexpr LutTable make_lut() {
  LutTable L{};
  for (int c = 0; c < 243; ++c) {
    int d[5] = {0, 0, 0, 0, 0};
    int x = c;
    for (int i = 0; i < 5; ++i) {
      d[i] = x % 3;
      x /= 3;
    }
    const uint32_t a = static_cast<uint32_t>(d[0] | (d[1] << 16) | (d[2] << 2) | (d[3] << 18) | (d[4] << 4));
    const uint32_t b = static_cast<uint32_t>((d[0] << 20) | (d[1] << 6) | (d[2] << 22) | (d[3] << 8) | (d[4] << 24));
    for (int l = 0; l < 32; ++l) {
      L.v[c * 32 + l] = a;
      L.v[243 * 32 + c * 32 + l] = b;
    }
  }
  return L;
}
__device__ const LutTable g_lut = make_lut();

struct Params {
  const uint32_t* codes;
  const uint16_t* scales;
  const uint16_t* x;
  float* y;
  float* partial;                  // [ksplit][B][N] when ksplit > 1
  unsigned long long* counters;    // [row groups]: (epoch << 16) | arrivals
  int* status;
  int N, K, P, ng, B, G;
  int wpc;                         // warps per CTA
  int upr;                         // K-units (32-word stages) per row
  int ups;                         // units per K-split
  int ksplit;
  int apply;                       // 1: block FWHT of x
  unsigned long long epoch;
  uint32_t xh_off, v_off, p2_off;  // shared-memory offsets: x^, per-group sums, per-group 2^(16+e)
};

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Base-3 word -> two registers of FP16-pair bit fields: R0 holds pairs 0..4 (trits 0..9) at field
// positions 0..4, R1 pairs 5..9 (trits 10..19).  Pair j of the word is (R & (0x00030003 << 2(j%5))).
__device__ __forceinline__ void b3_fields(uint32_t w, const uint32_t* __restrict__ lutA,
                                          const uint32_t* __restrict__ lutB, uint32_t& R0, uint32_t& R1) {
  const uint32_t v = min(w, kB3Max);
  const uint32_t hi = __umulhi(v + 1u, 2383401723u) >> 15;  // v / 3^10, exact for v < 3^20
  const uint32_t lo = v - hi * 59049u;
  const uint32_t bl = __umulhi(lo, 17675008u);                // lo / 243, exact for lo < 3^10
  const uint32_t al = lo - bl * 243u;
  const uint32_t bh = __umulhi(hi, 17675008u);
  const uint32_t ah = hi - bh * 243u;
  R0 = lutA[al * 32] | lutB[bl * 32];
  R1 = lutA[ah * 32] | lutB[bh * 32];
}

// ---------------------------------------------------------------------------------------------
// Prologue: x~ for this CTA's K-range, all batch rows, into shared memory in the layout of PACK.
// One warp per 128-block (round robin); the block exponent e is shared by the batch rows.
// ---------------------------------------------------------------------------------------------
template <int PACK>
__device__ __forceinline__ void prepare_x(const Params& p, uint8_t* smem, int k_start, int kr) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = p.B, G = p.G;
  uint16_t* xh = reinterpret_cast<uint16_t*>(smem + p.xh_off);
  float* V = reinterpret_cast<float*>(smem + p.v_off);
  float* P2 = reinterpret_cast<float*>(smem + p.p2_off);
  const int nblk = kr / kFwhtBlock;
  for (int blk = warp; blk < nblk; blk += p.wpc) {
    const int kb = k_start + blk * kFwhtBlock + 4 * lane;  // absolute trit index of this lane's 4 values
    float mx = 0.f;
    for (int b = 0; b < B; ++b) {
      float v[4];
      const uint2 raw = __ldg(reinterpret_cast<const uint2*>(p.x + static_cast<size_t>(b) * p.K + kb));
      v[0] = bf16_bits_to_float(static_cast<uint16_t>(raw.x & 0xffffu));
      v[1] = bf16_bits_to_float(static_cast<uint16_t>(raw.x >> 16));
      v[2] = bf16_bits_to_float(static_cast<uint16_t>(raw.y & 0xffffu));
      v[3] = bf16_bits_to_float(static_cast<uint16_t>(raw.y >> 16));
      if (p.apply) fwht128_warp(v);
#pragma unroll
      for (int j = 0; j < 4; ++j) mx = fmaxf(mx, fabsf(v[j]));
    }
    if (p.apply) mx *= 0.08838834764831845f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    int e = 0;
    if (mx > 0.f) {
      const int ex = (__float_as_int(mx) >> 23) & 0xff;
      e = (ex == 0 ? -126 : ex - 127) - 6;  // max |x~| * 2^-e in [64, 128)
      if (e > 100) {
        e = 100;
        if (lane == 0) record_error(p.status, TQ_ERR_RANGE);
      }
      e = max(e, -100);
    }
    const float down = __int_as_float((127 - e) << 23) * (p.apply ? 0.08838834764831845f : 1.f);
    const int prel = blk * kFwhtBlock + 4 * lane;  // trit index relative to k_start
    for (int b = 0; b < B; ++b) {
      float v[4];
      const uint2 raw = __ldg(reinterpret_cast<const uint2*>(p.x + static_cast<size_t>(b) * p.K + kb));
      v[0] = bf16_bits_to_float(static_cast<uint16_t>(raw.x & 0xffffu));
      v[1] = bf16_bits_to_float(static_cast<uint16_t>(raw.x >> 16));
      v[2] = bf16_bits_to_float(static_cast<uint16_t>(raw.y & 0xffffu));
      v[3] = bf16_bits_to_float(static_cast<uint16_t>(raw.y >> 16));
      if (p.apply) fwht128_warp(v);
      float vs = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int pr = prel + j;
        int pos, off;
        if (PACK == TQ_PACK_B3) {
          pos = ((pr % 20) % 10) >> 1;  // k_start is a multiple of 20
          const int m = pr >> 2, r4 = pr & 3;
          off = ((m * B + b) * 2 + (r4 >> 1)) * 2 + (r4 & 1);  // in halves
        } else {
          const int gi = pr / G, pg = pr % G, wg = pg >> 4, f = pg & 15, jj = f & 7;
          const int WPT = G / 64;
          pos = jj < 5 ? jj : jj - 5;
          const int qq = wg / WPT, u = wg % WPT;
          off = (((((gi * WPT + u) * 4 + (jj >> 1)) * B + b) * 4 + qq) * 2 + (jj & 1)) * 2 + (f >> 3);
        }
        const float F = __int_as_float((127 + 8 - 2 * pos) << 23);
        const __half h = __float2half_rn(v[j] * down * F);
        xh[off] = __half_as_ushort(h);
        vs += __half2float(h) * __int_as_float((127 - 8 + 2 * pos) << 23);
      }
      if (G == 128) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) vs += __shfl_xor_sync(0xffffffffu, vs, o);
      } else {
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) vs += __shfl_xor_sync(0xffffffffu, vs, o);
      }
      if ((lane & (G == 128 ? 31 : 15)) == 0) V[(prel / G) * B + b] = vs;
    }
    if (lane == 0) {
      const float p2 = __int_as_float((127 + 16 + e) << 23);  // 2^(16 + e)
      for (int gi = (blk * kFwhtBlock) / G; gi < (blk * kFwhtBlock + kFwhtBlock) / G; ++gi) P2[gi] = p2;
    }
  }
}

// ---------------------------------------------------------------------------------------------
// Output: one K-split writes y directly; several K-splits write partials and the last CTA of a row
// group (epoch-tagged arrival counter, reset by the last arriver) sums them in split order.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void store_out(const Params& p, int row, int b, float v) {
  if (row >= p.N || b >= p.B) return;
  if (p.ksplit == 1)
    p.y[static_cast<size_t>(b) * p.N + row] = v;
  else
    p.partial[(static_cast<size_t>(blockIdx.y) * p.B + b) * p.N + row] = v;
}

__device__ __forceinline__ void finish_splits(const Params& p, int row0, int rows, volatile int* s_flag) {
  if (p.ksplit == 1) return;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long* c = p.counters + blockIdx.x;
    unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(c), nw, got;
    int count;
    for (;;) {
      count = (old >> 16) == p.epoch ? static_cast<int>(old & 0xffffu) + 1 : 1;
      nw = (p.epoch << 16) | static_cast<unsigned long long>(count);
      got = atomicCAS(c, old, nw);
      if (got == old) break;
      old = got;
    }
    const int last = count == p.ksplit;
    if (last) atomicExch(c, 0ull);
    __threadfence();
    *s_flag = last;
  }
  __syncthreads();
  if (!*s_flag) return;
  for (int i = threadIdx.x; i < rows * p.B; i += blockDim.x) {
    const int b = i / rows, row = row0 + i % rows;
    if (row >= p.N) continue;
    float v = 0.f;
    for (int s = 0; s < p.ksplit; ++s) v += __ldcg(p.partial + (static_cast<size_t>(s) * p.B + b) * p.N + row);
    p.y[static_cast<size_t>(b) * p.N + row] = v;
  }
}

// ---------------------------------------------------------------------------------------------
// 2-bit, shared-row layout.  NT = number of 8-column batch tiles (1: B <= 8, 2: B <= 16).
// ---------------------------------------------------------------------------------------------
template <int G, int NT>
__global__ void __launch_bounds__(32 * kMaxWarps) gemv_2b_kernel(const __grid_constant__ Params p) {
  constexpr int WPT = G / 64;  // words per thread per group per row
  extern __shared__ __align__(16) uint8_t smem[];
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const int u_a = blockIdx.y * p.ups, u_b = min(u_a + p.ups, p.upr);
  const int k_start = u_a * Unit<TQ_PACK_2BIT>::TRITS;
  const int kr = min(u_b * Unit<TQ_PACK_2BIT>::TRITS, p.K) - k_start;
  const int ngr = kr / G;
  const int g_abs0 = k_start / G;
  pdl_wait();
  prepare_x<TQ_PACK_2BIT>(p, smem, k_start, kr);
  __syncthreads();

  const int row0 = blockIdx.x * p.wpc * 16 + warp * 16;
  const int rg = row0 + g, rg8 = rg + 8;
  const bool vg = rg < p.N, vg8 = rg8 < p.N;
  const uint32_t* cg = p.codes + static_cast<size_t>(vg ? rg : 0) * p.P + k_start / 16 + WPT * q;
  const uint32_t* cg8 = p.codes + static_cast<size_t>(vg8 ? rg8 : 0) * p.P + k_start / 16 + WPT * q;
  const uint16_t* sg = p.scales + static_cast<size_t>(vg ? rg : 0) * p.ng + g_abs0;
  const uint16_t* sg8 = p.scales + static_cast<size_t>(vg8 ? rg8 : 0) * p.ng + g_abs0;
  const uint32_t* xh = reinterpret_cast<const uint32_t*>(smem + p.xh_off);
  const float* V = reinterpret_cast<const float*>(smem + p.v_off);
  const float* P2 = reinterpret_cast<const float*>(smem + p.p2_off);
  constexpr int D = 4;  // groups of code words prefetched
  uint32_t buf[D][2 * WPT];
  uint16_t sbuf[D][2];
  auto fetch = [&](int gi, int slot) {
    if (gi < ngr) {
#pragma unroll
      for (int u = 0; u < WPT; ++u) {
        buf[slot][u] = vg ? __ldg(cg + gi * (G / 16) + u) : kB2Zero;
        buf[slot][WPT + u] = vg8 ? __ldg(cg8 + gi * (G / 16) + u) : kB2Zero;
      }
      sbuf[slot][0] = vg ? __ldg(sg + gi) : static_cast<uint16_t>(0);
      sbuf[slot][1] = vg8 ? __ldg(sg8 + gi) : static_cast<uint16_t>(0);
    }
  };
#pragma unroll
  for (int d = 0; d < D - 1; ++d) fetch(d, d);
  float acc[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[t][i] = 0.f;

  for (int gi0 = 0; gi0 < ngr; gi0 += D) {
#pragma unroll
    for (int d = 0; d < D; ++d) {
      const int gi = gi0 + d;
      if (gi >= ngr) break;
      fetch(gi + D - 1, (d + D - 1) % D);
      float c[NT][4];
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const int bA = min(8 * t + 2 * q, p.B - 1), bB = min(8 * t + 2 * q + 1, p.B - 1);
        const float vA = 8 * t + 2 * q < p.B ? -1.52587890625e-05f * V[gi * p.B + bA] : 0.f;
        const float vB = 8 * t + 2 * q + 1 < p.B ? -1.52587890625e-05f * V[gi * p.B + bB] : 0.f;
        c[t][0] = vA;
        c[t][1] = vB;
        c[t][2] = vA;
        c[t][3] = vB;
      }
#pragma unroll
      for (int u = 0; u < WPT; ++u) {
        const uint32_t w = buf[d][u], w8 = buf[d][WPT + u];
        const uint32_t w2 = w >> 10, w82 = w8 >> 10;
        uint32_t pr[8], pr8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          pr[j] = j < 5 ? (w & (0x00030003u << (2 * j))) : (w2 & (0x00030003u << (2 * (j - 5))));
          pr8[j] = j < 5 ? (w8 & (0x00030003u << (2 * j))) : (w82 & (0x00030003u << (2 * (j - 5))));
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const int b = 8 * t + g;
            const int bc = min(b, p.B - 1);
            const uint2 bv =
                *reinterpret_cast<const uint2*>(xh + ((((gi * WPT + u) * 4 + jj) * p.B + bc) * 4 + q) * 2);
            const uint32_t b0 = b < p.B ? bv.x : 0u, b1 = b < p.B ? bv.y : 0u;
            mma16816(c[t], pr[2 * jj], pr8[2 * jj], pr[2 * jj + 1], pr8[2 * jj + 1], b0, b1);
          }
        }
      }
      const float p2 = P2[gi];
      const float mg = half_bits_to_float(sbuf[d][0]) * p2, mg8 = half_bits_to_float(sbuf[d][1]) * p2;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        acc[t][0] = fmaf(mg, c[t][0], acc[t][0]);
        acc[t][1] = fmaf(mg, c[t][1], acc[t][1]);
        acc[t][2] = fmaf(mg8, c[t][2], acc[t][2]);
        acc[t][3] = fmaf(mg8, c[t][3], acc[t][3]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    store_out(p, rg, 8 * t + 2 * q, acc[t][0]);
    store_out(p, rg, 8 * t + 2 * q + 1, acc[t][1]);
    store_out(p, rg8, 8 * t + 2 * q, acc[t][2]);
    store_out(p, rg8, 8 * t + 2 * q + 1, acc[t][3]);
  }
  __shared__ int s_flag;
  finish_splits(p, blockIdx.x * p.wpc * 16, p.wpc * 16, &s_flag);
}

// ---------------------------------------------------------------------------------------------
// base-3, column layout.  NT = number of 2-row batch tiles (ceil(B / 2)).
// Thread (g, q) owns rows R = r0 + 4g + q and R + 32 of its warp's 64-row slab.
// ---------------------------------------------------------------------------------------------
template <int G, int NT, bool FULL>
__device__ __forceinline__ void b3_period(const Params& p, const uint32_t* __restrict__ cR,
                                          const uint32_t* __restrict__ cR2, bool vR, bool vR2,
                                          const uint32_t* __restrict__ lutA, const uint32_t* __restrict__ lutB,
                                          const uint32_t* __restrict__ xh, const float* __restrict__ V,
                                          const float* __restrict__ P2, const uint16_t* const (&srow)[4],
                                          const bool (&svalid)[4], int pi, int ngp, int lane, float (&acc)[NT][4]) {
  constexpr int GP = G / 2;      // pairs per group
  constexpr int GPS = 640 / G;   // groups per period
  const int g = lane >> 2, q = lane & 3;
  const int bq = q >> 1;         // batch within a tile held by this thread's accumulators
  const bool bsup = (g & 3) == q;  // this thread supplies B (x^) values
  const int bsel = g >> 2;         // batch within a tile it supplies
  float c[NT][4];
  uint4 cur = vR ? __ldg(reinterpret_cast<const uint4*>(cR)) : make_uint4(kB3Zero, kB3Zero, kB3Zero, kB3Zero);
  uint4 cur2 = vR2 ? __ldg(reinterpret_cast<const uint4*>(cR2)) : make_uint4(kB3Zero, kB3Zero, kB3Zero, kB3Zero);
#pragma unroll
  for (int step = 0; step < 8; ++step) {
    if (!FULL && (step * 80) / G >= ngp) break;
    uint4 nxt = cur, nxt2 = cur2;
    if (step < 7 && (FULL || ((step + 1) * 80) / G < ngp)) {  // never read past the row's last word
      if (vR) nxt = __ldg(reinterpret_cast<const uint4*>(cR) + step + 1);
      if (vR2) nxt2 = __ldg(reinterpret_cast<const uint4*>(cR2) + step + 1);
    }
    const uint32_t wr[4] = {cur.x, cur.y, cur.z, cur.w};
    const uint32_t wr2[4] = {cur2.x, cur2.y, cur2.z, cur2.w};
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      uint32_t A0, A1, C0, C1;
      b3_fields(wr[wi], lutA, lutB, A0, A1);
      b3_fields(wr2[wi], lutA, lutB, C0, C1);
#pragma unroll
      for (int mj = 0; mj < 5; ++mj) {
        const int pair = (step * 4 + wi) * 10 + 2 * mj;  // first pair of this MMA within the period
        const int gl = pair / GP;
        if (!FULL && gl >= ngp) break;
        if (pair % GP == 0) {
          // new group: accumulators start at -2^-16 * sum(x^) of the group for their batch
          const int gi = pi * GPS + gl;
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const int b = 2 * t + bq;
            const float v0 = b < p.B ? -1.52587890625e-05f * V[gi * p.B + b] : 0.f;
            c[t][0] = v0;
            c[t][1] = v0;
            c[t][2] = v0;
            c[t][3] = v0;
          }
        }
        const int j0 = (2 * mj) % 10, j1 = (2 * mj + 1) % 10;
        const uint32_t RA = j0 < 5 ? A0 : A1, RB = j1 < 5 ? A0 : A1;
        const uint32_t SA = j0 < 5 ? C0 : C1, SB = j1 < 5 ? C0 : C1;
        const uint32_t a0 = RA & (0x00030003u << (2 * (j0 % 5)));
        const uint32_t a2 = RB & (0x00030003u << (2 * (j1 % 5)));
        const uint32_t a1 = SA & (0x00030003u << (2 * (j0 % 5)));
        const uint32_t a3 = SB & (0x00030003u << (2 * (j1 % 5)));
        const int m = pi * 160 + pair / 2;  // MMA index within the K-range
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const int b = 2 * t + bsel;
          uint32_t b0 = 0u, b1 = 0u;
          if (bsup && b < p.B) {
            const uint2 bv = *reinterpret_cast<const uint2*>(xh + (m * p.B + b) * 2);
            b0 = bv.x;
            b1 = bv.y;
          }
          mma16816(c[t], a0, a1, a2, a3, b0, b1);
        }
        if ((pair + 2) % GP == 0) {
          const int gi = pi * GPS + gl;
          const float p2 = P2[gi];
          const int gabs = gi;  // srow pointers are offset to this CTA's first group
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float m_i = svalid[i] ? half_bits_to_float(__ldg(srow[i] + gabs)) * p2 : 0.f;
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[t][i] = fmaf(m_i, c[t][i], acc[t][i]);
          }
        }
      }
    }
    cur = nxt;
    cur2 = nxt2;
  }
}

template <int G, int NT>
__global__ void __launch_bounds__(32 * kMaxWarps) gemv_b3_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(16) uint8_t smem[];
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  // the chunk table into shared memory (it does not depend on earlier kernels)
  {
    const uint4* src = reinterpret_cast<const uint4*>(&g_lut);
    uint4* dst = reinterpret_cast<uint4*>(smem);
    for (int i = threadIdx.x; i < static_cast<int>(kLutWords / 4); i += blockDim.x) dst[i] = __ldg(src + i);
  }
  const int u_a = blockIdx.y * p.ups, u_b = min(u_a + p.ups, p.upr);
  const int k_start = u_a * 640;
  const int kr = min(u_b * 640, p.K) - k_start;
  const int g_abs0 = k_start / G;
  pdl_wait();
  prepare_x<TQ_PACK_B3>(p, smem, k_start, kr);
  __syncthreads();

  const int r0 = blockIdx.x * p.wpc * 64 + warp * 64;
  const int R = r0 + lane, R2 = R + 32;
  const bool vR = R < p.N, vR2 = R2 < p.N;
  const uint32_t* cR = p.codes + static_cast<size_t>(vR ? R : 0) * p.P + k_start / 20;
  const uint32_t* cR2 = p.codes + static_cast<size_t>(vR2 ? R2 : 0) * p.P + k_start / 20;
  // rows of the four accumulators this thread folds: threads (g, 2q%4) and (g, 2q%4 + 1), R and R+32
  const int cq = (2 * q) & 3;
  const int rows[4] = {r0 + 4 * g + cq, r0 + 4 * g + cq + 1, r0 + 32 + 4 * g + cq, r0 + 32 + 4 * g + cq + 1};
  const uint16_t* srow[4];
  bool svalid[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    svalid[i] = rows[i] < p.N;
    srow[i] = p.scales + static_cast<size_t>(svalid[i] ? rows[i] : 0) * p.ng + g_abs0;
  }
  const uint32_t* lutA = reinterpret_cast<const uint32_t*>(smem) + lane;
  const uint32_t* lutB = lutA + 243 * 32;
  const uint32_t* xh = reinterpret_cast<const uint32_t*>(smem + p.xh_off);
  const float* V = reinterpret_cast<const float*>(smem + p.v_off);
  const float* P2 = reinterpret_cast<const float*>(smem + p.p2_off);
  float acc[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[t][i] = 0.f;
  const int n_per = (kr + 639) / 640;
  for (int pi = 0; pi < n_per; ++pi) {
    const int ngp = min(640 / G, (kr - pi * 640) / G);
    if (ngp == 640 / G)
      b3_period<G, NT, true>(p, cR + pi * 32, cR2 + pi * 32, vR, vR2, lutA, lutB, xh, V, P2, srow, svalid, pi, ngp,
                             lane, acc);
    else
      b3_period<G, NT, false>(p, cR + pi * 32, cR2 + pi * 32, vR, vR2, lutA, lutB, xh, V, P2, srow, svalid, pi, ngp,
                              lane, acc);
  }
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int i = 0; i < 4; ++i) store_out(p, rows[i], 2 * t + (q >> 1), acc[t][i]);
  __shared__ int s_flag;
  finish_splits(p, blockIdx.x * p.wpc * 64, p.wpc * 64, &s_flag);
}

// ---------------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------------
constexpr int kRefSMs = 148;  // plans depend only on the problem, so workspace sizes are stable

struct Plan {
  int wpc, ksplit, ups, upr, n_rg, ut;
  size_t smem, xh_off, v_off, p2_off;
  size_t ws_part, ws_cnt, total;
};

Plan make_plan(const tq_desc* d, int B) {
  Plan pl{};
  const bool b3 = d->packing == TQ_PACK_B3;
  pl.ut = b3 ? 640 : 512;
  pl.upr = (d->K + pl.ut - 1) / pl.ut;
  const int slab = b3 ? 64 : 16;
  const int slabs = (d->N + slab - 1) / slab;
  // warps per CTA: 16 when there are enough slabs, fewer for narrow matrices
  pl.wpc = kMaxWarps;
  while (pl.wpc > 4 && slabs < pl.wpc * 8) pl.wpc /= 2;
  pl.n_rg = (slabs + pl.wpc - 1) / pl.wpc;
  // K-splits: enough CTAs to cover the SMs, and a K-range whose activations fit in shared memory
  const size_t lut = b3 ? kLutWords * 4 : 0;
  const size_t budget = 200 * 1024 - lut;
  int ks = std::max(1, (kRefSMs * (kMaxWarps / pl.wpc)) / pl.n_rg);
  ks = std::min(ks, pl.upr);
  auto xh_bytes = [&](int units) { return static_cast<size_t>(units) * pl.ut * 2 * B; };
  while (ks < pl.upr && xh_bytes((pl.upr + ks - 1) / ks) > budget) ++ks;
  pl.ups = (pl.upr + ks - 1) / ks;
  pl.ksplit = (pl.upr + pl.ups - 1) / pl.ups;
  const int kr = pl.ups * pl.ut;
  const int ngr = kr / d->group;
  pl.xh_off = lut;
  pl.v_off = pl.xh_off + align256(xh_bytes(pl.ups));
  pl.p2_off = pl.v_off + align256(static_cast<size_t>(ngr) * B * 4);
  pl.smem = pl.p2_off + align256(static_cast<size_t>(ngr) * 4);
  if (pl.ksplit > 1) {
    pl.ws_part = 0;
    pl.ws_cnt = align256(static_cast<size_t>(pl.ksplit) * B * d->N * 4);
    pl.total = pl.ws_cnt + align256(static_cast<size_t>(pl.n_rg) * 8);
  } else {
    pl.total = 256;
  }
  return pl;
}

int max_smem_optin() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 232448;
  if (!cache[dev]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess || v <= 0) v = 232448;
    cache[dev] = v;
  }
  return cache[dev];
}

unsigned long long next_epoch() {
  static unsigned long long e = 0x5eed1234ull;
  e = (e + 0x9E3779B97F4A7C15ull) & 0x0000ffffffffffffull;
  if (e == 0) e = 1;
  return e;
}

// Raises a kernel's dynamic shared-memory limit to at least `bytes` on the current device.  The
// attribute belongs to the (function, device) pair, so the largest value set so far is kept per pair.
cudaError_t ensure_smem_attr(const void* fn, size_t bytes) {
  struct Entry {
    const void* fn;
    int dev;
    size_t bytes;
  };
  static Entry table[256];
  static int used = 0;
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  Entry* ent = nullptr;
  for (int i = 0; i < used; ++i)
    if (table[i].fn == fn && table[i].dev == dev) ent = &table[i];
  if (ent && ent->bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  if (!ent && used < 256) ent = &table[used++];
  if (ent) *ent = Entry{fn, dev, bytes};
  return cudaSuccess;
}

template <typename Kern>
cudaError_t launch(Kern kern, const Params& prm, const Plan& pl, cudaStream_t s) {
  const int optin = max_smem_optin();
  if (pl.smem + 1024 > static_cast<size_t>(optin)) return cudaErrorInvalidConfiguration;
  if (cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), pl.smem); e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.n_rg, pl.ksplit);
  cfg.blockDim = dim3(32 * pl.wpc);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, prm);
}

template <int G>
cudaError_t launch_b3(const Params& prm, const Plan& pl, cudaStream_t s) {
  switch ((prm.B + 1) / 2) {
    case 1: return launch(gemv_b3_kernel<G, 1>, prm, pl, s);
    case 2: return launch(gemv_b3_kernel<G, 2>, prm, pl, s);
    case 3:
    case 4: return launch(gemv_b3_kernel<G, 4>, prm, pl, s);
    default: return launch(gemv_b3_kernel<G, 8>, prm, pl, s);
  }
}

template <int G>
cudaError_t launch_2b(const Params& prm, const Plan& pl, cudaStream_t s) {
  if (prm.B <= 8) return launch(gemv_2b_kernel<G, 1>, prm, pl, s);
  return launch(gemv_2b_kernel<G, 2>, prm, pl, s);
}

}  // namespace gemv

size_t gemv_workspace_bytes(const tq_desc* d, int batch) { return gemv::make_plan(d, batch).total; }

cudaError_t launch_gemv(const tq_desc* d, const uint32_t* codes, const uint16_t* scales, const uint16_t* x, int B,
                        float* y, void* ws, cudaStream_t s) {
  using namespace gemv;
  const Plan pl = make_plan(d, B);
  Params prm{};
  prm.codes = codes;
  prm.scales = scales;
  prm.x = x;
  prm.y = y;
  prm.partial = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + pl.ws_part);
  prm.counters = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(ws) + pl.ws_cnt);
  prm.status = status_ptr();
  prm.N = d->N;
  prm.K = d->K;
  prm.P = pitch_words(d->K, d->packing);
  prm.ng = d->K / d->group;
  prm.B = B;
  prm.G = d->group;
  prm.wpc = pl.wpc;
  prm.upr = pl.upr;
  prm.ups = pl.ups;
  prm.ksplit = pl.ksplit;
  prm.apply = d->fwht_block != 0;
  prm.epoch = next_epoch();
  prm.xh_off = static_cast<uint32_t>(pl.xh_off);
  prm.v_off = static_cast<uint32_t>(pl.v_off);
  prm.p2_off = static_cast<uint32_t>(pl.p2_off);
  if (d->packing == TQ_PACK_B3) return d->group == 128 ? launch_b3<128>(prm, pl, s) : launch_b3<64>(prm, pl, s);
  return d->group == 128 ? launch_2b<128>(prm, pl, s) : launch_2b<64>(prm, pl, s);
}

}  // namespace tq

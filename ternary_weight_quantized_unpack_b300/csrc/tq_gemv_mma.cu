// Decode GEMV: y[b][n] = sum_g s[n][g] sum_{k in g} t[n][k] x~[b][k], batch 1..16.
//
// The weights stream from HBM once; everything else is arranged so that the stream is the bottleneck:
//  * Decode is register-only.  A 2-bit digit d = t + 1 placed in mantissa bits 2i of an FP16 half
//    with a zero exponent is the subnormal d * 2^(2i-24), exactly, so one LOP3 turns a code word into
//    two FP16 tensor-core operands.  The position factor 2^(8-2i) and the offset t = d - 1 are folded
//    into the activations: x^ = x~ * 2^-e * 2^(8-2i) and, per group, the accumulator starts at
//    -2^-16 * sum(x~ 2^-e) (e: exponent of the 128-block, shared by the batch).
//  * Base-3 words (20 trits per uint32: the TurboQuant-MLX 1.58-bit Qwen3.6-35B-A3B page, "为什么 1.58bit 没变成乱码", point 3) are
//    split into four 5-trit chunks by two exact reciprocal multiplies; a 243-entry table (replicated
//    per lane, conflict-free) places the chunk's digits into those bit fields.
//  * The multiply-add runs on mma.sync m16n8k16 (FP16 x FP16 -> FP32).  On B300, tcgen05.mma costs
//    ~120 cycles per K=16 step whatever N is, so with N <= 16 it retires only ~17 trits/cycle/SM;
//    mma.sync m16n8k16 retires 126, above the ~100 the HBM rate requires.
//  * Each group of 64 or 128 weights has its own FP16 scale ("27B 大模型塞进 5.9GB",
//    section 二 ②): every MMA covers one group only, and the group's result is folded into the
//    output with one FMA per element.  The CTA's scales are staged in shared memory and
//    pre-multiplied by the block factor 2^(16+e).
//  * The block Walsh-Hadamard transform of the activations (same page, section 二 ①) goes straight
//    into the operand layout.  The 2-bit stream kernel transforms its own K-range inside each CTA up
//    to batch 4, and the expert-layer GEMVs do so for chunks of at most 2 tokens; otherwise a small
//    prep kernel transforms the activations once per call and every CTA bulk-copies
//    (cp.async.bulk) the slice of its K-range into shared memory.
//
// Work split: a CTA holds rs x kl warps: rs row slabs, each split over kl K-lanes of ppl units
// (a unit is 32 code words of a row: 640 trits base-3, 512 trits 2-bit; whole groups either way).
// When K is split over several CTAs (gridDim.y <= 8) they form one thread-block cluster.  Partial
// sums meet in shared memory: first over the K-lanes of a CTA, then over the cluster's CTAs through
// distributed shared memory, in a fixed order, so results are deterministic without global atomics.
// The plan is chosen per shape among those whose CTAs are all resident at once.
//
// Code words reach registers through a ring of plain 128-bit loads issued several steps ahead.  With
// TQ_STATIC_WEIGHTS the first loads and the scale staging are issued before the programmatic
// dependent-launch wait, so a chain of GEMVs keeps HBM busy across kernel boundaries.
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
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "tq_b3.cuh"
#include "tq_internal.cuh"
#include "tq_kernels.cuh"
#include "tq_sm100.cuh"
#include "tq_tmap.cuh"

namespace tq {
namespace gemv {

using namespace sm100;

constexpr int kMaxThreads = 512;
constexpr int kMaxCluster = 8;
// With static weights, every warp asks L2 for its whole code range before the dependent-launch wait,
// so HBM streams this call's weights while the preceding kernels finish.
constexpr bool kPrefetchL2 = true;
// Stream kernel: up to this batch the CTAs transform their own K-range of the activations (no prep
// kernel; measured on the 64-layer 2-bit stream: batch 4 4.39 -> 3.86 ms per token, batch 8 no
// better than the prep kernel, 5.11 -> 5.20 ms).  kEarlyStages: stages of the code ring issued before the dependent-launch wait (static
// weights).  Measured on the 64-layer batch-1 stream: 0 (activations requested before any weight
// stage) 3.43 ms per token, 1: 3.47 ms, 2: 3.72 ms; with static weights only the scales are read
// before the wait.
constexpr int kStreamFuseMaxB = 4;
constexpr int kEarlyStages = 0;
constexpr uint32_t kLutBytes = B3Lut<32>::kBytes;

template <int PACK>
struct Geo;
template <>
struct Geo<TQ_PACK_B3> {
  static constexpr int UT = 640;   // trits per unit (32 words; 5 groups of 128 or 10 of 64)
  static constexpr int SLAB = 64;  // rows per warp
};
template <>
struct Geo<TQ_PACK_2BIT> {
  static constexpr int UT = 512;
  static constexpr int SLAB = 16;
};
template <>
struct Geo<TQ_PACK_3BIT> {
  static constexpr int UT = 256;   // codes per unit (28 words = 4 blocks of 64; 2 groups of 128 or 4 of 64)
  static constexpr int SLAB = 64;  // rows per warp (column layout)
};
__host__ __device__ constexpr int unit_codes(int pack) { return pack == TQ_PACK_B3 ? 640 : pack == TQ_PACK_3BIT ? 256 : 512; }
__host__ __device__ constexpr int slab_rows(int pack) { return pack == TQ_PACK_2BIT ? 16 : 64; }

// Row length of VP[group][.]: V for each batch row, then zeros, then the block factor 2^(16+e) in the
// last slot; a multiple of 4 floats so that every group's row is a whole number of 16-byte chunks.
__host__ __device__ constexpr int vp_row(int B) { return (B + 1 + 3) & ~3; }

// Chunk lookup table (base-3), one copy per lane (32): lane l reads bank l.
using LutTable = B3Lut<32>;
__device__ const LutTable g_lut = make_b3_lut<32>();

// ---------------------------------------------------------------------------------------------
// Prep kernel: x^ and VP for the whole of K, one warp per 128-block, all batch rows in registers.
// x^ layout (halves), K-major so that any K-range is one contiguous slice starting at k * B:
//   base-3: ((((m >> 1) * B + b) * 2 + (m & 1)) * 4 + r  for trit k = 4m + r (an MMA pair shares
//           16 bytes);
//   3-bit : the same with m = 16 * (k / 64) + reg / 2 and r = 2 * (reg % 2) + half, where (reg, half)
//           is the operand register of the 64-block (0..31) and the FP16 half the code decodes into;
//   2-bit : ((((((gi*WPT + u)*2 + jj/2)*B + b)*4 + q)*2 + jj%2)*2 + pair%2)*2 + half for the trit at
//           word u of quad thread q in group gi, pair index jp (MMA jj = jp / 2), half = trit / 8.
// ---------------------------------------------------------------------------------------------
struct PrepParams {
  const uint16_t* x;  // modes 0, 1: bf16 rows
  const float* gu;    // mode 2: gate / up outputs, rows of 2K floats (gate then up)
  float* h_out;       // mode 2: optional copy of h = silu(gate) * up, rows of K floats
  uint16_t* xh;
  float* vp;
  int* status;
  int K, B, apply;
  // 0: batch row b is x row b.  With routed-token chunks (mode 1, 2) blockIdx.z selects a chunk
  // record {expert, count, rows[B]}: mode 1 reads x row rows[b] / topk, mode 2 forms
  // silu(gate) * up of gu row rows[b]; slots past count are zero.  Chunk z writes its own slice.
  int mode;
  const int* chunks;
  int topk;
  size_t xh_cstride, vp_cstride;  // halves / floats per chunk
};

__device__ __forceinline__ float silu(float z) { return z / (1.f + expf(-z)); }

// x^ and VP of one 128-block (absolute index blk) for batch slots 0..B-1 (slots past count are zero).
// xh / vpo point at the slice that starts at block blk0 (offsets are taken relative to it; blk0 is a
// multiple of 5, so word boundaries stay at the same offsets).  One warp; MAXB >= B.  XS: x (mode 0)
// is a shared-memory copy of the slice, rows of xs_stride values starting at trit blk0 * 128.
template <int PACK, int G, int MAXB, bool XS = false>
__device__ __forceinline__ void prep_block(const uint16_t* __restrict__ x, const float* __restrict__ gu, float* h_out,
                                           int* status, int K, int B, int apply, int mode, int topk, int blk,
                                           int blk0, int count, const int* rows, uint16_t* xh, float* vpo,
                                           int lane, int xs_stride = 0) {
  const int R = vp_row(B);
  const int kb = blk * kFwhtBlock + 4 * lane;   // absolute trit index of this lane's 4 values
  const int kr = kb - blk0 * kFwhtBlock;        // ... relative to the slice
  float v[MAXB][4];
  float mx = 0.f;
#pragma unroll
  for (int b = 0; b < MAXB; ++b) {
    if (b < B) {
      if (b >= count) {
        v[b][0] = v[b][1] = v[b][2] = v[b][3] = 0.f;
      } else if (mode == 2) {  // h = silu(gate) * up of the assignment's gate / up row
        const size_t a = static_cast<size_t>(rows[b]);
        const float4 gg = *reinterpret_cast<const float4*>(gu + a * 2 * K + kb);
        const float4 uu = *reinterpret_cast<const float4*>(gu + a * 2 * K + K + kb);
        v[b][0] = silu(gg.x) * uu.x;
        v[b][1] = silu(gg.y) * uu.y;
        v[b][2] = silu(gg.z) * uu.z;
        v[b][3] = silu(gg.w) * uu.w;
        if (h_out) *reinterpret_cast<float4*>(h_out + a * K + kb) = make_float4(v[b][0], v[b][1], v[b][2], v[b][3]);
      } else {
        const size_t r = mode == 1 ? static_cast<size_t>(rows[b] / topk) : static_cast<size_t>(b);
        const uint2 raw = XS ? *reinterpret_cast<const uint2*>(x + r * xs_stride + kr)
                             : __ldcg(reinterpret_cast<const uint2*>(x + r * K + kb));
        v[b][0] = bf16_bits_to_float(static_cast<uint16_t>(raw.x & 0xffffu));
        v[b][1] = bf16_bits_to_float(static_cast<uint16_t>(raw.x >> 16));
        v[b][2] = bf16_bits_to_float(static_cast<uint16_t>(raw.y & 0xffffu));
        v[b][3] = bf16_bits_to_float(static_cast<uint16_t>(raw.y >> 16));
      }
      if (apply) fwht128_warp(v[b]);
#pragma unroll
      for (int j = 0; j < 4; ++j) mx = fmaxf(mx, fabsf(v[b][j]));
    }
  }
  if (apply) mx *= 0.08838834764831845f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  int e = 0;
  if (mx > 0.f) {
    const int ex = (__float_as_int(mx) >> 23) & 0xff;
    e = (ex == 0 ? -126 : ex - 127) - 6;  // max |x~| * 2^-e in [64, 128)
    if (e > 100) {
      e = 100;
      if (lane == 0) record_error(status, TQ_ERR_RANGE);
    }
    e = max(e, -100);
  }
  const float down = __int_as_float((127 - e) << 23) * (apply ? 0.08838834764831845f : 1.f);
#pragma unroll
  for (int b = 0; b < MAXB; ++b) {
    if (b >= B) break;
    float vs = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int k = kr + j;
      int pb, off;  // pb: lowest mantissa bit of the weight's digit in its decoded FP16 half
      if (PACK == TQ_PACK_B3) {
        pb = 2 * (((k % 20) % 10) >> 1);
        const int m = k >> 2, r4 = k & 3;
        off = (((m >> 1) * B + b) * 2 + (m & 1)) * 4 + r4;
      } else if (PACK == TQ_PACK_3BIT) {
        // code c of its 64-block -> operand register r (0..31) of the block, half h, bit pb
        const int c = k & 63;
        int r, h;
        if (c < 60) {
          const int i = c / 10, jj = c - 10 * i;
          h = jj >= 5 ? 1 : 0;
          const int jr = jj - 5 * h;
          r = 5 * i + jr;
          pb = jr < 3 ? 3 * jr : 3 * jr - 8;
        } else {
          h = (c - 60) >> 1;
          r = 30 + ((c - 60) & 1);
          pb = 3 * ((c - 60) & 1);
        }
        const int m = (k >> 6) * 16 + (r >> 1), r4 = 2 * (r & 1) + h;
        off = (((m >> 1) * B + b) * 2 + (m & 1)) * 4 + r4;
      } else {
        constexpr int WPT = G / 64;
        const int gi = k / G, pg = k % G, wg = pg >> 4, f = pg & 15, jp = f & 7;
        pb = 2 * (jp < 5 ? jp : jp - 5);
        const int qq = wg / WPT, u = wg % WPT, jj = jp >> 1;
        off = ((((((gi * WPT + u) * 2 + (jj >> 1)) * B + b) * 4 + qq) * 2 + (jj & 1)) * 2 + (jp & 1)) * 2 + (f >> 3);
      }
      const float F = __int_as_float((127 + 8 - pb) << 23);
      const __half h = __float2half_rn(v[b][j] * down * F);
      xh[off] = __half_as_ushort(h);
      vs += __half2float(h) * __int_as_float((127 - 8 + pb) << 23);
    }
    if (G == 128) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) vs += __shfl_xor_sync(0xffffffffu, vs, o);
    } else {
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) vs += __shfl_xor_sync(0xffffffffu, vs, o);
    }
    // the digit offset: t = d - 1 (ternary), q = d - 4 (3-bit)
    constexpr float kOff = PACK == TQ_PACK_3BIT ? -4.f * 1.52587890625e-05f : -1.52587890625e-05f;
    if ((lane & (G == 128 ? 31 : 15)) == 0) vpo[(kr / G) * R + b] = kOff * vs;
  }
  if (lane < kFwhtBlock / G) {  // per group of the block: padding zeros and the block factor
    const int gi = (blk - blk0) * (kFwhtBlock / G) + lane;
    for (int b = B; b < R - 1; ++b) vpo[gi * R + b] = 0.f;
    vpo[gi * R + R - 1] = __int_as_float((127 + 16 + e) << 23);  // 2^(16 + e)
  }
}

// MAXB: the smallest of 1, 2, 4, 8, 16 that holds the batch (the per-row loops are unrolled over it).
template <int PACK, int G, int MAXB>
__global__ void __launch_bounds__(128) gemv_prep_kernel(const __grid_constant__ PrepParams p) {
  pdl_launch_dependents();
  pdl_wait();  // x may be the output of the preceding kernel; the previous call may still read xh
  const int lane = threadIdx.x & 31;
  const int blk = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (blk * kFwhtBlock >= p.K) return;
  int count = p.B;
  const int* rows = nullptr;
  uint16_t* xh = p.xh;
  float* vpo = p.vp;
  if (p.mode != 0) {
    const int z = static_cast<int>(blockIdx.z);
    if (z >= p.chunks[0]) return;
    const int* rec = p.chunks + 1 + static_cast<size_t>(z) * (2 + p.B);
    count = rec[1];
    rows = rec + 2;
    xh += static_cast<size_t>(z) * p.xh_cstride;
    vpo += static_cast<size_t>(z) * p.vp_cstride;
  }
  prep_block<PACK, G, MAXB>(p.x, p.gu, p.h_out, p.status, p.K, p.B, p.apply, p.mode, p.topk, blk, 0, count, rows,
                                 xh, vpo, lane);
}

// ---------------------------------------------------------------------------------------------
// GEMV kernels
// ---------------------------------------------------------------------------------------------
struct Params {
  CUtensorMap tm;  // 3-bit: the codes [N][P] as a 2-D map (box 28 words x 64 rows); unused otherwise
  const uint32_t* codes;
  const uint16_t* scales;
  const uint16_t* xh_g;  // prep output: x^ for all of K
  const float* vp_g;     // prep output: VP[group][R]
  float* y;
  int* status;
  int N, K, P, ng, B, R, G;
  int rs;     // row slabs per CTA
  int kl;     // K-lanes per CTA
  int ppl;    // units per K-lane
  int upr;    // units per row
  int early;  // 1: codes and scales may be read before the preceding kernel has completed
  int v8;     // base-3: rows and code base are 32-byte aligned, codes are read 32 bytes at a time
  uint32_t xh_off, vp_off, sw_off, bar_off;  // shared-memory offsets: x^, VP, per-warp scales, barriers
  uint32_t ring_off;                         // 3-bit: per-warp code rings
  // Routed-token chunks (nullptr: one dense matrix).  blockIdx.z selects record {expert, count,
  // rows[B]} of chunks[1 + z * (2 + B)] (chunks[0] = number of records); the expert's codes and
  // scales start expert * *_estride elements in, the chunk's prep slice z * *_cstride in, and batch
  // slot b (< count) is stored to output row rows[b].
  const int* chunks;
  size_t codes_estride, scales_estride, xh_cstride, vp_cstride;
  // fused = 1: no prep kernel; each CTA forms x^ / VP of its own K-range in shared memory from these
  // inputs (the prep kernel's modes, see PrepParams).
  int fused, mode, topk, apply;
  const uint16_t* x;
  const float* gu;
  float* h_out;
  // Fused combine of the expert layer (count == nullptr: none); see ChunkCombine.
  int* cmb_count;
  const float* cmb_gate;
  float* cmb_y;
};

// Operands of this CTA: the whole call, or one chunk of routed tokens.
struct Sel {
  const uint32_t* codes;
  const uint16_t* scales;
  const uint16_t* xh;
  const float* vp;
  const int* rows;  // output row of each batch slot, or nullptr (slot b -> row b)
  int count;        // batch slots holding data
};

// false: this CTA has no chunk (the grid covers the largest possible number of chunks).  With chunks
// the record is written by the preceding kernel, so this runs after the dependent-launch wait.
__device__ __forceinline__ bool select_operands(const Params& p, Sel& s) {
  s.codes = p.codes;
  s.scales = p.scales;
  s.xh = p.xh_g;
  s.vp = p.vp_g;
  s.rows = nullptr;
  s.count = p.B;
  if (!p.chunks) return true;
  pdl_wait();
  const int z = static_cast<int>(blockIdx.z);
  if (z >= p.chunks[0]) return false;
  const int* rec = p.chunks + 1 + static_cast<size_t>(z) * (2 + p.B);
  s.codes += static_cast<size_t>(rec[0]) * p.codes_estride;
  s.scales += static_cast<size_t>(rec[0]) * p.scales_estride;
  s.xh += static_cast<size_t>(z) * p.xh_cstride;
  s.vp += static_cast<size_t>(z) * p.vp_cstride;
  s.rows = rec + 2;
  s.count = rec[1];
  return true;
}

// Where this thread's CTA and warp sit in the problem.
struct Cta {
  int warp, lane, slab, kln;
  int RT;       // rows per CTA
  int row0;     // first row of the CTA
  int u0;       // first unit of the CTA
  int k_start;  // first trit of the CTA's K-range
  int kr;       // trits in the CTA's K-range (a multiple of 128)
  int ngr;      // groups in the CTA's K-range
  int g_abs0;   // first group of the CTA's K-range
  int ua, ub;   // this warp's units [ua, ub) (empty: idle K-lane)
};

template <int PACK>
__device__ __forceinline__ Cta cta_geometry(const Params& p) {
  constexpr int UT = Geo<PACK>::UT, SLAB = Geo<PACK>::SLAB;
  Cta c;
  c.warp = threadIdx.x >> 5;
  c.lane = threadIdx.x & 31;
  c.slab = c.warp % p.rs;
  c.kln = c.warp / p.rs;
  c.RT = p.rs * SLAB;
  c.row0 = blockIdx.x * c.RT;
  c.u0 = blockIdx.y * p.kl * p.ppl;
  const int u1 = min(c.u0 + p.kl * p.ppl, p.upr);
  c.k_start = c.u0 * UT;
  c.kr = min(u1 * UT, p.K) - c.k_start;
  c.ngr = c.kr / p.G;
  c.g_abs0 = c.k_start / p.G;
  c.ua = c.u0 + c.kln * p.ppl;
  c.ub = min(c.ua + p.ppl, u1);
  return c;
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Scales of one unit of one warp (SR rows x NG groups), loaded one unit ahead into registers (two
// halves per register) and staged in the warp's own shared-memory area as halves [group][row
// position].  PERM stores rows r and r + 8 of a 16-row slab next to each other (2-bit layout).
// Rows past N and groups past the unit load a clamped (valid) address: their values feed only
// outputs that are never stored, which keeps the hot loops free of divergent branches.
template <int SR, int NG, bool PERM>
struct UnitScales {
  static constexpr int PER_LANE = SR * NG / 32;
  static_assert(PER_LANE % 2 == 0, "scales are packed in pairs");
  uint32_t v[PER_LANE / 2];

  __device__ __forceinline__ void load(const Params& p, const uint16_t* scales, int row_w0, int u, int ngp, int lane) {
#pragma unroll
    for (int j = 0; j < PER_LANE; ++j) {
      const int e = lane + 32 * j, r = e / NG, g = min(e % NG, ngp - 1), row = min(row_w0 + r, p.N - 1);
      const uint32_t h = __ldg(scales + static_cast<size_t>(row) * p.ng + u * NG + g);
      if (j & 1)
        v[j >> 1] |= h << 16;
      else
        v[j >> 1] = h;
    }
  }
  __device__ __forceinline__ void store(uint16_t* sw, int lane) const {
#pragma unroll
    for (int j = 0; j < PER_LANE; ++j) {
      const int e = lane + 32 * j, r = e / NG, g = e % NG;
      const int pos = PERM ? (((r & 7) << 1) | (r >> 3)) : r;
      sw[g * SR + pos] = static_cast<uint16_t>((j & 1) ? (v[j >> 1] >> 16) : (v[j >> 1] & 0xffffu));
    }
  }
};

// Two adjacent staged scales times the block factor, as fp32.
__device__ __forceinline__ float2 scale_pair(const uint16_t* sw, float p2) {
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(sw));
  return make_float2(f.x * p2, f.y * p2);
}

// Shared-memory setup common to both kernels: mbarriers and the prep output slice of this CTA (after
// the dependent-launch wait).
struct Bars {
  uint64_t lut, x;
  uint32_t zero[4];  // 16 zero bytes: the B operand of lanes that supply none
};

__device__ __forceinline__ void init_bars(Bars* bars) {
  if (threadIdx.x == 0) {
    mbar_init(&bars->lut, 1);
    mbar_init(&bars->x, 1);
    fence_mbar_init();
#pragma unroll
    for (int i = 0; i < 4; ++i) bars->zero[i] = 0u;
  }
  __syncthreads();
}

__device__ __forceinline__ void copy_prep_slice(const Params& p, const Cta& c, const Sel& sel, uint8_t* smem,
                                                Bars* bars) {
  if (threadIdx.x == 0) {
    const uint32_t xb = static_cast<uint32_t>(c.kr) * p.B * 2u;
    const uint32_t vb = static_cast<uint32_t>(c.ngr) * p.R * 4u;
    mbar_arrive_expect_tx(&bars->x, xb + vb);
    bulk_g2s(smem + p.xh_off, sel.xh + static_cast<size_t>(c.k_start) * p.B, xb, &bars->x);
    bulk_g2s(smem + p.vp_off, sel.vp + static_cast<size_t>(c.g_abs0) * p.R, vb, &bars->x);
  }
}

__device__ __forceinline__ void wait_bar(const Params& p, uint64_t* bar) {
  if (!mbar_wait(bar, 0) && (threadIdx.x & 31) == 0) record_error(p.status, TQ_ERR_TIMEOUT);
}

// Fused alternative to the prep kernel: the CTA's warps form x^ and VP of its K-range, one 128-block
// per warp at a time, straight into shared memory.
template <int PACK, int G>
__device__ __forceinline__ void fused_prologue(const Params& p, const Cta& c, const Sel& sel, uint8_t* smem) {
  const int blk0 = c.k_start / kFwhtBlock, nblk = c.kr / kFwhtBlock;
  const int nw = static_cast<int>(blockDim.x >> 5);
  for (int i = c.warp; i < nblk; i += nw)
    prep_block<PACK, G, 2>(p.x, p.gu, p.h_out, p.status, p.K, p.B, p.apply, p.mode, p.topk, blk0 + i, blk0, sel.count,
                           sel.rows, reinterpret_cast<uint16_t*>(smem + p.xh_off),
                           reinterpret_cast<float*>(smem + p.vp_off), c.lane);
  __syncthreads();
}

// ---------------------------------------------------------------------------------------------
// Partial sums red[kl][RT][B] (in shared memory) -> y.  K-lanes are added in lane order, then the
// cluster's CTAs in rank order through distributed shared memory.  Every thread calls this.
// ---------------------------------------------------------------------------------------------
// The expert layer's combine, fused into the down projection: count this CTA's finished slot for each
// of its tokens; for the tokens whose topk slots are now all finished, add the slots' outputs (rows of
// this tile) in slot order, weighted by the gates.  flags: shared scratch (one int per batch slot).
// The CTA's output stores precede the count (barrier, then a device-scope fence by the counting
// thread); the combining CTA fences after reading the count, before it loads the other slots' rows.
__device__ __forceinline__ void combine_tokens(const Params& p, const Cta& c, const Sel& sel, int* flags) {
  __syncthreads();  // every thread's stores (and, before this, any use of the scratch) are done
  const int tile = static_cast<int>(blockIdx.x), tiles = static_cast<int>(gridDim.x);
  if (threadIdx.x == 0) {
    __threadfence();
    for (int b = 0; b < p.B; ++b) {
      flags[b] = -1;
      if (b >= sel.count) continue;
      const int t = sel.rows[b] / p.topk;
      if (atomicAdd(p.cmb_count + static_cast<size_t>(t) * tiles + tile, 1) == p.topk - 1) flags[b] = t;
    }
    __threadfence();
  }
  __syncthreads();
  for (int b = 0; b < p.B; ++b) {
    const int t = flags[b];
    if (t < 0) continue;
    const float* gate = p.cmb_gate + static_cast<size_t>(t) * p.topk;
    for (int rl = threadIdx.x; rl < c.RT; rl += blockDim.x) {
      const int row = c.row0 + rl;
      if (row >= p.N) continue;
      float acc = 0.f;
      for (int j = 0; j < p.topk; ++j)
        acc = fmaf(gate[j], __ldcg(p.y + (static_cast<size_t>(t) * p.topk + j) * p.N + row), acc);
      p.cmb_y[static_cast<size_t>(t) * p.N + row] = acc;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0)
    for (int b = 0; b < p.B; ++b)
      if (flags[b] >= 0) p.cmb_count[static_cast<size_t>(flags[b]) * tiles + tile] = 0;
}

__device__ __forceinline__ void reduce_store(const Params& p, const Cta& c, const Sel& sel, float* red) {
  const int E = c.RT * p.B;
  if (p.kl > 1) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      float v = red[e];
      for (int l = 1; l < p.kl; ++l) v += red[l * E + e];
      red[e] = v;
    }
    __syncthreads();
  }
  const int ks = static_cast<int>(gridDim.y);
  if (ks == 1) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      const int rl = e / p.B, b = e - rl * p.B, row = c.row0 + rl;
      if (row < p.N && b < sel.count) p.y[static_cast<size_t>(sel.rows ? sel.rows[b] : b) * p.N + row] = red[e];
    }
    if (p.cmb_count) combine_tokens(p, c, sel, reinterpret_cast<int*>(red));
    return;
  }
  cluster_sync();  // every CTA's red[0] is complete
  const int rank = static_cast<int>(cluster_ctarank());
  const int chunk = (E + ks - 1) / ks;
  const int e0 = rank * chunk, e1 = min(E, e0 + chunk);
  const uint32_t base = smem_addr(red);
  for (int e = e0 + static_cast<int>(threadIdx.x); e < e1; e += blockDim.x) {
    float part[kMaxCluster];  // all remote loads in flight at once, then summed in rank order
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r)
      part[r] = r < ks ? ld_cluster_f32(cluster_map(base + 4u * static_cast<uint32_t>(e), static_cast<uint32_t>(r)))
                       : 0.f;
    float v = 0.f;
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r)
      if (r < ks) v += part[r];
    const int rl = e / p.B, b = e - rl * p.B, row = c.row0 + rl;
    if (row < p.N && b < sel.count) p.y[static_cast<size_t>(sel.rows ? sel.rows[b] : b) * p.N + row] = v;
  }
  cluster_sync();  // keep this CTA's shared memory alive until the peers have read it; and every
                   // rank's stores precede the combine count of rank 0
  if (p.cmb_count && rank == 0) combine_tokens(p, c, sel, reinterpret_cast<int*>(red));
}

// ---------------------------------------------------------------------------------------------
// 2-bit, shared-row layout.  NT = number of 8-column batch tiles (1: B <= 8, 2: B <= 16).
// ---------------------------------------------------------------------------------------------
template <int G, int NT>
__global__ void __launch_bounds__(kMaxThreads) gemv_2b_kernel(const __grid_constant__ Params p) {
  constexpr int WPT = G / 64;          // words per thread per group per row
  constexpr int GPU = 512 / G;         // groups per unit
  constexpr int D = G == 128 ? 6 : 8;  // ring of groups in flight
  extern __shared__ __align__(16) uint8_t smem[];
  pdl_launch_dependents();
  const Cta c = cta_geometry<TQ_PACK_2BIT>(p);
  Sel sel;
  if (!select_operands(p, sel)) return;
  Bars* bars = reinterpret_cast<Bars*>(smem + p.bar_off);
  init_bars(bars);
  const int g = c.lane >> 2, q = c.lane & 3;
  const int rg = c.row0 + c.slab * 16 + g, rg8 = rg + 8;
  const bool vg = rg < p.N, vg8 = rg8 < p.N;  // rows past N compute on row 0 and are not stored
  // this warp's groups, relative to the CTA's first group
  const int gl_a = (c.ua - c.u0) * GPU;
  const int gl_b = max(gl_a, min((c.ub - c.u0) * GPU, c.ngr));
  const uint32_t* cg = sel.codes + static_cast<size_t>(vg ? rg : 0) * p.P + c.k_start / 16 + WPT * q;
  const uint32_t* cg8 = sel.codes + static_cast<size_t>(vg8 ? rg8 : 0) * p.P + c.k_start / 16 + WPT * q;
  const int row_w0 = c.row0 + c.slab * 16;
  uint16_t* sw = reinterpret_cast<uint16_t*>(smem + p.sw_off) + c.warp * (GPU * 16);
  UnitScales<16, GPU, true> us;
  auto unit_groups = [&](int u) { return min(GPU, (min((u + 1) * 512, p.K) - u * 512) / G); };
  uint32_t buf[D][2 * WPT];
#pragma unroll
  for (int d = 0; d < D; ++d)
#pragma unroll
    for (int u = 0; u < 2 * WPT; ++u) buf[d][u] = kB2Zero;
  // rows past N read row 0 (their outputs are not stored); groups past the range re-read the last
  auto fetch = [&](int gl, int slot) {
    const int gc = min(gl, gl_b - 1);
    if (WPT == 2) {  // words 2q, 2q + 1 of the group: one 8-byte load per row (rows and offsets are even)
      const uint2 a = __ldg(reinterpret_cast<const uint2*>(cg + gc * (G / 16)));
      const uint2 b = __ldg(reinterpret_cast<const uint2*>(cg8 + gc * (G / 16)));
      buf[slot][0] = a.x;
      buf[slot][1] = a.y;
      buf[slot][WPT] = b.x;
      buf[slot][WPT + 1] = b.y;
    } else {
#pragma unroll
      for (int u = 0; u < WPT; ++u) {
        buf[slot][u] = __ldg(cg + gc * (G / 16) + u);
        buf[slot][WPT + u] = __ldg(cg8 + gc * (G / 16) + u);
      }
    }
  };
  auto prime = [&]() {
    if (gl_a < gl_b) {
#pragma unroll
      for (int d = 0; d < D - 1; ++d) fetch(gl_a + d, d);
      us.load(p, sel.scales, row_w0, c.ua, unit_groups(c.ua), c.lane);
    }
  };
  if (kPrefetchL2 && p.early && gl_a < gl_b && c.lane < 16 && row_w0 + c.lane < p.N)
    bulk_prefetch_l2(sel.codes + static_cast<size_t>(row_w0 + c.lane) * p.P + c.k_start / 16 + gl_a * (G / 16),
                     static_cast<uint32_t>(gl_b - gl_a) * (G / 4));
  if (p.early) prime();
  pdl_wait();
  if (!p.fused) copy_prep_slice(p, c, sel, smem, bars);
  if (!p.early) prime();
  if (p.fused) {
    fused_prologue<TQ_PACK_2BIT, G>(p, c, sel, smem);
  } else {
    wait_bar(p, &bars->x);
  }

  const uint32_t* xh = reinterpret_cast<const uint32_t*>(smem + p.xh_off);
  const float* V = reinterpret_cast<const float*>(smem + p.vp_off);
  float acc[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[t][i] = 0.f;

  for (int gi0 = gl_a; gi0 < gl_b; gi0 += D) {
#pragma unroll
    for (int d = 0; d < D; ++d) {
      const int gl = gi0 + d;
      if (gl >= gl_b) break;
      fetch(gl + D - 1, (d + D - 1) % D);
      const int gu = (gl - gl_a) & (GPU - 1);  // group within the unit
      if (gu == 0) {  // a new unit: its scales into the warp's area, the next unit's into registers
        const int u = c.ua + (gl - gl_a) / GPU;
        __syncwarp();
        us.store(sw, c.lane);
        __syncwarp();
        if (u + 1 < c.ub) us.load(p, sel.scales, row_w0, u + 1, unit_groups(u + 1), c.lane);
      }
      float cc[NT][4];
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        // batch columns past B read a valid slot: they land only in columns that are not stored
        const int b = min(8 * t + 2 * q, p.R - 2);
        const float2 v = *reinterpret_cast<const float2*>(V + gl * p.R + b);
        cc[t][0] = v.x;
        cc[t][1] = v.y;
        cc[t][2] = v.x;
        cc[t][3] = v.y;
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
        uint4 bp[NT];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const int b = min(8 * t + g, p.B - 1);  // columns past B: not stored
            if ((jj & 1) == 0)
              bp[t] = *reinterpret_cast<const uint4*>(xh + ((((gl * WPT + u) * 2 + (jj >> 1)) * p.B + b) * 4 + q) * 4);
            const uint32_t b0 = (jj & 1) ? bp[t].z : bp[t].x, b1 = (jj & 1) ? bp[t].w : bp[t].y;
            mma16816(cc[t], pr[2 * jj], pr8[2 * jj], pr[2 * jj + 1], pr8[2 * jj + 1], b0, b1);
          }
        }
      }
      const float2 m = scale_pair(sw + gu * 16 + 2 * g, V[gl * p.R + p.R - 1]);  // rows g, g + 8
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        acc[t][0] = fmaf(m.x, cc[t][0], acc[t][0]);
        acc[t][1] = fmaf(m.x, cc[t][1], acc[t][1]);
        acc[t][2] = fmaf(m.y, cc[t][2], acc[t][2]);
        acc[t][3] = fmaf(m.y, cc[t][3], acc[t][3]);
      }
    }
  }

  __syncthreads();  // the partial sums reuse the x^ region
  float* red = reinterpret_cast<float*>(smem);
  const int rl = c.slab * 16 + g;
  float* r0 = red + (c.kln * c.RT + rl) * p.B;
  float* r8 = red + (c.kln * c.RT + rl + 8) * p.B;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int b = 8 * t + 2 * q;
    if (b < p.B) {
      r0[b] = acc[t][0];
      r8[b] = acc[t][2];
    }
    if (b + 1 < p.B) {
      r0[b + 1] = acc[t][1];
      r8[b + 1] = acc[t][3];
    }
  }
  __syncthreads();
  reduce_store(p, c, sel, red);
}

// ---------------------------------------------------------------------------------------------
// base-3, column layout.  NT = number of 2-row batch tiles (ceil(B / 2)).
// Thread (g, q) owns rows R = r0 + 4g + q and R + 32 of its warp's 64-row slab.
// ---------------------------------------------------------------------------------------------

template <int G, int NT, bool FULL>
__device__ __forceinline__ void b3_unit(const Params& p, const Cta& c, int u, int ngp, const uint4* __restrict__ cR,
                                        const uint4* __restrict__ cR2, int s_last, uint4 (&ra)[4], uint4 (&rb)[4],
                                        const uint32_t* __restrict__ lutA, const uint32_t* __restrict__ lutB,
                                        const uint32_t* const (&bptr)[NT], const int (&bstr)[NT],
                                        const float* __restrict__ V, const uint16_t* __restrict__ swr,
                                        float (&acc)[NT][4]) {
  constexpr int GP = G / 2;     // pairs per group
  constexpr int GPS = 640 / G;  // groups per unit
  const int q = c.lane & 3;
  const int bq = q >> 1;    // batch within a tile held by this thread's accumulators
  const int ul = u - c.u0;  // unit index within the CTA
  float cc[NT][4];
  uint4 bp[NT];
#pragma unroll
  for (int st = 0; st < 8; ++st) {
    if (!FULL && (st * 80) / G >= ngp) break;
    if (p.v8) {  // 32-byte loads of two steps, two steps ahead (past this warp's range: its last two)
      if ((st & 1) == 0) {
        const int s = min(u * 8 + st + 2, s_last - 1);
        ldg_v8(cR + s, ra[(st + 2) & 3], ra[(st + 3) & 3]);
        ldg_v8(cR2 + s, rb[(st + 2) & 3], rb[(st + 3) & 3]);
      }
    } else {  // keep the ring three steps ahead (past this warp's range: re-read its last step)
      const int s = min(u * 8 + st + 3, s_last);
      ra[(st + 3) & 3] = __ldg(cR + s);
      rb[(st + 3) & 3] = __ldg(cR2 + s);
    }
    const uint4 cur = ra[st & 3], cur2 = rb[st & 3];
    const uint32_t wr[4] = {cur.x, cur.y, cur.z, cur.w};
    const uint32_t wr2[4] = {cur2.x, cur2.y, cur2.z, cur2.w};
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      uint32_t La[4], Lb[4];
      b3_chunks<32>(wr[wi], lutA, lutB, La);
      b3_chunks<32>(wr2[wi], lutA, lutB, Lb);
#pragma unroll
      for (int mj = 0; mj < 5; ++mj) {
        const int pair = (st * 4 + wi) * 10 + 2 * mj;  // first pair of this MMA within the unit
        const int gl = pair / GP;
        if (!FULL && gl >= ngp) break;
        const int gla = ul * GPS + gl;  // group index within the CTA
        if (pair % GP == 0) {
          // new group: accumulators start at -2^-16 * sum(x^) of the group for their batch
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const float v0 = V[gla * p.R + min(2 * t + bq, p.B - 1)];  // columns past B are not stored
            cc[t][0] = v0;
            cc[t][1] = v0;
            cc[t][2] = v0;
            cc[t][3] = v0;
          }
        }
        const int mloc = (st * 4 + wi) * 5 + mj;  // MMA index within the unit
        if ((mloc & 1) == 0) {
          const int mp = ul * 80 + (mloc >> 1);  // MMA pair index within the CTA
#pragma unroll
          for (int t = 0; t < NT; ++t) bp[t] = *reinterpret_cast<const uint4*>(bptr[t] + mp * bstr[t]);
        }
        const uint32_t a0 = b3_pair(La, 2 * mj), a2 = b3_pair(La, 2 * mj + 1);
        const uint32_t a1 = b3_pair(Lb, 2 * mj), a3 = b3_pair(Lb, 2 * mj + 1);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const uint32_t b0 = (mloc & 1) ? bp[t].z : bp[t].x, b1 = (mloc & 1) ? bp[t].w : bp[t].y;
          mma16816(cc[t], a0, a1, a2, a3, b0, b1);
        }
        if ((pair + 2) % GP == 0) {
          const float p2 = V[gla * p.R + p.R - 1];
          const float2 m01 = scale_pair(swr + gl * 64, p2);       // rows of the accumulators 0, 1
          const float2 m23 = scale_pair(swr + gl * 64 + 32, p2);  // rows + 32
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            acc[t][0] = fmaf(m01.x, cc[t][0], acc[t][0]);
            acc[t][1] = fmaf(m01.y, cc[t][1], acc[t][1]);
            acc[t][2] = fmaf(m23.x, cc[t][2], acc[t][2]);
            acc[t][3] = fmaf(m23.y, cc[t][3], acc[t][3]);
          }
        }
      }
    }
  }
}

template <int G, int NT>
__global__ void __launch_bounds__(kMaxThreads) gemv_b3_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(16) uint8_t smem[];
  pdl_launch_dependents();
  const Cta c = cta_geometry<TQ_PACK_B3>(p);
  Sel sel;
  if (!select_operands(p, sel)) return;
  Bars* bars = reinterpret_cast<Bars*>(smem + p.bar_off);
  init_bars(bars);
  const int g = c.lane >> 2, q = c.lane & 3;
  if (threadIdx.x == 0) {  // the chunk table (constant data of this library)
    mbar_arrive_expect_tx(&bars->lut, kLutBytes);
    bulk_g2s(smem, &g_lut, kLutBytes, &bars->lut);
  }
  // rows past N compute on row 0 and are not stored
  const int R = c.row0 + c.slab * 64 + c.lane, R2 = R + 32;
  const uint4* cR = reinterpret_cast<const uint4*>(sel.codes + static_cast<size_t>(R < p.N ? R : 0) * p.P);
  const uint4* cR2 = reinterpret_cast<const uint4*>(sel.codes + static_cast<size_t>(R2 < p.N ? R2 : 0) * p.P);
  const int s_begin = c.ua * 8;
  const int s_last = min(c.ub * 8, p.P >> 2) - 1;  // this warp's last 4-word step (a row has P / 4)
  constexpr int GPS = 640 / G;
  const int row_w0 = c.row0 + c.slab * 64;
  uint16_t* sw = reinterpret_cast<uint16_t*>(smem + p.sw_off) + c.warp * (GPS * 64);
  UnitScales<64, GPS, false> us;
  auto unit_groups = [&](int u) { return min(GPS, (min((u + 1) * 640, p.K) - u * 640) / G); };
  uint4 ra[4], rb[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    ra[i] = make_uint4(kB3Zero, kB3Zero, kB3Zero, kB3Zero);
    rb[i] = ra[i];
  }
  auto prime = [&]() {
    if (c.ua < c.ub) {
      if (p.v8) {
#pragma unroll
        for (int i = 0; i < 4; i += 2) {
          ldg_v8(cR + min(s_begin + i, s_last - 1), ra[i], ra[i + 1]);
          ldg_v8(cR2 + min(s_begin + i, s_last - 1), rb[i], rb[i + 1]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 3; ++i) {
          ra[i] = __ldg(cR + min(s_begin + i, s_last));
          rb[i] = __ldg(cR2 + min(s_begin + i, s_last));
        }
      }
      us.load(p, sel.scales, row_w0, c.ua, unit_groups(c.ua), c.lane);
    }
  };
  if (kPrefetchL2 && p.early && c.ua < c.ub) {
    const uint32_t bytes = static_cast<uint32_t>(min(c.ub * 8, p.P >> 2) - s_begin) * 16u;
    if (R < p.N) bulk_prefetch_l2(cR + s_begin, bytes);
    if (R2 < p.N) bulk_prefetch_l2(cR2 + s_begin, bytes);
  }
  if (p.early) prime();
  pdl_wait();
  if (!p.fused) copy_prep_slice(p, c, sel, smem, bars);
  if (!p.early) prime();
  if (p.fused) {
    fused_prologue<TQ_PACK_B3, G>(p, c, sel, smem);
  } else {
    wait_bar(p, &bars->x);
  }
  wait_bar(p, &bars->lut);

  const uint32_t* lutA = reinterpret_cast<const uint32_t*>(smem) + c.lane;
  const uint32_t* lutB = lutA + 243 * 32;
  const uint32_t* xh = reinterpret_cast<const uint32_t*>(smem + p.xh_off);
  const float* V = reinterpret_cast<const float*>(smem + p.vp_off);
  // B operand: lane (g, q) supplies batch 2t + g/4 of tile t when g % 4 == q, else 16 zero bytes;
  // batch rows past B read row B - 1 (their columns are not stored)
  const uint32_t* bptr[NT];
  int bstr[NT];
  {
    const bool bsup = (g & 3) == q;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      bptr[t] = bsup ? xh + min(2 * t + (g >> 2), p.B - 1) * 4 : bars->zero;
      bstr[t] = bsup ? p.B * 4 : 0;  // words per MMA pair: 4 halves per (pair, batch row) x 2 MMAs
    }
  }
  // accumulator rows: threads (g, cq) and (g, cq + 1) of the slab, R and R + 32
  const int cq = (2 * q) & 3;
  const int rl0 = c.slab * 64 + 4 * g + cq;
  const uint16_t* swr = sw + 4 * g + cq;  // this thread's accumulator rows within the warp's slab
  float acc[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[t][i] = 0.f;
  for (int u = c.ua; u < c.ub; ++u) {
    const int ngp = unit_groups(u);
    // this unit's scales into the warp's area, the next unit's into registers
    __syncwarp();
    us.store(sw, c.lane);
    __syncwarp();
    if (u + 1 < c.ub) us.load(p, sel.scales, row_w0, u + 1, unit_groups(u + 1), c.lane);
    if (ngp == GPS)
      b3_unit<G, NT, true>(p, c, u, ngp, cR, cR2, s_last, ra, rb, lutA, lutB, bptr, bstr, V, swr, acc);
    else
      b3_unit<G, NT, false>(p, c, u, ngp, cR, cR2, s_last, ra, rb, lutA, lutB, bptr, bstr, V, swr, acc);
  }

  __syncthreads();  // the partial sums reuse the table / x^ region
  float* red = reinterpret_cast<float*>(smem);
  const int rows[4] = {rl0, rl0 + 1, rl0 + 32, rl0 + 33};
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int b = 2 * t + (q >> 1);
    if (b < p.B) {
#pragma unroll
      for (int i = 0; i < 4; ++i) red[(c.kln * c.RT + rows[i]) * p.B + b] = acc[t][i];
    }
  }
  __syncthreads();
  reduce_store(p, c, sel, red);
}

// ---------------------------------------------------------------------------------------------
// 3-bit codes, column layout (the base-3 kernel's thread / row / accumulator arrangement).
// A 64-code block is 7 words; word i < 6 yields five operand registers and word 6 two, 32 in all:
// register j < 3 of a word is w & (7 << 3j | 7 << (16 + 3j)) (codes of slots j and j + 5 at bit 3j of
// their halves), j = 3, 4 take the same mask of w >> 8 (bit 3j - 8).  A digit d at bit p of a zero-
// exponent half is d * 2^(p - 24); the prep kernel folds 2^(8 - p) into the activations and the
// offset q = d - 4 into the group's starting value.  MMA m of a block takes registers 2m, 2m + 1 of
// both rows of the thread, so a block is 16 MMAs and a group 16 (G = 64) or 32 (G = 128).
// A unit is 28 words (7 steps of four).  A warp's codes arrive one unit at a time as a 2-D TMA box
// (its 64 rows x 112 bytes) in a two-slot shared-memory ring, the next unit in flight while this one
// is decoded: one request per box instead of 32 scattered 16-byte requests per warp-wide load (the
// L1 would take those one 128-byte line at a time).  Lane l reads rows l and l + 32 of the box (a row
// stride of 112 bytes keeps 16-byte reads free of bank conflicts).
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t q3_reg(uint32_t w, int i, int j) {
  if (i == 6) return w & (j == 0 ? 0x00070007u : 0x00380038u);
  return j < 3 ? (w & (0x00070007u << (3 * j))) : ((w >> 8) & (0x00070007u << (3 * j - 8)));
}

constexpr int kQ3Steps = 7;                       // 16-byte steps per unit
constexpr int kQ3UnitWords = 28;
constexpr uint32_t kQ3Box = 64u * kQ3UnitWords * 4u;  // one unit of the warp's 64 rows: 7168 bytes
constexpr uint32_t kQ3WarpRing = 2u * kQ3Box + 128u;  // two slots, then the two slots' mbarriers

template <int G, int NT, bool FULL>
__device__ __forceinline__ void q3_unit(const Params& p, const Cta& c, int u, int ngp,
                                        const uint4* __restrict__ box, const uint32_t* const (&bptr)[NT],
                                        const int (&bstr)[NT], const float* __restrict__ V,
                                        const uint16_t* __restrict__ swr, float (&acc)[NT][4]) {
  constexpr int GM = G / 4;     // MMAs per group
  constexpr int GPS = 256 / G;  // groups per unit
  const int bq = (c.lane & 3) >> 1;
  const int ul = u - c.u0;
  float cc[NT][4];
  uint4 bp[NT];
  uint32_t ea = 0u, eb = 0u;  // the even register of the MMA being formed (rows R, R + 32)
#pragma unroll
  for (int st = 0; st < kQ3Steps; ++st) {
    const uint4 cur = box[st], cur2 = box[32 * kQ3Steps + st];  // rows l and l + 32 of the box
    const uint32_t wr[4] = {cur.x, cur.y, cur.z, cur.w};
    const uint32_t wr2[4] = {cur2.x, cur2.y, cur2.z, cur2.w};
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      const int w = 4 * st + wi, blk = w / 7, i = w % 7;
#pragma unroll
      for (int j = 0; j < (i < 6 ? 5 : 2); ++j) {
        const int reg = 5 * i + j;  // operand register of the block
        const uint32_t xa = q3_reg(wr[wi], i, j), xb = q3_reg(wr2[wi], i, j);
        if ((reg & 1) == 0) {
          ea = xa;
          eb = xb;
          continue;
        }
        const int mloc = blk * 16 + (reg >> 1);  // MMA index within the unit
        const int gl = mloc / GM;
        if (!FULL && gl >= ngp) continue;
        const int gla = ul * GPS + gl;  // group index within the CTA
        if (mloc % GM == 0) {
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const float v0 = V[gla * p.R + min(2 * t + bq, p.B - 1)];  // columns past B are not stored
            cc[t][0] = v0;
            cc[t][1] = v0;
            cc[t][2] = v0;
            cc[t][3] = v0;
          }
        }
        if ((mloc & 1) == 0) {
          const int mp = ul * 32 + (mloc >> 1);  // MMA pair index within the CTA
#pragma unroll
          for (int t = 0; t < NT; ++t) bp[t] = *reinterpret_cast<const uint4*>(bptr[t] + mp * bstr[t]);
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const uint32_t b0 = (mloc & 1) ? bp[t].z : bp[t].x, b1 = (mloc & 1) ? bp[t].w : bp[t].y;
          mma16816(cc[t], ea, eb, xa, xb, b0, b1);
        }
        if ((mloc + 1) % GM == 0) {
          const float p2 = V[gla * p.R + p.R - 1];
          const float2 m01 = scale_pair(swr + gl * 64, p2);
          const float2 m23 = scale_pair(swr + gl * 64 + 32, p2);
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            acc[t][0] = fmaf(m01.x, cc[t][0], acc[t][0]);
            acc[t][1] = fmaf(m01.y, cc[t][1], acc[t][1]);
            acc[t][2] = fmaf(m23.x, cc[t][2], acc[t][2]);
            acc[t][3] = fmaf(m23.y, cc[t][3], acc[t][3]);
          }
        }
      }
    }
  }
}

template <int G, int NT>
__global__ void __launch_bounds__(kMaxThreads) gemv_q3_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(16) uint8_t smem[];
  pdl_launch_dependents();
  const Cta c = cta_geometry<TQ_PACK_3BIT>(p);
  Sel sel;
  if (!select_operands(p, sel)) return;
  Bars* bars = reinterpret_cast<Bars*>(smem + p.bar_off);
  init_bars(bars);
  const int g = c.lane >> 2, q = c.lane & 3;
  // rows past N are zero-filled by the TMA box, computed and not stored
  constexpr int GPS = 256 / G;
  const int row_w0 = c.row0 + c.slab * 64;
  uint16_t* sw = reinterpret_cast<uint16_t*>(smem + p.sw_off) + c.warp * (GPS * 64);
  UnitScales<64, GPS, false> us;
  auto unit_groups = [&](int u) { return min(GPS, (min((u + 1) * 256, p.K) - u * 256) / G); };
  uint8_t* wring = smem + p.ring_off + c.warp * kQ3WarpRing;
  uint64_t* ubar = reinterpret_cast<uint64_t*>(wring + 2 * kQ3Box);
  if (c.lane == 0) {
    mbar_init(&ubar[0], 1);
    mbar_init(&ubar[1], 1);
    fence_mbar_init();
  }
  __syncwarp();
  auto issue = [&](int u) {  // unit u of the warp's rows into slot (u - ua) & 1
    if (c.lane == 0) {
      const int slot = (u - c.ua) & 1;
      mbar_arrive_expect_tx(&ubar[slot], kQ3Box);
      tma_load_2d(wring + slot * kQ3Box, &p.tm, kQ3UnitWords * u, row_w0, &ubar[slot]);
    }
  };
  auto prime = [&]() {
    if (c.ua < c.ub) {
      issue(c.ua);
      if (c.ua + 1 < c.ub) issue(c.ua + 1);
      us.load(p, sel.scales, row_w0, c.ua, unit_groups(c.ua), c.lane);
    }
  };
  if (p.early) prime();
  pdl_wait();
  if (!p.fused) copy_prep_slice(p, c, sel, smem, bars);
  if (!p.early) prime();
  if (p.fused) {
    fused_prologue<TQ_PACK_3BIT, G>(p, c, sel, smem);
  } else {
    wait_bar(p, &bars->x);
  }

  const uint32_t* xh = reinterpret_cast<const uint32_t*>(smem + p.xh_off);
  const float* V = reinterpret_cast<const float*>(smem + p.vp_off);
  // B operand: lane (g, q) supplies batch 2t + g/4 of tile t when g % 4 == q, else 16 zero bytes
  const uint32_t* bptr[NT];
  int bstr[NT];
  {
    const bool bsup = (g & 3) == q;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      bptr[t] = bsup ? xh + min(2 * t + (g >> 2), p.B - 1) * 4 : bars->zero;
      bstr[t] = bsup ? p.B * 4 : 0;
    }
  }
  const int cq = (2 * q) & 3;
  const int rl0 = c.slab * 64 + 4 * g + cq;
  const uint16_t* swr = sw + 4 * g + cq;
  float acc[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[t][i] = 0.f;
  for (int u = c.ua; u < c.ub; ++u) {
    const int ngp = unit_groups(u);
    __syncwarp();
    us.store(sw, c.lane);
    __syncwarp();
    if (u + 1 < c.ub) us.load(p, sel.scales, row_w0, u + 1, unit_groups(u + 1), c.lane);
    const int slot = (u - c.ua) & 1;
    if (!mbar_wait(&ubar[slot], ((u - c.ua) >> 1) & 1) && c.lane == 0) record_error(p.status, TQ_ERR_TIMEOUT);
    const uint4* box = reinterpret_cast<const uint4*>(wring + slot * kQ3Box) + c.lane * kQ3Steps;
    if (ngp == GPS)
      q3_unit<G, NT, true>(p, c, u, ngp, box, bptr, bstr, V, swr, acc);
    else
      q3_unit<G, NT, false>(p, c, u, ngp, box, bptr, bstr, V, swr, acc);
    if (u + 2 < c.ub) {  // the slot is free once every lane has read it
      __syncwarp();
      fence_proxy_async_smem();
      issue(u + 2);
    }
  }

  __syncthreads();  // the partial sums reuse the x^ region
  float* red = reinterpret_cast<float*>(smem);
  const int rows[4] = {rl0, rl0 + 1, rl0 + 32, rl0 + 33};
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int b = 2 * t + (q >> 1);
    if (b < p.B) {
#pragma unroll
      for (int i = 0; i < 4; ++i) red[(c.kln * c.RT + rows[i]) * p.B + b] = acc[t][i];
    }
  }
  __syncthreads();
  reduce_store(p, c, sel, red);
}

// ---------------------------------------------------------------------------------------------
// 2-bit dense decode, streamed ("stream" kernel).  One CTA per SM: nw consumer warps, each owning a
// 16-row slab of the CTA's 16*nw-row block, and one producer warp whose elected lane streams the
// block's codes through a ring of S shared-memory stages with 2-D TMA (32 words = 512 trits x 16*nw
// rows per stage, 128-byte swizzle, L2 evict-first).  The activations are requested first after the
// dependent-launch wait (kEarlyStages code stages may go out before it with static weights).
// K may be split over the ks CTAs of a cluster: the other ranks push their partial sums into the
// leader's shared memory and arrive on the cluster barrier; the leader adds them in rank order.
// The activations of the CTA's K-range are transformed in the CTA (batch <= kStreamFuseMaxB) or
// bulk-copied from the prep kernel's output.  Decode, MMA and scale folding are those of the
// shared-row layout above.
// ---------------------------------------------------------------------------------------------
struct SParams {
  const uint16_t* scales;
  const uint16_t* x;     // bf16 rows [B][K] (fused prologue)
  const uint16_t* xh_g;  // prep kernel output (not fused)
  const float* vp_g;
  float* y;
  int* status;
  int N, K, ng, B, R;
  int gpc;  // groups per CTA K-range (whole 128-blocks)
  int nw;   // consumer warps
  int S;    // ring stages
  int fused, early, apply;
  uint32_t stage_bytes;
  uint32_t xh_off, vp_off, sc_off, red_off, bar_off, xs_off;  // offsets from the 1024-aligned base
};

// The scales of one stage of one warp (16 rows x NG groups starting at absolute group ga), held two
// halves per register and staged as halves [group][row position] (rows r and r + 8 adjacent).
template <int NG>
struct StageScales {
  static constexpr int PER_LANE = 16 * NG / 32;
  uint32_t v[PER_LANE / 2];
  __device__ __forceinline__ void load(const uint16_t* scales, int N, int ng, int row_w0, int ga, int ngs, int lane) {
#pragma unroll
    for (int j = 0; j < PER_LANE; ++j) {
      const int e = lane + 32 * j, r = e / NG, g = min(e % NG, ngs - 1), row = min(row_w0 + r, N - 1);
      const uint32_t h = __ldg(scales + static_cast<size_t>(row) * ng + ga + g);
      if (j & 1)
        v[j >> 1] |= h << 16;
      else
        v[j >> 1] = h;
    }
  }
  __device__ __forceinline__ void store(uint16_t* sw, int lane) const {
#pragma unroll
    for (int j = 0; j < PER_LANE; ++j) {
      const int e = lane + 32 * j, r = e / NG, g = e % NG;
      sw[g * 16 + (((r & 7) << 1) | (r >> 3))] = static_cast<uint16_t>((j & 1) ? (v[j >> 1] >> 16) : (v[j >> 1] & 0xffffu));
    }
  }
};

template <int G, int NT>
__global__ void __launch_bounds__(17 * 32) gemv_2b_stream_kernel(const __grid_constant__ CUtensorMap tm,
                                                                  const __grid_constant__ SParams p) {
  constexpr int WPT = G / 64;   // words per thread per group per row
  constexpr int GPS = 512 / G;  // groups per stage
  constexpr int MAXB = 8 * NT;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  pdl_launch_dependents();
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
  const int nw = p.nw, BR = 16 * nw;
  const int row0 = static_cast<int>(blockIdx.x) * BR;
  const int g0 = static_cast<int>(blockIdx.y) * p.gpc;
  const int ngc = min(p.gpc, p.ng - g0);  // groups of this CTA (> 0)
  const int nst = (ngc + GPS - 1) / GPS;
  const int kw0 = g0 * (G / 16);          // first code word of the K-range
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  uint64_t* empty = full + p.S;
  uint64_t* xbar = empty + p.S;
  const int ks = static_cast<int>(gridDim.y);
  if (threadIdx.x == 0) {
    for (int i = 0; i < p.S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], nw);
    }
    mbar_init(xbar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (ks > 1) cluster_arrive_relaxed();  // waited on before the first remote access

  if (warp == nw) {  // ---------------- producer ----------------
    if (lane == 0) tma_prefetch_desc(&tm);
    // fused: the CTA's columns of x (rows of kr bf16 values), once the preceding kernel is done
    auto copy_x = [&]() {
      const uint32_t rb = static_cast<uint32_t>(ngc) * G * 2u;
      mbar_arrive_expect_tx(xbar, rb * p.B);
      for (int b = 0; b < p.B; ++b)
        bulk_g2s(smem + p.xs_off + static_cast<size_t>(b) * rb, p.x + static_cast<size_t>(b) * p.K + g0 * G, rb,
                 xbar);
    };
    // not fused: this CTA's slices of the prep kernel's output
    auto copy_slices = [&]() {
      const uint32_t xb = static_cast<uint32_t>(ngc) * G * p.B * 2u;
      const uint32_t vb = static_cast<uint32_t>(ngc) * p.R * 4u;
      mbar_arrive_expect_tx(xbar, xb + vb);
      bulk_g2s(smem + p.xh_off, p.xh_g + static_cast<size_t>(g0) * G * p.B, xb, xbar);
      bulk_g2s(smem + p.vp_off, p.vp_g + static_cast<size_t>(g0) * p.R, vb, xbar);
    };
    auto wait_and_copy = [&]() {
      pdl_wait();
      if (lane == 0) {
        if (p.fused)
          copy_x();
        else
          copy_slices();
      }
    };
    const uint64_t pol = l2_evict_first_policy();  // codes are read once per call
    // Static weights: the first kEarlyStages stages go out before the dependent-launch wait; the
    // activations are requested next, ahead of the rest of the ring, so that they do not queue
    // behind the whole ring's weight traffic.
    const int early_st = p.early ? min(nst, kEarlyStages) : 0;
    for (int s = 0; s < nst; ++s) {
      const int slot = s % p.S;
      if (s == early_st) wait_and_copy();
      if (s >= p.S && !mbar_wait(&empty[slot], ((s / p.S) + 1) & 1)) {
        if (lane == 0) record_error(p.status, TQ_ERR_TIMEOUT);
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&full[slot], p.stage_bytes);
        tma_load_2d_hint(smem + static_cast<size_t>(slot) * p.stage_bytes, &tm, kw0 + 32 * s, row0, &full[slot], pol);
      }
    }
    if (early_st == nst) wait_and_copy();
    __syncwarp();
  } else {  // ---------------- consumers ----------------
    const int g = lane >> 2, q = lane & 3;
    const int row_w0 = row0 + 16 * warp;
    uint16_t* sw = reinterpret_cast<uint16_t*>(smem + p.sc_off) + warp * (GPS * 16);
    // scales two stages ahead: stage s uses usA (s even) or usB (s odd)
    StageScales<GPS> usA, usB;
    auto load_scales = [&](StageScales<GPS>& us, int s) {
      us.load(p.scales, p.N, p.ng, row_w0, g0 + s * GPS, min(GPS, ngc - s * GPS), lane);
    };
    if (!p.early) pdl_wait();
    load_scales(usA, 0);
    if (nst > 1) load_scales(usB, 1);
    if (p.early) pdl_wait();
    uint16_t* xhs = reinterpret_cast<uint16_t*>(smem + p.xh_off);
    float* vps = reinterpret_cast<float*>(smem + p.vp_off);
    const int k_start = g0 * G, kr = ngc * G;
    if (p.fused) {
      if (!mbar_wait(xbar, 0) && lane == 0) record_error(p.status, TQ_ERR_TIMEOUT);
      const int blk0 = k_start / kFwhtBlock, nblk = kr / kFwhtBlock;
      const uint16_t* xs = reinterpret_cast<const uint16_t*>(smem + p.xs_off);
      for (int i = warp; i < nblk; i += nw)
        prep_block<TQ_PACK_2BIT, G, MAXB, true>(xs, nullptr, nullptr, p.status, p.K, p.B, p.apply, 0, 0, blk0 + i,
                                                blk0, p.B, nullptr, xhs, vps, lane, kr);
      named_bar_sync(1, 32 * nw);
    } else {
      if (!mbar_wait(xbar, 0) && lane == 0) record_error(p.status, TQ_ERR_TIMEOUT);
    }
    const uint32_t* xh = reinterpret_cast<const uint32_t*>(xhs);
    const float* V = vps;
    float acc[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[t][i] = 0.f;
    // this thread's bytes within a stage row: words WPT*q .. of each group, 128-byte swizzle
    const uint32_t rA = static_cast<uint32_t>(16 * warp + g) * 128u, rB = rA + 8u * 128u;
    auto stage = [&](int s, StageScales<GPS>& us) {
      const int slot = s % p.S;
      const int ngs = min(GPS, ngc - s * GPS);
      __syncwarp();
      us.store(sw, lane);
      __syncwarp();
      if (s + 2 < nst) load_scales(us, s + 2);
      if (!mbar_wait(&full[slot], (s / p.S) & 1) && lane == 0) record_error(p.status, TQ_ERR_TIMEOUT);
      const uint8_t* st = smem + static_cast<size_t>(slot) * p.stage_bytes;
#pragma unroll
      for (int j = 0; j < GPS; ++j) {
        if (j >= ngs) break;
        const int gl = s * GPS + j;  // group within the CTA's K-range
        uint32_t w[2 * WPT];
        if (WPT == 2) {
          const uint32_t off = (static_cast<uint32_t>((2 * j + (q >> 1)) ^ g) << 4) + 8u * (q & 1);
          const uint2 a = *reinterpret_cast<const uint2*>(st + rA + off);
          const uint2 b = *reinterpret_cast<const uint2*>(st + rB + off);
          w[0] = a.x;
          w[1] = a.y;
          w[2] = b.x;
          w[3] = b.y;
        } else {
          const uint32_t off = (static_cast<uint32_t>(j ^ g) << 4) + 4u * q;
          w[0] = *reinterpret_cast<const uint32_t*>(st + rA + off);
          w[1] = *reinterpret_cast<const uint32_t*>(st + rB + off);
        }
        float cc[NT][4];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const int b = min(8 * t + 2 * q, p.R - 2);  // columns past B read a valid slot, never stored
          const float2 v = *reinterpret_cast<const float2*>(V + gl * p.R + b);
          cc[t][0] = v.x;
          cc[t][1] = v.y;
          cc[t][2] = v.x;
          cc[t][3] = v.y;
        }
#pragma unroll
        for (int u = 0; u < WPT; ++u) {
          const uint32_t wa = w[u], w8 = w[WPT + u];
          const uint32_t w2 = wa >> 10, w82 = w8 >> 10;
          uint32_t pr[8], pr8[8];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            pr[jj] = jj < 5 ? (wa & (0x00030003u << (2 * jj))) : (w2 & (0x00030003u << (2 * (jj - 5))));
            pr8[jj] = jj < 5 ? (w8 & (0x00030003u << (2 * jj))) : (w82 & (0x00030003u << (2 * (jj - 5))));
          }
          uint4 bp[NT];
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              const int b = min(8 * t + g, p.B - 1);  // columns past B: not stored
              if ((jj & 1) == 0)
                bp[t] = *reinterpret_cast<const uint4*>(xh + ((((gl * WPT + u) * 2 + (jj >> 1)) * p.B + b) * 4 + q) * 4);
              const uint32_t b0 = (jj & 1) ? bp[t].z : bp[t].x, b1 = (jj & 1) ? bp[t].w : bp[t].y;
              mma16816(cc[t], pr[2 * jj], pr8[2 * jj], pr[2 * jj + 1], pr8[2 * jj + 1], b0, b1);
            }
          }
        }
        const float2 m = scale_pair(sw + j * 16 + 2 * g, V[gl * p.R + p.R - 1]);  // rows g, g + 8
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          acc[t][0] = fmaf(m.x, cc[t][0], acc[t][0]);
          acc[t][1] = fmaf(m.x, cc[t][1], acc[t][1]);
          acc[t][2] = fmaf(m.y, cc[t][2], acc[t][2]);
          acc[t][3] = fmaf(m.y, cc[t][3], acc[t][3]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    };
    for (int s = 0; s < nst; s += 2) {
      stage(s, usA);
      if (s + 1 < nst) stage(s + 1, usB);
    }
    const int rg = row_w0 + g, rg8 = rg + 8;
    const int rl = 16 * warp + g;
    if (ks > 1 && blockIdx.y != 0) {
      // push the partial sums into the cluster leader's buffer (slot rank - 1), then arrive on the
      // cluster barrier (release); the leader waits on it and adds them to its own in rank order
      cluster_wait();
      const uint32_t slot0 = smem_addr(smem + p.red_off) + 4u * static_cast<uint32_t>((blockIdx.y - 1) * BR * p.B);
      const uint32_t base = cluster_map(slot0, 0);
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const int b = 8 * t + 2 * q;
        if (b < p.B) {
          st_cluster_f32(base + 4u * static_cast<uint32_t>(rl * p.B + b), acc[t][0]);
          st_cluster_f32(base + 4u * static_cast<uint32_t>((rl + 8) * p.B + b), acc[t][2]);
        }
        if (b + 1 < p.B) {
          st_cluster_f32(base + 4u * static_cast<uint32_t>(rl * p.B + b + 1), acc[t][1]);
          st_cluster_f32(base + 4u * static_cast<uint32_t>((rl + 8) * p.B + b + 1), acc[t][3]);
        }
      }
      cluster_arrive_release();
    } else {
      if (ks > 1) {
        cluster_wait();
        cluster_arrive_release();  // second phase: complete once every rank has pushed (or exited)
        cluster_wait();
        const float* red = reinterpret_cast<const float*>(smem + p.red_off);
        const int E = BR * p.B;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const int b = min(8 * t + 2 * q, p.B - 1), b1 = min(b + 1, p.B - 1);
          for (int r = 1; r < ks; ++r) {
            const float* rr = red + (r - 1) * E;
            acc[t][0] += rr[rl * p.B + b];
            acc[t][1] += rr[rl * p.B + b1];
            acc[t][2] += rr[(rl + 8) * p.B + b];
            acc[t][3] += rr[(rl + 8) * p.B + b1];
          }
        }
      }
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const int b = 8 * t + 2 * q;
        if (rg < p.N) {
          if (b < p.B) p.y[static_cast<size_t>(b) * p.N + rg] = acc[t][0];
          if (b + 1 < p.B) p.y[static_cast<size_t>(b + 1) * p.N + rg] = acc[t][1];
        }
        if (rg8 < p.N) {
          if (b < p.B) p.y[static_cast<size_t>(b) * p.N + rg8] = acc[t][2];
          if (b + 1 < p.B) p.y[static_cast<size_t>(b + 1) * p.N + rg8] = acc[t][3];
        }
      }
    }
  }
  if (ks > 1 && warp == nw) cluster_wait();  // the producer warp completes its barrier phase too
}

// ---------------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------------
constexpr int kSMs = 148;  // B300
constexpr size_t kSmemLimit = 227 * 1024;

struct Plan {
  bool ok;
  int rs, kl, ppl, ks, upr, n_rg;
  size_t smem, xh_off, vp_off, sw_off, bar_off, ring_off;
};

// Shared-memory layout of a candidate split; returns the total bytes.  The partial-sum buffer of
// the epilogue reuses the table / x^ region.
size_t layout(Plan& pl, int pack, int B, int G, int K) {
  const int UT = unit_codes(pack), SLAB = slab_rows(pack);
  const int RT = pl.rs * SLAB;
  const int kr = std::min(pl.kl * pl.ppl * UT, K);
  const int ngr = kr / G;
  pl.xh_off = pack == TQ_PACK_B3 ? kLutBytes : 0;
  const size_t main = pl.xh_off + align256(static_cast<size_t>(kr) * B * 2);
  const size_t red = static_cast<size_t>(pl.kl) * RT * B * 4;
  pl.vp_off = align256(std::max(main, red));
  pl.sw_off = pl.vp_off + align256(static_cast<size_t>(ngr) * vp_row(B) * 4);
  pl.bar_off = pl.sw_off + align256(static_cast<size_t>(pl.rs) * pl.kl * (UT / G) * SLAB * 2);
  pl.ring_off = pl.bar_off + 256;
  pl.smem = pl.ring_off + (pack == TQ_PACK_3BIT ? static_cast<size_t>(pl.rs) * pl.kl * kQ3WarpRing : 0);
  return pl.smem;
}

// Candidate splits in order of estimated time: per-warp units x busiest-SM warps (at least 12, 24 for
// 3-bit codes, below which a warp's own latency dominates); ties go to fewer CTAs, then to smaller
// clusters.
std::vector<Plan> candidates(const tq_desc* d, int B) {
  const int UT = unit_codes(d->packing), SLAB = slab_rows(d->packing);
  // the 3-bit kernel (a serial chain per warp, one TMA box per unit) keeps gaining up to ~24 warps
  const double min_warps = d->packing == TQ_PACK_3BIT ? 24.0 : 12.0;
  const int upr = (d->K + UT - 1) / UT;
  const int slabs = (d->N + SLAB - 1) / SLAB;
  std::vector<std::tuple<double, int, int, Plan>> list;
  for (int kl = 1; kl <= 16; ++kl) {
    for (int rs = 1; rs * kl <= 16; rs *= 2) {
      for (int ks = 1; ks <= kMaxCluster; ++ks) {
        Plan pl{};
        pl.upr = upr;
        pl.kl = kl;
        pl.rs = rs;
        pl.ks = ks;
        pl.ppl = (upr + kl * ks - 1) / (kl * ks);
        if ((ks - 1) * kl * pl.ppl >= upr) continue;  // a CTA without work
        if (kl > 1 && (kl - 1) * pl.ppl >= upr) continue;  // a K-lane that can never have work
        pl.n_rg = (slabs + rs - 1) / rs;
        if (layout(pl, d->packing, B, d->group, d->K) > kSmemLimit) continue;
        const long long C = static_cast<long long>(pl.n_rg) * ks;
        const long long k = (C + kSMs - 1) / kSMs;
        const double cost = pl.ppl * std::max<double>(static_cast<double>(k * rs * kl), min_warps);
        list.emplace_back(cost, static_cast<int>(C), ks, pl);
      }
    }
  }
  std::stable_sort(list.begin(), list.end(), [](const auto& a, const auto& b) {
    if (std::get<0>(a) != std::get<0>(b)) return std::get<0>(a) < std::get<0>(b);
    if (std::get<1>(a) != std::get<1>(b)) return std::get<1>(a) < std::get<1>(b);
    return std::get<2>(a) < std::get<2>(b);
  });
  std::vector<Plan> out;
  for (auto& t : list) out.push_back(std::get<3>(t));
  return out;
}

// Raises a kernel's dynamic shared-memory limit to at least `bytes` on the current device.  The
// attribute belongs to the (function, device) pair, so the largest value set so far is kept per pair.
cudaError_t ensure_smem_attr(const void* fn, size_t bytes) {
  static std::map<std::pair<const void*, int>, size_t> done;
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  size_t& have = done[{fn, dev}];
  if (have >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  have = bytes;
  return cudaSuccess;
}

cudaLaunchConfig_t launch_config(const Plan& pl, cudaStream_t s, cudaLaunchAttribute (&attr)[2], int zdim = 1) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.n_rg, pl.ks, zdim);
  cfg.blockDim = dim3(32 * pl.rs * pl.kl);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = s;
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (pl.ks > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 1;
    attr[na].val.clusterDim.y = pl.ks;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cfg;
}

// The first candidate whose CTAs (or clusters) can all be resident at once on this device; plans
// are cached per (kernel, shape, device).
cudaError_t choose_plan(const void* kern, const tq_desc* d, int B, Plan* out) {
  static std::map<std::tuple<const void*, int, int, int, int, int>, Plan> cache;
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const auto key = std::make_tuple(kern, d->N, d->K, d->group, B, dev);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *out = it->second;
      return cudaSuccess;
    }
  }
  int sms = kSMs;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) sms = kSMs;
  int optin = 0;
  if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
  Plan chosen{};
  for (const Plan& pl : candidates(d, B)) {
    if (pl.smem > static_cast<size_t>(optin)) continue;
    if ((e = ensure_smem_attr(kern, pl.smem)) != cudaSuccess) return e;
    bool fits = false;
    if (pl.ks > 1) {
      cudaLaunchAttribute attr[2];
      cudaLaunchConfig_t cfg = launch_config(pl, nullptr, attr);
      int nc = 0;
      if (cudaOccupancyMaxActiveClusters(&nc, kern, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        continue;
      }
      fits = nc >= pl.n_rg;
    } else {
      int bps = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kern, 32 * pl.rs * pl.kl, pl.smem) != cudaSuccess) {
        (void)cudaGetLastError();
        continue;
      }
      fits = bps > 0 && static_cast<long long>(pl.n_rg) <= static_cast<long long>(bps) * sms;
    }
    if (fits) {
      chosen = pl;
      chosen.ok = true;
      break;
    }
  }
  if (!chosen.ok) {  // nothing fits in one wave: take the best plan that launches at all
    for (const Plan& pl : candidates(d, B)) {
      if (pl.smem <= static_cast<size_t>(optin) && pl.ks == 1) {
        chosen = pl;
        chosen.ok = true;
        break;
      }
    }
  }
  if (!chosen.ok) return cudaErrorInvalidConfiguration;
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = chosen;
  *out = chosen;
  return cudaSuccess;
}

template <int PACK, int G>
cudaError_t launch_prep(const PrepParams& pp, cudaStream_t s, int zdim) {
  cudaLaunchConfig_t cfg = {};
  const int nblk = pp.K / kFwhtBlock;
  cfg.gridDim = dim3((nblk + 3) / 4, 1, zdim);
  cfg.blockDim = dim3(128);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (pp.B <= 1) return cudaLaunchKernelEx(&cfg, gemv_prep_kernel<PACK, G, 1>, pp);
  if (pp.B <= 2) return cudaLaunchKernelEx(&cfg, gemv_prep_kernel<PACK, G, 2>, pp);
  if (pp.B <= 4) return cudaLaunchKernelEx(&cfg, gemv_prep_kernel<PACK, G, 4>, pp);
  if (pp.B <= 8) return cudaLaunchKernelEx(&cfg, gemv_prep_kernel<PACK, G, 8>, pp);
  return cudaLaunchKernelEx(&cfg, gemv_prep_kernel<PACK, G, kMaxBatch>, pp);
}

// The decode kernel for a shape: packing, group and batch tiles.
template <int G>
const void* kernel_b3(int B) {
  switch ((B + 1) / 2) {
    case 1: return reinterpret_cast<const void*>(gemv_b3_kernel<G, 1>);
    case 2: return reinterpret_cast<const void*>(gemv_b3_kernel<G, 2>);
    case 3:
    case 4: return reinterpret_cast<const void*>(gemv_b3_kernel<G, 4>);
    default: return reinterpret_cast<const void*>(gemv_b3_kernel<G, 8>);
  }
}
template <int G>
const void* kernel_q3(int B) {
  switch ((B + 1) / 2) {
    case 1: return reinterpret_cast<const void*>(gemv_q3_kernel<G, 1>);
    case 2: return reinterpret_cast<const void*>(gemv_q3_kernel<G, 2>);
    case 3:
    case 4: return reinterpret_cast<const void*>(gemv_q3_kernel<G, 4>);
    default: return reinterpret_cast<const void*>(gemv_q3_kernel<G, 8>);
  }
}
template <int G>
const void* kernel_2b(int B) {
  return B <= 8 ? reinterpret_cast<const void*>(gemv_2b_kernel<G, 1>) : reinterpret_cast<const void*>(gemv_2b_kernel<G, 2>);
}
const void* gemv_kernel(const tq_desc* d, int B) {
  if (d->packing == TQ_PACK_B3) return d->group == 128 ? kernel_b3<128>(B) : kernel_b3<64>(B);
  if (d->packing == TQ_PACK_3BIT) return d->group == 128 ? kernel_q3<128>(B) : kernel_q3<64>(B);
  return d->group == 128 ? kernel_2b<128>(B) : kernel_2b<64>(B);
}

// Prep output of one matrix (or one chunk): x^ (K x batch halves) then VP (groups x vp_row(batch)
// floats).  Both are multiples of 256 bytes.
size_t xh_bytes(const tq_desc* d, int B) { return align256(static_cast<size_t>(d->K) * B * 2); }
size_t vp_bytes(const tq_desc* d, int B) { return align256(static_cast<size_t>(d->K / d->group) * vp_row(B) * 4); }

// Prep kernel (or the fused prologue) then decode kernel; pp and prm carry everything but the
// shape-derived fields.  For the expert layer's chunks of at most 2 tokens the prologue is fused into
// the decode kernel (one kernel boundary less in a chain of several launches; measured faster at
// 1 and 8 tokens); dense calls use one prep kernel that transforms the activations once for all
// CTAs (measured faster on the decode stream).
// ---- stream kernel (2-bit dense) ----


struct SPlan {
  bool ok;
  int nw, ks, gpc, S, n_rb;
  size_t smem;
  uint32_t stage_bytes, xh_off, vp_off, sc_off, red_off, bar_off, xs_off;
};

// Shared-memory layout (offsets from the 1024-aligned base): ring, x^, VP, per-warp scales, partial
// sums, barriers.  The ring takes what the rest leaves, up to 8 stages.
bool stream_layout(SPlan& pl, int B, int G) {
  const int BR = 16 * pl.nw, GPS = 512 / G;
  pl.stage_bytes = static_cast<uint32_t>(BR) * 128u;
  const size_t xh = align256(static_cast<size_t>(pl.gpc) * G * B * 2);
  const size_t vp = align256(static_cast<size_t>(pl.gpc) * vp_row(B) * 4);
  const size_t sw = align256(static_cast<size_t>(pl.nw) * GPS * 16 * 2);  // per-warp scale staging
  const size_t red = align256(static_cast<size_t>(pl.ks - 1) * BR * B * 4);
  const size_t xs = B <= kStreamFuseMaxB ? align256(static_cast<size_t>(pl.gpc) * G * B * 2) : 0;
  const size_t bars = 256;
  const size_t fixed = xh + vp + sw + red + xs + bars + 1024;  // + alignment slack of the base
  if (fixed + 2 * static_cast<size_t>(pl.stage_bytes) > kSmemLimit) return false;
  pl.S = static_cast<int>(std::min<size_t>(8, (kSmemLimit - fixed) / pl.stage_bytes));
  size_t off = static_cast<size_t>(pl.S) * pl.stage_bytes;
  pl.xh_off = static_cast<uint32_t>(off);
  off += xh;
  pl.vp_off = static_cast<uint32_t>(off);
  off += vp;
  pl.sc_off = static_cast<uint32_t>(off);
  off += sw;
  pl.red_off = static_cast<uint32_t>(off);
  off += red;
  pl.xs_off = static_cast<uint32_t>(off);
  off += xs;
  pl.bar_off = static_cast<uint32_t>(off);
  off += bars;
  pl.smem = off + 1024;
  return true;
}

// Candidate splits, cheapest first: 16*nw-row blocks x ks K-ranges (whole 128-blocks), at most one
// CTA per SM.  Cost: groups per warp x warps per SM (the decode loop is issue-bound once ~6 warps
// share an SM); ties go to fewer CTAs.
std::vector<SPlan> stream_candidates(const tq_desc* d, int B, int sms) {
  const int G = d->group, ng = d->K / G, bpg = kFwhtBlock / G;
  std::vector<std::pair<double, SPlan>> list;
  for (int nw : {16, 8}) {
    const int BR = 16 * nw, n_rb = (d->N + BR - 1) / BR;
    for (int ks = 1; ks <= kMaxCluster && n_rb * ks <= sms; ++ks) {
      int gpc = (ng + ks - 1) / ks;
      gpc = (gpc + bpg - 1) / bpg * bpg;
      if ((ks - 1) * gpc >= ng) continue;  // a CTA without work
      SPlan pl{};
      pl.nw = nw;
      pl.ks = ks;
      pl.gpc = gpc;
      pl.n_rb = n_rb;
      if (!stream_layout(pl, B, G)) continue;
      pl.ok = true;
      list.emplace_back(static_cast<double>(gpc) * std::max(nw, 6), pl);
    }
  }
  std::stable_sort(list.begin(), list.end(), [](const auto& a, const auto& b) {
    if (a.first != b.first) return a.first < b.first;
    return a.second.n_rb * a.second.ks < b.second.n_rb * b.second.ks;
  });
  std::vector<SPlan> out;
  for (auto& e : list) out.push_back(e.second);
  return out;
}

template <int G, int NT>
const void* stream_kernel_t() {
  return reinterpret_cast<const void*>(gemv_2b_stream_kernel<G, NT>);
}
const void* stream_kernel(int G, int B) {
  if (G == 128) return B <= 8 ? stream_kernel_t<128, 1>() : stream_kernel_t<128, 2>();
  return B <= 8 ? stream_kernel_t<64, 1>() : stream_kernel_t<64, 2>();
}

// Tensor map over a code matrix [N][P] (uint32), box 32 words x BR rows, 128-byte swizzle; cached per
// (address, N, P, BR).
bool codes_tmap(const uint32_t* codes, int N, int P, int BR, CUtensorMap* out) {
  static std::map<std::tuple<const void*, int, int, int>, CUtensorMap> cache;
  static std::mutex mu;
  const auto key = std::make_tuple(static_cast<const void*>(codes), N, P, BR);
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) {
    *out = it->second;
    return true;
  }
  CUtensorMap m;
  if (!make_tmap_2d(&m, codes, CU_TENSOR_MAP_DATA_TYPE_UINT32, static_cast<uint64_t>(P), static_cast<uint64_t>(N),
                    static_cast<uint64_t>(P) * 4u, 32u, static_cast<uint32_t>(BR), CU_TENSOR_MAP_SWIZZLE_128B))
    return false;
  if (cache.size() > 4096) cache.clear();
  cache[key] = m;
  *out = m;
  return true;
}

// The stream kernel's plan for a shape on the current device (cached), or !ok when it does not apply.
cudaError_t choose_stream_plan(const tq_desc* d, int B, SPlan* out) {
  static std::map<std::tuple<int, int, int, int, int, int>, SPlan> cache;  // per packing: only 2-bit streams
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const auto key = std::make_tuple(d->N, d->K, d->group, B, dev, d->packing);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *out = it->second;
      return cudaSuccess;
    }
  }
  int sms = kSMs, optin = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) sms = kSMs;
  if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
  SPlan pl{};
  if (d->packing == TQ_PACK_2BIT && d->K % kFwhtBlock == 0 && B <= kMaxBatch) {
    // the first candidate whose CTAs (clusters) are all resident at once
    const void* kern = stream_kernel(d->group, B);
    for (const SPlan& c : stream_candidates(d, B, sms)) {
      if (c.smem > static_cast<size_t>(optin)) continue;
      if ((e = ensure_smem_attr(kern, c.smem)) != cudaSuccess) return e;
      bool fits = false;
      if (c.ks > 1) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(c.n_rb, c.ks, 1);
        cfg.blockDim = dim3(32 * (c.nw + 1));
        cfg.dynamicSmemBytes = c.smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = c.ks;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int nc = 0;
        if (cudaOccupancyMaxActiveClusters(&nc, kern, &cfg) != cudaSuccess) {
          (void)cudaGetLastError();
          continue;
        }
        fits = nc >= c.n_rb;
      } else {
        fits = c.n_rb <= sms;
      }
      if (fits) {
        pl = c;
        break;
      }
    }
  }
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = pl;
  *out = pl;
  return cudaSuccess;
}

// Dense 2-bit GEMV through the stream kernel (plus the prep kernel above kStreamFuseMaxB).
cudaError_t launch_stream(const tq_desc* d, const SPlan& pl, const uint32_t* codes, const uint16_t* scales,
                          const uint16_t* x, int B, float* y, void* ws, bool early, cudaStream_t s) {
  const int G = d->group;
  const int P = pitch_words(d->K, d->packing);
  CUtensorMap tm;
  if (!codes_tmap(codes, d->N, P, 16 * pl.nw, &tm)) return cudaErrorInvalidValue;
  SParams sp{};
  sp.scales = scales;
  sp.x = x;
  sp.xh_g = static_cast<const uint16_t*>(ws);
  sp.vp_g = reinterpret_cast<const float*>(static_cast<const uint8_t*>(ws) + xh_bytes(d, B));
  sp.y = y;
  sp.status = status_ptr();
  sp.N = d->N;
  sp.K = d->K;
  sp.ng = d->K / G;
  sp.B = B;
  sp.R = vp_row(B);
  sp.gpc = pl.gpc;
  sp.nw = pl.nw;
  sp.S = pl.S;
  sp.fused = B <= kStreamFuseMaxB;
  sp.early = early;
  sp.apply = d->fwht_block != 0;
  sp.stage_bytes = pl.stage_bytes;
  sp.xh_off = pl.xh_off;
  sp.vp_off = pl.vp_off;
  sp.sc_off = pl.sc_off;
  sp.red_off = pl.red_off;
  sp.bar_off = pl.bar_off;
  sp.xs_off = pl.xs_off;
  cudaError_t e;
  if (!sp.fused) {
    PrepParams pp{};
    pp.x = x;
    pp.xh = static_cast<uint16_t*>(ws);
    pp.vp = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + xh_bytes(d, B));
    pp.status = sp.status;
    pp.K = d->K;
    pp.B = B;
    pp.apply = sp.apply;
    e = G == 128 ? launch_prep<TQ_PACK_2BIT, 128>(pp, s, 1) : launch_prep<TQ_PACK_2BIT, 64>(pp, s, 1);
    if (e != cudaSuccess) return e;
  }
  const void* kern = stream_kernel(G, B);
  if ((e = ensure_smem_attr(kern, pl.smem)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.n_rb, pl.ks, 1);
  cfg.blockDim = dim3(32 * (pl.nw + 1));
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (pl.ks > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 1;
    attr[na].val.clusterDim.y = pl.ks;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  void* args[] = {&tm, &sp};
  return cudaLaunchKernelExC(&cfg, kern, args);
}

cudaError_t launch_pair(const tq_desc* d, PrepParams pp, Params prm, int B, int zdim, cudaStream_t s) {
  pp.status = status_ptr();
  pp.K = d->K;
  pp.B = B;
  pp.apply = d->fwht_block != 0;
  const bool b3 = d->packing == TQ_PACK_B3;
  const void* kern = gemv_kernel(d, B);
  Plan pl{};
  cudaError_t e = choose_plan(kern, d, B, &pl);
  if (e != cudaSuccess) return e;
  if ((e = ensure_smem_attr(kern, pl.smem)) != cudaSuccess) return e;
  prm.fused = B <= 2 && prm.chunks != nullptr;
  if (prm.fused) {
    prm.mode = pp.mode;
    prm.topk = pp.topk;
    prm.apply = pp.apply;
    prm.x = pp.x;
    prm.gu = pp.gu;
    prm.h_out = pp.h_out;
  } else {
    const bool g128 = d->group == 128;
    if (b3)
      e = g128 ? launch_prep<TQ_PACK_B3, 128>(pp, s, zdim) : launch_prep<TQ_PACK_B3, 64>(pp, s, zdim);
    else if (d->packing == TQ_PACK_3BIT)
      e = g128 ? launch_prep<TQ_PACK_3BIT, 128>(pp, s, zdim) : launch_prep<TQ_PACK_3BIT, 64>(pp, s, zdim);
    else
      e = g128 ? launch_prep<TQ_PACK_2BIT, 128>(pp, s, zdim) : launch_prep<TQ_PACK_2BIT, 64>(pp, s, zdim);
    if (e != cudaSuccess) return e;
  }
  prm.xh_g = pp.xh;
  prm.vp_g = pp.vp;
  prm.status = pp.status;
  prm.N = d->N;
  prm.K = d->K;
  prm.P = pitch_words(d->K, d->packing);
  prm.ng = d->K / d->group;
  prm.B = B;
  prm.R = vp_row(B);
  prm.G = d->group;
  prm.rs = pl.rs;
  prm.kl = pl.kl;
  prm.ppl = pl.ppl;
  prm.upr = pl.upr;
  prm.xh_off = static_cast<uint32_t>(pl.xh_off);
  prm.vp_off = static_cast<uint32_t>(pl.vp_off);
  prm.sw_off = static_cast<uint32_t>(pl.sw_off);
  prm.bar_off = static_cast<uint32_t>(pl.bar_off);
  prm.ring_off = static_cast<uint32_t>(pl.ring_off);
  if (d->packing == TQ_PACK_3BIT &&
      !make_tmap_2d(&prm.tm, prm.codes, CU_TENSOR_MAP_DATA_TYPE_UINT32, static_cast<uint64_t>(prm.P),
                    static_cast<uint64_t>(d->N), static_cast<uint64_t>(prm.P) * 4u, kQ3UnitWords, 64,
                    CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  prm.v8 = b3 && prm.P % 8 == 0 && reinterpret_cast<uintptr_t>(prm.codes) % 32 == 0 &&
           (!prm.chunks || prm.codes_estride % 8 == 0);
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = launch_config(pl, s, attr, zdim);
  void* args[] = {&prm};
  return cudaLaunchKernelExC(&cfg, kern, args);
}

}  // namespace gemv

size_t gemv_workspace_bytes(const tq_desc* d, int batch) {
  using namespace gemv;
  // the smallest split (one slab, one K-lane, eight CTAs along K) must fit shared memory
  Plan pl{};
  pl.upr = (d->K + unit_codes(d->packing) - 1) / unit_codes(d->packing);
  pl.rs = 1;
  pl.kl = 1;
  pl.ks = std::min(kMaxCluster, pl.upr);
  pl.ppl = (pl.upr + pl.ks - 1) / pl.ks;
  if (layout(pl, d->packing, batch, d->group, d->K) > kSmemLimit) return 0;
  return xh_bytes(d, batch) + vp_bytes(d, batch);
}

cudaError_t launch_gemv(const tq_desc* d, const uint32_t* codes, const uint16_t* scales, const uint16_t* x, int B,
                        float* y, void* ws, cudaStream_t s) {
  using namespace gemv;
  PrepParams pp{};
  pp.x = x;
  pp.xh = static_cast<uint16_t*>(ws);
  pp.vp = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + xh_bytes(d, B));
  SPlan spl{};
  if (const cudaError_t e = choose_stream_plan(d, B, &spl); e != cudaSuccess) return e;
  if (spl.ok) return launch_stream(d, spl, codes, scales, x, B, y, ws, (d->flags & TQ_STATIC_WEIGHTS) != 0, s);
  Params prm{};
  prm.codes = codes;
  prm.scales = scales;
  prm.y = y;
  prm.early = (d->flags & TQ_STATIC_WEIGHTS) != 0;
  return launch_pair(d, pp, prm, B, 1, s);
}

int gemv_kernel_count(const tq_desc* d, int B) {
  using namespace gemv;
  SPlan spl{};
  if (choose_stream_plan(d, B, &spl) != cudaSuccess) {
    (void)cudaGetLastError();
    return -1;
  }
  return spl.ok && B <= kStreamFuseMaxB ? 1 : 2;
}

size_t gemv_chunks_workspace_bytes(const tq_desc* d, int B, int max_chunks) {
  using namespace gemv;
  if (gemv_workspace_bytes(d, B) == 0) return 0;
  return static_cast<size_t>(max_chunks) * (xh_bytes(d, B) + vp_bytes(d, B));
}

int gemv_chunks_row_tiles(const tq_desc* d, int B) {
  using namespace gemv;
  if (gemv_workspace_bytes(d, B) == 0) return -1;
  Plan pl{};
  if (choose_plan(gemv_kernel(d, B), d, B, &pl) != cudaSuccess) return -1;
  return pl.n_rg;
}

cudaError_t launch_gemv_chunks(const tq_desc* d, const uint32_t* codes, const uint16_t* scales, size_t codes_estride,
                               size_t scales_estride, int mode, const uint16_t* x, const float* gu, float* h_out,
                               int topk, const int* chunks, int B, int max_chunks, float* y, void* ws,
                               cudaStream_t s, const ChunkCombine* combine) {
  using namespace gemv;
  PrepParams pp{};
  pp.x = x;
  pp.gu = gu;
  pp.h_out = h_out;
  pp.xh = static_cast<uint16_t*>(ws);
  pp.vp = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + static_cast<size_t>(max_chunks) * xh_bytes(d, B));
  pp.mode = mode;
  pp.chunks = chunks;
  pp.topk = topk;
  pp.xh_cstride = xh_bytes(d, B) / 2;
  pp.vp_cstride = vp_bytes(d, B) / 4;
  Params prm{};
  prm.codes = codes;
  prm.scales = scales;
  prm.y = y;
  prm.early = 0;  // the expert of a chunk is known only after routing
  prm.chunks = chunks;
  prm.codes_estride = codes_estride;
  prm.scales_estride = scales_estride;
  prm.xh_cstride = pp.xh_cstride;
  prm.vp_cstride = pp.vp_cstride;
  prm.topk = topk;
  if (combine) {
    prm.cmb_count = combine->count;
    prm.cmb_gate = combine->gate;
    prm.cmb_y = combine->y;
  }
  return launch_pair(d, pp, prm, B, max_chunks, s);
}

}  // namespace tq

// Decode GEMV on the 5th-generation tensor cores: y[b][n] = sum_g s[n][g] sum_{k in g} t[n][k] x~[b][k].
//
// Why tensor cores for a bandwidth-bound GEMV: at the HBM rate each SM must retire ~80 trits per
// cycle (base-3, 0.2 B/trit at ~6.5 TB/s over 148 SMs), i.e. ~1.5 issue slots per trit in total.
// Turning a trit into a float and adding it on the CUDA cores costs 3+ slots; here a trit costs
// about one slot of integer decode and the multiply-add goes to tcgen05.mma.
//
// Data flow per CTA (one CTA per SM, persistent, stream-K partition of (128-row tile, stage)):
//   producer warp : cp.async.bulk of 128 rows x 32 code words (one "stage") + the stage's block of
//                   prepared activations x^ into a shared-memory ring;
//   4 decode warps: thread = row.  Decode code words into pairs of FP16 values and write them to
//                   tensor memory (tcgen05.st) as the A operand, one 128-trit (or 64-trit) group at a
//                   time; after the MMA of a group, read its 128 x 16 fp32 result (tcgen05.ld) and
//                   fold in the group's FP16 scale (one FMA per batch column).
//   MMA thread    : per group, G/16 MMAs (M=128, N=16, K=16, A from TMEM, B = x^ in shared memory)
//                   plus one MMA that subtracts sum(x^) (see below), into a fresh accumulator.
//
// Decoding without arithmetic: a 2-bit digit d = t + 1 placed in mantissa bits 2i of an FP16 half
// with a zero exponent field is the subnormal d * 2^(2i-24), exactly.  Masking a code word with
// 0x00030003 << 2i therefore yields two FP16 operands (one per half-word) in one LOP3; the position
// factor 2^(8-2i) and the offset (t = d - 1) are folded into the activations: the preparation
// kernel stores x^ = x~ * 2^-e * 2^(8-2i) and, per group, -sum(x~ * 2^-e) as an extra K-slot
// multiplied by a constant A of 2^-16.  Base-3 words are split into four 5-trit chunks (two exact
// reciprocal multiplies) and a 243-entry lookup table (replicated per lane, conflict-free) places
// the digits into those bit fields.
//   base-3: tantan.ink/?p=490, section "为什么 1.58bit 没变成乱码", point 3 (20 trits per uint32);
//   group scale: cosmocat.dev "27B 大模型塞进 5.9GB", section 二 ② (one FP16 scale per 128 weights);
//   rotation: same page, section 二 ① (matching O(n log n) transform on the activations).
#include <algorithm>

#include "tq_internal.cuh"
#include "tq_kernels.cuh"
#include "tq_sm100.cuh"

namespace tq {
namespace gemv_tc {

using namespace sm100;

constexpr int kRows = 128;                // rows per tile = MMA M = TMEM lanes
constexpr int kStageWords = 32;           // code words per row per stage (128 bytes)
constexpr int kRowPitchSmem = 144;        // 128 B + 16 B padding: conflict-free 16-byte row reads
constexpr int kCodeStageBytes = kRows * kRowPitchSmem;
constexpr int kRing = 4;                  // groups in flight between the decode warps and the MMA
constexpr int kThreads = 192;             // warps 0-3 decode, 4 producer, 5 MMA + TMEM owner
constexpr uint32_t kLutBytes = 2u * 243u * 32u * 4u;
constexpr int kMaxStages = 6;

template <int PACK>
struct Geo;
template <>
struct Geo<TQ_PACK_B3> {
  static constexpr int kStageTrits = 640;  // 32 words x 20 trits = 5 groups of 128
};
template <>
struct Geo<TQ_PACK_2BIT> {
  static constexpr int kStageTrits = 512;  // 32 words x 16 trits = 4 groups of 128
};

template <int PACK, int G>
struct Cfg {
  static constexpr int ST = Geo<PACK>::kStageTrits;
  static constexpr int GP = G / 2;        // TMEM columns (FP16 pairs) per group
  static constexpr int GPS = ST / G;      // groups per stage
  static constexpr int SLICES = G / 16;   // K=16 MMAs per group
  static constexpr int A_COLS = kRing * GP;
  static constexpr int D_COL0 = A_COLS;
  static constexpr int C_COL0 = A_COLS + kRing * 16;
  static constexpr int TMEM_COLS = (C_COL0 + 8) <= 256 ? 256 : 512;
  static constexpr uint32_t LUT_BYTES = PACK == TQ_PACK_B3 ? kLutBytes : 0u;
};

// Chunk lookup table: for a 5-trit chunk c (digits d0..d4 of c in base 3) the "A" entry places the
// digits at FP16 pair fields (lo0, hi0, lo1, hi1, lo2) and the "B" entry at (hi2, lo3, hi3, lo4, hi4),
// where loI / hiI are bits 2I / 16 + 2I.  Each entry is replicated 32 times so lane l reads bank l.
struct LutTable {
  uint32_t v[2 * 243 * 32];
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
  const uint8_t* xhat;      // prepared activations, one block per stage
  const float* pow2g;       // 2^(16 + e) per group (e = exponent of the group's block)
  float* y;
  float* partial;           // [tile][part][B][128] partial outputs of split tiles
  int* counters;            // [tile] arrivals of split tiles (zeroed by the preparation kernel)
  int* status;
  int N, K, P, ng, B, n_tiles, spr, units;
  uint32_t xhat_stage_bytes;  // bytes of one stage block of x^ (main + correction + zero chunk)
  uint32_t corr_offset;       // offset of the correction chunks inside a stage block
  uint32_t stage_smem;        // shared-memory bytes per pipeline stage
  int stages;                 // pipeline depth
};

__device__ __forceinline__ void fail(const Params& p, volatile int* s_abort) {
  record_error(p.status, TQ_ERR_TIMEOUT);
  *s_abort = 1;
}

// CTA that owns unit u under the static partition u_c = floor(c * units / grid).
__device__ __forceinline__ int cta_of_unit(long long u, long long units, long long grid) {
  return static_cast<int>(((u + 1) * grid + units - 1) / units - 1);
}

// Sink of decoded pairs for one decode thread: stages 16 pairs in registers, writes them to the
// current group's A slot in TMEM, hands finished groups to the MMA and folds finished MMAs into acc.
template <int PACK, int G, int NB>
struct Decoder {
  using C = Cfg<PACK, G>;
  uint32_t lane_tmem;   // TMEM address of this warp's lane quarter, column 0
  uint64_t* a_full;
  uint64_t* mma_done;
  float* m_ring;        // [kRing][128] per-thread multipliers of groups in flight
  volatile int* s_abort;
  const Params* p;
  int r, lane;
  int gc, consumed;
  bool ok;
  float acc[NB];
  uint32_t stg[16];

  __device__ __forceinline__ uint32_t slot_col() const { return lane_tmem + (gc % kRing) * C::GP; }

  __device__ __forceinline__ void consume_one() {
    const int q = consumed;
    const int slot = q % kRing;
    bool w = mbar_wait(mma_done + slot, (q / kRing) & 1);
    w = __all_sync(0xffffffffu, w);
    if (!w) {
      ok = false;
      if (lane == 0) fail(*p, s_abort);
      return;
    }
    tc_fence_after();
    uint32_t d[NB];
    tmem_ld<NB>(lane_tmem + C::D_COL0 + slot * 16, d);
    tmem_wait_ld();
    const float m = m_ring[slot * kRows + r];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = fmaf(m, __uint_as_float(d[b]), acc[b]);
    ++consumed;
  }
  __device__ __forceinline__ void begin_group() {
    while (ok && gc - consumed >= kRing) consume_one();
  }
  __device__ __forceinline__ void end_group(float m) {
    tmem_wait_st();
    tc_fence_before();
    m_ring[(gc % kRing) * kRows + r] = m;
    __syncwarp();
    if (lane == 0) mbar_arrive(a_full + (gc % kRing));
    ++gc;
  }
  __device__ __forceinline__ void drain() {
    while (ok && consumed < gc) consume_one();
  }
};

// Decode one stage (32 words) of base-3 codes: natural-order pairs (t_2j, t_2j+1).
template <int G, int NB>
__device__ __forceinline__ void decode_stage_b3(Decoder<TQ_PACK_B3, G, NB>& D, const uint32_t (&w)[32],
                                                const uint32_t* __restrict__ lutA, const uint32_t* __restrict__ lutB,
                                                int ngs, const float (&mg)[Cfg<TQ_PACK_B3, G>::GPS]) {
  using C = Cfg<TQ_PACK_B3, G>;
  uint32_t col = 0;
#pragma unroll
  for (int wi = 0; wi < 32; ++wi) {
    if ((wi * 10) / C::GP >= ngs) break;
    const uint32_t v = min(w[wi], kB3Max);
    const uint32_t hi = __umulhi(v + 1u, 2383401723u) >> 15;    // v / 3^10, exact for v < 3^20
    const uint32_t lo = v - hi * 59049u;
    const uint32_t bl = __umulhi(lo, 17675008u);                  // lo / 243, exact for lo < 3^10
    const uint32_t al = lo - bl * 243u;
    const uint32_t bh = __umulhi(hi, 17675008u);
    const uint32_t ah = hi - bh * 243u;
    const uint32_t A0 = lutA[al * 32], B0 = lutB[bl * 32], A1 = lutA[ah * 32], B1 = lutB[bh * 32];
#pragma unroll
    for (int j = 0; j < 10; ++j) {
      const int q = wi * 10 + j;
      const int gl = q / C::GP;
      if (gl < ngs) {
        if (q % C::GP == 0) {
          D.begin_group();
          col = D.slot_col();
        }
        const uint32_t mask = 0x00030003u << (2 * (j % 5));
        D.stg[q % 16] = j < 5 ? ((A0 | B0) & mask) : ((A1 | B1) & mask);
        if (q % 16 == 15) tmem_st16(col + (q % C::GP) - 15, D.stg);
        if (q % C::GP == C::GP - 1) D.end_group(mg[gl]);
      }
    }
  }
}

// Decode one stage (32 words) of 2-bit codes: pair j of a word = fields (j, j + 8).
template <int G, int NB>
__device__ __forceinline__ void decode_stage_2b(Decoder<TQ_PACK_2BIT, G, NB>& D, const uint32_t (&w)[32], int ngs,
                                                const float (&mg)[Cfg<TQ_PACK_2BIT, G>::GPS]) {
  using C = Cfg<TQ_PACK_2BIT, G>;
  uint32_t col = 0;
#pragma unroll
  for (int wi = 0; wi < 32; ++wi) {
    if ((wi * 8) / C::GP >= ngs) break;
    const uint32_t v = w[wi];
    const uint32_t v2 = v >> 10;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int q = wi * 8 + j;
      const int gl = q / C::GP;
      if (q % C::GP == 0) {
        D.begin_group();
        col = D.slot_col();
      }
      D.stg[q % 16] = j < 5 ? (v & (0x00030003u << (2 * j))) : (v2 & (0x00030003u << (2 * (j - 5))));
      if (q % 16 == 15) tmem_st16(col + (q % C::GP) - 15, D.stg);
      if (q % C::GP == C::GP - 1) D.end_group(mg[gl]);
    }
  }
}

template <int PACK, int G, int NB>
__global__ void __launch_bounds__(kThreads, 1) gemv_tc_kernel(const __grid_constant__ Params p) {
  using C = Cfg<PACK, G>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long grid = gridDim.x;
  const int u0 = static_cast<int>(static_cast<long long>(blockIdx.x) * p.units / grid);
  const int u1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * p.units / grid);
  const int S = p.stages;

  uint8_t* lut_smem = smem;
  uint8_t* stages = smem + C::LUT_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(stages + static_cast<size_t>(S) * p.stage_smem);
  uint64_t* codes_full = bars;
  uint64_t* xhat_full = bars + S;
  uint64_t* empty = bars + 2 * S;
  uint64_t* a_full = bars + 3 * S;
  uint64_t* mma_done = a_full + kRing;
  uint64_t* lut_bar = mma_done + kRing;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(lut_bar + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* m_ring = reinterpret_cast<float*>(lut_bar + 3);  // 16-byte aligned: bars start 16-aligned

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(codes_full + i, 1);
      mbar_init(xhat_full + i, 1);
      mbar_init(empty + i, 5);  // 4 decode warps (codes read) + 1 MMA commit (x^ read)
    }
    for (int i = 0; i < kRing; ++i) {
      mbar_init(a_full + i, 4);
      mbar_init(mma_done + i, 1);
    }
    mbar_init(lut_bar, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp < 4) {
    // ------------------------------------------------------------------ decode warps (thread = row)
    Decoder<PACK, G, NB> D;
    D.lane_tmem = tbase + (static_cast<uint32_t>(warp * 32) << 16);
    D.a_full = a_full;
    D.mma_done = mma_done;
    D.m_ring = m_ring;
    D.s_abort = s_abort;
    D.p = &p;
    D.r = threadIdx.x;
    D.lane = lane;
    D.gc = 0;
    D.consumed = 0;
    D.ok = true;
    {
      // constant A of the correction MMA: K-slots 0 and 1 hold 2^-16 (FP16 0x0100), the rest 0
      uint32_t cv[8] = {0x01000100u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
      tmem_st8(D.lane_tmem + C::C_COL0, cv);
    }
    const uint32_t* lutA = reinterpret_cast<const uint32_t*>(lut_smem) + lane;
    const uint32_t* lutB = lutA + 243 * 32;
    if (PACK == TQ_PACK_B3) {
      bool w = mbar_wait(lut_bar, 0);
      w = __all_sync(0xffffffffu, w);
      if (!w) {
        D.ok = false;
        if (lane == 0) fail(p, s_abort);
      }
    }
    pdl_wait();  // pow2g and the split counters come from the preparation kernel
    int seg_tile = -1, seg_first = 0;
    for (int u = u0; u < u1 && D.ok; ++u) {
      if (__any_sync(0xffffffffu, *s_abort != 0)) break;
      const int it = u - u0, i = it % S;
      const int t = u / p.spr, st = u % p.spr;
      if (t != seg_tile) {
        seg_tile = t;
        seg_first = st;
#pragma unroll
        for (int b = 0; b < NB; ++b) D.acc[b] = 0.f;
      }
      const int row = t * kRows + threadIdx.x;
      const int ngs = min(C::GPS, p.ng - st * C::GPS);
      float mg[C::GPS];
#pragma unroll
      for (int gl = 0; gl < C::GPS; ++gl) {
        const int g = st * C::GPS + gl;
        mg[gl] = (gl < ngs && row < p.N)
                     ? half_bits_to_float(__ldg(p.scales + static_cast<size_t>(row) * p.ng + g)) * __ldg(p.pow2g + g)
                     : 0.f;
      }
      bool w = mbar_wait(codes_full + i, (it / S) & 1);
      w = __all_sync(0xffffffffu, w);
      if (!w) {
        D.ok = false;
        if (lane == 0) fail(p, s_abort);
        break;
      }
      uint32_t cw[32];
      if (row < p.N) {
        const uint4* src = reinterpret_cast<const uint4*>(stages + static_cast<size_t>(i) * p.stage_smem +
                                                          threadIdx.x * kRowPitchSmem);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 v = src[q];
          cw[4 * q] = v.x;
          cw[4 * q + 1] = v.y;
          cw[4 * q + 2] = v.z;
          cw[4 * q + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int q = 0; q < 32; ++q) cw[q] = PACK == TQ_PACK_B3 ? kB3Zero : kB2Zero;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + i);
      if constexpr (PACK == TQ_PACK_B3)
        decode_stage_b3<G, NB>(D, cw, lutA, lutB, ngs, mg);
      else
        decode_stage_2b<G, NB>(D, cw, ngs, mg);
      if (!D.ok) break;
      // end of this CTA's segment of tile t: fold in the remaining groups, then write
      if (u == u1 - 1 || (u + 1) / p.spr != t) {
        D.drain();
        if (!D.ok) break;
        if (seg_first == 0 && st == p.spr - 1) {
          if (row < p.N)
#pragma unroll
            for (int b = 0; b < NB; ++b)
              if (b < p.B) p.y[static_cast<size_t>(b) * p.N + row] = D.acc[b];
        } else {
          const long long first_u = static_cast<long long>(t) * p.spr;
          const int c_first = cta_of_unit(first_u, p.units, grid);
          const int n_parts = cta_of_unit(first_u + p.spr - 1, p.units, grid) - c_first + 1;
          const int part = static_cast<int>(blockIdx.x) - c_first;
          float* pp = p.partial + (static_cast<size_t>(t) * p.spr + part) * p.B * kRows;
#pragma unroll
          for (int b = 0; b < NB; ++b)
            if (b < p.B) pp[b * kRows + threadIdx.x] = D.acc[b];
          // last-arriving warp (over all parts of the tile) sums the parts in K order: deterministic
          __threadfence();
          __syncwarp();
          int last = 0;
          if (lane == 0) {
            const int old = atomicAdd(p.counters + t, 1);
            last = old == 4 * n_parts - 1;
            if (last) p.counters[t] = 0;
            __threadfence();
          }
          last = __shfl_sync(0xffffffffu, last, 0);
          if (last) {
            for (int rr = lane; rr < kRows; rr += 32) {
              const int rrow = t * kRows + rr;
              if (rrow >= p.N) break;
              for (int b = 0; b < p.B; ++b) {
                float v = 0.f;
                for (int q = 0; q < n_parts; ++q)
                  v += __ldcg(p.partial + ((static_cast<size_t>(t) * p.spr + q) * p.B + b) * kRows + rr);
                p.y[static_cast<size_t>(b) * p.N + rrow] = v;
              }
            }
          }
        }
      }
    }
    D.drain();
  } else if (warp == 4) {
    // ------------------------------------------------------------------ producer warp
    if (PACK == TQ_PACK_B3 && lane == 0) {
      mbar_arrive_expect_tx(lut_bar, kLutBytes);
      bulk_g2s(lut_smem, &g_lut, kLutBytes, lut_bar);
    }
    bool pdl_done = false;
    for (int u = u0; u < u1; ++u) {
      if (*s_abort) break;
      const int it = u - u0, i = it % S;
      bool w = true;
      if (lane == 0) w = mbar_wait(empty + i, ((it / S) & 1) ^ 1);
      w = __shfl_sync(0xffffffffu, w, 0);
      if (!w) {
        if (lane == 0) fail(p, s_abort);
        break;
      }
      const int t = u / p.spr, st = u % p.spr;
      const int rows = min(kRows, p.N - t * kRows);
      const int words = min(kStageWords, p.P - st * kStageWords);
      uint8_t* cs = stages + static_cast<size_t>(i) * p.stage_smem;
      if (lane == 0) mbar_arrive_expect_tx(codes_full + i, static_cast<uint32_t>(rows * words * 4));
      __syncwarp();
      const uint32_t* src = p.codes + static_cast<size_t>(t) * kRows * p.P + st * kStageWords;
      for (int rr = lane; rr < rows; rr += 32)
        bulk_g2s(cs + rr * kRowPitchSmem, src + static_cast<size_t>(rr) * p.P, static_cast<uint32_t>(words * 4),
                 codes_full + i);
      if (lane == 0) {
        if (!pdl_done) {
          pdl_wait();
          pdl_done = true;
        }
        mbar_arrive_expect_tx(xhat_full + i, p.xhat_stage_bytes);
        bulk_g2s(cs + kCodeStageBytes, p.xhat + static_cast<size_t>(st) * p.xhat_stage_bytes, p.xhat_stage_bytes,
                 xhat_full + i);
      }
    }
  } else if (lane == 0) {
    // ------------------------------------------------------------------ MMA issuer (one thread)
    const uint32_t idesc = idesc_f16_f32(kRows, 16);
    const uint32_t lbo = 16u * static_cast<uint32_t>(p.B), sbo = 128u;
    int gc = 0;
    bool alive = true;
    for (int u = u0; u < u1 && alive; ++u) {
      if (*s_abort) break;
      const int it = u - u0, i = it % S;
      if (!mbar_wait(xhat_full + i, (it / S) & 1)) {
        fail(p, s_abort);
        break;
      }
      tc_fence_after();
      const int st = u % p.spr;
      const int ngs = min(C::GPS, p.ng - st * C::GPS);
      const uint32_t xs = smem_addr(stages + static_cast<size_t>(i) * p.stage_smem + kCodeStageBytes);
      const uint32_t cs = xs + p.corr_offset;
      for (int gl = 0; gl < ngs; ++gl) {
        const int slot = gc % kRing;
        if (!mbar_wait(a_full + slot, (gc / kRing) & 1)) {
          fail(p, s_abort);
          alive = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tbase + C::D_COL0 + slot * 16;
#pragma unroll
        for (int s = 0; s < C::SLICES; ++s) {
          const uint32_t a = tbase + slot * C::GP + s * 8;
          const uint64_t bd = smem_desc_noswizzle(xs + ((gl * G + 16 * s) >> 3) * lbo, lbo, sbo);
          mma_f16_ts(d, a, bd, idesc, s > 0 ? 1u : 0u);
        }
        mma_f16_ts(d, tbase + C::C_COL0, smem_desc_noswizzle(cs + gl * lbo, lbo, sbo), idesc, 1u);
        mma_commit(mma_done + slot);
        ++gc;
      }
      mma_commit(empty + i);
    }
  }

  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------------------------
// Preparation: x (bf16 [B][K]) -> x^ blocks per stage, per-group correction, 2^(16+e) per group.
// One warp per 128-block of K handling every batch row; e is shared by the block's rows.
// ---------------------------------------------------------------------------------------------
template <int PACK>
__global__ void __launch_bounds__(256) xprep_kernel(const uint16_t* __restrict__ x, int B, int K, int G, int apply,
                                                    uint8_t* __restrict__ xhat, uint32_t stage_bytes,
                                                    uint32_t corr_off, float* __restrict__ pow2g,
                                                    int* __restrict__ counters, int n_counters, int* status) {
  constexpr int ST = Geo<PACK>::kStageTrits;
  pdl_launch_dependents();
  const int gtid = blockIdx.x * blockDim.x + threadIdx.x;
  for (int i = gtid; i < n_counters; i += gridDim.x * blockDim.x) counters[i] = 0;
  const int wid = gtid >> 5, lane = threadIdx.x & 31;
  if (wid >= K / kFwhtBlock) return;
  const int kb0 = wid * kFwhtBlock;
  const int GPS = ST / G;
  const int ng = K / G;
  float v[kMaxBatch][4];
  float mx = 0.f;
#pragma unroll
  for (int b = 0; b < kMaxBatch; ++b) {
    if (b < B) {
      const uint2 raw = *reinterpret_cast<const uint2*>(x + static_cast<size_t>(b) * K + kb0 + 4 * lane);
      v[b][0] = bf16_bits_to_float(static_cast<uint16_t>(raw.x & 0xffffu));
      v[b][1] = bf16_bits_to_float(static_cast<uint16_t>(raw.x >> 16));
      v[b][2] = bf16_bits_to_float(static_cast<uint16_t>(raw.y & 0xffffu));
      v[b][3] = bf16_bits_to_float(static_cast<uint16_t>(raw.y >> 16));
      if (apply) {
        fwht128_warp(v[b]);
#pragma unroll
        for (int j = 0; j < 4; ++j) v[b][j] *= 0.08838834764831845f;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) mx = fmaxf(mx, fabsf(v[b][j]));
    }
  }
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
  const float down = __int_as_float((127 - e) << 23);  // 2^-e
  const int st = kb0 / ST;
  const int kin = kb0 - st * ST;
  uint8_t* sbase = xhat + static_cast<size_t>(st) * stage_bytes;
#pragma unroll
  for (int b = 0; b < kMaxBatch; ++b) {
    if (b < B) {
      float vsum = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int k = kb0 + 4 * lane + j;
        const int kk = kin + 4 * lane + j;
        int pos, slot;
        if (PACK == TQ_PACK_B3) {
          pos = ((k % 20) % 10) >> 1;
          slot = kk;
        } else {
          const int f = k & 15, jj = f & 7;
          pos = jj < 5 ? jj : jj - 5;
          slot = (kk & ~15) + 2 * jj + (f >> 3);
        }
        const float F = __int_as_float((127 + 8 - 2 * pos) << 23);     // 2^(8 - 2 pos)
        const float Finv = __int_as_float((127 - 8 + 2 * pos) << 23);  // 2^(2 pos - 8)
        const __half h = __float2half_rn(v[b][j] * down * F);
        vsum += __half2float(h) * Finv;
        *reinterpret_cast<uint16_t*>(sbase + (slot >> 3) * 16 * B + b * 16 + (slot & 7) * 2) = __half_as_ushort(h);
      }
      if (G == 128) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) vsum += __shfl_xor_sync(0xffffffffu, vsum, o);
      } else {
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) vsum += __shfl_xor_sync(0xffffffffu, vsum, o);
      }
      if ((lane & (G == 128 ? 31 : 15)) == 0) {
        const int g = kb0 / G + (G == 64 ? (lane >> 4) : 0);
        const int gl = g - st * GPS;
        const __half hi = __float2half_rn(-vsum);
        const __half lo = __float2half_rn(-vsum - __half2float(hi));
        const uint4 cv = make_uint4(static_cast<uint32_t>(__half_as_ushort(hi)) |
                                        (static_cast<uint32_t>(__half_as_ushort(lo)) << 16),
                                    0u, 0u, 0u);
        *reinterpret_cast<uint4*>(sbase + corr_off + gl * 16 * B + b * 16) = cv;
      }
    }
  }
  if (lane == 0) {
    const float p2 = __int_as_float((127 + 16 + e) << 23);  // 2^(16 + e)
    for (int g = kb0 / G; g < (kb0 + kFwhtBlock) / G; ++g) pow2g[g] = p2;
  }
  if (kin == 0) {
    // correction chunks of groups that do not exist in this stage, and the trailing zero chunk
    const int ngs = min(GPS, ng - st * GPS);
    const int n16 = (GPS + 1 - ngs) * B;
    uint4* z = reinterpret_cast<uint4*>(sbase + corr_off + ngs * 16 * B);
    for (int i = lane; i < n16; i += 32) z[i] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// ---------------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------------
struct Plan {
  int ST, GPS, spr, n_tiles, units, ng;
  uint32_t stage_bytes, corr_off;
  size_t off_pow2, off_cnt, off_part, total;
};

Plan make_plan(const tq_desc* d, int B) {
  Plan pl{};
  pl.ST = d->packing == TQ_PACK_B3 ? 640 : 512;
  pl.GPS = pl.ST / d->group;
  pl.spr = (d->K + pl.ST - 1) / pl.ST;
  pl.n_tiles = (d->N + kRows - 1) / kRows;
  pl.units = pl.n_tiles * pl.spr;
  pl.ng = d->K / d->group;
  pl.corr_off = static_cast<uint32_t>(pl.ST * 2 * B);
  pl.stage_bytes = pl.corr_off + static_cast<uint32_t>((pl.GPS + 1) * 16 * B);
  size_t off = align256(static_cast<size_t>(pl.spr) * pl.stage_bytes);
  pl.off_pow2 = off;
  off += align256(static_cast<size_t>(pl.ng) * 4);
  pl.off_cnt = off;
  off += align256(static_cast<size_t>(pl.n_tiles) * 4);
  pl.off_part = off;
  off += align256(static_cast<size_t>(pl.n_tiles) * pl.spr * B * kRows * 4);
  pl.total = off;
  return pl;
}

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cache[dev]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
    cache[dev] = v;
  }
  return cache[dev];
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

template <int PACK, int G, int NB>
cudaError_t launch_main(const Params& prm0, int grid, cudaStream_t s) {
  using C = Cfg<PACK, G>;
  Params prm = prm0;
  const size_t fixed = C::LUT_BYTES + 8 * (3 * kMaxStages + 2 * kRing + 1) + 32 + kRing * kRows * 4 + 1024;
  const int optin = max_smem_optin();
  int S = kMaxStages;
  while (S > 2 && fixed + static_cast<size_t>(S) * prm.stage_smem > static_cast<size_t>(optin)) --S;
  prm.stages = S;
  const size_t smem = C::LUT_BYTES + static_cast<size_t>(S) * prm.stage_smem + 8 * (3 * S + 2 * kRing + 1) + 32 +
                      kRing * kRows * 4;
  if (smem > static_cast<size_t>(optin)) return cudaErrorInvalidConfiguration;
  // ask for more than half of the SM's shared memory so that exactly one CTA runs per SM (each
  // CTA holds up to 512 TMEM columns)
  const size_t smem_req = std::max(smem, static_cast<size_t>(optin / 2 + 1024));
  auto kern = gemv_tc_kernel<PACK, G, NB>;
  static bool attr_set = false;  // per instantiation
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_req;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, prm);
}

template <int PACK, int G>
cudaError_t launch_nb(const Params& prm, int grid, cudaStream_t s) {
  const int B = prm.B;
  if (B <= 1) return launch_main<PACK, G, 1>(prm, grid, s);
  if (B <= 2) return launch_main<PACK, G, 2>(prm, grid, s);
  if (B <= 4) return launch_main<PACK, G, 4>(prm, grid, s);
  if (B <= 8) return launch_main<PACK, G, 8>(prm, grid, s);
  return launch_main<PACK, G, 16>(prm, grid, s);
}

}  // namespace gemv_tc

size_t gemv_tc_workspace_bytes(const tq_desc* d, int batch) { return gemv_tc::make_plan(d, batch).total; }

cudaError_t launch_gemv_tc(const tq_desc* d, const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                           int B, float* y, void* ws, cudaStream_t s) {
  using namespace gemv_tc;
  const Plan pl = make_plan(d, B);
  uint8_t* base = static_cast<uint8_t*>(ws);
  Params prm{};
  prm.codes = codes;
  prm.scales = scales;
  prm.xhat = base;
  prm.pow2g = reinterpret_cast<float*>(base + pl.off_pow2);
  prm.y = y;
  prm.partial = reinterpret_cast<float*>(base + pl.off_part);
  prm.counters = reinterpret_cast<int*>(base + pl.off_cnt);
  prm.status = status_ptr();
  prm.N = d->N;
  prm.K = d->K;
  prm.P = pitch_words(d->K, d->packing);
  prm.ng = pl.ng;
  prm.B = B;
  prm.n_tiles = pl.n_tiles;
  prm.spr = pl.spr;
  prm.units = pl.units;
  prm.xhat_stage_bytes = pl.stage_bytes;
  prm.corr_offset = pl.corr_off;
  prm.stage_smem = static_cast<uint32_t>(kCodeStageBytes + ((pl.stage_bytes + 256 + 127) / 128) * 128);
  const int warps = d->K / kFwhtBlock;
  const int xblocks = (warps * 32 + 255) / 256;
  const int apply = d->fwht_block != 0;
  if (d->packing == TQ_PACK_B3)
    xprep_kernel<TQ_PACK_B3><<<xblocks, 256, 0, s>>>(x, B, d->K, d->group, apply, base, pl.stage_bytes, pl.corr_off,
                                                      const_cast<float*>(prm.pow2g), prm.counters, pl.n_tiles,
                                                      prm.status);
  else
    xprep_kernel<TQ_PACK_2BIT><<<xblocks, 256, 0, s>>>(x, B, d->K, d->group, apply, base, pl.stage_bytes,
                                                        pl.corr_off, const_cast<float*>(prm.pow2g), prm.counters,
                                                        pl.n_tiles, prm.status);
  cudaError_t e = cudaPeekAtLastError();
  if (e != cudaSuccess) return e;
  const int grid = std::min(num_sms(), pl.units);
  if (d->packing == TQ_PACK_B3)
    return d->group == 128 ? launch_nb<TQ_PACK_B3, 128>(prm, grid, s) : launch_nb<TQ_PACK_B3, 64>(prm, grid, s);
  return d->group == 128 ? launch_nb<TQ_PACK_2BIT, 128>(prm, grid, s) : launch_nb<TQ_PACK_2BIT, 64>(prm, grid, s);
}

}  // namespace tq

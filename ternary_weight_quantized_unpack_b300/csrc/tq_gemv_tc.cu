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
#include "tq_tmap.cuh"

namespace tq {
namespace gemv_tc {

using namespace sm100;

constexpr int kRows = 128;                // rows per tile = MMA M = TMEM lanes
constexpr int kStageWords = 32;           // code words per row per stage (128 bytes)
constexpr int kCodeStageBytes = kRows * kStageWords * 4;  // 16 KB, 128B-swizzled by the TMA
constexpr int kKLanes = 4;                // decode warp groups working on different stages
constexpr int kDecodeWarps = 4 * kKLanes; // 4 lane quarters x 4 K-lanes
constexpr int kProducerWarp = kDecodeWarps;  // also owns the TMEM allocation
constexpr int kThreads = 32 * (kDecodeWarps + 1);
constexpr uint32_t kLutBytes = 2u * 243u * 32u * 4u;
constexpr int kMaxStages = 8;

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
  static constexpr int GPS = ST / G;        // groups per stage
  static constexpr int CPG = G / 64;        // 64-trit chunks (32 TMEM columns) per group
  static constexpr int CPS = ST / 64;       // chunks per stage
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

// TMEM columns (512 allocated): K-lane j owns A chunk slots [64j, 64j+64) (2 x 32 columns) and
// D slots [256 + 32j, 256 + 32j + 32) (2 x 16 columns); the constant correction A is at 384.
constexpr int kTmemCols = 512;
constexpr int kDCol0 = 256;
constexpr int kCCol = 384;

struct Params {
  CUtensorMap tmap;         // codes [N][P] uint32, box 32 words x 128 rows, 128B swizzle
  const uint16_t* scales;
  const uint8_t* xhat;      // prepared activations, one block per stage (x^, corrections, 2^(16+e))
  float* y;
  float* partial;           // [unit][B][128] partial outputs, indexed by the first unit of a part
  int* counters;            // [tile] arrivals (zeroed by the preparation kernel, reset by the last arriver)
  int* status;
  int N, K, P, ng, B, n_tiles, spr, units;
  uint32_t xhat_stage_bytes;  // bytes of one stage block
  uint32_t corr_offset;       // offset of the correction chunks inside a stage block
  uint32_t pow2_offset;       // offset of the per-group 2^(16+e) floats inside a stage block
  uint32_t stage_smem;        // shared-memory bytes per pipeline stage (multiple of 1024)
  int stages;                 // pipeline depth
};

__device__ __forceinline__ void fail(const Params& p, volatile int* s_abort) {
  record_error(p.status, TQ_ERR_TIMEOUT);
  *s_abort = 1;
}

// Static stream-K partition: CTA c owns units [floor(c U / G), floor((c+1) U / G)); inside a CTA,
// K-lane j owns the contiguous run [first + floor(j n / 4), first + floor((j+1) n / 4)).  Stages are
// loaded into the ring round-robin over K-lanes (m-th unit of K-lane 0, 1, 2, 3, then m+1, ...).
__device__ __forceinline__ int cta_first_unit(int c, int units, int grid) {
  return static_cast<int>(static_cast<unsigned>(c) * static_cast<unsigned>(units) / static_cast<unsigned>(grid));
}
__device__ __forceinline__ int cta_of_unit(int u, int units, int grid) {
  return static_cast<int>((static_cast<unsigned>(u + 1) * static_cast<unsigned>(grid) + units - 1) /
                          static_cast<unsigned>(units)) - 1;
}
__device__ __forceinline__ int klane_begin(int j, int n) { return (j * n) >> 2; }
// Ring position of the m-th unit of K-lane j, given the K-lane run lengths len[4].
__device__ __forceinline__ int ring_pos(int j, int m, const int (&len)[kKLanes]) {
  int pos = 0;
#pragma unroll
  for (int q = 0; q < kKLanes; ++q) pos += min(len[q], m) + ((q < j && m < len[q]) ? 1 : 0);
  return pos;
}
// A part is the run of units of one tile decoded by one K-lane of one CTA; unit u starts a part when
// it begins a tile or begins a K-lane run.
__device__ __forceinline__ bool starts_part(int u, int spr, int units, int grid) {
  if (u % spr == 0) return true;
  const int c = cta_of_unit(u, units, grid);
  const int first = cta_first_unit(c, units, grid);
  const int n = cta_first_unit(c + 1, units, grid) - first;
  const int d = u - first;
  return d == 0 || d == klane_begin(1, n) || d == klane_begin(2, n) || d == klane_begin(3, n);
}
// Bit k set <=> unit t * spr + k starts a part (spr <= 64).  Whole warp.
__device__ __forceinline__ unsigned long long part_mask(int t, int spr, int units, int grid, int lane) {
  const bool a = lane < spr && starts_part(t * spr + lane, spr, units, grid);
  const bool b = lane + 32 < spr && starts_part(t * spr + lane + 32, spr, units, grid);
  return static_cast<unsigned long long>(__ballot_sync(0xffffffffu, a)) |
         (static_cast<unsigned long long>(__ballot_sync(0xffffffffu, b)) << 32);
}

// One decode thread of one K-lane.  Produces 64-trit chunks of FP16 pairs into its K-lane's two
// TMEM chunk slots.  When the K-lane's four warps have written a chunk, the K-lane leader (lane 0 of
// its first warp) issues the chunk's MMAs.  Chunk completions are consumed in order; when the last
// chunk of a group completes, its 128 x 16 result is folded into acc with the group's multiplier.
template <int PACK, int G, int NB>
struct Lane {
  using C = Cfg<PACK, G>;
  uint32_t tm;          // TMEM address of this warp's lane quarter, column 0
  uint32_t tbase;       // TMEM address of lane 0, column 0 (MMA operands)
  uint64_t* a_full;     // [2] of this K-lane
  uint64_t* mma_done;   // [2] of this K-lane
  uint64_t* empty_bar;  // the current stage's "empty" barrier
  float* m_ring;        // [2][128] multipliers of the groups in flight (this K-lane)
  volatile int* s_abort;
  const Params* p;
  uint32_t xs;          // shared address of the current stage's x^ block
  uint32_t lbo;
  int stage_chunks;     // chunks in the current stage
  int j, r, lane;
  bool leader;
  int cc, waited;       // chunks produced / chunks whose MMA completion has been consumed
  bool ok;
  float acc[NB];
  uint32_t stg[16];

  __device__ __forceinline__ uint32_t a_col() const { return tm + 64u * j + 32u * (cc & 1); }

  __device__ __forceinline__ void wait_next() {
    const int n = waited;
    bool w = mbar_wait(mma_done + (n & 1), (n >> 1) & 1);
    w = __all_sync(0xffffffffu, w);
    if (!w) {
      ok = false;
      if (lane == 0) fail(*p, s_abort);
      return;
    }
    if (n % C::CPG == C::CPG - 1) {  // last chunk of a group: its accumulator is final
      const int g = n / C::CPG;
      tc_fence_after();
      uint32_t d[NB];
      tmem_ld<NB>(tm + kDCol0 + 32u * j + 16u * (g & 1), d);
      tmem_wait_ld();
      const float m = m_ring[(g & 1) * kRows + r];
#pragma unroll
      for (int b = 0; b < NB; ++b) acc[b] = fmaf(m, __uint_as_float(d[b]), acc[b]);
    }
    ++waited;
  }
  __device__ __forceinline__ void begin_chunk() {
    while (ok && waited <= cc - 2) wait_next();
  }
  // c = chunk index within the stage; group_end: last chunk of its group, m = the group's multiplier
  __device__ __forceinline__ void end_chunk(int c, bool group_end, float m) {
    tmem_wait_st();
    tc_fence_before();
    if (group_end) m_ring[((cc / C::CPG) & 1) * kRows + r] = m;
    __syncwarp();
    if (lane == 0) mbar_arrive(a_full + (cc & 1));
    if (leader) {
      if (!mbar_wait(a_full + (cc & 1), (cc >> 1) & 1)) {
        fail(*p, s_abort);
      } else {
        tc_fence_after();
        const uint32_t idesc = idesc_f16_f32(kRows, 16);
        const int gl = c / C::CPG, half = c % C::CPG;
        const uint32_t d = tbase + kDCol0 + 32u * j + 16u * ((cc / C::CPG) & 1);
        const uint32_t a = tbase + 64u * j + 32u * (cc & 1);
#pragma unroll
        for (int s4 = 0; s4 < 4; ++s4) {
          const int slot = gl * G + half * 64 + 16 * s4;
          mma_f16_ts(d, a + 8u * s4, smem_desc_noswizzle(xs + (slot >> 3) * lbo, lbo, 128u), idesc,
                     (half == 0 && s4 == 0) ? 0u : 1u);
        }
        if (half == C::CPG - 1)
          mma_f16_ts(d, tbase + kCCol, smem_desc_noswizzle(xs + p->corr_offset + gl * lbo, lbo, 128u), idesc, 1u);
        mma_commit(mma_done + (cc & 1));
        if (c == stage_chunks - 1) mma_commit(empty_bar);  // every MMA reading this stage's x^ is issued
      }
    }
    __syncwarp();
    ++cc;
  }
  __device__ __forceinline__ void drain() {
    while (ok && waited < cc) wait_next();
  }
};

// Per-pair work shared by both decoders: stage 16 pairs, store, close chunks.
template <int PACK, int G, int NB, bool FULL>
__device__ __forceinline__ void put_pair(Lane<PACK, G, NB>& L, int q, uint32_t v, int ngs,
                                         const float (&mg)[Cfg<PACK, G>::GPS]) {
  const int gl = (2 * q) / G;  // group of pair q (pairs are 2 trits)
  if (!FULL && gl >= ngs) return;
  if (q % 32 == 0) L.begin_chunk();
  L.stg[q % 16] = v;
  if (q % 16 == 15) tmem_st16(L.a_col() + (q % 32) - 15, L.stg);
  if (q % 32 == 31) L.end_chunk(q / 32, (2 * q + 2) % G == 0, (2 * q + 2) % G == 0 ? mg[gl] : 0.f);
}

// Decode one stage (32 words) of base-3 codes: natural-order pairs (t_2j, t_2j+1).
template <int G, int NB, bool FULL>
__device__ __forceinline__ void decode_stage_b3(Lane<TQ_PACK_B3, G, NB>& L, const uint32_t (&w)[32],
                                                const uint32_t* __restrict__ lutA, const uint32_t* __restrict__ lutB,
                                                int ngs, const float (&mg)[Cfg<TQ_PACK_B3, G>::GPS]) {
#pragma unroll
  for (int wi = 0; wi < 32; ++wi) {
    if (!FULL && (wi * 20) / G >= ngs) break;
    const uint32_t v = min(w[wi], kB3Max);
    const uint32_t hi = __umulhi(v + 1u, 2383401723u) >> 15;  // v / 3^10, exact for v < 3^20
    const uint32_t lo = v - hi * 59049u;
    const uint32_t bl = __umulhi(lo, 17675008u);                // lo / 243, exact for lo < 3^10
    const uint32_t al = lo - bl * 243u;
    const uint32_t bh = __umulhi(hi, 17675008u);
    const uint32_t ah = hi - bh * 243u;
    const uint32_t P0 = lutA[al * 32] | lutB[bl * 32];
    const uint32_t P1 = lutA[ah * 32] | lutB[bh * 32];
#pragma unroll
    for (int jj = 0; jj < 10; ++jj)
      put_pair<TQ_PACK_B3, G, NB, FULL>(L, wi * 10 + jj, (jj < 5 ? P0 : P1) & (0x00030003u << (2 * (jj % 5))), ngs,
                                        mg);
  }
}

// Decode one stage (32 words) of 2-bit codes: pair j of a word = fields (j, j + 8).
template <int G, int NB, bool FULL>
__device__ __forceinline__ void decode_stage_2b(Lane<TQ_PACK_2BIT, G, NB>& L, const uint32_t (&w)[32], int ngs,
                                                const float (&mg)[Cfg<TQ_PACK_2BIT, G>::GPS]) {
#pragma unroll
  for (int wi = 0; wi < 32; ++wi) {
    if (!FULL && (wi * 16) / G >= ngs) break;
    const uint32_t v = w[wi];
    const uint32_t v2 = v >> 10;
#pragma unroll
    for (int jj = 0; jj < 8; ++jj)
      put_pair<TQ_PACK_2BIT, G, NB, FULL>(
          L, wi * 8 + jj, jj < 5 ? (v & (0x00030003u << (2 * jj))) : (v2 & (0x00030003u << (2 * (jj - 5)))), ngs, mg);
  }
}

template <int PACK, int G, int NB>
__global__ void __launch_bounds__(kThreads, 1) gemv_tc_kernel(const __grid_constant__ Params p) {
  using C = Cfg<PACK, G>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grid = static_cast<int>(gridDim.x);
  const int u0 = cta_first_unit(blockIdx.x, p.units, grid);
  const int n_units = cta_first_unit(blockIdx.x + 1, p.units, grid) - u0;
  const int S = p.stages;
  int kl_len[kKLanes];
#pragma unroll
  for (int q = 0; q < kKLanes; ++q) kl_len[q] = klane_begin(q + 1, n_units) - klane_begin(q, n_units);
  int max_len = 0;
#pragma unroll
  for (int q = 0; q < kKLanes; ++q) max_len = max(max_len, kl_len[q]);

  uint8_t* stages = smem;                                               // 1024-aligned stage buffers
  uint8_t* lut_smem = smem + static_cast<size_t>(S) * p.stage_smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(lut_smem + C::LUT_BYTES);
  uint64_t* codes_full = bars;
  uint64_t* xhat_full = bars + S;
  uint64_t* empty = bars + 2 * S;
  uint64_t* a_full = bars + 3 * S;            // [kKLanes][2]
  uint64_t* mma_done = a_full + 2 * kKLanes;  // [kKLanes][2]
  uint64_t* lut_bar = mma_done + 2 * kKLanes;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(lut_bar + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* m_ring = reinterpret_cast<float*>(lut_bar + 3);  // [kKLanes][2][128]

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(codes_full + i, 1);
      mbar_init(xhat_full + i, 1);
      mbar_init(empty + i, 5);  // the 4 warps of the stage's K-lane (codes read) + the leader's commit (x^ read)
    }
    for (int i = 0; i < 2 * kKLanes; ++i) {
      mbar_init(a_full + i, 4);
      mbar_init(mma_done + i, 1);
    }
    mbar_init(lut_bar, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
    if (lane == 0) tma_prefetch_desc(&p.tmap);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  if (warp < 4) {
    // constant A of the correction MMA: K-slots 0 and 1 hold 2^-16 (FP16 0x0100), the rest 0
    uint32_t cv[8] = {0x01000100u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    tmem_st8(tbase + (static_cast<uint32_t>(warp * 32) << 16) + kCCol, cv);
    tmem_wait_st();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();

  if (warp < kDecodeWarps) {
    // ------------------------------------------------------------- decode warps: K-lane j, quarter q
    const int q = warp & 3, j = warp >> 2;
    Lane<PACK, G, NB> L;
    L.tm = tbase + (static_cast<uint32_t>(q * 32) << 16);
    L.tbase = tbase;
    L.a_full = a_full + 2 * j;
    L.mma_done = mma_done + 2 * j;
    L.m_ring = m_ring + j * 2 * kRows;
    L.s_abort = s_abort;
    L.p = &p;
    L.lbo = 16u * static_cast<uint32_t>(p.B);
    L.j = j;
    L.r = q * 32 + lane;
    L.lane = lane;
    L.leader = q == 0 && lane == 0;
    L.cc = 0;
    L.waited = 0;
    L.ok = true;
    const uint32_t* lutA = reinterpret_cast<const uint32_t*>(lut_smem) + lane;
    const uint32_t* lutB = lutA + 243 * 32;
    if (PACK == TQ_PACK_B3) {
      bool w = mbar_wait(lut_bar, 0);
      w = __all_sync(0xffffffffu, w);
      if (!w) {
        L.ok = false;
        if (lane == 0) fail(p, s_abort);
      }
    }
    const int kbeg = u0 + klane_begin(j, n_units);
    const int klen = kl_len[j];
    int seg_first = kbeg;
    float sc[C::GPS];
    auto load_scales = [&](int u) {
      const int t = u / p.spr, st = u % p.spr;
      const int row = t * kRows + L.r;
      const int ngs = min(C::GPS, p.ng - st * C::GPS);
#pragma unroll
      for (int gl = 0; gl < C::GPS; ++gl)
        sc[gl] = (gl < ngs && row < p.N)
                     ? half_bits_to_float(__ldg(p.scales + static_cast<size_t>(row) * p.ng + st * C::GPS + gl))
                     : 0.f;
    };
    if (klen > 0) load_scales(kbeg);
#pragma unroll
    for (int b = 0; b < NB; ++b) L.acc[b] = 0.f;
    const int swz = L.r & 7;
    for (int m = 0; m < klen && L.ok; ++m) {
      if (__any_sync(0xffffffffu, *s_abort != 0)) break;
      const int u = kbeg + m;
      const int pos = ring_pos(j, m, kl_len);
      const int i = pos % S;
      const uint32_t par = (pos / S) & 1;
      const int t = u / p.spr, st = u % p.spr;
      const int row = t * kRows + L.r;
      const int ngs = min(C::GPS, p.ng - st * C::GPS);
      float cur[C::GPS];
#pragma unroll
      for (int gl = 0; gl < C::GPS; ++gl) cur[gl] = sc[gl];
      if (m + 1 < klen) load_scales(u + 1);  // prefetch for the next unit
      bool w = mbar_wait(codes_full + i, par);
      w = __all_sync(0xffffffffu, w);
      if (!w) {
        L.ok = false;
        if (lane == 0) fail(p, s_abort);
        break;
      }
      uint32_t cw[32];
      {
        // row r of the 128B-swizzled tile: 16-byte chunk k sits at position k ^ (r & 7)
        const uint8_t* rowp = stages + static_cast<size_t>(i) * p.stage_smem + L.r * 128;
#pragma unroll
        for (int k4 = 0; k4 < 8; ++k4) {
          const uint4 v = *reinterpret_cast<const uint4*>(rowp + ((k4 ^ swz) << 4));
          cw[4 * k4] = v.x;
          cw[4 * k4 + 1] = v.y;
          cw[4 * k4 + 2] = v.z;
          cw[4 * k4 + 3] = v.w;
        }
      }
      if (row >= p.N) {
#pragma unroll
        for (int k4 = 0; k4 < 32; ++k4) cw[k4] = PACK == TQ_PACK_B3 ? kB3Zero : kB2Zero;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + i);
      // per-group multipliers s * 2^(16+e): 2^(16+e) travels with the stage's x^ block
      w = mbar_wait(xhat_full + i, par);
      w = __all_sync(0xffffffffu, w);
      if (!w) {
        L.ok = false;
        if (lane == 0) fail(p, s_abort);
        break;
      }
      uint8_t* xblk = stages + static_cast<size_t>(i) * p.stage_smem + kCodeStageBytes;
      const float* pw = reinterpret_cast<const float*>(xblk + p.pow2_offset);
      float mg[C::GPS];
#pragma unroll
      for (int gl = 0; gl < C::GPS; ++gl) mg[gl] = cur[gl] * pw[gl];
      L.xs = smem_addr(xblk);
      L.empty_bar = empty + i;
      L.stage_chunks = ngs * C::CPG;
      if constexpr (PACK == TQ_PACK_B3) {
        if (ngs == C::GPS)
          decode_stage_b3<G, NB, true>(L, cw, lutA, lutB, ngs, mg);
        else
          decode_stage_b3<G, NB, false>(L, cw, lutA, lutB, ngs, mg);
      } else {
        if (ngs == C::GPS)
          decode_stage_2b<G, NB, true>(L, cw, ngs, mg);
        else
          decode_stage_2b<G, NB, false>(L, cw, ngs, mg);
      }
      if (!L.ok) break;
      // end of this K-lane's part of tile t: fold in its last groups, then publish
      if (m + 1 == klen || (u + 1) % p.spr == 0) {
        L.drain();
        if (!L.ok) break;
        const unsigned long long mask = part_mask(t, p.spr, p.units, grid, lane);
        const int n_parts = __popcll(mask);
        if (n_parts == 1) {
          if (row < p.N)
#pragma unroll
            for (int b = 0; b < NB; ++b)
              if (b < p.B) p.y[static_cast<size_t>(b) * p.N + row] = L.acc[b];
        } else {
          float* pp = p.partial + static_cast<size_t>(seg_first) * p.B * kRows;
#pragma unroll
          for (int b = 0; b < NB; ++b)
            if (b < p.B) pp[b * kRows + L.r] = L.acc[b];
          __threadfence();
          __syncwarp();
          int last = 0;
          if (lane == 0) {
            const int old = atomicAdd(p.counters + t, 1);
            last = old == 4 * n_parts - 1;  // 4 warps (lane quarters) per part
            if (last) p.counters[t] = 0;
            __threadfence();
          }
          last = __shfl_sync(0xffffffffu, last, 0);
          if (last) {
            // this warp sums every part of the tile, in unit order: deterministic
            for (int rr = lane; rr < kRows; rr += 32) {
              const int rrow = t * kRows + rr;
              if (rrow >= p.N) break;
              for (int b = 0; b < p.B; ++b) {
                float v = 0.f;
                unsigned long long mm = mask;
                while (mm) {
                  const int k = __ffsll(static_cast<long long>(mm)) - 1;
                  mm &= mm - 1;
                  v += __ldcg(p.partial + (static_cast<size_t>(t * p.spr + k) * p.B + b) * kRows + rr);
                }
                p.y[static_cast<size_t>(b) * p.N + rrow] = v;
              }
            }
          }
        }
        seg_first = u + 1;
#pragma unroll
        for (int b = 0; b < NB; ++b) L.acc[b] = 0.f;
      }
    }
    L.drain();
  } else {
    // ------------------------------------------------------------- producer warp (lane 0)
    if (lane == 0) {
      if (PACK == TQ_PACK_B3) {
        mbar_arrive_expect_tx(lut_bar, kLutBytes);
        bulk_g2s(lut_smem, &g_lut, kLutBytes, lut_bar);
      }
      bool pdl_done = false;
      int pos = 0;
      bool alive = true;
      for (int m = 0; m < max_len && alive; ++m) {
        for (int jj = 0; jj < kKLanes; ++jj) {
          if (m >= kl_len[jj]) continue;
          if (*s_abort) {
            alive = false;
            break;
          }
          const int u = u0 + klane_begin(jj, n_units) + m;
          const int i = pos % S;
          if (!mbar_wait(empty + i, ((pos / S) & 1) ^ 1)) {
            fail(p, s_abort);
            alive = false;
            break;
          }
          const int t = u / p.spr, st = u % p.spr;
          uint8_t* cs = stages + static_cast<size_t>(i) * p.stage_smem;
          mbar_arrive_expect_tx(codes_full + i, static_cast<uint32_t>(kCodeStageBytes));
          tma_load_2d(cs, &p.tmap, st * kStageWords, t * kRows, codes_full + i);
          if (!pdl_done) {
            pdl_wait();  // x^ comes from the preparation kernel
            pdl_done = true;
          }
          mbar_arrive_expect_tx(xhat_full + i, p.xhat_stage_bytes);
          bulk_g2s(cs + kCodeStageBytes, p.xhat + static_cast<size_t>(st) * p.xhat_stage_bytes, p.xhat_stage_bytes,
                   xhat_full + i);
          ++pos;
        }
      }
    }
  }

  __syncthreads();
  if (warp == kProducerWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

// ---------------------------------------------------------------------------------------------
// Preparation: x (bf16 [B][K]) -> x^ blocks per stage, per-group correction, 2^(16+e) per group.
// One warp per 128-block of K handling every batch row; e is shared by the block's rows.
// ---------------------------------------------------------------------------------------------
template <int PACK>
__global__ void __launch_bounds__(256) xprep_kernel(const uint16_t* __restrict__ x, int B, int K, int G, int apply,
                                                    uint8_t* __restrict__ xhat, uint32_t stage_bytes,
                                                    uint32_t corr_off, uint32_t pow2_off,
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
    for (int g = kb0 / G; g < (kb0 + kFwhtBlock) / G; ++g)
      reinterpret_cast<float*>(sbase + pow2_off)[g - st * GPS] = p2;
  }
  if (kin == 0) {
    // correction chunks of groups that do not exist in this stage, the trailing zero chunk, and
    // the multipliers of the missing groups
    const int ngs = min(GPS, ng - st * GPS);
    const int n16 = (GPS + 1 - ngs) * B;
    uint4* z = reinterpret_cast<uint4*>(sbase + corr_off + ngs * 16 * B);
    for (int i = lane; i < n16; i += 32) z[i] = make_uint4(0u, 0u, 0u, 0u);
    for (int gl = ngs + lane; gl < GPS; gl += 32) reinterpret_cast<float*>(sbase + pow2_off)[gl] = 0.f;
  }
}

// ---------------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------------
struct Plan {
  int ST, GPS, spr, n_tiles, units, ng;
  uint32_t stage_bytes, corr_off, pow2_off;
  size_t off_cnt, off_part, total;
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
  pl.pow2_off = pl.corr_off + static_cast<uint32_t>((pl.GPS + 1) * 16 * B);
  pl.stage_bytes = pl.pow2_off + static_cast<uint32_t>(((pl.GPS * 4 + 15) / 16) * 16);
  size_t off = align256(static_cast<size_t>(pl.spr) * pl.stage_bytes);
  pl.off_cnt = off;
  off += align256(static_cast<size_t>(pl.n_tiles) * 4);
  pl.off_part = off;
  off += align256(static_cast<size_t>(pl.units) * B * kRows * 4);
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
  auto smem_for = [&](int S) {
    return static_cast<size_t>(S) * prm.stage_smem + C::LUT_BYTES + 8 * (3 * S + 4 * kKLanes + 1) + 24 +
           kKLanes * 2 * kRows * 4;
  };
  const int optin = max_smem_optin();
  int S = kMaxStages;
  while (S > 2 && smem_for(S) > static_cast<size_t>(optin)) --S;
  prm.stages = S;
  const size_t smem = smem_for(S);
  if (smem > static_cast<size_t>(optin)) return cudaErrorInvalidConfiguration;
  // more than half of the SM's shared memory: exactly one CTA (and one 512-column TMEM block) per SM
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
  if (!make_tmap_2d(&prm.tmap, codes, CU_TENSOR_MAP_DATA_TYPE_UINT32, static_cast<uint64_t>(pitch_words(d->K, d->packing)),
                    static_cast<uint64_t>(d->N), static_cast<uint64_t>(pitch_words(d->K, d->packing)) * 4,
                    kStageWords, kRows, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  prm.scales = scales;
  prm.xhat = base;
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
  prm.pow2_offset = pl.pow2_off;
  prm.stage_smem = static_cast<uint32_t>(((kCodeStageBytes + pl.stage_bytes + 256 + 1023) / 1024) * 1024);
  const int warps = d->K / kFwhtBlock;
  const int xblocks = (warps * 32 + 255) / 256;
  const int apply = d->fwht_block != 0;
  if (d->packing == TQ_PACK_B3)
    xprep_kernel<TQ_PACK_B3><<<xblocks, 256, 0, s>>>(x, B, d->K, d->group, apply, base, pl.stage_bytes, pl.corr_off,
                                                      pl.pow2_off, prm.counters, pl.n_tiles, prm.status);
  else
    xprep_kernel<TQ_PACK_2BIT><<<xblocks, 256, 0, s>>>(x, B, d->K, d->group, apply, base, pl.stage_bytes,
                                                        pl.corr_off, pl.pow2_off, prm.counters, pl.n_tiles,
                                                        prm.status);
  cudaError_t e = cudaPeekAtLastError();
  if (e != cudaSuccess) return e;
  const int grid = std::min(num_sms(), pl.units);
  if (d->packing == TQ_PACK_B3)
    return d->group == 128 ? launch_nb<TQ_PACK_B3, 128>(prm, grid, s) : launch_nb<TQ_PACK_B3, 64>(prm, grid, s);
  return d->group == 128 ? launch_nb<TQ_PACK_2BIT, 128>(prm, grid, s) : launch_nb<TQ_PACK_2BIT, 64>(prm, grid, s);
}

}  // namespace tq

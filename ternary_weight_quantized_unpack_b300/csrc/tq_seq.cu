// Decode step: a sequence of dependent 2-bit or base-3 ternary GEMVs in one persistent launch (the
// base-3 kernel, further down, shares everything but the item decode).
//
// Decoding one token runs every linear of the model once, each on the previous one's output.  Issued
// as separate kernels, every call pays a launch, an activation fetch and transform, and a tail in
// which the weight stream stops.  Here one cooperative launch (one CTA per SM, all resident) runs the
// whole chain:
//
//  * Every warp streams its own weight tiles with 2-D TMA (32 rows x 32 code words = 512 trits of
//    each row, 128-byte swizzle, plus the matching 32 x 8 FP16 scales) into a private ring of
//    shared-memory stages.  The ring runs ahead across call boundaries: while the grid waits on a
//    barrier and the next input is being transformed, the next call's weights are already in flight.
//  * After a call's items, one grid-wide barrier (a counter in the workspace, bounded wait): every
//    partial sum of the call is written.  Each CTA then turns its share of the call's output rows
//    into final values (partial sums added in K order, times the output scale) and hands them over:
//    at batch 1 and 2 as (epoch, value) words that the next call's readers poll directly, at batch 4
//    and 8 by raising a ready flag for which those readers wait (bounded) before loading the rows.
//    Partial sums and sums of squares alternate between two buffers by the parity of the call, so a
//    CTA may start the next call while others still finalize this one.
//  * Work split, K-major: the items (32-row unit ru, 512-trit K slice ku) of a call are ordered by
//    ku, then ru, and divided into equal contiguous ranges, one per CTA (and each into ranges for
//    its warps).  A CTA therefore works on one or two K slices of many row units: it transforms only
//    the activations of its own slices, and every item writes its own partial sums (32 rows x batch)
//    to the workspace; the CTA that finalizes an output row adds its K slices' partial sums in ku
//    order, so results do not depend on timing.
//  * Decode and multiply-add are those of the 2-bit decode GEMV: a digit d = t + 1 in mantissa bits
//    2i of an FP16 half is the subnormal d * 2^(2i-24), one LOP3 per operand register, mma.sync
//    m16n8k16 with FP32 accumulation.  Each group of 64 or 128 weights has its own FP16 scale
//    ("27B 大模型塞进 5.9GB", section 二 ②); every MMA covers one group.  The MMA's eight columns are
//    shared by batch rows and groups: column c holds group (c / Bp) of the cycle for batch row
//    c % Bp, so at batch 1 four (group 128) or eight (group 64) groups accumulate side by side and
//    the scale is folded once per cycle rather than once per group.
//  * The input of each call is the block Walsh-Hadamard transform (same page, section 二 ①) of a bf16
//    vector, of the previous call's output, of that output divided by its root mean square (the
//    normalisation a pre-norm decoder applies before its attention and FFN projections), or of
//    silu(gate) * up of the previous call's output (the SwiGLU of a stacked gate/up projection).
//    The RMS factor is a per-call scalar: the call computes W * FWHT(input) and the finalize step
//    multiplies by 1 / rms, formed from per-block sums of squares the input transform stores.
#include <algorithm>
#include <cstring>
#include <new>
#include <vector>

#include "tq_b3.cuh"
#include "tq_internal.cuh"
#include "tq_kernels.cuh"
#include "tq_sm100.cuh"
#include "tq_tmap.cuh"

namespace tq {
namespace seq {

using namespace sm100;

constexpr int kNW = 12;                        // warps per CTA
// Ring stages per warp: three while the batch is small, two at four or eight batch rows.
__host__ __device__ constexpr int ring_depth(int Bp) { return Bp <= 2 ? 3 : 2; }
constexpr int kGatherKu = 12;                  // partial sums one thread adds in one go
constexpr int kRows = 32;                      // rows per item: two 16-row MMA slabs
constexpr int kItemTrits = 512;                // trits per item along K: 32 code words of a row
constexpr uint32_t kCodeStage = kRows * 128u;  // one item's codes: 4 KB (128-byte swizzled rows)
constexpr uint32_t kScaleStage = kRows * 16u;  // 8 FP16 scales per row: 512 B
constexpr uint32_t kStageBytes = kCodeStage + kScaleStage;
constexpr size_t kSmemLimit = 227 * 1024;
constexpr float kRmsEps = 1e-6f;  // RMS normalisation of an input: x / sqrt(mean(x^2) + eps)

// Device copy of one call; 128-byte aligned, tensor maps first (they must be 64-byte aligned).
struct alignas(128) CallDev {
  CUtensorMap tm_codes;   // codes [N][P] uint32, box {32 words, 32 rows}, 128-byte swizzle
  CUtensorMap tm_scales;  // scales [N][ng] FP16, box {8 groups, 32 rows}
  const uint16_t* x;      // mode 0: bf16 [B][K]
  const uint16_t* scales; // FP16 [N][ng] (base-3: read with plain loads; 2-bit: through tm_scales)
  float* y;               // [B][N]
  int T;                  // items = nru * nku (T * grid < 2^31)
  int N, K, ng, mode, apply;
  int nru, nku, gp;       // 32-row units, 512-trit K slices, CTAs taking part
};
static_assert(sizeof(CallDev) % 128 == 0, "call records are 128-byte aligned");

// The fields of a call the kernel reads repeatedly, kept in registers.
struct CallLite {
  const uint16_t* x;
  const uint16_t* scales;
  float* y;
  int T, N, K, ng, mode, apply, nru, nku, gp;
  __device__ __forceinline__ explicit CallLite(const CallDev& c)
      : x(c.x), scales(c.scales), y(c.y), T(c.T), N(c.N), K(c.K), ng(c.ng), mode(c.mode), apply(c.apply), nru(c.nru), nku(c.nku),
        gp(c.gp) {}
};

struct Params {
  const CallDev* calls;
  int ncalls, B;
  int* status;
  unsigned* sync;         // [0]: barrier arrivals, [1]: CTAs that have exited, [2]: launches completed,
                          // [64 + cta]: ready flags
  float* part;            // partial sums: [2][items][Bp][32] (parity of the call)
  uint64_t* hand;         // batch 1-2: each call's output as (epoch << 32 | value bits): [2][Bp][N]
  size_t hand_stride;     // words per parity of hand
  float* ssq;             // per 128-block sums of squares of an RMS-normalised input: [2][blocks][Bp]
  size_t part_stride;     // floats per parity of part
  int ssq_stride;         // floats per parity of ssq
  int nkc;                // K slices one CTA may cover (x^ capacity)
  uint32_t off_scales, off_xh, off_zero, off_v, off_f, off_bar, off_misc, off_lut;
};

// ---- static work split (K-major) ---------------------------------------------------------------
__host__ __device__ __forceinline__ int cta_start(int T, int gp, int cta) {
  return static_cast<int>(static_cast<unsigned>(T) * static_cast<unsigned>(cta) / static_cast<unsigned>(gp));
}

// This warp's items [a, b) of call c: the CTA's equal share of the call's items, split evenly over
// its nw warps.
__device__ __forceinline__ void warp_items(const CallLite& c, int cta, int warp, int nw, int& a, int& b) {
  if (cta >= c.gp) {
    a = b = 0;
    return;
  }
  const int ca = cta_start(c.T, c.gp, cta), cb = cta_start(c.T, c.gp, cta + 1), tc = cb - ca;
  a = ca + (tc * warp) / nw;
  b = ca + (tc * (warp + 1)) / nw;
}

// ---- waits ---------------------------------------------------------------------------------------
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid barrier number k (after call k), in two halves so that work that does not depend on it can
// run in between: grid_arrive_release (thread 0, after a CTA barrier: adds one with release
// semantics, so every write of the CTA before the barrier is visible to a thread that acquires the
// count) and grid_wait (every thread; thread 0 waits with acquire loads until every CTA has arrived,
// false if limit_ns passed first).
__device__ __forceinline__ void grid_arrive_release(unsigned* sync) {
  asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(sync) : "memory");
}
__device__ __forceinline__ bool grid_wait(unsigned* sync, unsigned k, int* flag, uint64_t limit_ns = kWaitNs) {
  if (threadIdx.x == 0) {
    *flag = 1;
    const unsigned target = (k + 1) * gridDim.x;
    if (ld_acquire(sync) < target) {
      const uint64_t t0 = global_timer_ns();
      for (uint32_t i = 0;; ++i) {
        if (ld_acquire(sync) >= target) break;
        if ((i & 63u) == 63u && global_timer_ns() - t0 > limit_ns) {
          *flag = 0;
          break;
        }
      }
    }
  }
  __syncthreads();  // the acquire above and this barrier order every thread's later reads
  return *flag != 0;
}

// Ready flags: CTA c stores j + 1 in flags[c] (release, after a CTA barrier) once its rows of call
// j's output are final.
constexpr int kFlagBase = 64;  // flags start at this word of the sync area
__device__ __forceinline__ void st_release(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Rows [fr0, fr1) of an N-row output that CTA c of `grid` finalizes.
__device__ __forceinline__ void fin_rows(int N, int c, int grid, int& fr0, int& fr1) {
  fr0 = (c * (N / 4)) / grid * 4;
  fr1 = ((c + 1) * (N / 4)) / grid * 4;
}
// The CTA whose fin_rows range holds row r (a multiple of 4): the least c with r < fr1(c).
__device__ __forceinline__ int fin_owner(int N, int grid, int r) {
  return static_cast<int>((static_cast<long long>(r / 4 + 1) * grid - 1) / (N / 4));
}
// One thread waits (bounded) until a ready flag reaches `want`; its later loads are ordered after the
// acquire.  False on timeout.
__device__ __forceinline__ bool wait_flag(const unsigned* flag, unsigned want) {
  if (ld_acquire(flag) >= want) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 0;; ++i) {
    if (ld_acquire(flag) >= want) return true;
    if ((i & 63u) == 63u && global_timer_ns() - t0 > kWaitNs) return false;
  }
}

// ---- handoff of a finished call's output (batch 1 and 2) -------------------------------------------
// The lanes that finalize an output value also write it with its call's epoch in one 64-bit word
// (epoch in the high half, the float's bits in the low half; launch-unique: launches completed x
// calls + call + 1).  A consumer polls the words it reads: a word whose epoch matches carries the
// value itself, so reading needs one L2 round trip where a ready flag and then the rows took two.
// One 64-bit access is single-copy atomic, so a value is never seen with another call's epoch.  A
// CTA barrier still follows the finalize, so that no warp polls while its own CTA finalizes (without
// it the spinning warps took the finalizing warps' issue slots: 3.4 instead of 3.0 ms per 2-bit
// token).  Batch 4 and 8 keep the ready flags: their first polls would need too many registers.
__host__ __device__ constexpr bool hand_batch(int Bp) { return Bp <= 2; }
__device__ __forceinline__ void st_hand2(uint64_t* p, uint64_t a, uint64_t b) {
  asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}
__device__ __forceinline__ void ld_hand2(const uint64_t* p, uint64_t& a, uint64_t& b) {
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ bool hand_ready(const uint64_t (&w)[4], uint32_t epoch) {
  return static_cast<uint32_t>(w[0] >> 32) == epoch && static_cast<uint32_t>(w[1] >> 32) == epoch &&
         static_cast<uint32_t>(w[2] >> 32) == epoch && static_cast<uint32_t>(w[3] >> 32) == epoch;
}
// Four consecutive values (rows k..k+3 of one batch row) whose first poll was w: poll again until
// all four carry `epoch` (bounded; *abort on timeout), and return them.
__device__ __forceinline__ float4 hand_take(const uint64_t* h, uint32_t epoch, uint64_t (&w)[4], int* abort) {
  if (!hand_ready(w, epoch)) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 0;; ++i) {
      ld_hand2(h, w[0], w[1]);
      ld_hand2(h + 2, w[2], w[3]);
      if (hand_ready(w, epoch)) break;
      if ((i & 63u) == 63u && global_timer_ns() - t0 > kWaitNs) {
        *abort = 1;
        break;
      }
    }
  }
  return make_float4(__uint_as_float(static_cast<uint32_t>(w[0])), __uint_as_float(static_cast<uint32_t>(w[1])),
                     __uint_as_float(static_cast<uint32_t>(w[2])), __uint_as_float(static_cast<uint32_t>(w[3])));
}

// ---- finalizing a call's output rows -------------------------------------------------------------
// Output scale of an RMS-mode call for batch row b (1 / rms of its own input), for the lane's b; one
// warp, every batch row's loads in flight together.  The per-block sums of squares are added in a
// fixed order, so every warp gets the same bits.
template <int BP>
__device__ __forceinline__ float out_scale_warp(const CallLite& c, const float* ssq, int B, int b, int lane) {
  float t[BP];
#pragma unroll
  for (int bb = 0; bb < BP; ++bb) t[bb] = 0.f;
  const int nblk = c.K / kFwhtBlock;
  for (int k = lane; k < nblk; k += 32)
#pragma unroll
    for (int bb = 0; bb < BP; ++bb)
      if (bb < B) t[bb] += __ldcg(ssq + k * BP + bb);
  float sc = 1.f;
#pragma unroll
  for (int bb = 0; bb < BP; ++bb) {
    const float x = rsqrtf(warp_sum(t[bb]) / static_cast<float>(c.K) + kRmsEps);
    if (bb == b) sc = x;
  }
  return sc;
}

// Rows [fr0, fr0 + nr) (multiples of 4) of call c, for every batch row: the K slices' partial sums
// added in ku order, times the output scale, stored to y.  A group of nsp adjacent lanes shares one
// 4-row chunk: lane s adds the slices [s * per, (s + 1) * per) (all its loads issued before the
// adds), then the group combines its sums by a fixed butterfly.  The result does not depend on which
// CTA computes it, and the partial sums and the sums of squares of the scale are in flight together.
template <int BP, int ROWS, bool HAND>
__device__ __forceinline__ void finalize(const CallLite& c, const float* ppart, const float* ssq, int B, int fr0,
                                         int nr, uint64_t* hand, uint32_t epoch) {
  const int lane = static_cast<int>(threadIdx.x & 31);
  int nsp = 1;
  while (nsp * kGatherKu < c.nku) nsp <<= 1;  // lanes per chunk (a power of two up to 32)
  const int per = (c.nku + nsp - 1) / nsp;    // slices per lane (<= kGatherKu)
  const size_t step = static_cast<size_t>(c.nru) * BP * ROWS;
  const int total = (nr / 4) * B;
  const int nthr = (total * nsp + 31) & ~31;  // whole warps, so every lane takes part in the shuffles
  for (int t = threadIdx.x; t < nthr; t += blockDim.x) {
    const int s = t % nsp, u = t / nsp;
    const bool valid = u < total;
    const int b = valid ? u % B : 0, c4 = valid ? u / B : 0;
    const int k = fr0 + 4 * c4;
    const float* p0 = ppart + (static_cast<size_t>(k / ROWS) * BP + b) * ROWS + (k % ROWS);
    const int ku0 = s * per;
    float4 v[kGatherKu];
#pragma unroll
    for (int i = 0; i < kGatherKu; ++i)
      if (valid && i < per && ku0 + i < c.nku) v[i] = __ldcg(reinterpret_cast<const float4*>(p0 + (ku0 + i) * step));
    const float sc = c.mode == 3 ? out_scale_warp<BP>(c, ssq, B, b, lane) : 1.f;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < kGatherKu; ++i)
      if (valid && i < per && ku0 + i < c.nku) {
        a.x += v[i].x;
        a.y += v[i].y;
        a.z += v[i].z;
        a.w += v[i].w;
      }
    for (int m = 1; m < nsp; m <<= 1) {
      a.x += __shfl_xor_sync(0xffffffffu, a.x, m);
      a.y += __shfl_xor_sync(0xffffffffu, a.y, m);
      a.z += __shfl_xor_sync(0xffffffffu, a.z, m);
      a.w += __shfl_xor_sync(0xffffffffu, a.w, m);
    }
    if (valid && s == 0) {
      const float4 r = make_float4(a.x * sc, a.y * sc, a.z * sc, a.w * sc);
      *reinterpret_cast<float4*>(c.y + static_cast<size_t>(b) * c.N + k) = r;
      if constexpr (HAND) {
        uint64_t* h = hand + static_cast<size_t>(b) * c.N + k;
        const uint64_t e = static_cast<uint64_t>(epoch) << 32;
        st_hand2(h, e | __float_as_uint(r.x), e | __float_as_uint(r.y));
        st_hand2(h + 2, e | __float_as_uint(r.z), e | __float_as_uint(r.w));
      }
    }
  }
}

// ---- the activation transform ------------------------------------------------------------------
// Halves of x^ for batch row b of group gi: [word slot u][pair p][quad thread q][8 halves] = 2G bytes.
// The half at position h = 4 (m & 1) + 2 (j & 1) + (f >> 3) of the 16-byte chunk (u, p = m >> 1, q)
// multiplies field f of word WPT * q + u, where j = f & 7 and m = j >> 1: the two B registers of
// MMA m.  Its value is x~ * 2^-e * 2^(8 - 2 pos), pos = j < 5 ? j : j - 5 (the field's place in the
// FP16 mantissa), e the exponent of the 128-block and batch row.
template <int G>
__device__ __forceinline__ uint32_t xh_offset(int t_in, int& pos) {
  constexpr int WPT = G / 64;
  const int wd = t_in >> 4, f = t_in & 15, j = f & 7, m = j >> 1;
  const int q = wd / WPT, u = wd % WPT, p = m >> 1;
  const int h = ((m & 1) << 2) | ((j & 1) << 1) | (f >> 3);
  pos = j < 5 ? j : j - 5;
  return static_cast<uint32_t>((((u * 2 + p) * 4 + q) << 4) + (h << 1));
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.f + __expf(-z)); }

// Per-lane constants of the x^ layout (the same for every block): byte offsets of the lane's four
// values in a group's block of halves, and the position factors 2^(8 - 2 pos) and 2^(2 pos - 8).
template <int G>
struct LaneLayout {
  uint32_t off[4];
  float up[4], dn[4];
  __device__ __forceinline__ explicit LaneLayout(int lane) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      int pos;
      off[i] = xh_offset<G>((4 * lane + i) % G, pos);
      up[i] = __int_as_float((127 + 8 - 2 * pos) << 23);
      dn[i] = __int_as_float((127 - 8 + 2 * pos) << 23);
    }
  }
};

// x^ and V / F of one 128-block (absolute index blk, local group index lg0 of its first group) for
// all batch rows; one warp.  Modes other than 0 read the previous call pc's final output: the CTAs
// that finalized the block's 128 rows (SwiGLU: and the 128 matching rows of the up half) form one
// or two contiguous ranges; one lane per CTA waits (bounded) for its flag, raising *abort on timeout,
// and the warp barrier then orders every lane's reads after those acquires.  ssq: RMS mode, where
// the block's sums of squares go (global).  PACK selects the x^ layout of the decode loop (2-bit:
// LaneLayout; base-3: MMA order, see the base-3 kernel).
template <int PACK, int G, int BP>
__device__ __forceinline__ void prep_block(const Params& p, const CallLite& c, const CallLite& pc, unsigned want,
                                           int* abort, int blk, int lg0, const LaneLayout<G>& L, uint8_t* xh,
                                           float* V, float* Fv, float* ssq, int lane, const uint64_t* hand_prev,
                                           uint32_t epoch_prev) {
  const int k0 = blk * kFwhtBlock + 4 * lane;
  // handoff (batch 1-2): the previous output's words, all first polls in flight together
  constexpr bool HAND = hand_batch(BP);
  constexpr int HB = HAND ? BP : 1;
  uint64_t hw[HB][2][4];
  if constexpr (HAND) {
    if (c.mode != 0) {
#pragma unroll
      for (int b = 0; b < BP; ++b)
#pragma unroll
        for (int sg = 0; sg < 2; ++sg)
          if (b < p.B && (sg == 0 || c.mode == 2)) {
            const uint64_t* h = hand_prev + static_cast<size_t>(b) * pc.N + (sg ? c.K : 0) + k0;
            ld_hand2(h, hw[b][sg][0], hw[b][sg][1]);
            ld_hand2(h + 2, hw[b][sg][2], hw[b][sg][3]);
          }
    }
  }
  if (!HAND && c.mode != 0) {
    const unsigned* flags = p.sync + kFlagBase;
    const int grid = static_cast<int>(gridDim.x), kb = blk * kFwhtBlock;
    const int lo = fin_owner(pc.N, grid, kb), n1 = fin_owner(pc.N, grid, kb + kFwhtBlock - 4) - lo + 1;
    const int lo2 = c.mode == 2 ? fin_owner(pc.N, grid, c.K + kb) : 0;
    const int n2 = c.mode == 2 ? fin_owner(pc.N, grid, c.K + kb + kFwhtBlock - 4) - lo2 + 1 : 0;
    bool ok = true;
    for (int i = lane; i < n1 + n2; i += 32) ok = wait_flag(flags + (i < n1 ? lo + i : lo2 + i - n1), want) && ok;
    if (!ok) *abort = 1;
    __syncwarp();
  }
  float v[BP][4];
#pragma unroll
  for (int b = 0; b < BP; ++b) {
    v[b][0] = v[b][1] = v[b][2] = v[b][3] = 0.f;
    if (b >= p.B) continue;
    if (c.mode == 0) {
      const uint2 raw = __ldcg(reinterpret_cast<const uint2*>(c.x + static_cast<size_t>(b) * c.K + k0));
      v[b][0] = bf16_bits_to_float(static_cast<uint16_t>(raw.x & 0xffffu));
      v[b][1] = bf16_bits_to_float(static_cast<uint16_t>(raw.x >> 16));
      v[b][2] = bf16_bits_to_float(static_cast<uint16_t>(raw.y & 0xffffu));
      v[b][3] = bf16_bits_to_float(static_cast<uint16_t>(raw.y >> 16));
    } else if (c.mode == 2) {
      float4 g4, u4;
      if constexpr (HAND) {
        const uint64_t* h = hand_prev + static_cast<size_t>(b) * pc.N + k0;
        g4 = hand_take(h, epoch_prev, hw[b][0], abort);
        u4 = hand_take(h + c.K, epoch_prev, hw[b][1], abort);
      } else {
        const float* yb = pc.y + static_cast<size_t>(b) * pc.N;
        g4 = __ldcg(reinterpret_cast<const float4*>(yb + k0));
        u4 = __ldcg(reinterpret_cast<const float4*>(yb + c.K + k0));
      }
      v[b][0] = silu_f(g4.x) * u4.x;
      v[b][1] = silu_f(g4.y) * u4.y;
      v[b][2] = silu_f(g4.z) * u4.z;
      v[b][3] = silu_f(g4.w) * u4.w;
    } else {
      float4 a;
      if constexpr (HAND)
        a = hand_take(hand_prev + static_cast<size_t>(b) * pc.N + k0, epoch_prev, hw[b][0], abort);
      else
        a = __ldcg(reinterpret_cast<const float4*>(pc.y + static_cast<size_t>(b) * pc.N + k0));
      v[b][0] = a.x, v[b][1] = a.y, v[b][2] = a.z, v[b][3] = a.w;
    }
  }
  if (c.mode == 3) {  // sums of squares of the block's input, for the output scale of this call
#pragma unroll
    for (int b = 0; b < BP; ++b) {
      const float t = warp_sum(v[b][0] * v[b][0] + v[b][1] * v[b][1] + v[b][2] * v[b][2] + v[b][3] * v[b][3]);
      if (lane == 0 && b < p.B) ssq[blk * BP + b] = t;
    }
  }
  if (c.apply) {
#pragma unroll
    for (int b = 0; b < BP; ++b)
      if (b < p.B) fwht128_warp(v[b]);
  }
  const float norm = c.apply ? 0.08838834764831845f : 1.f;  // 1 / sqrt(128)
  const int lg = lg0 + (4 * lane) / G;                      // local group of this lane's values
#pragma unroll
  for (int b = 0; b < BP; ++b) {
    // per batch row: exponent of the block, max |x~| * 2^-e in [64, 128)
    float mx = fmaxf(fmaxf(fabsf(v[b][0]), fabsf(v[b][1])), fmaxf(fabsf(v[b][2]), fabsf(v[b][3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    mx *= norm;
    int e = 0;
    if (mx > 0.f) {
      const int ex = (__float_as_int(mx) >> 23) & 0xff;
      e = (ex == 0 ? -126 : ex - 127) - 6;
      if (e > 100) {
        e = 100;
        if (lane == 0) record_error(p.status, TQ_ERR_RANGE);
      }
      e = max(e, -100);
    }
    const float down = __int_as_float((127 - e) << 23) * norm;
    float vs = 0.f;
    if constexpr (PACK == TQ_PACK_2BIT) {
      uint8_t* gbase = xh + (static_cast<size_t>(lg) * BP + b) * (2 * G);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half h = __float2half_rn(v[b][i] * down * L.up[i]);
        *reinterpret_cast<__half*>(gbase + L.off[i]) = h;
        vs += __half2float(h) * L.dn[i];
      }
    } else {
      // base-3: trit k of the CTA's slice (which starts on a word boundary) is half k % 4 of MMA
      // m = k / 4; its digit sits at bit pb = 2 ((k % 20 % 10) / 2) of the decoded half
      const int kr = lg0 * G + 4 * lane, m = kr >> 2;
      uint32_t hw[2];
#pragma unroll
      for (int i = 0; i < 4; i += 2) {
        const int pb0 = 2 * (((kr + i) % 20 % 10) >> 1), pb1 = 2 * (((kr + i + 1) % 20 % 10) >> 1);
        const __half h0 = __float2half_rn(v[b][i] * down * __int_as_float((127 + 8 - pb0) << 23));
        const __half h1 = __float2half_rn(v[b][i + 1] * down * __int_as_float((127 + 8 - pb1) << 23));
        vs += __half2float(h0) * __int_as_float((127 - 8 + pb0) << 23) +
              __half2float(h1) * __int_as_float((127 - 8 + pb1) << 23);
        hw[i >> 1] = static_cast<uint32_t>(__half_as_ushort(h0)) | (static_cast<uint32_t>(__half_as_ushort(h1)) << 16);
      }
      *reinterpret_cast<uint2*>(xh + ((static_cast<size_t>(m >> 1) * BP + b) * 2 + (m & 1)) * 8) = make_uint2(hw[0], hw[1]);
    }
    constexpr int lanes_per_group = G / 4;
#pragma unroll
    for (int o = lanes_per_group / 2; o > 0; o >>= 1) vs += __shfl_xor_sync(0xffffffffu, vs, o);
    if ((lane & (lanes_per_group - 1)) == 0) {
      V[lg * BP + b] = -1.52587890625e-05f * vs;                                   // -2^-16 * sum
      Fv[lg * BP + b] = b < p.B ? __int_as_float((127 + 16 + e) << 23) : 0.f;  // 2^(16 + e)
    }
  }
}

// ---- MMA -------------------------------------------------------------------------------------------
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---- leaving a launch ------------------------------------------------------------------------------
// After an abort, wait (bounded) for this warp's copies still in flight into its ring of kD stages.
__device__ __forceinline__ void drain_ring(uint64_t* full, int kD, unsigned consumed, unsigned issued, int cst,
                                           uint32_t cph) {
  for (; consumed < issued; ++consumed) {
    if (!mbar_wait(&full[cst], cph)) break;
    if (++cst == kD) {
      cst = 0;
      cph ^= 1u;
    }
  }
}
// Every thread: the last CTA to leave resets the barrier words and the flags for the next launch and
// advances the count of completed launches (not after an abort: tq_seq_upload resets them then).
__device__ __forceinline__ void leave_launch(const Params& p, bool abort, unsigned launch_seq) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(p.sync + 1, 1u);
    if (prev == gridDim.x - 1 && !abort) {
      for (unsigned c2 = 0; c2 < gridDim.x; ++c2) p.sync[kFlagBase + c2] = 0u;
      p.sync[0] = 0u;
      p.sync[1] = 0u;
      p.sync[2] = launch_seq + 1u;
      __threadfence();
    }
  }
}

// ---- the kernel ----------------------------------------------------------------------------------
template <int G, int BP>
__global__ void __launch_bounds__(kNW * 32, 1) gemv_seq_kernel(const __grid_constant__ Params p) {
  constexpr int WPT = G / 64;             // code words per quad thread per group per row
  constexpr int GPI = kItemTrits / G;     // groups per item
  constexpr int CPG = GPI < 8 / BP ? GPI : 8 / BP;  // groups per accumulation cycle
  constexpr int NCYC = GPI / CPG;
  constexpr int BPI = kItemTrits / kFwhtBlock;     // 128-blocks per item
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  constexpr int kD = ring_depth(BP);
  const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
  const int g = lane >> 2, q = lane & 3;
  const int cta = static_cast<int>(blockIdx.x);
  uint8_t* codes_st = smem + static_cast<size_t>(warp) * kD * kCodeStage;
  const uint16_t* scales_st = reinterpret_cast<const uint16_t*>(smem + p.off_scales) + warp * kD * (kScaleStage / 2);
  uint8_t* scales_w = smem + p.off_scales + static_cast<size_t>(warp) * kD * kScaleStage;
  uint8_t* xh = smem + p.off_xh;
  const uint8_t* zero = smem + p.off_zero;
  float* V = reinterpret_cast<float*>(smem + p.off_v);
  float* Fv = reinterpret_cast<float*>(smem + p.off_f);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.off_bar) + warp * kD;
  int* s_flag = reinterpret_cast<int*>(smem + p.off_misc);  // [0] abort, [1] barrier result

  for (uint32_t i = threadIdx.x; i < 64; i += blockDim.x) reinterpret_cast<uint32_t*>(smem + p.off_zero)[i] = 0u;
  const int vcap = (p.nkc * GPI + 8) * BP;
  for (int i = threadIdx.x; i < vcap; i += blockDim.x) V[i] = Fv[i] = 0.f;
  if (lane == 0)
    for (int s = 0; s < kD; ++s) mbar_init(&full[s], 1);
  if (threadIdx.x == 0) s_flag[0] = 0;
  fence_mbar_init();
  __syncthreads();

  auto warp_range = [&](const CallLite& c, int& a, int& b) { warp_items(c, cta, warp, kNW, a, b); };

  // ---- producer state (lane 0 issues; the cursor is kept warp-uniform) ----
  int pcall = 0, pidx = 0, pend = 0, pru = 0, pku = 0, pnru = 0;
  auto set_call = [&]() {
    const CallLite c(p.calls[pcall]);
    warp_range(c, pidx, pend);
    pnru = c.nru;
    pku = pidx / c.nru;
    pru = pidx - pku * c.nru;
  };
  set_call();
  unsigned issued = 0, consumed = 0;
  int ist = 0;                 // stage of the next copy
  int cst = 0;                 // stage of the next item to consume
  uint32_t cph = 0;            // its phase parity
  const uint64_t pol = l2_evict_first_policy();
  auto issue_next = [&]() {
    while (pidx >= pend) {
      if (++pcall >= p.ncalls) return;
      set_call();
    }
    const CallDev* cd = p.calls + pcall;
    const int s = ist;
    ist = ist + 1 == kD ? 0 : ist + 1;
    if (lane == 0) {
      mbar_arrive_expect_tx(&full[s], kStageBytes);
      tma_load_2d_hint(codes_st + static_cast<size_t>(s) * kCodeStage, &cd->tm_codes, pku * 32, pru * kRows, &full[s],
                       pol);
      tma_load_2d(scales_w + static_cast<size_t>(s) * kScaleStage, &cd->tm_scales, (pku * GPI) & ~7, pru * kRows,
                  &full[s]);
    }
    ++issued;
    ++pidx;
    if (++pru == pnru) {
      pru = 0;
      ++pku;
    }
  };
  for (int s = 0; s < kD; ++s) issue_next();

  bool abort = false;
  const LaneLayout<G> L(lane);
  unsigned nbar = 0;  // grid barriers passed
  const uint32_t launch_seq = __ldcg(p.sync + 2);  // launches completed (advanced by the last CTA out)
  const uint32_t epoch0 = launch_seq * static_cast<uint32_t>(p.ncalls);
  for (int j = 0; j < p.ncalls && !abort; ++j) {
    const CallLite c(p.calls[j]);
    const CallLite pc(p.calls[j > 0 ? j - 1 : 0]);
    float* part = p.part + static_cast<size_t>(j & 1) * p.part_stride;
    float* ssq = p.ssq + (j & 1) * p.ssq_stride;
    // ---- this CTA's items and the K slices they cover ----
    int ca = 0, cb = 0, ku_lo = 0, ku_hi = -1;
    if (cta < c.gp) {
      ca = cta_start(c.T, c.gp, cta);
      cb = cta_start(c.T, c.gp, cta + 1);
      ku_lo = ca / c.nru;
      if (cb > ca) ku_hi = (cb - 1) / c.nru;
    }
    // ---- input transform of this CTA's K slices (reading the previous call's final output as each
    //      warp's rows become ready) ----
    if (cb > ca) {
      const int blk0 = ku_lo * BPI;
      const int blk1 = min((ku_hi + 1) * BPI, c.K / kFwhtBlock);
      for (int blk = blk0 + warp; blk < blk1; blk += kNW)
        prep_block<TQ_PACK_2BIT, G, BP>(p, c, pc, static_cast<unsigned>(j), s_flag, blk, (blk - blk0) * (kFwhtBlock / G), L, xh,
                          V, Fv, ssq, lane, p.hand + static_cast<size_t>((j - 1) & 1) * p.hand_stride, epoch0 + j);
    }
    __syncthreads();
    if (s_flag[0] != 0) {  // a ready flag did not come in time
      if (threadIdx.x == 0) record_error(p.status, TQ_ERR_TIMEOUT);
      abort = true;
      break;
    }

    // ---- this warp's items ----
    int wa = 0, wb = 0;
    warp_range(c, wa, wb);
    const int my_slot = g / BP, my_b = g % BP;  // B operand: this lane supplies column g = slot * BP + b
    const uint32_t rA = static_cast<uint32_t>(g) * 128u;
    int ku = wb > wa ? wa / c.nru : 0, ru = wa - ku * c.nru;
    for (int it = wa; it < wb; ++it) {
      const int st = cst;
      if (!mbar_wait(&full[st], cph)) {
        if (lane == 0) record_error(p.status, TQ_ERR_TIMEOUT);
        abort = true;
        break;
      }
      const uint8_t* cs = codes_st + static_cast<size_t>(st) * kCodeStage;
      const uint16_t* ss = scales_st + st * (kScaleStage / 2);
      const int g_item0 = ku * GPI;                  // first group of the item
      const int lg_item0 = (ku - ku_lo) * GPI;       // ... in this CTA's x^
      constexpr int ngi = GPI;  // groups in the item: K is a multiple of 8 groups, so items are whole
      const int gofs = g_item0 & 7;                  // its column in the scale box
      float acc[2][4];
#pragma unroll
      for (int s = 0; s < 2; ++s)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[s][i] = 0.f;
#pragma unroll
      for (int cy = 0; cy < NCYC; ++cy) {
        const int gb = cy * CPG;
        if (gb >= ngi) break;
        const int col0 = 2 * q;
        // independent accumulator chains per slab (batch 1: two, by word slot u or group parity)
        constexpr int NCH = BP == 1 ? 2 : 1;
        float cc[2][NCH][4];
        {
          // start values: -2^-16 * sum x^ for the columns of groups present in this cycle
          const float2 v2 = *reinterpret_cast<const float2*>(V + (lg_item0 + gb) * BP + col0);
          const bool ok0 = col0 < CPG * BP && gb + col0 / BP < ngi;
          const bool ok1 = col0 + 1 < CPG * BP && gb + (col0 + 1) / BP < ngi;
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            cc[s][0][0] = cc[s][0][2] = ok0 ? v2.x : 0.f;
            cc[s][0][1] = cc[s][0][3] = ok1 ? v2.y : 0.f;
#pragma unroll
            for (int ch = 1; ch < NCH; ++ch)
#pragma unroll
              for (int i = 0; i < 4; ++i) cc[s][ch][i] = 0.f;
          }
        }
#pragma unroll
        for (int gl = 0; gl < CPG; ++gl) {
          const int jj = gb + gl;  // group within the item
          if (jj >= ngi) break;
          uint32_t wv[2][2][WPT];  // [slab][row g / g + 8][word]
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            const uint8_t* r0 = cs + rA + static_cast<uint32_t>(s) * 2048u;
            if constexpr (WPT == 2) {
              const uint32_t off = (static_cast<uint32_t>((2 * jj + (q >> 1)) ^ g) << 4) + 8u * (q & 1);
              const uint2 a = *reinterpret_cast<const uint2*>(r0 + off);
              const uint2 b = *reinterpret_cast<const uint2*>(r0 + 1024u + off);
              wv[s][0][0] = a.x;
              wv[s][0][WPT - 1] = a.y;
              wv[s][1][0] = b.x;
              wv[s][1][WPT - 1] = b.y;
            } else {
              const uint32_t off = (static_cast<uint32_t>(jj ^ g) << 4) + 4u * q;
              wv[s][0][0] = *reinterpret_cast<const uint32_t*>(r0 + off);
              wv[s][1][0] = *reinterpret_cast<const uint32_t*>(r0 + 1024u + off);
            }
          }
          const uint8_t* bbase = (my_slot == gl && my_b < p.B)
                                     ? xh + (static_cast<size_t>(lg_item0 + jj) * BP + my_b) * (2 * G)
                                     : zero;
#pragma unroll
          for (int u = 0; u < WPT; ++u) {
            uint4 bq[2];
#pragma unroll
            for (int pp = 0; pp < 2; ++pp)
              bq[pp] = *reinterpret_cast<const uint4*>(bbase + (((u * 2 + pp) * 4 + q) << 4));
#pragma unroll
            for (int s = 0; s < 2; ++s) {
              const uint32_t w = wv[s][0][u], w8 = wv[s][1][u];
              const uint32_t w2 = w >> 10, w82 = w8 >> 10;
              uint32_t pr[8], pr8[8];
#pragma unroll
              for (int f = 0; f < 8; ++f) {
                pr[f] = f < 5 ? (w & (0x00030003u << (2 * f))) : (w2 & (0x00030003u << (2 * (f - 5))));
                pr8[f] = f < 5 ? (w8 & (0x00030003u << (2 * f))) : (w82 & (0x00030003u << (2 * (f - 5))));
              }
              const int ch = NCH == 1 ? 0 : WPT == 2 ? u : (gl & 1);
#pragma unroll
              for (int m = 0; m < 4; ++m) {
                const uint4 b = bq[m >> 1];
                mma16816(cc[s][ch], pr[2 * m], pr8[2 * m], pr[2 * m + 1], pr8[2 * m + 1], (m & 1) ? b.z : b.x,
                         (m & 1) ? b.w : b.y);
              }
            }
          }
        }
        // fold the cycle: acc += scale(row, group) * 2^(16 + e) * cc for each column
        {
          const float2 f2 = *reinterpret_cast<const float2*>(Fv + (lg_item0 + gb) * BP + col0);
          const int sl0 = min(col0 / BP, CPG - 1), sl1 = min((col0 + 1) / BP, CPG - 1);
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            const uint16_t* sr = ss + (16 * s + g) * 8 + gofs + gb;
            const float s00 = half_bits_to_float(sr[sl0]), s01 = half_bits_to_float(sr[sl1]);
            const float s80 = half_bits_to_float(sr[64 + sl0]), s81 = half_bits_to_float(sr[64 + sl1]);
            float t[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              t[i] = cc[s][0][i];
#pragma unroll
              for (int ch = 1; ch < NCH; ++ch) t[i] += cc[s][ch][i];
            }
            acc[s][0] = fmaf(s00 * f2.x, t[0], acc[s][0]);
            acc[s][1] = fmaf(s01 * f2.y, t[1], acc[s][1]);
            acc[s][2] = fmaf(s80 * f2.x, t[2], acc[s][2]);
            acc[s][3] = fmaf(s81 * f2.y, t[3], acc[s][3]);
          }
        }
      }
      __syncwarp();
      ++consumed;
      if (++cst == kD) {
        cst = 0;
        cph ^= 1u;
      }
      fence_proxy_async_smem();  // this stage's reads before the copy that refills it
      issue_next();
      // the item's partial sums: per (row, batch row), summed over the columns of that batch row
      {
        float o[2][4];
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          if (BP == 1) {
            o[s][0] = acc[s][0] + acc[s][1];
            o[s][2] = acc[s][2] + acc[s][3];
            o[s][1] = o[s][3] = 0.f;
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) o[s][i] = acc[s][i];
          }
#pragma unroll
          for (int m = 1; m < 4; m <<= 1) {
            if ((2 * m) % BP != 0) continue;  // lanes q and q ^ m hold the same batch rows
#pragma unroll
            for (int i = 0; i < 4; ++i) o[s][i] += __shfl_xor_sync(0xffffffffu, o[s][i], m);
          }
        }
        constexpr int nwq = BP >= 2 ? BP / 2 : 1;  // quad threads holding distinct batch rows
        if (q < nwq) {
          float* dst = part + (static_cast<size_t>(ku) * c.nru + ru) * BP * kRows;
#pragma unroll
          for (int s = 0; s < 2; ++s)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              if (BP == 1 && (i & 1)) continue;
              const int r = 16 * s + g + (i >= 2 ? 8 : 0);
              const int b = BP == 1 ? 0 : 2 * q + (i & 1);
              __stcg(dst + b * kRows + r, o[s][i]);
            }
        }
      }
      if (++ru == c.nru) {
        ru = 0;
        ++ku;
      }
    }
    abort = __syncthreads_or(abort) != 0;
    if (abort) break;
    // ---- barrier: every partial sum and sum of squares of this call is written (the CTA barrier
    //      just passed orders them before thread 0's release) ----
    if (threadIdx.x == 0) grid_arrive_release(p.sync);
    if (!grid_wait(p.sync, nbar++, s_flag + 1)) {
      if (threadIdx.x == 0) record_error(p.status, TQ_ERR_TIMEOUT);
      abort = true;
      break;
    }
    // ---- this CTA's share of the call's output rows: partial sums in ku order, times the output
    //      scale ----
    {
      int fr0, fr1;
      fin_rows(c.N, cta, static_cast<int>(gridDim.x), fr0, fr1);
      finalize<BP, kRows, hand_batch(BP)>(c, part, ssq, p.B, fr0, fr1 - fr0,
                                                        p.hand + static_cast<size_t>(j & 1) * p.hand_stride,
                                                        epoch0 + j + 1);
    }
    // ---- this CTA's rows are final: raise its flag (with the handoff only the CTA barrier: warps
    //      do not start polling for the next input while their CTA still finalizes) ----
    __syncthreads();
    if (!hand_batch(BP) && threadIdx.x == 0)
      st_release(p.sync + kFlagBase + cta, static_cast<unsigned>(j + 1));
  }

  if (abort) drain_ring(full, kD, consumed, issued, cst, cph);
  leave_launch(p, abort, launch_seq);
}

// ---- base-3 --------------------------------------------------------------------------------------
// The same step over base-3 codes (20 trits per 32-bit word: the TurboQuant-MLX 1.58-bit Qwen3.6-35B-A3B
// page, "为什么 1.58bit 没变成乱码", point 3), in the column layout of the per-call base-3 decode: a warp owns 64 rows, lane l
// decodes rows l and l + 32 word by word (two reciprocal multiplies split a word into four 5-trit
// chunks, a table in shared memory places each chunk's digits in FP16 pair fields, one mask per
// pair gives an operand register), and the B operand of an MMA is zero except in the column of the
// lane that supplies a batch row, so each column of the m16n8k16 accumulator holds one row's dot
// product.  An item is a warp's 64 rows x 640 trits (32 words of each row: one 2-D TMA box of 64 x
// 128 bytes, 128-byte swizzle); scales are loaded one item ahead into registers and staged per warp
// as [group][row].  Boundaries, work split, finalize and flags are those of the 2-bit kernel.
namespace b3 {
constexpr int kNW = 8;                         // warps per CTA (255 registers each; the rings and the table fill shared memory)
constexpr int kD = 2;                          // ring stages per warp
constexpr int kRows = 64;                      // rows per item
constexpr int kItemTrits = 640;                // trits per item along K: 32 words, five 128-blocks
constexpr uint32_t kCodeStage = kRows * 128u;  // one item's codes: 8 KB
constexpr int kLutRep = 16;                    // table copies (lanes l and l + 16 share one)
constexpr uint32_t kLutBytes = B3Lut<kLutRep>::kBytes;
}  // namespace b3

__device__ const B3Lut<b3::kLutRep> g_seq_lut = make_b3_lut<b3::kLutRep>();

// Scales of one item (64 rows x GPI groups), loaded into registers one item ahead (two halves per
// register) and staged in the warp's area as halves [group][row].  Rows past N and groups past the
// matrix read a clamped (valid) address; their values reach only outputs that are never stored.
template <int GPI>
struct ItemScales {
  static constexpr int PER_LANE = 64 * GPI / 32;
  uint32_t v[PER_LANE / 2];
  __device__ __forceinline__ void load(const CallLite& c, int ku, int ru, int lane) {
#pragma unroll
    for (int j = 0; j < PER_LANE; ++j) {
      const int e = lane + 32 * j, r = e / GPI, g = e % GPI;
      const int row = min(ru * 64 + r, c.N - 1), grp = min(ku * GPI + g, c.ng - 1);
      const uint32_t h = __ldg(c.scales + static_cast<size_t>(row) * c.ng + grp);
      if (j & 1)
        v[j >> 1] |= h << 16;
      else
        v[j >> 1] = h;
    }
  }
  __device__ __forceinline__ void store(uint16_t* sw, int lane) const {
#pragma unroll
    for (int j = 0; j < PER_LANE; ++j) {
      const int e = lane + 32 * j, r = e / GPI, g = e % GPI;
      sw[g * 64 + r] = static_cast<uint16_t>((j & 1) ? (v[j >> 1] >> 16) : (v[j >> 1] & 0xffffu));
    }
  }
};

// One item: the warp's 64 rows x the item's ngi groups, folded into acc (rows rl0, rl0 + 1, rl0 + 32,
// rl0 + 33 of the item for batch row 2t + bq of tile t).  box: the item's swizzled codes; bptr / bstr:
// where this lane's B operand of tile t comes from and its stride per MMA pair (x^ of the CTA's slice,
// MMA pair mp and batch row b at words (mp * BP + b) * 4, or the zero chunk with stride 0); mp0: the
// item's first MMA pair in the slice; V / Fv of local group lg = lg_item0 + gl, batch row b at
// lg * BP + b; swr: the staged scales at this lane's first accumulator row.
template <int G, int BP, bool FULL>
__device__ __forceinline__ void b3_item(const uint4* __restrict__ box, int lane, int ngi, const uint32_t* __restrict__ lutA,
                                        const uint32_t* __restrict__ lutB, const uint32_t* const (&bptr)[(BP + 1) / 2],
                                        const int (&bstr)[(BP + 1) / 2], int mp0, const float* __restrict__ V,
                                        const float* __restrict__ Fv, int lg_item0, const uint16_t* __restrict__ swr,
                                        float (&acc)[(BP + 1) / 2][4]) {
  constexpr int NT = (BP + 1) / 2;
  constexpr int GP = G / 2;  // pairs per group
  const int bq = (lane & 3) >> 1;
  const int sl = lane & 7;   // 128-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ (r % 8)
  float cc[NT][4];
  uint4 bp[NT];
#pragma unroll
  for (int st = 0; st < 8; ++st) {
    if (!FULL && (st * 80) / G >= ngi) break;
    const uint4 cur = box[lane * 8 + (st ^ sl)], cur2 = box[(lane + 32) * 8 + (st ^ sl)];
    const uint32_t wr[4] = {cur.x, cur.y, cur.z, cur.w};
    const uint32_t wr2[4] = {cur2.x, cur2.y, cur2.z, cur2.w};
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      uint32_t La[4], Lb[4];
      b3_chunks<b3::kLutRep>(wr[wi], lutA, lutB, La);
      b3_chunks<b3::kLutRep>(wr2[wi], lutA, lutB, Lb);
#pragma unroll
      for (int mj = 0; mj < 5; ++mj) {
        const int pair = (st * 4 + wi) * 10 + 2 * mj;  // first pair of this MMA within the item
        const int gl = pair / GP;
        if (!FULL && gl >= ngi) break;
        const int lg = lg_item0 + gl;
        if (pair % GP == 0) {  // a new group: the sum starts at -2^-16 * sum(x^) of its batch row
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const int b = 2 * t + bq;
            const float v0 = b < BP ? V[lg * BP + b] : 0.f;
            cc[t][0] = cc[t][1] = cc[t][2] = cc[t][3] = v0;
          }
        }
        const int mloc = (st * 4 + wi) * 5 + mj;  // MMA index within the item
        if ((mloc & 1) == 0) {
#pragma unroll
          for (int t = 0; t < NT; ++t)
            bp[t] = *reinterpret_cast<const uint4*>(bptr[t] + (mp0 + (mloc >> 1)) * bstr[t]);
        }
        const uint32_t a0 = b3_pair(La, 2 * mj), a2 = b3_pair(La, 2 * mj + 1);
        const uint32_t a1 = b3_pair(Lb, 2 * mj), a3 = b3_pair(Lb, 2 * mj + 1);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const uint32_t b0 = (mloc & 1) ? bp[t].z : bp[t].x, b1 = (mloc & 1) ? bp[t].w : bp[t].y;
          mma16816(cc[t], a0, a1, a2, a3, b0, b1);
        }
        if ((pair + 2) % GP == 0) {  // the group's last MMA: fold scale(row, group) * 2^(16 + e) * cc
          const float2 s01 = __half22float2(*reinterpret_cast<const __half2*>(swr + gl * 64));
          const float2 s23 = __half22float2(*reinterpret_cast<const __half2*>(swr + gl * 64 + 32));
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const int b = 2 * t + bq;
            const float f = b < BP ? Fv[lg * BP + b] : 0.f;
            acc[t][0] = fmaf(s01.x * f, cc[t][0], acc[t][0]);
            acc[t][1] = fmaf(s01.y * f, cc[t][1], acc[t][1]);
            acc[t][2] = fmaf(s23.x * f, cc[t][2], acc[t][2]);
            acc[t][3] = fmaf(s23.y * f, cc[t][3], acc[t][3]);
          }
        }
      }
    }
  }
}

template <int G, int BP>
__global__ void __launch_bounds__(b3::kNW * 32, 1) gemv_seq_b3_kernel(const __grid_constant__ Params p) {
  using b3::kD;
  using b3::kNW;
  using b3::kRows;
  using b3::kItemTrits;
  using b3::kCodeStage;
  constexpr int GPI = kItemTrits / G;           // groups per item (5 or 10)
  constexpr int BPI = kItemTrits / kFwhtBlock;  // 128-blocks per item
  constexpr int NT = (BP + 1) / 2;              // two-row batch tiles
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
  const int g = lane >> 2, q = lane & 3;
  const int cta = static_cast<int>(blockIdx.x);
  uint8_t* codes_st = smem + static_cast<size_t>(warp) * kD * kCodeStage;
  uint16_t* sw = reinterpret_cast<uint16_t*>(smem + p.off_scales) + warp * (GPI * 64);
  uint8_t* xh = smem + p.off_xh;
  const uint32_t* zero = reinterpret_cast<const uint32_t*>(smem + p.off_zero);
  float* V = reinterpret_cast<float*>(smem + p.off_v);
  float* Fv = reinterpret_cast<float*>(smem + p.off_f);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.off_bar) + warp * kD;
  uint64_t* lut_bar = reinterpret_cast<uint64_t*>(smem + p.off_bar) + kNW * kD;
  int* s_flag = reinterpret_cast<int*>(smem + p.off_misc);  // [0] abort, [1] barrier result
  uint32_t* lut = reinterpret_cast<uint32_t*>(smem + p.off_lut);

  for (uint32_t i = threadIdx.x; i < 64; i += blockDim.x) reinterpret_cast<uint32_t*>(smem + p.off_zero)[i] = 0u;
  const int vcap = (p.nkc * GPI + 8) * BP;
  for (int i = threadIdx.x; i < vcap; i += blockDim.x) V[i] = Fv[i] = 0.f;
  if (lane == 0)
    for (int s = 0; s < kD; ++s) mbar_init(&full[s], 1);
  if (threadIdx.x == 0) {
    s_flag[0] = 0;
    mbar_init(lut_bar, 1);
  }
  fence_mbar_init();
  __syncthreads();
  if (threadIdx.x == 0) {  // the chunk table (constant data of this library)
    mbar_arrive_expect_tx(lut_bar, b3::kLutBytes);
    bulk_g2s(lut, &g_seq_lut, b3::kLutBytes, lut_bar);
  }

  auto warp_range = [&](const CallLite& c, int& a, int& b) { warp_items(c, cta, warp, kNW, a, b); };

  // ---- producer state (lane 0 issues; the cursor is kept warp-uniform) ----
  int pcall = 0, pidx = 0, pend = 0, pru = 0, pku = 0, pnru = 0;
  auto set_call = [&]() {
    const CallLite c(p.calls[pcall]);
    warp_range(c, pidx, pend);
    pnru = c.nru;
    pku = pidx / c.nru;
    pru = pidx - pku * c.nru;
  };
  set_call();
  unsigned issued = 0, consumed = 0;
  int ist = 0, cst = 0;
  uint32_t cph = 0;
  const uint64_t pol = l2_evict_first_policy();
  auto issue_next = [&]() {
    while (pidx >= pend) {
      if (++pcall >= p.ncalls) return;
      set_call();
    }
    const CallDev* cd = p.calls + pcall;
    const int s = ist;
    ist = ist + 1 == kD ? 0 : ist + 1;
    if (lane == 0) {
      mbar_arrive_expect_tx(&full[s], kCodeStage);
      tma_load_2d_hint(codes_st + static_cast<size_t>(s) * kCodeStage, &cd->tm_codes, pku * 32, pru * kRows, &full[s],
                       pol);
    }
    ++issued;
    ++pidx;
    if (++pru == pnru) {
      pru = 0;
      ++pku;
    }
  };
  for (int s = 0; s < kD; ++s) issue_next();

  bool abort = !mbar_wait(lut_bar, 0);
  if (abort && threadIdx.x == 0) record_error(p.status, TQ_ERR_TIMEOUT);
  abort = __syncthreads_or(abort) != 0;
  const LaneLayout<G> L(lane);
  const uint32_t* lutA = lut + (lane & (b3::kLutRep - 1));
  const uint32_t* lutB = lutA + 243 * b3::kLutRep;
  // B operand: lane (g, q) supplies batch row 2t + g / 4 of tile t when g % 4 == q, else 16 zero bytes
  const uint32_t* bptr[NT];
  int bstr[NT];
  const int bq = q >> 1;
  const int rl0 = 4 * g + ((2 * q) & 3);  // this lane's accumulator rows: rl0, rl0 + 1, rl0 + 32, rl0 + 33
  ItemScales<GPI> us;
  unsigned nbar = 0;
  // epochs of this launch's calls: launches completed (stable during a launch) x calls + call + 1
  const uint32_t launch_seq = __ldcg(p.sync + 2);
  const uint32_t epoch0 = launch_seq * static_cast<uint32_t>(p.ncalls);
  for (int j = 0; j < p.ncalls && !abort; ++j) {
    const CallLite c(p.calls[j]);
    const CallLite pc(p.calls[j > 0 ? j - 1 : 0]);
    float* part = p.part + static_cast<size_t>(j & 1) * p.part_stride;
    float* ssq = p.ssq + (j & 1) * p.ssq_stride;
    int ca = 0, cb = 0, ku_lo = 0, ku_hi = -1;
    if (cta < c.gp) {
      ca = cta_start(c.T, c.gp, cta);
      cb = cta_start(c.T, c.gp, cta + 1);
      ku_lo = ca / c.nru;
      if (cb > ca) ku_hi = (cb - 1) / c.nru;
    }
    int wa = 0, wb = 0;
    warp_range(c, wa, wb);
    int ku = wb > wa ? wa / c.nru : 0, ru = wa - ku * c.nru;
    if (wb > wa) us.load(c, ku, ru, lane);  // the first item's scales, in flight during the transform
    // ---- input transform of this CTA's K slices ----
    if (cb > ca) {
      const int blk0 = ku_lo * BPI;
      const int blk1 = min((ku_hi + 1) * BPI, c.K / kFwhtBlock);
      for (int blk = blk0 + warp; blk < blk1; blk += kNW)
        prep_block<TQ_PACK_B3, G, BP>(p, c, pc, static_cast<unsigned>(j), s_flag, blk, (blk - blk0) * (kFwhtBlock / G),
                                      L, xh, V, Fv, ssq, lane,
                                      p.hand + static_cast<size_t>((j - 1) & 1) * p.hand_stride, epoch0 + j);
    }
    __syncthreads();
    if (s_flag[0] != 0) {  // a ready flag did not come in time
      if (threadIdx.x == 0) record_error(p.status, TQ_ERR_TIMEOUT);
      abort = true;
      break;
    }
    {
      const bool bsup = (g & 3) == q;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const int b = 2 * t + (g >> 2);
        bptr[t] = bsup && b < p.B ? reinterpret_cast<const uint32_t*>(xh) + b * 4 : zero;
        bstr[t] = bsup && b < p.B ? BP * 4 : 0;  // words per MMA pair: 8 halves per batch row
      }
    }
    // ---- this warp's items ----
    for (int it = wa; it < wb; ++it) {
      const int st = cst;
      if (!mbar_wait(&full[st], cph)) {
        if (lane == 0) record_error(p.status, TQ_ERR_TIMEOUT);
        abort = true;
        break;
      }
      __syncwarp();
      us.store(sw, lane);
      __syncwarp();
      if (it + 1 < wb) {
        const int nru2 = ru + 1 == c.nru ? 0 : ru + 1, nku2 = ru + 1 == c.nru ? ku + 1 : ku;
        us.load(c, nku2, nru2, lane);
      }
      const uint4* box = reinterpret_cast<const uint4*>(codes_st + static_cast<size_t>(st) * kCodeStage);
      const int ngi = min(GPI, c.ng - ku * GPI);
      float acc[NT][4];
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
      const int lg_item0 = (ku - ku_lo) * GPI, mp0 = (ku - ku_lo) * (kItemTrits / 8);
      if (ngi == GPI)
        b3_item<G, BP, true>(box, lane, ngi, lutA, lutB, bptr, bstr, mp0, V, Fv, lg_item0, sw + rl0, acc);
      else
        b3_item<G, BP, false>(box, lane, ngi, lutA, lutB, bptr, bstr, mp0, V, Fv, lg_item0, sw + rl0, acc);
      __syncwarp();
      ++consumed;
      if (++cst == kD) {
        cst = 0;
        cph ^= 1u;
      }
      fence_proxy_async_smem();  // this stage's reads before the copy that refills it
      issue_next();
      // the item's partial sums: each (row, batch row) is held by one lane
      float* dst = part + static_cast<size_t>(ku * c.nru + ru) * BP * kRows;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const int b = 2 * t + bq;
        if (b < p.B) {
          __stcg(reinterpret_cast<float2*>(dst + b * kRows + rl0), make_float2(acc[t][0], acc[t][1]));
          __stcg(reinterpret_cast<float2*>(dst + b * kRows + rl0 + 32), make_float2(acc[t][2], acc[t][3]));
        }
      }
      if (++ru == c.nru) {
        ru = 0;
        ++ku;
      }
    }
    abort = __syncthreads_or(abort) != 0;
    if (abort) break;
    // ---- barrier: every partial sum and sum of squares of this call is written ----
    if (threadIdx.x == 0) grid_arrive_release(p.sync);
    if (!grid_wait(p.sync, nbar++, s_flag + 1)) {
      if (threadIdx.x == 0) record_error(p.status, TQ_ERR_TIMEOUT);
      abort = true;
      break;
    }
    {
      int fr0, fr1;
      fin_rows(c.N, cta, static_cast<int>(gridDim.x), fr0, fr1);
      finalize<BP, kRows, hand_batch(BP)>(c, part, ssq, p.B, fr0, fr1 - fr0,
                                                      p.hand + static_cast<size_t>(j & 1) * p.hand_stride, epoch0 + j + 1);
    }
    // ---- this CTA's rows are final: raise its flag (with the handoff only the CTA barrier) ----
    __syncthreads();
    if (!hand_batch(BP) && threadIdx.x == 0)
      st_release(p.sync + kFlagBase + cta, static_cast<unsigned>(j + 1));
  }

  if (abort) drain_ring(full, kD, consumed, issued, cst, cph);
  leave_launch(p, abort, launch_seq);
}

}  // namespace seq
}  // namespace tq

// ---------------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------------
using namespace tq;
using namespace tq::seq;

struct tq_seq {
  std::vector<CallDev> calls;
  int ncalls = 0, B = 0, Bp = 0, G = 0, grid = 0, nkc = 0, dev = 0, pack = 0, nw = 0;
  size_t smem = 0;
  uint32_t off_scales = 0, off_xh = 0, off_zero = 0, off_v = 0, off_f = 0, off_bar = 0, off_misc = 0, off_lut = 0;
  size_t ws_calls = 0, ws_sync = 0, ws_part = 0, ws_ssq = 0, ws_hand = 0, ws_bytes = 0, part_stride = 0, hand_stride = 0;
  int ssq_stride = 0;
  const void* kern = nullptr;
};

namespace {

template <int PACK, int G, int BP>
const void* seq_kernel_t() {
  if constexpr (PACK == TQ_PACK_B3) return reinterpret_cast<const void*>(gemv_seq_b3_kernel<G, BP>);
  return reinterpret_cast<const void*>(gemv_seq_kernel<G, BP>);
}
template <int PACK>
const void* seq_kernel_p(int G, int Bp) {
  if (G == 128) {
    switch (Bp) {
      case 1: return seq_kernel_t<PACK, 128, 1>();
      case 2: return seq_kernel_t<PACK, 128, 2>();
      case 4: return seq_kernel_t<PACK, 128, 4>();
      default: return seq_kernel_t<PACK, 128, 8>();
    }
  }
  switch (Bp) {
    case 1: return seq_kernel_t<PACK, 64, 1>();
    case 2: return seq_kernel_t<PACK, 64, 2>();
    case 4: return seq_kernel_t<PACK, 64, 4>();
    default: return seq_kernel_t<PACK, 64, 8>();
  }
}
const void* seq_kernel(int pack, int G, int Bp) {
  return pack == TQ_PACK_B3 ? seq_kernel_p<TQ_PACK_B3>(G, Bp) : seq_kernel_p<TQ_PACK_2BIT>(G, Bp);
}

}  // namespace

extern "C" tq_status tq_seq_create(const tq_seq_call* calls, int ncalls, int batch, tq_seq** out) {
  if (!out) return TQ_ERR_INVALID_ARG;
  *out = nullptr;
  if (!calls || ncalls < 1 || batch < 1 || batch > 8) return TQ_ERR_INVALID_ARG;
  const int G = calls[0].d.group, pack = calls[0].d.packing;
  int Kmax = 0;
  for (int j = 0; j < ncalls; ++j) {
    const tq_seq_call& c = calls[j];
    tq_status st = check_linear_desc(&c.d);
    if (st != TQ_OK) return st;
    if (c.d.packing != pack || c.d.group != G) return TQ_ERR_UNSUPPORTED;
    // 2-bit: FP16 scales are fetched by TMA, so a scale row must be a multiple of 16 bytes
    if ((pack == TQ_PACK_2BIT && (c.d.K / c.d.group) % 8 != 0) || c.d.N % 4 != 0) return TQ_ERR_UNSUPPORTED;
    if (!c.codes || !c.scales || !c.y) return TQ_ERR_INVALID_ARG;
    if (!aligned(c.codes, 16) || !aligned(c.scales, 16) || !aligned(c.y, 16)) return TQ_ERR_MISALIGNED;
    if (c.x_src == TQ_SEQ_X_BF16) {
      if (!c.x) return TQ_ERR_INVALID_ARG;
      if (!aligned(c.x, 16)) return TQ_ERR_MISALIGNED;
    } else if (c.x_src == TQ_SEQ_X_PREV || c.x_src == TQ_SEQ_X_RMS_PREV) {
      if (j == 0 || calls[j - 1].d.N < c.d.K) return TQ_ERR_INVALID_ARG;
    } else if (c.x_src == TQ_SEQ_X_SWIGLU_PREV) {
      if (j == 0 || calls[j - 1].d.N != 2 * c.d.K) return TQ_ERR_INVALID_ARG;
    } else {
      return TQ_ERR_INVALID_ARG;
    }
    Kmax = std::max(Kmax, c.d.K);
  }
  int dev = 0, sms = 0, optin = 0, coop = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e);
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return cuda_fail(e);
  if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
    return cuda_fail(e);
  if ((e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev)) != cudaSuccess) return cuda_fail(e);
  if (!coop) return TQ_ERR_UNSUPPORTED;

  tq_seq* s = new (std::nothrow) tq_seq();
  if (!s) return TQ_ERR_INVALID_ARG;
  s->ncalls = ncalls;
  s->B = batch;
  s->Bp = batch <= 1 ? 1 : batch <= 2 ? 2 : batch <= 4 ? 4 : 8;
  s->G = G;
  s->grid = sms;
  s->dev = dev;
  s->pack = pack;
  const bool b3p = pack == TQ_PACK_B3;
  const int rows = b3p ? b3::kRows : kRows, item = b3p ? b3::kItemTrits : kItemTrits;
  s->nw = b3p ? b3::kNW : kNW;
  // per-call work split; the most K slices any CTA covers, the largest item count
  s->calls.resize(ncalls);
  long long Tmax = 0;
  for (int j = 0; j < ncalls; ++j) {
    const tq_seq_call& c = calls[j];
    CallDev& d = s->calls[j];
    std::memset(&d, 0, sizeof(d));
    d.x = c.x_src == TQ_SEQ_X_BF16 ? c.x : nullptr;
    d.scales = c.scales;
    d.y = c.y;
    d.N = c.d.N;
    d.K = c.d.K;
    d.ng = c.d.K / G;
    d.mode = c.x_src;
    d.apply = c.d.fwht_block != 0;
    d.nru = (c.d.N + rows - 1) / rows;
    d.nku = (c.d.K + item - 1) / item;
    const long long T = static_cast<long long>(d.nru) * d.nku;
    if (T * sms >= (1ll << 31)) {
      delete s;
      return TQ_ERR_UNSUPPORTED;
    }
    d.T = static_cast<int>(T);
    d.gp = std::min(sms, d.T);
    Tmax = std::max(Tmax, T);
    for (int cta = 0; cta < d.gp; ++cta) {
      const int a = cta_start(d.T, d.gp, cta), b = cta_start(d.T, d.gp, cta + 1);
      if (b > a) s->nkc = std::max(s->nkc, (b - 1) / d.nru - a / d.nru + 1);
    }
  }
  // shared memory: rings, scales (2-bit: their ring; base-3: a per-warp staging area), x^ of the CTA's K
  // slices, zero chunk, V, F, barriers, flags, and for base-3 the chunk table
  const int GPI = item / G;
  const int kD = b3p ? b3::kD : ring_depth(s->Bp);
  const size_t xh = align256(static_cast<size_t>(s->nkc) * GPI * s->Bp * 2 * G);
  const size_t vf = align256(static_cast<size_t>(s->nkc * GPI + 8) * s->Bp * 4);
  auto layout = [&]() {
    size_t off = static_cast<size_t>(s->nw) * kD * (b3p ? b3::kCodeStage : kCodeStage);
    s->off_scales = static_cast<uint32_t>(off);
    off += b3p ? align256(static_cast<size_t>(s->nw) * GPI * 64 * 2) : static_cast<size_t>(kNW) * kD * kScaleStage;
    s->off_xh = static_cast<uint32_t>(off);
    off += xh;
    s->off_zero = static_cast<uint32_t>(off);
    off += 256;
    s->off_v = static_cast<uint32_t>(off);
    off += vf;
    s->off_f = static_cast<uint32_t>(off);
    off += vf;
    s->off_bar = static_cast<uint32_t>(off);
    off += align256(static_cast<size_t>(s->nw) * kD * 8 + 8);  // base-3: one more, the table copy's
    s->off_misc = static_cast<uint32_t>(off);
    off += 256;
    if (b3p) {
      s->off_lut = static_cast<uint32_t>(off);
      off += align256(b3::kLutBytes);
    }
    s->smem = off + 1024;  // alignment slack of the base
  };
  layout();
  if (s->smem > kSmemLimit || s->smem > static_cast<size_t>(optin)) {
    delete s;
    return TQ_ERR_UNSUPPORTED;  // the activations of the widest CTA range do not fit shared memory
  }
  s->kern = seq_kernel(pack, G, s->Bp);
  if ((e = cudaFuncSetAttribute(s->kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(s->smem))) !=
      cudaSuccess) {
    delete s;
    return cuda_fail(e);
  }
  int bps = 0;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, s->kern, s->nw * 32, s->smem)) != cudaSuccess ||
      bps < 1) {
    delete s;
    return e != cudaSuccess ? cuda_fail(e) : TQ_ERR_UNSUPPORTED;
  }
  for (int j = 0; j < ncalls; ++j) {
    const tq_seq_call& c = calls[j];
    CallDev& d = s->calls[j];
    const int P = pitch_words(c.d.K, c.d.packing);
    // codes: box of 32 words x one item's rows, 128-byte swizzle; 2-bit scales: box of 8 groups
    if (!make_tmap_2d(&d.tm_codes, c.codes, CU_TENSOR_MAP_DATA_TYPE_UINT32, static_cast<uint64_t>(P),
                      static_cast<uint64_t>(c.d.N), static_cast<uint64_t>(P) * 4u, 32u, static_cast<uint32_t>(rows),
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
        (!b3p && !make_tmap_2d(&d.tm_scales, c.scales, CU_TENSOR_MAP_DATA_TYPE_UINT16, static_cast<uint64_t>(d.ng),
                               static_cast<uint64_t>(c.d.N), static_cast<uint64_t>(d.ng) * 2u, 8u, kRows,
                               CU_TENSOR_MAP_SWIZZLE_NONE))) {
      delete s;
      return TQ_ERR_CUDA;
    }
  }
  s->part_stride = static_cast<size_t>(Tmax) * s->Bp * rows;
  s->ssq_stride = (Kmax / kFwhtBlock) * s->Bp;
  s->ws_calls = align256(sizeof(CallDev) * ncalls);
  s->ws_sync = align256((kFlagBase + static_cast<size_t>(sms)) * 4);
  s->ws_part = align256(2 * s->part_stride * 4);
  s->ws_ssq = align256(static_cast<size_t>(2) * s->ssq_stride * 4);
  if (hand_batch(s->Bp)) {  // each call's output with its epoch, two parities
    int Nmax = 0;
    for (int j = 0; j < ncalls; ++j) Nmax = std::max(Nmax, calls[j].d.N);
    s->hand_stride = static_cast<size_t>(s->Bp) * Nmax;
    s->ws_hand = align256(2 * s->hand_stride * 8);
  }
  s->ws_bytes = s->ws_calls + s->ws_sync + s->ws_part + s->ws_ssq + s->ws_hand;
  *out = s;
  return TQ_OK;
}

extern "C" size_t tq_seq_workspace_bytes(const tq_seq* s) { return s ? s->ws_bytes : 0; }

extern "C" tq_status tq_seq_upload(const tq_seq* s, void* workspace, size_t workspace_bytes) {
  if (!s || !workspace) return TQ_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return TQ_ERR_MISALIGNED;
  if (workspace_bytes < s->ws_bytes) return TQ_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t e = cudaMemcpy(ws, s->calls.data(), sizeof(CallDev) * s->ncalls, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e);
  if ((e = cudaMemset(ws + s->ws_calls, 0, s->ws_sync)) != cudaSuccess) return cuda_fail(e);
  // no stale epochs: the handoff words start at epoch 0, which no call of a run uses
  if (s->ws_hand &&
      (e = cudaMemset(ws + s->ws_calls + s->ws_sync + s->ws_part + s->ws_ssq, 0, s->ws_hand)) != cudaSuccess)
    return cuda_fail(e);
  return TQ_OK;
}

extern "C" tq_status tq_seq_run(const tq_seq* s, void* workspace, void* stream) {
  if (!s || !workspace) return TQ_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return TQ_ERR_MISALIGNED;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev != s->dev) return TQ_ERR_INVALID_ARG;
  int* status = status_ptr();
  if (!status) return TQ_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  Params prm{};
  prm.calls = reinterpret_cast<const CallDev*>(ws);
  prm.ncalls = s->ncalls;
  prm.B = s->B;
  prm.status = status;
  prm.sync = reinterpret_cast<unsigned*>(ws + s->ws_calls);
  prm.part = reinterpret_cast<float*>(ws + s->ws_calls + s->ws_sync);
  prm.ssq = reinterpret_cast<float*>(ws + s->ws_calls + s->ws_sync + s->ws_part);
  prm.hand = s->ws_hand ? reinterpret_cast<uint64_t*>(ws + s->ws_calls + s->ws_sync + s->ws_part + s->ws_ssq) : nullptr;
  prm.hand_stride = s->hand_stride;
  prm.part_stride = s->part_stride;
  prm.ssq_stride = s->ssq_stride;
  prm.nkc = s->nkc;
  prm.off_scales = s->off_scales;
  prm.off_xh = s->off_xh;
  prm.off_zero = s->off_zero;
  prm.off_v = s->off_v;
  prm.off_f = s->off_f;
  prm.off_bar = s->off_bar;
  prm.off_misc = s->off_misc;
  prm.off_lut = s->off_lut;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(s->grid);
  cfg.blockDim = dim3(s->nw * 32);
  cfg.dynamicSmemBytes = s->smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&prm};
  if ((e = cudaLaunchKernelExC(&cfg, s->kern, args)) != cudaSuccess) return cuda_fail(e);
  return TQ_OK;
}

extern "C" int tq_seq_kernel_count(const tq_seq* s) { return s ? 1 : -1; }

extern "C" void tq_seq_destroy(tq_seq* s) { delete s; }

// ---- self-test of the bounded waits ------------------------------------------------------------
namespace tq {
namespace seq {

// One CTA waits, with a short limit, on what nothing will complete: kind 0 an mbarrier that is
// never arrived on (the form of every TMA-ring wait), kind 1 a grid barrier that no CTA arrives at
// (the form of the call-boundary wait above).  The wait gives up, the kernel records TQ_ERR_TIMEOUT
// exactly as the production kernels do and returns.
__global__ void selftest_wait_kernel(int kind, unsigned long long limit_ns, unsigned* counter, int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  bool ok;
  if (kind == 0) {
    ok = mbar_wait(&bar, 0, limit_ns);
  } else {
    ok = grid_wait(counter, 0, &flag, limit_ns);  // counter is 0 and nothing adds to it
  }
  if (!ok && threadIdx.x == 0) record_error(status, TQ_ERR_TIMEOUT);
}

}  // namespace seq
}  // namespace tq

extern "C" tq_status tq_selftest_wait(int kind, long long limit_ns, void* workspace, void* stream) {
  using namespace tq;
  if ((kind != 0 && kind != 1) || limit_ns <= 0 || limit_ns > 1000000000ll) return TQ_ERR_INVALID_ARG;
  if (kind == 1 && !workspace) return TQ_ERR_INVALID_ARG;
  if (workspace && !aligned(workspace, 256)) return TQ_ERR_MISALIGNED;
  int* status = status_ptr();
  if (!status) return TQ_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned* counter = static_cast<unsigned*>(workspace);
  cudaError_t e;
  if (counter && (e = cudaMemsetAsync(counter, 0, sizeof(unsigned), st)) != cudaSuccess) return cuda_fail(e);
  seq::selftest_wait_kernel<<<1, 32, 0, st>>>(kind, static_cast<unsigned long long>(limit_ns), counter, status);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);
  return TQ_OK;
}

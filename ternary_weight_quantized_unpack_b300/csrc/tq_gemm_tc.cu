// Batched prefill: Y[m][n] = bf16( sum_k x~[m][k] * s[n][k/group] * t[n][k] ), fp32 accumulation.
//
// Prefill is a dense contraction (M = 2048..4096 tokens), so it runs on the 5th-generation tensor
// cores (tcgen05.mma kind::f16, accumulators in tensor memory).  The ternary weights are decoded
// once per call into exact FP16 products s * t (t in {-1, 0, 1}, so s * t is s, -s or 0): decoding
// inside the MMA loop would cost about one instruction per weight, and with 256 tokens of reuse per
// weight tile the SM would need ~16 decoded weights per cycle to keep the tensor pipe busy, far above
// its issue rate.  The one-off decode streams the packed weights from HBM (0.25 B per weight, 2-bit)
// and writes 2 B per weight; its cost is amortised over all M tokens.
//
// GEMM kernel: persistent, one CTA per SM, 128-token x 256-weight-row output tiles, K in steps of 64:
//   warp 0     TMA producer: 128B-swizzled tiles of x~ (128 x 64) and W (256 x 64) into a 4-stage
//              ring, running ahead across tiles
//   warp 1     MMA issuer (one thread): 4 x tcgen05.mma M128 N256 K16 per stage into one of two
//              TMEM accumulators (2 x 256 columns); a commit frees the stage, another marks the
//              accumulator full
//   warps 2-5  epilogue: tcgen05.ld of a full accumulator, bf16 conversion, stores; then the
//              accumulator is released, so one tile's epilogue overlaps the next tile's MMAs
// Every mbarrier wait is bounded; a wait that runs out records TQ_ERR_TIMEOUT and the warp stops.
//
// Grouped mode (the expert layer at prefill sizes): instead of the M x N tile grid the kernel walks a
// tile list written on the device - {first A row, valid rows, first B row, first output column} -
// so one launch covers every routed expert: A holds the tokens sorted by expert, B the decoded
// weights of all experts stacked, and rows past an expert's token count are computed but not stored.
// Output fp32.
// Activations are the block Walsh-Hadamard transform of x in FP16 ("27B 大模型塞进
// 5.9GB", section 二 ①); group scales per 64 or 128 weights (same page, section 二 ②).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <algorithm>
#include <map>
#include <mutex>

#include "tq_internal.cuh"
#include "tq_kernels.cuh"
#include "tq_sm100.cuh"
#include "tq_tmap.cuh"

namespace tq {
namespace gemm {

using namespace sm100;

constexpr int BM = 128;  // tokens per tile (MMA M, TMEM lanes)
constexpr int BN = 256;  // weight rows per tile (MMA N, TMEM columns)
constexpr int BK = 64;   // K per stage: one 128-byte swizzle row of FP16 ...
constexpr int BK8 = 128; // ... or of FP8
constexpr int STAGES = 4;
constexpr uint32_t kABytes = BM * BK * 2;
constexpr uint32_t kBBytes = BN * BK * 2;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;  // two 128 x 256 fp32 accumulators

struct Smem {
  uint8_t a[STAGES][kABytes];  // each 1024-byte aligned (sizes are multiples of 1024)
  uint8_t b[STAGES][kBBytes];
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t acc_full[2];   // MMA issuer -> epilogue
  uint64_t acc_empty[2];  // epilogue (one arrival per warp) -> MMA issuer
  uint32_t tmem;
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;  // + alignment of the base to 1024

// v * 2^e: one multiply by the exact power of two while 2^e is a normal float (one rounding only where
// the product leaves the normal range, as ldexpf), ldexpf beyond.
__device__ __forceinline__ float scale2(float v, int e) {
  return e >= -126 && e <= 127 ? v * __int_as_float((127 + e) << 23) : ldexpf(v, e);
}

// Tile list of the grouped mode (tiles == nullptr: the plain M x N grid).
struct GroupedTiles {
  const int4* tiles;  // {A row, valid rows, B row, output column}
  const int* count;   // number of tiles
  float* y;           // fp32 output, row r at y + r * ldy
  int ldy;
};

__device__ __forceinline__ void tile_of(const GroupedTiles& gt, int t, int n_mt, int& m0, int& rows, int& nb, int& no) {
  if (gt.tiles) {
    const int4 v = gt.tiles[t];
    m0 = v.x;
    rows = v.y;
    nb = v.z;
    no = v.w;
  } else {
    m0 = (t % n_mt) * BM;
    rows = BM;
    nb = no = (t / n_mt) * BN;
  }
}

// F8: operands FP8 E4M3 (kind::f8f6f4), each row of x~ and of W under its own power-of-two factor
// fa[m] = 2^ea[m] / fb[n] = 2^eb[n] (floats), which the epilogue applies as one exact power of two.
template <bool F8>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w, uint16_t* y,
                   int M, int N, int K, int* status, const __grid_constant__ GroupedTiles gt, const float* fa,
                   const float* fb) {
  constexpr int BKE = F8 ? BK8 : BK;  // K elements per stage
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = K / BKE;
  const int n_mt = (M + BM - 1) / BM;
  const int n_tiles = gt.tiles ? *gt.count : n_mt * ((N + BN - 1) / BN);
  // tile t: token tile t % n_mt, weight tile t / n_mt (the CTAs running together share few weight tiles)
  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.acc_full[b], 1);
      mbar_init(&sm.acc_empty[b], 4);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem;

  if (warp == 0 && lane == 0) {
    int g = 0;  // K steps issued so far, over all tiles
    bool ok = true;
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
      int m0, rows, nb, no;
      tile_of(gt, t, n_mt, m0, rows, nb, no);
      for (int kb = 0; kb < nk; ++kb, ++g) {
        const int s = g % STAGES;
        if (g >= STAGES && !mbar_wait(&sm.empty[s], ((g / STAGES) & 1) ^ 1)) {
          record_error(status, TQ_ERR_TIMEOUT);
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&sm.full[s], kABytes + kBBytes);
        tma_load_2d(sm.a[s], &tm_x, kb * BKE, m0, &sm.full[s]);
        tma_load_2d(sm.b[s], &tm_w, kb * BKE, nb, &sm.full[s]);
      }
    }
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
    int g = 0, it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++it) {
      const int b = it & 1;
      if (it >= 2 && !mbar_wait(&sm.acc_empty[b], ((it >> 1) - 1) & 1)) {  // epilogue of tile it - 2 done
        record_error(status, TQ_ERR_TIMEOUT);
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem + static_cast<uint32_t>(b * BN);
      for (int kb = 0; kb < nk; ++kb, ++g) {
        const int s = g % STAGES;
        if (!mbar_wait(&sm.full[s], (g / STAGES) & 1)) {
          record_error(status, TQ_ERR_TIMEOUT);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_addr(sm.a[s]), b0 = smem_addr(sm.b[s]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {  // 32 bytes of K each: 16 FP16 or 32 FP8
          if (F8)
            mma_f8_ss(d, smem_desc_sw128(a0 + 32u * k), smem_desc_sw128(b0 + 32u * k), idesc, (kb | k) != 0);
          else
            mma_f16_ss(d, smem_desc_sw128(a0 + 32u * k), smem_desc_sw128(b0 + 32u * k), idesc, (kb | k) != 0);
        }
        mma_commit(&sm.empty[s]);  // the stage is free once these MMAs have read it
      }
      mma_commit(&sm.acc_full[b]);
    }
  } else if (warp >= 2) {
    const int q = warp & 3;  // a warp reads TMEM lanes 32 (warp % 4) .. + 31
    const bool vec = (N & 7) == 0;
    int it = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++it) {
      const int b = it & 1;
      int m0, rows, nb, n0;
      tile_of(gt, t, n_mt, m0, rows, nb, n0);
      if (!mbar_wait(&sm.acc_full[b], (it >> 1) & 1)) {
        if (lane == 0) record_error(status, TQ_ERR_TIMEOUT);
        break;
      }
      tc_fence_after();
      const int m = m0 + 32 * q + lane;
      const float fam = F8 && m < M ? fa[m] : 1.f;
#pragma unroll 1
      for (int c = 0; c < BN; c += 32) {
        uint32_t v[32];
        tmem_ld<32>(tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(b * BN + c), v);
        tmem_wait_ld();
        const int n = n0 + c;
        if (F8) {  // y = acc * (2^ea[m] * 2^eb[n]): the factor is an exact power of two, one rounding
#pragma unroll
          for (int j = 0; j < 32; ++j)
            v[j] = __float_as_uint(__uint_as_float(v[j]) * (fam * (n + j < N ? __ldg(fb + n + j) : 1.f)));
        }
        if (gt.tiles) {
          if (32 * q + lane < rows) {
            float4* dst = reinterpret_cast<float4*>(gt.y + static_cast<size_t>(m) * gt.ldy + n);
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              dst[j / 4] = make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]), __uint_as_float(v[j + 2]),
                                       __uint_as_float(v[j + 3]));
          }
        } else if (m < M && n < N) {
          uint16_t* dst = y + static_cast<size_t>(m) * N + n;
          if (vec && n + 32 <= N) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              uint4 o;
              uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const __nv_bfloat162 h =
                    __floats2bfloat162_rn(__uint_as_float(v[j + 2 * i]), __uint_as_float(v[j + 2 * i + 1]));
                ow[i] = *reinterpret_cast<const uint32_t*>(&h);
              }
              *reinterpret_cast<uint4*>(dst + j) = o;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if (n + j < N) {
                const __nv_bfloat16 h = __float2bfloat16_rn(__uint_as_float(v[j]));
                dst[j] = *reinterpret_cast<const uint16_t*>(&h);
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.acc_empty[b]);  // this warp is done with the accumulator
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------------------------
// Decode: codes -> W[n][k] = s[n][k / G] * t[n][k] as FP16 (exact: s, -s or 0).
// 2-bit: one thread per word (16 trits, one group), two 16-byte stores.
// base-3: one thread per 4 words (80 trits), digits by exact reciprocal multiplies.
// ---------------------------------------------------------------------------------------------
// The output of a CTA's threads is one contiguous range of W (threads take consecutive words or quads
// of consecutive rows), so each thread writes its 16-byte pieces into shared memory at their offset
// in that range and the CTA then stores the range with consecutive lanes on consecutive 16 bytes:
// whole 32-byte sectors per store instead of half sectors.
constexpr int kDecThreads = 256;

__device__ __forceinline__ void flush_stage(const uint4* stage, uint16_t* w, long long base, long long end) {
  __syncthreads();
  uint4* out = reinterpret_cast<uint4*>(w + base);
  const int nchunks = static_cast<int>((end - base) / 8);
  for (int c = threadIdx.x; c < nchunks; c += blockDim.x) out[c] = stage[c];
}

// Pair tables: a pair of trits becomes two FP16 halves (t0 in the low half) as (mask & s2) ^ sign,
// s2 = the scale in both halves: mask has 0xFFFF in a half whose trit is non-zero, sign 0x8000 (the
// FP16 sign bit, flipped) in a half whose trit is -1.  2-bit: indexed by the pair's 4 code bits (field 3 reads as t = 0, as
// tq_unpack reads it); base-3: by the pair's value d0 + 3 d1 (0..8, d = t + 1).
__device__ __forceinline__ void pair_entry(int t0, int t1, uint32_t& mask, uint32_t& sign) {
  mask = (t0 != 0 ? 0x0000FFFFu : 0u) | (t1 != 0 ? 0xFFFF0000u : 0u);
  sign = (t0 < 0 ? 0x00008000u : 0u) | (t1 < 0 ? 0x80000000u : 0u);
}

// 2-bit: one thread per word (16 weights of one group), eight pairs, two 16-byte pieces.
__global__ void __launch_bounds__(kDecThreads) decode_2b_kernel(const uint32_t* __restrict__ codes,
                                                                const uint16_t* __restrict__ scales,
                                                                uint16_t* __restrict__ w, int N, int K, int P, int ng,
                                                                int G) {
  __shared__ uint4 stage[kDecThreads * 2];
  __shared__ uint2 pairs[16];
  if (threadIdx.x < 16) {
    const int f0 = threadIdx.x & 3, f1 = threadIdx.x >> 2;
    uint32_t m, sg;
    pair_entry(f0 == 3 ? 0 : f0 - 1, f1 == 3 ? 0 : f1 - 1, m, sg);
    pairs[threadIdx.x] = make_uint2(m, sg);
  }
  __syncthreads();
  const int wpr = K / 16;  // words with data per row
  const long long total = static_cast<long long>(N) * wpr;
  const long long i0 = static_cast<long long>(blockIdx.x) * blockDim.x;
  const long long i = i0 + threadIdx.x;
  // word i writes W[16 i .. 16 i + 15] (rows are K = 16 * wpr wide): the CTA's range is contiguous
  const long long base = 16 * i0, end = 16 * min(total, i0 + blockDim.x);
  if (i < total) {
    const int n = static_cast<int>(i / wpr), j = static_cast<int>(i - static_cast<long long>(n) * wpr);
    const uint32_t word = __ldg(codes + static_cast<size_t>(n) * P + j);
    const uint32_t s = __ldg(scales + static_cast<size_t>(n) * ng + (16 * j) / G);
    const uint32_t s2 = s | (s << 16);
    uint32_t o[8];
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      const uint2 e = pairs[(word >> (4 * h)) & 15u];
      o[h] = (e.x & s2) ^ e.y;
    }
    stage[2 * threadIdx.x] = make_uint4(o[0], o[1], o[2], o[3]);
    stage[2 * threadIdx.x + 1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
  flush_stage(stage, w, base, end);
}

// base-3: one thread per 2 words (40 trits, 80 bytes of output) of a row; a pair of trits is the
// word's value mod 9, taken by an exact reciprocal multiply.  K is a multiple of 8 here (the FWHT
// block), so every piece and the row tail are whole 16-byte pieces and go through the staging above.
constexpr int kB3DecWords = 2;
__global__ void __launch_bounds__(kDecThreads) decode_b3_kernel(const uint32_t* __restrict__ codes,
                                                                const uint16_t* __restrict__ scales,
                                                                uint16_t* __restrict__ w, int N, int K, int P, int ng,
                                                                int G) {
  constexpr int kT = 20 * kB3DecWords;  // trits per thread
  __shared__ uint4 stage[kDecThreads * (kT / 8)];
  __shared__ uint2 pairs[9];
  if (threadIdx.x < 9) {
    uint32_t m, sg;
    pair_entry(static_cast<int>(threadIdx.x % 3) - 1, static_cast<int>(threadIdx.x / 3) - 1, m, sg);
    pairs[threadIdx.x] = make_uint2(m, sg);
  }
  __syncthreads();
  const int ppr = (K + kT - 1) / kT;  // pieces per row
  const long long total = static_cast<long long>(N) * ppr;
  const long long i0 = static_cast<long long>(blockIdx.x) * blockDim.x;
  const long long i = i0 + threadIdx.x;
  auto out_of = [&](long long q) {  // first element of W that piece q writes
    const long long n = q / ppr;
    return n * K + static_cast<long long>(kT) * (q - n * ppr);
  };
  const long long base = out_of(i0);
  const long long last = min(total, i0 + blockDim.x) - 1;
  const long long end = out_of(last) + min(kT, K - kT * static_cast<int>(last % ppr));
  if (i < total) {
    const int n = static_cast<int>(i / ppr), j = static_cast<int>(i - static_cast<long long>(n) * ppr);
    const int k0 = kT * j, kn = min(kT, K - k0);
    const uint16_t* srow = scales + static_cast<size_t>(n) * ng;
    // the (at most two) groups the piece touches (groups are 64 or 128 >= 40), and where the second
    // starts (relative to k0)
    const int g0 = k0 / G;
    const int b1 = (g0 + 1) * G - k0;
    const uint32_t sa = __ldg(srow + g0);
    const uint32_t sb = b1 < kn ? __ldg(srow + g0 + 1) : sa;
    const uint32_t s2a = sa | (sa << 16), s2b = sb | (sb << 16);
    uint32_t wv[kB3DecWords];
#pragma unroll
    for (int wi = 0; wi < kB3DecWords; ++wi)
      wv[wi] = 20 * wi < kn ? min(__ldg(codes + static_cast<size_t>(n) * P + kB3DecWords * j + wi), kB3Max) : kB3Zero;
    uint4* st = stage + (out_of(i) - base) / 8;
#pragma unroll
    for (int c = 0; c < kT / 8; ++c) {
      uint32_t o[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int pr = 4 * c + h;        // pair within the piece
        const int wi = pr / 10;          // its word
        const uint32_t v = wv[wi];
        const uint32_t q = __umulhi(v, 0x38E38E39u) >> 1;  // v / 9, exact for every 32-bit v
        wv[wi] = q;
        const uint2 e = pairs[v - 9u * q];
        o[h] = (e.x & (2 * pr < b1 ? s2a : s2b)) ^ e.y;
      }
      if (8 * c < kn) st[c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
  flush_stage(stage, w, base, end);
}

// ---------------------------------------------------------------------------------------------
// FP8 operands.  Row factors: ea[m] = floor(log2 max_k |x~[m][k]|) - 7 and eb[n] = floor(log2
// max_g |s[n][g]|) - 7 (0 for an all-zero row), so each row's largest magnitude lands in [128, 256),
// below the E4M3 maximum 448; values are rounded to E4M3 to nearest even (cvt .satfinite).
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ int row_exponent(float mx) {
  if (!(mx > 0.f)) return 0;
  int ex = 0;
  (void)frexpf(mx, &ex);  // mx = f * 2^ex, f in [0.5, 1)
  return ex - 1 - 7;
}

__device__ __forceinline__ uint8_t to_e4m3(float v) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

// One CTA per token row: the block transform of the row (bf16 in, fp32), its largest magnitude, then
// the E4M3 values of x~ * 2^-ea (the transform is recomputed in the second pass from the bf16 input).
constexpr int kActThreads = 256;
__global__ void __launch_bounds__(kActThreads) fp8_act_kernel(const uint16_t* __restrict__ x, uint8_t* __restrict__ xq,
                                                              float* __restrict__ fa, int K, int apply, int* status) {
  __shared__ float red[kActThreads / 32];
  const int m = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nblk = K / kFwhtBlock;
  const uint16_t* xr = x + static_cast<size_t>(m) * K;
  auto block_values = [&](int blk, float (&v)[4]) {
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(xr + blk * kFwhtBlock + 4 * lane));
    v[0] = bf16_bits_to_float(static_cast<uint16_t>(raw.x & 0xffffu));
    v[1] = bf16_bits_to_float(static_cast<uint16_t>(raw.x >> 16));
    v[2] = bf16_bits_to_float(static_cast<uint16_t>(raw.y & 0xffffu));
    v[3] = bf16_bits_to_float(static_cast<uint16_t>(raw.y >> 16));
    if (apply) {
      fwht128_warp(v);
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] *= 0.08838834764831845f;
    }
  };
  float mx = 0.f;
  for (int blk = warp; blk < nblk; blk += kActThreads / 32) {
    float v[4];
    block_values(blk, v);
#pragma unroll
    for (int j = 0; j < 4; ++j) mx = fmaxf(mx, fabsf(v[j]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  mx = red[0];
#pragma unroll
  for (int w = 1; w < kActThreads / 32; ++w) mx = fmaxf(mx, red[w]);
  if (!(mx <= 3.0e38f)) {  // inf or NaN in the row
    if (threadIdx.x == 0) record_error(status, TQ_ERR_RANGE);
    mx = 0.f;
  }
  const int e = row_exponent(mx);
  if (threadIdx.x == 0) fa[m] = ldexpf(1.f, e);
  for (int blk = warp; blk < nblk; blk += kActThreads / 32) {
    float v[4];
    block_values(blk, v);
    uint32_t o = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) o |= static_cast<uint32_t>(to_e4m3(scale2(v[j], -e))) << (8 * j);
    *reinterpret_cast<uint32_t*>(xq + static_cast<size_t>(m) * K + blk * kFwhtBlock + 4 * lane) = o;
  }
}

// The same in one pass over the input: the row's transformed values wait in shared memory (K floats)
// while the CTA takes the maximum; then each thread converts and stores 16 consecutive values.
constexpr int kActSmemThreads = 512;
__global__ void __launch_bounds__(kActSmemThreads) fp8_act_smem_kernel(const uint16_t* __restrict__ x,
                                                                   uint8_t* __restrict__ xq, float* __restrict__ fa,
                                                                   int K, int apply, int* status) {
  extern __shared__ float4 xs4[];
  __shared__ float red[kActSmemThreads / 32];
  const int m = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nblk = K / kFwhtBlock;
  const uint16_t* xr = x + static_cast<size_t>(m) * K;
  float mx = 0.f;
  constexpr int kNWarps = kActSmemThreads / 32, kBatch = 8;  // a warp's blocks, 8 loads in flight at a time
  for (int base = warp; base < nblk; base += kNWarps * kBatch) {
    uint2 raw[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int blk = base + kNWarps * i;
      if (blk < nblk) raw[i] = __ldg(reinterpret_cast<const uint2*>(xr + blk * kFwhtBlock + 4 * lane));
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int blk = base + kNWarps * i;
      if (blk >= nblk) break;
      float v[4] = {bf16_bits_to_float(static_cast<uint16_t>(raw[i].x & 0xffffu)),
                    bf16_bits_to_float(static_cast<uint16_t>(raw[i].x >> 16)),
                    bf16_bits_to_float(static_cast<uint16_t>(raw[i].y & 0xffffu)),
                    bf16_bits_to_float(static_cast<uint16_t>(raw[i].y >> 16))};
      if (apply) {
        fwht128_warp(v);
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] *= 0.08838834764831845f;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) mx = fmaxf(mx, fabsf(v[j]));
      xs4[blk * (kFwhtBlock / 4) + lane] = make_float4(v[0], v[1], v[2], v[3]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  mx = red[0];
#pragma unroll
  for (int w = 1; w < kActSmemThreads / 32; ++w) mx = fmaxf(mx, red[w]);
  if (!(mx <= 3.0e38f)) {  // inf or NaN in the row
    if (threadIdx.x == 0) record_error(status, TQ_ERR_RANGE);
    mx = 0.f;
  }
  const int e = row_exponent(mx);
  if (threadIdx.x == 0) fa[m] = ldexpf(1.f, e);
  uint4* out = reinterpret_cast<uint4*>(xq + static_cast<size_t>(m) * K);
  for (int c = threadIdx.x; c < K / 16; c += kActSmemThreads) {
    uint32_t o[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float4 v = xs4[4 * c + w];
      o[w] = static_cast<uint32_t>(to_e4m3(scale2(v.x, -e))) | (static_cast<uint32_t>(to_e4m3(scale2(v.y, -e))) << 8) |
             (static_cast<uint32_t>(to_e4m3(scale2(v.z, -e))) << 16) |
             (static_cast<uint32_t>(to_e4m3(scale2(v.w, -e))) << 24);
    }
    out[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}
constexpr int kActSmemMaxK = 200 * 1024 / 4;  // K up to which the one-pass kernel is used

// eb[n] from the row's scales (one thread per row).
__global__ void fp8_wexp_kernel(const uint16_t* __restrict__ scales, int* __restrict__ eb, float* __restrict__ fb,
                                int N, int ng, int* status) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  float mx = 0.f;
  for (int g = 0; g < ng; ++g) mx = fmaxf(mx, fabsf(__half2float(__ushort_as_half(__ldg(scales + static_cast<size_t>(n) * ng + g)))));
  if (!(mx <= 65504.f)) {
    record_error(status, TQ_ERR_RANGE);
    mx = 0.f;
  }
  const int e = row_exponent(mx);
  eb[n] = e;
  fb[n] = ldexpf(1.f, e);
}

// E4M3 of +-s * 2^-eb: the byte for +s; -s flips the sign bit, t = 0 is the byte 0.
__device__ __forceinline__ uint8_t signed_e4m3(int t, uint8_t pos) {
  return t == 0 ? static_cast<uint8_t>(0) : (t > 0 ? pos : static_cast<uint8_t>(pos ^ 0x80u));
}

// 2-bit: a warp takes 128 consecutive words (of the flattened [N][K/16] word grid), lane l the words
// l + 32 q (q < 4): every load and every 16-byte store of the warp is one contiguous 128- / 512-byte
// range, and each lane has four independent loads in flight.  A word is 16 weights of one group.
// A byte of a code word (four 2-bit fields) becomes four output bytes through two tables built in
// shared memory: nz (0xFF where t != 0) and neg (0x80 where t = -1); out = (nz & 4 x pos) ^ neg, pos
// the E4M3 byte of s * 2^-eb (the sign bit flips for t = -1, whatever the sign of s).
constexpr int kF8WordsPerLane = 4;
__global__ void __launch_bounds__(kDecThreads) decode_2b_f8_kernel(const uint32_t* __restrict__ codes,
                                                                   const uint16_t* __restrict__ scales,
                                                                   const int* __restrict__ eb, uint8_t* __restrict__ w,
                                                                   int N, int K, int P, int ng, int G) {
  __shared__ uint32_t nz_t[256], neg_t[256];
  {
    const uint32_t b = threadIdx.x;  // kDecThreads == 256: one entry per thread
    uint32_t nz = 0, ng8 = 0;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const uint32_t f = (b >> (2 * h)) & 3u;  // field 1 is t = 0, field 3 reads as t = 0
      if (f == 0u || f == 2u) nz |= 0xFFu << (8 * h);
      if (f == 0u) ng8 |= 0x80u << (8 * h);
    }
    nz_t[b] = nz;
    neg_t[b] = ng8;
  }
  __syncthreads();
  const int wpr = K / 16;
  const unsigned total = static_cast<unsigned>(N) * static_cast<unsigned>(wpr);  // < 2^31 (checked on the host)
  const unsigned base = (blockIdx.x * blockDim.x + (threadIdx.x & ~31u)) * kF8WordsPerLane + (threadIdx.x & 31u);
  uint32_t word[kF8WordsPerLane];
  float sv[kF8WordsPerLane];
  int ev[kF8WordsPerLane];
#pragma unroll
  for (int q = 0; q < kF8WordsPerLane; ++q) {
    const unsigned i = min(base + 32u * q, total - 1u);
    const unsigned n = i / static_cast<unsigned>(wpr), j = i - n * static_cast<unsigned>(wpr);
    word[q] = __ldg(codes + static_cast<size_t>(n) * P + j);
    sv[q] = __half2float(__ushort_as_half(__ldg(scales + static_cast<size_t>(n) * ng + (16 * j) / G)));
    ev[q] = __ldg(eb + n);
  }
#pragma unroll
  for (int q = 0; q < kF8WordsPerLane; ++q) {
    const unsigned i = base + 32u * q;
    if (i >= total) break;
    const uint32_t pos4 = static_cast<uint32_t>(to_e4m3(ldexpf(sv[q], -ev[q]))) * 0x01010101u;
    uint32_t o[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t b = (word[q] >> (8 * c)) & 0xFFu;
      o[c] = (nz_t[b] & pos4) ^ neg_t[b];
    }
    // word i of the flattened grid is weights 16 i .. 16 i + 15 of W (rows are K = 16 * wpr wide)
    *reinterpret_cast<uint4*>(w + 16 * static_cast<size_t>(i)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// base-3: one thread per 4 words (80 weights) of a row; K is a multiple of 128, so every 80-weight
// piece and the row tail are whole 16-byte pieces.
__global__ void __launch_bounds__(kDecThreads) decode_b3_f8_kernel(const uint32_t* __restrict__ codes,
                                                                   const uint16_t* __restrict__ scales,
                                                                   const int* __restrict__ eb, uint8_t* __restrict__ w,
                                                                   int N, int K, int P, int ng, int G) {
  const int per_row = (K + 79) / 80;
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<long long>(N) * per_row) return;
  const int n = static_cast<int>(i / per_row), j = static_cast<int>(i - static_cast<long long>(n) * per_row);
  const int k0 = 80 * j, kn = min(80, K - k0);
  const uint16_t* srow = scales + static_cast<size_t>(n) * ng;
  const int e = __ldg(eb + n);
  const int g0 = k0 / G;
  const int b1 = (g0 + 1) * G - k0, b2 = b1 + G;
  const uint8_t pa = to_e4m3(ldexpf(__half2float(__ushort_as_half(__ldg(srow + g0))), -e));
  const uint8_t pb = b1 < kn ? to_e4m3(ldexpf(__half2float(__ushort_as_half(__ldg(srow + g0 + 1))), -e)) : pa;
  const uint8_t pc = b2 < kn ? to_e4m3(ldexpf(__half2float(__ushort_as_half(__ldg(srow + g0 + 2))), -e)) : pb;
  uint32_t o[20];
#pragma unroll
  for (int wi = 0; wi < 4; ++wi) {
    uint32_t v = 20 * wi < kn ? min(__ldg(codes + static_cast<size_t>(n) * P + 4 * j + wi), kB3Max) : kB3Zero;
#pragma unroll
    for (int d4 = 0; d4 < 5; ++d4) {
      uint32_t out = 0;
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const uint32_t qd = __umulhi(v, 0xAAAAAAABu) >> 1;  // v / 3, exact for every 32-bit v
        const int t = static_cast<int>(v - 3u * qd) - 1;
        v = qd;
        const int k = 20 * wi + 4 * d4 + h;
        out |= static_cast<uint32_t>(signed_e4m3(t, k < b1 ? pa : (k < b2 ? pb : pc))) << (8 * h);
      }
      o[5 * wi + d4] = out;
    }
  }
  uint4* dst = reinterpret_cast<uint4*>(w + static_cast<size_t>(n) * K + k0);
#pragma unroll
  for (int c = 0; c < 5; ++c)
    if (16 * c < kn) dst[c] = make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
}

// ---------------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------------
template <bool F8>
cudaError_t ensure_attr() {
  static std::map<int, bool> done;
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(gemm_tc_kernel<F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kSmemBytes));
  if (e == cudaSuccess) done[dev] = true;
  return e;
}

int sm_count() {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    sms = 148;
  }
  return sms;
}

}  // namespace gemm

size_t gemm_workspace_bytes(const tq_desc* d, int M) {
  return align256(static_cast<size_t>(M) * d->K * 2) + align256(static_cast<size_t>(d->N) * d->K * 2);
}

cudaError_t launch_gemm(const tq_desc* d, const uint32_t* codes, const uint16_t* scales, const uint16_t* x, int M,
                        uint16_t* y, void* ws, cudaStream_t s) {
  using namespace gemm;
  const int N = d->N, K = d->K, G = d->group, P = pitch_words(K, d->packing), ng = K / G;
  uint16_t* xa = static_cast<uint16_t*>(ws);
  uint16_t* wa = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + align256(static_cast<size_t>(M) * K * 2));
  // x~ in FP16 (values beyond the FP16 range record TQ_ERR_RANGE)
  cudaError_t e = launch_fwht_bf16(x, xa, 1, M, K, d->fwht_block != 0, s);
  if (e != cudaSuccess) return e;
  // W = s * t in FP16
  if (d->packing == TQ_PACK_2BIT) {
    const long long n = static_cast<long long>(N) * (K / 16);
    decode_2b_kernel<<<static_cast<unsigned>((n + kDecThreads - 1) / kDecThreads), kDecThreads, 0, s>>>(codes, scales, wa, N, K, P, ng, G);
  } else {
    const long long n = static_cast<long long>(N) * ((K + 20 * kB3DecWords - 1) / (20 * kB3DecWords));
    decode_b3_kernel<<<static_cast<unsigned>((n + kDecThreads - 1) / kDecThreads), kDecThreads, 0, s>>>(codes, scales, wa, N, K, P, ng, G);
  }
  if ((e = cudaPeekAtLastError()) != cudaSuccess) return e;
  CUtensorMap tm_x, tm_w;
  if (!make_tmap_2d(&tm_x, xa, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, K, M, static_cast<uint64_t>(K) * 2, BK, BM,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tm_w, wa, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, K, N, static_cast<uint64_t>(K) * 2, BK, BN,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if ((e = ensure_attr<false>()) != cudaSuccess) return e;
  // persistent: one CTA per SM, each walking the tiles with a stride of the grid
  int dev = 0, sms = 148;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) sms = 148;
  const long long tiles = static_cast<long long>((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  const unsigned grid = static_cast<unsigned>(std::min<long long>(tiles, sms));
  gemm_tc_kernel<false><<<grid, kThreads, kSmemBytes, s>>>(tm_x, tm_w, y, M, N, K, status_ptr(), GroupedTiles{},
                                                           nullptr, nullptr);
  return cudaPeekAtLastError();
}

cudaError_t launch_gemm_grouped(const uint16_t* xa, int a_rows, const uint16_t* wa, int w_rows, int K, const int* tiles,
                                const int* count, int max_tiles, float* y, int ldy, cudaStream_t s) {
  using namespace gemm;
  CUtensorMap tm_x, tm_w;
  if (!make_tmap_2d(&tm_x, xa, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, K, a_rows, static_cast<uint64_t>(K) * 2, BK, BM,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tm_w, wa, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, K, w_rows, static_cast<uint64_t>(K) * 2, BK, BN,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  cudaError_t e;
  if ((e = ensure_attr<false>()) != cudaSuccess) return e;
  int dev = 0, sms = 148;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) sms = 148;
  const unsigned grid = static_cast<unsigned>(std::max(1, std::min(max_tiles, sms)));
  const GroupedTiles gt{reinterpret_cast<const int4*>(tiles), count, y, ldy};
  gemm_tc_kernel<false><<<grid, kThreads, kSmemBytes, s>>>(tm_x, tm_w, nullptr, a_rows, 0, K, status_ptr(), gt,
                                                           nullptr, nullptr);
  return cudaPeekAtLastError();
}

cudaError_t launch_decode(const tq_desc* d, const uint32_t* codes, const uint16_t* scales, uint16_t* w, cudaStream_t s) {
  using namespace gemm;
  const int N = d->N, K = d->K, G = d->group, P = pitch_words(K, d->packing), ng = K / G;
  if (d->packing == TQ_PACK_2BIT) {
    const long long n = static_cast<long long>(N) * (K / 16);
    decode_2b_kernel<<<static_cast<unsigned>((n + kDecThreads - 1) / kDecThreads), kDecThreads, 0, s>>>(codes, scales, w, N, K, P, ng, G);
  } else {
    const long long n = static_cast<long long>(N) * ((K + 20 * kB3DecWords - 1) / (20 * kB3DecWords));
    decode_b3_kernel<<<static_cast<unsigned>((n + kDecThreads - 1) / kDecThreads), kDecThreads, 0, s>>>(codes, scales, w, N, K, P, ng, G);
  }
  return cudaPeekAtLastError();
}

size_t gemm_fp8_workspace_bytes(const tq_desc* d, int M) {
  return align256(static_cast<size_t>(M) * d->K) + align256(static_cast<size_t>(d->N) * d->K) +
         align256(static_cast<size_t>(M) * 4) + 2 * align256(static_cast<size_t>(d->N) * 4);
}

cudaError_t launch_gemm_fp8(const tq_desc* d, const uint32_t* codes, const uint16_t* scales, const uint16_t* x, int M,
                            uint16_t* y, void* ws, cudaStream_t s) {
  using namespace gemm;
  const int N = d->N, K = d->K, G = d->group, P = pitch_words(K, d->packing), ng = K / G;
  uint8_t* xq = static_cast<uint8_t*>(ws);
  uint8_t* wq = xq + align256(static_cast<size_t>(M) * K);
  float* fa = reinterpret_cast<float*>(wq + align256(static_cast<size_t>(N) * K));
  int* eb = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(fa) + align256(static_cast<size_t>(M) * 4));
  float* fb = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(eb) + align256(static_cast<size_t>(N) * 4));
  int* status = status_ptr();
  cudaError_t e;
  if (K <= kActSmemMaxK) {
    const size_t sm = static_cast<size_t>(K) * 4;
    static std::map<int, size_t> attr_done;
    static std::mutex attr_mu;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    {
      std::lock_guard<std::mutex> lock(attr_mu);
      if (attr_done[dev] < sm) {
        if ((e = cudaFuncSetAttribute(fp8_act_smem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(sm))) != cudaSuccess)
          return e;
        attr_done[dev] = sm;
      }
    }
    fp8_act_smem_kernel<<<M, kActSmemThreads, sm, s>>>(x, xq, fa, K, d->fwht_block != 0, status);
  } else {
    fp8_act_kernel<<<M, kActThreads, 0, s>>>(x, xq, fa, K, d->fwht_block != 0, status);
  }
  fp8_wexp_kernel<<<(N + 255) / 256, 256, 0, s>>>(scales, eb, fb, N, ng, status);
  if (d->packing == TQ_PACK_2BIT) {
    const long long n = static_cast<long long>(N) * (K / 16);
    const long long per_cta = static_cast<long long>(kDecThreads) * kF8WordsPerLane;
    decode_2b_f8_kernel<<<static_cast<unsigned>((n + per_cta - 1) / per_cta), kDecThreads, 0, s>>>(
        codes, scales, eb, wq, N, K, P, ng, G);
  } else {
    const long long n = static_cast<long long>(N) * ((K + 79) / 80);
    decode_b3_f8_kernel<<<static_cast<unsigned>((n + kDecThreads - 1) / kDecThreads), kDecThreads, 0, s>>>(
        codes, scales, eb, wq, N, K, P, ng, G);
  }
  e = cudaPeekAtLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap tm_x, tm_w;
  if (!make_tmap_2d(&tm_x, xq, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, M, static_cast<uint64_t>(K), BK8, BM,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tm_w, wq, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, N, static_cast<uint64_t>(K), BK8, BN,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if ((e = ensure_attr<true>()) != cudaSuccess) return e;
  const long long tiles = static_cast<long long>((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  const unsigned grid = static_cast<unsigned>(std::min<long long>(tiles, sm_count()));
  gemm_tc_kernel<true><<<grid, kThreads, kSmemBytes, s>>>(tm_x, tm_w, y, M, N, K, status, GroupedTiles{}, fa, fb);
  return cudaPeekAtLastError();
}

}  // namespace tq

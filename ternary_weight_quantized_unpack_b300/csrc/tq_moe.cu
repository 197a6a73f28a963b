// Routed MoE expert layer at decode time: top-k routing of 256 experts (8 active per token, router
// in full precision - the TurboQuant-MLX 1.58-bit Qwen3.6-35B-A3B page, section "为什么 1.58bit 没变成乱码", point 1), then the
// ternary SwiGLU experts, in three launches:
//  1. one CTA routes every token (warp per token), counts the assignments per expert, scans the
//     per-expert chunk counts and writes the chunk table: the (token, slot) assignments of each
//     expert in ascending order, cut into chunks of 1 token (a single token) or 2 tokens;
//  2. the gate/up projection as the decode GEMV over those chunks (blockIdx.z = chunk), each chunk
//     streaming its expert's packed codes once and transforming its tokens' inputs itself;
//  3. the down projection the same way on FWHT(silu(gate) * up); as each CTA stores its rows it
//     counts the finished slot of each of its tokens, and the CTA that finishes a token's last slot
//     adds the slots' rows in slot order, weighted by the gates (deterministic).
//
// At prefill sizes (tq_moe_gemm) the layer is a grouped GEMM instead: the assignments are sorted by
// expert, the tokens' transformed inputs gathered in that order (FP16), every expert's weights
// decoded to FP16 s * t, and one persistent tcgen05 launch per projection walks a tile list that
// covers each expert's rows of the sorted inputs against that expert's weights; silu(gate) * up and
// its transform, the down projection the same way, and the combine in slot order.
#include <float.h>

#include <algorithm>

#include "tq_internal.cuh"
#include "tq_kernels.cuh"
#include "tq_sm100.cuh"

namespace tq {
namespace {

constexpr int kMaxExperts = 256;
constexpr int kMaxTopk = 8;

// Token t, one warp: k rounds of a warp-wide argmax with the order (logit descending, expert index
// ascending); gate = softmax over the chosen logits, summed in slot order.  s_idx (optional): a
// shared-memory copy of the token's expert indices, at the same offsets as idx.
__device__ __forceinline__ void route_token(const float* __restrict__ logits, int t, int E, int topk,
                                            int* __restrict__ idx, float* __restrict__ gate, int lane,
                                            int* s_idx = nullptr) {
  float v[kMaxExperts / 32];
#pragma unroll
  for (int i = 0; i < kMaxExperts / 32; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? logits[static_cast<size_t>(t) * E + e] : -FLT_MAX;
  }
  unsigned taken = 0;
  float sel_v[kMaxTopk];
  int sel_i[kMaxTopk];
#pragma unroll
  for (int j = 0; j < kMaxTopk; ++j) {
    if (j >= topk) break;
    float bv = 0.f;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < kMaxExperts / 32; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && (bi == 0x7fffffff || v[i] > bv)) { bv = v[i]; bi = e; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      const bool take = (oi != 0x7fffffff) && (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi));
      if (take) { bv = ov; bi = oi; }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    sel_v[j] = bv;
    sel_i[j] = bi;
  }
  if (lane == 0) {
    const float m = sel_v[0];
    float ex[kMaxTopk];
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxTopk; ++j)
      if (j < topk) { ex[j] = expf(sel_v[j] - m); sum += ex[j]; }
#pragma unroll
    for (int j = 0; j < kMaxTopk; ++j)
      if (j < topk) {
        idx[static_cast<size_t>(t) * topk + j] = sel_i[j];
        gate[static_cast<size_t>(t) * topk + j] = ex[j] / sum;
        if (s_idx) s_idx[t * topk + j] = sel_i[j];
      }
  }
}

__global__ void route_kernel(const float* __restrict__ logits, int T, int E, int topk, int* __restrict__ idx,
                             float* __restrict__ gate) {
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t < T) route_token(logits, t, E, topk, idx, gate, threadIdx.x & 31);
}

constexpr int kPlanThreads = 1024;
constexpr int kPlanSmemAssign = 8192;  // assignments kept in shared memory (larger batches read global)

// Step 1 of the expert layer, one CTA: route every token, then the chunk table.  table[0] = number of
// chunks; chunk c is the record table[1 + c * (2 + CB)] = {expert, count, a_0 .. a_(CB-1)}, chunks
// in expert order and each expert's assignments in ascending order (unused slots repeat a_0; they
// are never read as data).  Also zeroes the combine counts.  Deterministic: counts are order-free
// and each assignment's place follows from the number of earlier assignments to its expert.
__global__ void __launch_bounds__(kPlanThreads) moe_plan_kernel(const float* __restrict__ logits, int T, int E,
                                                                int topk, int CB, int* __restrict__ idx,
                                                                float* __restrict__ gate, int* __restrict__ table,
                                                                int* __restrict__ count, int ncount) {
  extern __shared__ int s_assign[];  // min(A, kPlanSmemAssign) expert indices
  __shared__ int s_cnt[kMaxExperts], s_off[kMaxExperts], s_wsum[kMaxExperts / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, A = T * topk;
  const bool in_smem = A <= kPlanSmemAssign;
  for (int t = warp; t < T; t += kPlanThreads / 32)
    route_token(logits, t, E, topk, idx, gate, lane, in_smem ? s_assign : nullptr);
  for (int i = threadIdx.x; i < ncount; i += kPlanThreads) count[i] = 0;
  for (int e = threadIdx.x; e < kMaxExperts; e += kPlanThreads) s_cnt[e] = 0;
  __syncthreads();  // idx is complete (in shared memory, or global writes of this CTA read back below)
  for (int a = threadIdx.x; a < A; a += kPlanThreads) {
    const int e = in_smem ? s_assign[a] : __ldcg(idx + a);
    atomicAdd(&s_cnt[e], 1);
  }
  __syncthreads();
  // exclusive scan of the chunk counts over the experts: per warp, then across warps
  if (threadIdx.x < kMaxExperts) {
    const int e = threadIdx.x;
    const int nch = e < E ? (s_cnt[e] + CB - 1) / CB : 0;
    int incl = nch;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) s_wsum[warp] = incl;
    s_off[e] = incl - nch;
  }
  __syncthreads();
  if (threadIdx.x < kMaxExperts) {
    int base = 0;
    for (int w = 0; w < warp; ++w) base += s_wsum[w];
    s_off[threadIdx.x] += base;
    if (threadIdx.x == kMaxExperts - 1) {
      int total = 0;
      for (int w = 0; w < kMaxExperts / 32; ++w) total += s_wsum[w];
      table[0] = total;
    }
  }
  __syncthreads();
  if (in_smem) {
    // one thread per assignment: its rank among the earlier assignments to the same expert gives its
    // chunk and slot
    for (int a = threadIdx.x; a < A; a += kPlanThreads) {
      const int e = s_assign[a];
      int rank = 0;
      for (int b = 0; b < a; ++b) rank += s_assign[b] == e;
      const int ci = rank / CB, slot = rank - ci * CB;
      int* rec = table + 1 + static_cast<size_t>(s_off[e] + ci) * (2 + CB);
      rec[2 + slot] = a;
      if (slot == 0) {
        const int n = min(CB, s_cnt[e] - ci * CB);
        rec[0] = e;
        rec[1] = n;
        for (int j = n; j < CB; ++j) rec[2 + j] = a;
      }
    }
  } else if (threadIdx.x < E && s_cnt[threadIdx.x] > 0) {
    // large batches: one thread per expert places its assignments, in order
    const int e = threadIdx.x;
    int chunk = s_off[e], slot = 0;
    int* rec = table + 1 + static_cast<size_t>(chunk) * (2 + CB);
    for (int a = 0; a < A; ++a) {
      if (__ldcg(idx + a) != e) continue;
      rec[2 + slot] = a;
      if (++slot == CB) {
        rec[0] = e;
        rec[1] = CB;
        ++chunk;
        slot = 0;
        rec = table + 1 + static_cast<size_t>(chunk) * (2 + CB);
      }
    }
    if (slot > 0) {
      rec[0] = e;
      rec[1] = slot;
      for (int j = slot; j < CB; ++j) rec[2 + j] = rec[2];
    }
  }
}

// Tokens per chunk: one token never routes twice to an expert; larger batches share an expert's
// weights between 2 routed tokens per pass (the GEMV then transforms its inputs itself: no separate
// transform launch).
int chunk_batch(int T) { return T == 1 ? 1 : 2; }

// Row tiles of the down projection's chunked GEMV are at most H / 16 (one 16-row slab each).
size_t combine_count_ints(int T, int H) { return static_cast<size_t>(T) * ((H + 15) / 16); }

struct MoeWs {
  int* table;   // chunk records
  float* gu;    // gate / up outputs per assignment [T * topk][2F]
  float* ypart; // down outputs per assignment [T * topk][H]
  int* count;   // combine counts [T][row tiles]
  void* prep;   // prep output of the current stage (shared by both stages)
  size_t bytes;
};

// Sizes assume groups of 64 (more groups than 128, so enough for both).
MoeWs moe_ws_layout(void* base, int T, int topk, int H, int F) {
  MoeWs w{};
  char* p = static_cast<char*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) { char* q = p ? p + off : nullptr; off += align256(bytes); return q; };
  const int A = T * topk, CB = chunk_batch(T);
  w.table = reinterpret_cast<int*>(take((1 + static_cast<size_t>(A) * (2 + CB)) * 4));
  w.gu = reinterpret_cast<float*>(take(static_cast<size_t>(A) * 2 * F * 4));
  w.ypart = reinterpret_cast<float*>(take(static_cast<size_t>(A) * H * 4));
  w.count = reinterpret_cast<int*>(take(combine_count_ints(T, H) * 4));
  const tq_desc gu{2 * F, H, 64, TQ_PACK_B3, kFwhtBlock, 0}, dn{H, F, 64, TQ_PACK_B3, kFwhtBlock, 0};
  const size_t prep = std::max(gemv_chunks_workspace_bytes(&gu, CB, A), gemv_chunks_workspace_bytes(&dn, CB, A));
  w.prep = take(prep);
  w.bytes = prep == 0 ? 0 : off;
  return w;
}

// ---- expert layer at prefill sizes ----------------------------------------------------------------
constexpr int kSortThreads = 1024;
constexpr int kTileM = 128;  // token rows per GEMM tile (the grouped GEMM's M)
constexpr int kTileN = 256;  // weight rows per GEMM tile

// One CTA: counts per expert, sorted positions (an expert's assignments are contiguous; their order
// within the expert does not change any result, since every row's products are independent), and
// the two tile lists {A row, valid rows, B row, output column} for gate/up (NTgu column tiles per
// expert, Ngu weight rows per expert) and down (NTd, Nd).
__global__ void __launch_bounds__(kSortThreads) moe_sort_kernel(const int* __restrict__ idx, int A, int E, int* perm,
                                                                int* ipos, int4* tiles_gu, int* count_gu,
                                                                int NTgu, int Ngu, int4* tiles_d, int* count_d,
                                                                int NTd, int Nd) {
  __shared__ int s_cnt[kMaxExperts], s_off[kMaxExperts], s_moff[kMaxExperts], s_cur[kMaxExperts];
  __shared__ int s_w[2][kMaxExperts / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e = threadIdx.x; e < kMaxExperts; e += kSortThreads) s_cnt[e] = s_cur[e] = 0;
  __syncthreads();
  for (int a = threadIdx.x; a < A; a += kSortThreads) atomicAdd(&s_cnt[idx[a]], 1);
  __syncthreads();
  if (threadIdx.x < kMaxExperts) {  // exclusive scans of the counts and of the m-tiles per expert
    const int e = threadIdx.x;
    const int c = e < E ? s_cnt[e] : 0, mt = (c + kTileM - 1) / kTileM;
    int ic = c, im = mt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int vc = __shfl_up_sync(0xffffffffu, ic, o), vm = __shfl_up_sync(0xffffffffu, im, o);
      if (lane >= o) {
        ic += vc;
        im += vm;
      }
    }
    if (lane == 31) {
      s_w[0][warp] = ic;
      s_w[1][warp] = im;
    }
    s_off[e] = ic - c;
    s_moff[e] = im - mt;
  }
  __syncthreads();
  if (threadIdx.x < kMaxExperts) {
    int bc = 0, bm = 0;
    for (int w = 0; w < warp; ++w) {
      bc += s_w[0][w];
      bm += s_w[1][w];
    }
    s_off[threadIdx.x] += bc;
    s_moff[threadIdx.x] += bm;
    if (threadIdx.x == kMaxExperts - 1) {
      int tm = 0;
      for (int w = 0; w < kMaxExperts / 32; ++w) tm += s_w[1][w];
      *count_gu = tm * NTgu;
      *count_d = tm * NTd;
    }
  }
  __syncthreads();
  for (int a = threadIdx.x; a < A; a += kSortThreads) {
    const int e = idx[a];
    const int pos = s_off[e] + atomicAdd(&s_cur[e], 1);
    perm[pos] = a;
    ipos[a] = pos;
  }
  if (threadIdx.x < E) {
    const int e = threadIdx.x, c = s_cnt[e];
    for (int i = 0; i * kTileM < c; ++i) {
      const int m0 = s_off[e] + i * kTileM, rows = min(kTileM, c - i * kTileM), mi = s_moff[e] + i;
      for (int j = 0; j < NTgu; ++j) tiles_gu[mi * NTgu + j] = make_int4(m0, rows, e * Ngu + j * kTileN, j * kTileN);
      for (int j = 0; j < NTd; ++j) tiles_d[mi * NTd + j] = make_int4(m0, rows, e * Nd + j * kTileN, j * kTileN);
    }
  }
}

// Sorted row r: the FP16 block transform of x row perm[r] / topk.  One warp per (row, 128-block).
__global__ void moe_gather_fwht_kernel(const uint16_t* __restrict__ x, const int* __restrict__ perm, int topk, int A,
                                       int K, int apply, uint16_t* __restrict__ out, int* status) {
  const long long wid = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int nb = K / kFwhtBlock;
  if (wid >= static_cast<long long>(A) * nb) return;
  const int r = static_cast<int>(wid / nb), blk = static_cast<int>(wid % nb), lane = threadIdx.x & 31;
  const int src = perm[r] / topk;
  const uint2 raw = __ldg(reinterpret_cast<const uint2*>(x + static_cast<size_t>(src) * K + blk * kFwhtBlock + 4 * lane));
  float v[4] = {bf16_bits_to_float(static_cast<uint16_t>(raw.x & 0xffffu)),
                bf16_bits_to_float(static_cast<uint16_t>(raw.x >> 16)),
                bf16_bits_to_float(static_cast<uint16_t>(raw.y & 0xffffu)),
                bf16_bits_to_float(static_cast<uint16_t>(raw.y >> 16))};
  if (apply) {
    fwht128_warp(v);
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] *= 0.08838834764831845f;
  }
  __half h[4];
  bool overflow = false;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    h[j] = __float2half_rn(v[j]);
    overflow |= __hisinf(h[j]) != 0;
  }
  if (overflow) record_error(status, TQ_ERR_RANGE);
  uint2 o;
  o.x = static_cast<uint32_t>(__half_as_ushort(h[0])) | (static_cast<uint32_t>(__half_as_ushort(h[1])) << 16);
  o.y = static_cast<uint32_t>(__half_as_ushort(h[2])) | (static_cast<uint32_t>(__half_as_ushort(h[3])) << 16);
  *reinterpret_cast<uint2*>(out + static_cast<size_t>(r) * K + blk * kFwhtBlock + 4 * lane) = o;
}

// Sorted row r: h = silu(gate) * up from the gate/up output (fp32 [A][2F]); optionally h to h_out row
// perm[r] (assignment order); then its FP16 block transform.  One warp per (row, 128-block).
__global__ void moe_swiglu_fwht_kernel(const float* __restrict__ gu, const int* __restrict__ perm, int A, int F,
                                       int apply, float* __restrict__ h_out, uint16_t* __restrict__ out,
                                       int* status) {
  const long long wid = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int nb = F / kFwhtBlock;
  if (wid >= static_cast<long long>(A) * nb) return;
  const int r = static_cast<int>(wid / nb), blk = static_cast<int>(wid % nb), lane = threadIdx.x & 31;
  const int k0 = blk * kFwhtBlock + 4 * lane;
  const float4 g = *reinterpret_cast<const float4*>(gu + static_cast<size_t>(r) * 2 * F + k0);
  const float4 u = *reinterpret_cast<const float4*>(gu + static_cast<size_t>(r) * 2 * F + F + k0);
  float v[4] = {g.x / (1.f + expf(-g.x)) * u.x, g.y / (1.f + expf(-g.y)) * u.y, g.z / (1.f + expf(-g.z)) * u.z,
                g.w / (1.f + expf(-g.w)) * u.w};
  if (h_out)
    *reinterpret_cast<float4*>(h_out + static_cast<size_t>(perm[r]) * F + k0) = make_float4(v[0], v[1], v[2], v[3]);
  if (apply) {
    fwht128_warp(v);
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] *= 0.08838834764831845f;
  }
  __half h[4];
  bool overflow = false;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    h[j] = __float2half_rn(v[j]);
    overflow |= __hisinf(h[j]) != 0;
  }
  if (overflow) record_error(status, TQ_ERR_RANGE);
  uint2 o;
  o.x = static_cast<uint32_t>(__half_as_ushort(h[0])) | (static_cast<uint32_t>(__half_as_ushort(h[1])) << 16);
  o.y = static_cast<uint32_t>(__half_as_ushort(h[2])) | (static_cast<uint32_t>(__half_as_ushort(h[3])) << 16);
  *reinterpret_cast<uint2*>(out + static_cast<size_t>(r) * F + k0) = o;
}

// y[t][n] = sum_j gate[t][j] * yp[ipos[t * topk + j]][n], slots in order.
__global__ void moe_combine_kernel(const float* __restrict__ yp, const int* __restrict__ ipos,
                                   const float* __restrict__ gate, int T, int H, int topk, float* __restrict__ y) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<long long>(T) * (H / 4)) return;
  const int t = static_cast<int>(i / (H / 4)), n = 4 * static_cast<int>(i % (H / 4));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < topk; ++j) {
    const float gj = gate[static_cast<size_t>(t) * topk + j];
    const float4 v = *reinterpret_cast<const float4*>(yp + static_cast<size_t>(ipos[t * topk + j]) * H + n);
    acc.x = fmaf(gj, v.x, acc.x);
    acc.y = fmaf(gj, v.y, acc.y);
    acc.z = fmaf(gj, v.z, acc.z);
    acc.w = fmaf(gj, v.w, acc.w);
  }
  *reinterpret_cast<float4*>(y + static_cast<size_t>(t) * H + n) = acc;
}

// Workspace of the prefill expert layer.
struct MoeGemmWs {
  int *perm, *ipos, *tiles_gu, *tiles_d, *counts;
  uint16_t *xs, *wgu, *hs, *wd;
  float *gu, *yp;
  int max_tiles_gu, max_tiles_d;
  size_t bytes;
};

MoeGemmWs moe_gemm_ws_layout(void* base, int T, int E, int topk, int H, int F) {
  MoeGemmWs w{};
  char* p = static_cast<char*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) { char* q = p ? p + off : nullptr; off += align256(bytes); return q; };
  const int A = T * topk;
  const int mt = (A + kTileM - 1) / kTileM + E;  // m-tiles: at most one partial tile per expert
  w.max_tiles_gu = mt * (2 * F / kTileN);
  w.max_tiles_d = mt * (H / kTileN);
  w.perm = reinterpret_cast<int*>(take(static_cast<size_t>(A) * 4));
  w.ipos = reinterpret_cast<int*>(take(static_cast<size_t>(A) * 4));
  w.tiles_gu = reinterpret_cast<int*>(take(static_cast<size_t>(w.max_tiles_gu) * 16));
  w.tiles_d = reinterpret_cast<int*>(take(static_cast<size_t>(w.max_tiles_d) * 16));
  w.counts = reinterpret_cast<int*>(take(2 * 4));
  w.xs = reinterpret_cast<uint16_t*>(take(static_cast<size_t>(A) * H * 2));
  w.wgu = reinterpret_cast<uint16_t*>(take(static_cast<size_t>(E) * 2 * F * H * 2));
  w.gu = reinterpret_cast<float*>(take(static_cast<size_t>(A) * 2 * F * 4));
  w.hs = reinterpret_cast<uint16_t*>(take(static_cast<size_t>(A) * F * 2));
  w.wd = reinterpret_cast<uint16_t*>(take(static_cast<size_t>(E) * H * F * 2));
  w.yp = reinterpret_cast<float*>(take(static_cast<size_t>(A) * H * 4));
  w.bytes = off;
  return w;
}

cudaError_t launch_route(const float* logits, int T, int E, int topk, int* idx, float* gate, cudaStream_t s) {
  const unsigned blocks = static_cast<unsigned>((T + 7) / 8);
  route_kernel<<<blocks, 256, 0, s>>>(logits, T, E, topk, idx, gate);
  return cudaPeekAtLastError();
}

}  // namespace
}  // namespace tq

using namespace tq;

extern "C" tq_status tq_moe_route(const float* logits, int T, int E, int topk, int32_t* idx, float* gate,
                                  void* stream) {
  if (!logits || !idx || !gate || T < 1 || E < 1 || topk < 1) return TQ_ERR_INVALID_ARG;
  if (E > kMaxExperts || topk > kMaxTopk || topk > E) return TQ_ERR_UNSUPPORTED;
  if (!aligned(logits, 4) || !aligned(idx, 4) || !aligned(gate, 4)) return TQ_ERR_MISALIGNED;
  const cudaError_t e = launch_route(logits, T, E, topk, idx, gate, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return TQ_OK;
}

extern "C" size_t tq_moe_workspace_bytes(int T, int E, int topk, int H, int F) {
  if (T < 1 || E < 1 || E > kMaxExperts || topk < 1 || topk > kMaxTopk || topk > E || H < 1 || F < 1) return 0;
  if (H % kFwhtBlock != 0 || F % kFwhtBlock != 0) return 0;
  return moe_ws_layout(nullptr, T, topk, H, F).bytes;
}

extern "C" tq_status tq_moe_gemv(const tq_desc* gate_up, const tq_desc* down, int E, int topk,
                                 const uint32_t* gu_codes, const uint16_t* gu_scales, const uint32_t* d_codes,
                                 const uint16_t* d_scales, const float* router_logits, const uint16_t* x, int T,
                                 int32_t* topk_idx, float* topk_gate, float* h_out, float* y, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  tq_status st;
  if ((st = check_linear_desc(gate_up)) != TQ_OK) return st;
  if ((st = check_linear_desc(down)) != TQ_OK) return st;
  const int H = gate_up->K, F = down->K;
  if (gate_up->N != 2 * F || down->N != H) return TQ_ERR_INVALID_ARG;
  if (gate_up->packing != down->packing || gate_up->group != down->group || gate_up->fwht_block != down->fwht_block)
    return TQ_ERR_UNSUPPORTED;
  if (T < 1 || E < 1 || topk < 1) return TQ_ERR_INVALID_ARG;
  if (E > kMaxExperts || topk > kMaxTopk || topk > E) return TQ_ERR_UNSUPPORTED;
  if (!gu_codes || !gu_scales || !d_codes || !d_scales || !router_logits || !x || !topk_idx || !topk_gate || !y ||
      !workspace)
    return TQ_ERR_INVALID_ARG;
  if (!aligned(gu_codes, 16) || !aligned(gu_scales, 16) || !aligned(d_codes, 16) || !aligned(d_scales, 16) ||
      !aligned(x, 16) || !aligned(y, 16) || !aligned(router_logits, 4) || !aligned(topk_idx, 4) ||
      !aligned(topk_gate, 4) || (h_out && !aligned(h_out, 16)) || !aligned(workspace, 256))
    return TQ_ERR_MISALIGNED;
  if (workspace_bytes < tq_moe_workspace_bytes(T, E, topk, H, F)) return TQ_ERR_WORKSPACE;
  if (!status_ptr()) return TQ_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MoeWs w = moe_ws_layout(workspace, T, topk, H, F);
  const int G = gate_up->group, A = T * topk, CB = chunk_batch(T);
  const int tiles = gemv_chunks_row_tiles(down, CB);
  if (tiles < 1 || static_cast<size_t>(T) * tiles > combine_count_ints(T, H)) return TQ_ERR_UNSUPPORTED;
  cudaError_t e;
  const int A_smem = std::min(A, kPlanSmemAssign);
  moe_plan_kernel<<<1, kPlanThreads, static_cast<size_t>(A_smem) * 4, s>>>(router_logits, T, E, topk, CB, topk_idx,
                                                                           topk_gate, w.table, w.count, T * tiles);
  if ((e = cudaPeekAtLastError()) != cudaSuccess) return cuda_fail(e);
  // gate / up: chunk slot b holds assignment a, fed with x row a / topk; output row a of gu
  e = launch_gemv_chunks(gate_up, gu_codes, gu_scales, static_cast<size_t>(2 * F) * pitch_words(H, gate_up->packing),
                         static_cast<size_t>(2 * F) * (H / G), 1, x, nullptr, nullptr, topk, w.table, CB, A, w.gu,
                         w.prep, s);
  if (e != cudaSuccess) return cuda_fail(e);
  // down: fed with FWHT(silu(gate) * up) of assignment a; output row a of ypart; the combine into y
  // is done by the CTA that finishes a token's last slot
  const ChunkCombine cmb{w.count, topk_gate, y};
  e = launch_gemv_chunks(down, d_codes, d_scales, static_cast<size_t>(H) * pitch_words(F, down->packing),
                         static_cast<size_t>(H) * (F / G), 2, nullptr, w.gu, h_out, topk, w.table, CB, A, w.ypart,
                         w.prep, s, &cmb);
  if (e != cudaSuccess) return cuda_fail(e);
  return TQ_OK;
}

extern "C" size_t tq_moe_gemm_workspace_bytes(int T, int E, int topk, int H, int F) {
  if (T < 1 || E < 1 || E > kMaxExperts || topk < 1 || topk > kMaxTopk || topk > E || H < 1 || F < 1) return 0;
  if (H % kTileN != 0 || (2 * F) % kTileN != 0 || F % kFwhtBlock != 0) return 0;
  if (static_cast<long long>(T) * topk >= (1ll << 24)) return 0;
  return moe_gemm_ws_layout(nullptr, T, E, topk, H, F).bytes;
}

extern "C" tq_status tq_moe_gemm(const tq_desc* gate_up, const tq_desc* down, int E, int topk,
                                 const uint32_t* gu_codes, const uint16_t* gu_scales, const uint32_t* d_codes,
                                 const uint16_t* d_scales, const float* router_logits, const uint16_t* x, int T,
                                 int32_t* topk_idx, float* topk_gate, float* h_out, float* y, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  tq_status st;
  if ((st = check_linear_desc(gate_up)) != TQ_OK) return st;
  if ((st = check_linear_desc(down)) != TQ_OK) return st;
  const int H = gate_up->K, F = down->K;
  if (gate_up->N != 2 * F || down->N != H) return TQ_ERR_INVALID_ARG;
  if (gate_up->packing != down->packing || gate_up->group != down->group || gate_up->fwht_block != down->fwht_block)
    return TQ_ERR_UNSUPPORTED;
  if (T < 1 || E < 1 || topk < 1) return TQ_ERR_INVALID_ARG;
  if (E > kMaxExperts || topk > kMaxTopk || topk > E) return TQ_ERR_UNSUPPORTED;
  if (H % kTileN != 0 || (2 * F) % kTileN != 0) return TQ_ERR_UNSUPPORTED;
  if (!gu_codes || !gu_scales || !d_codes || !d_scales || !router_logits || !x || !topk_idx || !topk_gate || !y ||
      !workspace)
    return TQ_ERR_INVALID_ARG;
  if (!aligned(gu_codes, 16) || !aligned(gu_scales, 16) || !aligned(d_codes, 16) || !aligned(d_scales, 16) ||
      !aligned(x, 16) || !aligned(y, 16) || !aligned(router_logits, 4) || !aligned(topk_idx, 4) ||
      !aligned(topk_gate, 4) || (h_out && !aligned(h_out, 16)) || !aligned(workspace, 256))
    return TQ_ERR_MISALIGNED;
  const size_t need = tq_moe_gemm_workspace_bytes(T, E, topk, H, F);
  if (need == 0) return TQ_ERR_UNSUPPORTED;
  if (workspace_bytes < need) return TQ_ERR_WORKSPACE;
  int* status = status_ptr();
  if (!status) return TQ_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MoeGemmWs w = moe_gemm_ws_layout(workspace, T, E, topk, H, F);
  const int A = T * topk, apply = gate_up->fwht_block != 0;
  cudaError_t e;
  if ((e = launch_route(router_logits, T, E, topk, topk_idx, topk_gate, s)) != cudaSuccess) return cuda_fail(e);
  moe_sort_kernel<<<1, kSortThreads, 0, s>>>(topk_idx, A, E, w.perm, w.ipos, reinterpret_cast<int4*>(w.tiles_gu),
                                             w.counts, 2 * F / kTileN, 2 * F, reinterpret_cast<int4*>(w.tiles_d),
                                             w.counts + 1, H / kTileN, H);
  if ((e = cudaPeekAtLastError()) != cudaSuccess) return cuda_fail(e);
  {
    const long long warps = static_cast<long long>(A) * (H / kFwhtBlock);
    moe_gather_fwht_kernel<<<static_cast<unsigned>((warps + 7) / 8), 256, 0, s>>>(x, w.perm, topk, A, H, apply, w.xs,
                                                                                   status);
    if ((e = cudaPeekAtLastError()) != cudaSuccess) return cuda_fail(e);
  }
  // every expert's gate/up rows as one stacked matrix [E * 2F][H], decoded to FP16
  const tq_desc gu_all{E * 2 * F, H, gate_up->group, gate_up->packing, gate_up->fwht_block, 0};
  if ((e = launch_decode(&gu_all, gu_codes, gu_scales, w.wgu, s)) != cudaSuccess) return cuda_fail(e);
  if ((e = launch_gemm_grouped(w.xs, A, w.wgu, E * 2 * F, H, w.tiles_gu, w.counts, w.max_tiles_gu, w.gu, 2 * F, s)) !=
      cudaSuccess)
    return cuda_fail(e);
  {
    const long long warps = static_cast<long long>(A) * (F / kFwhtBlock);
    moe_swiglu_fwht_kernel<<<static_cast<unsigned>((warps + 7) / 8), 256, 0, s>>>(w.gu, w.perm, A, F, apply, h_out,
                                                                                   w.hs, status);
    if ((e = cudaPeekAtLastError()) != cudaSuccess) return cuda_fail(e);
  }
  const tq_desc d_all{E * H, F, down->group, down->packing, down->fwht_block, 0};
  if ((e = launch_decode(&d_all, d_codes, d_scales, w.wd, s)) != cudaSuccess) return cuda_fail(e);
  if ((e = launch_gemm_grouped(w.hs, A, w.wd, E * H, F, w.tiles_d, w.counts + 1, w.max_tiles_d, w.yp, H, s)) !=
      cudaSuccess)
    return cuda_fail(e);
  {
    const long long n = static_cast<long long>(T) * (H / 4);
    moe_combine_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(w.yp, w.ipos, topk_gate, T, H, topk, y);
    if ((e = cudaPeekAtLastError()) != cudaSuccess) return cuda_fail(e);
  }
  return TQ_OK;
}

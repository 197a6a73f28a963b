// Routed MoE expert layer at decode time: top-k routing of 256 experts (8 active per token, router
// in full precision - tantan.ink/?p=490, section "为什么 1.58bit 没变成乱码", point 1), then the
// ternary SwiGLU experts, each reading its packed codes once for all tokens routed to it.
#include <float.h>

#include "tq_internal.cuh"
#include "tq_kernels.cuh"
#include "tq_simple.cuh"

namespace tq {
namespace {

constexpr int kMaxExperts = 256;
constexpr int kMaxTopk = 8;

// One warp per token: k rounds of a warp-wide argmax with the order (logit descending, expert
// index ascending); gate = softmax over the chosen logits, summed in slot order.
__global__ void route_kernel(const float* __restrict__ logits, int T, int E, int topk, int* __restrict__ idx,
                             float* __restrict__ gate) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + warp;
  if (t >= T) return;
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
      }
  }
}

// One block: per-expert counts, offsets and the (token, slot) assignment list grouped by expert,
// each expert's entries in ascending (token, slot) order - deterministic.
__global__ void lists_kernel(const int* __restrict__ idx, int n_assign, int E, int* __restrict__ counts,
                             int* __restrict__ offsets, int* __restrict__ list) {
  __shared__ int s_off[kMaxExperts + 1];
  const int e = threadIdx.x;
  int c = 0;
  if (e < E)
    for (int a = 0; a < n_assign; ++a) c += idx[a] == e;
  if (e < kMaxExperts) s_off[e + 1] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    s_off[0] = 0;
    for (int i = 0; i < E; ++i) s_off[i + 1] += s_off[i];
  }
  __syncthreads();
  if (e < E) {
    counts[e] = c;
    offsets[e] = s_off[e];
    int pos = s_off[e];
    for (int a = 0; a < n_assign && pos < s_off[e] + c; ++a)
      if (idx[a] == e) list[pos++] = a;
  }
  if (threadIdx.x == 0) offsets[E] = s_off[E];
}

__device__ __forceinline__ float silu(float z) { return z / (1.f + expf(-z)); }

// gate/up GEMV + SwiGLU: block (expert, 8 rows), warp per row r; for every assignment routed to
// the expert: h = silu(Wg[r] x~) * (Wu[r] x~).
template <int PACKING>
__global__ void __launch_bounds__(256) gate_up_kernel(const uint32_t* __restrict__ gu_codes,
                                                      const uint16_t* __restrict__ gu_scales,
                                                      const float* __restrict__ xt, const int* __restrict__ counts,
                                                      const int* __restrict__ offsets, const int* __restrict__ list,
                                                      int H, int F, int G, int topk, float* __restrict__ h,
                                                      float* __restrict__ h_out) {
  const int e = blockIdx.x;
  const int cnt = counts[e];
  if (cnt == 0) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.y * 8 + warp;
  if (r >= F) return;
  const int P = pitch_words(H, PACKING), ng = groups_of(H, G);
  const uint32_t* wg = gu_codes + (static_cast<size_t>(e) * 2 * F + r) * P;
  const uint32_t* wu = gu_codes + (static_cast<size_t>(e) * 2 * F + F + r) * P;
  const uint16_t* sg = gu_scales + (static_cast<size_t>(e) * 2 * F + r) * ng;
  const uint16_t* su = gu_scales + (static_cast<size_t>(e) * 2 * F + F + r) * ng;
  const int off = offsets[e];
  for (int i = 0; i < cnt; ++i) {
    const int a = list[off + i];
    const float* xa = xt + static_cast<size_t>(a / topk) * H;
    float ag[1] = {0.f}, au[1] = {0.f};
    row_dot_accumulate<PACKING, 1>(wg, sg, xa, H, H, G, 1, lane, ag);
    row_dot_accumulate<PACKING, 1>(wu, su, xa, H, H, G, 1, lane, au);
    const float g = warp_sum(ag[0]), u = warp_sum(au[0]);
    if (lane == 0) {
      const float hv = silu(g) * u;
      h[static_cast<size_t>(a) * F + r] = hv;
      if (h_out) h_out[static_cast<size_t>(a) * F + r] = hv;
    }
  }
}

template <int PACKING>
__global__ void __launch_bounds__(256) down_kernel(const uint32_t* __restrict__ d_codes,
                                                   const uint16_t* __restrict__ d_scales,
                                                   const float* __restrict__ ht, const int* __restrict__ counts,
                                                   const int* __restrict__ offsets, const int* __restrict__ list,
                                                   int H, int F, int G, float* __restrict__ ypart) {
  const int e = blockIdx.x;
  const int cnt = counts[e];
  if (cnt == 0) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.y * 8 + warp;
  if (r >= H) return;
  const int P = pitch_words(F, PACKING), ng = groups_of(F, G);
  const uint32_t* wd = d_codes + (static_cast<size_t>(e) * H + r) * P;
  const uint16_t* sd = d_scales + (static_cast<size_t>(e) * H + r) * ng;
  const int off = offsets[e];
  for (int i = 0; i < cnt; ++i) {
    const int a = list[off + i];
    float acc[1] = {0.f};
    row_dot_accumulate<PACKING, 1>(wd, sd, ht + static_cast<size_t>(a) * F, F, F, G, 1, lane, acc);
    const float v = warp_sum(acc[0]);
    if (lane == 0) ypart[static_cast<size_t>(a) * H + r] = v;
  }
}

// y[t][r] = sum_j gate[t][j] * ypart[t*topk + j][r], summed in slot order j = 0..topk-1.
__global__ void combine_kernel(const float* __restrict__ ypart, const float* __restrict__ gate, int T, int H,
                               int topk, float* __restrict__ y) {
  const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<size_t>(T) * H) return;
  const int t = static_cast<int>(i / H), r = static_cast<int>(i % H);
  float acc = 0.f;
  for (int j = 0; j < topk; ++j)
    acc = fmaf(gate[static_cast<size_t>(t) * topk + j], ypart[(static_cast<size_t>(t) * topk + j) * H + r], acc);
  y[i] = acc;
}

struct MoeWs {
  float* xt;
  int* counts;
  int* offsets;
  int* list;
  float* h;
  float* ht;
  float* ypart;
  size_t bytes;
};

MoeWs moe_ws_layout(void* base, int T, int E, int topk, int H, int F) {
  MoeWs w{};
  char* p = static_cast<char*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) { char* q = p ? p + off : nullptr; off += align256(bytes); return q; };
  const size_t A = static_cast<size_t>(T) * topk;
  w.xt = reinterpret_cast<float*>(take(static_cast<size_t>(T) * H * 4));
  w.counts = reinterpret_cast<int*>(take(static_cast<size_t>(E) * 4));
  w.offsets = reinterpret_cast<int*>(take(static_cast<size_t>(E + 1) * 4));
  w.list = reinterpret_cast<int*>(take(A * 4));
  w.h = reinterpret_cast<float*>(take(A * F * 4));
  w.ht = reinterpret_cast<float*>(take(A * F * 4));
  w.ypart = reinterpret_cast<float*>(take(A * H * 4));
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
  return moe_ws_layout(nullptr, T, E, topk, H, F).bytes;
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
  MoeWs w = moe_ws_layout(workspace, T, E, topk, H, F);
  const int G = gate_up->group;
  const int apply = gate_up->fwht_block != 0;
  const int n_assign = T * topk;
  if (launch_route(router_logits, T, E, topk, topk_idx, topk_gate, s) != cudaSuccess) goto fail;
  lists_kernel<<<1, kMaxExperts, 0, s>>>(topk_idx, n_assign, E, w.counts, w.offsets, w.list);
  if (cudaPeekAtLastError() != cudaSuccess) goto fail;
  if (launch_fwht_bf16(x, w.xt, 0, T, H, apply, s) != cudaSuccess) goto fail;
  {
    dim3 grid(E, (F + 7) / 8);
    if (gate_up->packing == TQ_PACK_B3)
      gate_up_kernel<TQ_PACK_B3><<<grid, 256, 0, s>>>(gu_codes, gu_scales, w.xt, w.counts, w.offsets, w.list, H, F, G,
                                                      topk, w.h, h_out);
    else
      gate_up_kernel<TQ_PACK_2BIT><<<grid, 256, 0, s>>>(gu_codes, gu_scales, w.xt, w.counts, w.offsets, w.list, H, F,
                                                        G, topk, w.h, h_out);
    if (cudaPeekAtLastError() != cudaSuccess) goto fail;
  }
  if (apply) {
    if (launch_fwht_f32(w.h, w.ht, n_assign, F, s) != cudaSuccess) goto fail;
  } else if (cudaMemcpyAsync(w.ht, w.h, static_cast<size_t>(n_assign) * F * 4, cudaMemcpyDeviceToDevice, s) !=
             cudaSuccess) {
    goto fail;
  }
  {
    dim3 grid(E, (H + 7) / 8);
    if (down->packing == TQ_PACK_B3)
      down_kernel<TQ_PACK_B3><<<grid, 256, 0, s>>>(d_codes, d_scales, w.ht, w.counts, w.offsets, w.list, H, F, G,
                                                   w.ypart);
    else
      down_kernel<TQ_PACK_2BIT><<<grid, 256, 0, s>>>(d_codes, d_scales, w.ht, w.counts, w.offsets, w.list, H, F, G,
                                                     w.ypart);
    if (cudaPeekAtLastError() != cudaSuccess) goto fail;
  }
  {
    const size_t n = static_cast<size_t>(T) * H;
    combine_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(w.ypart, topk_gate, T, H, topk, y);
    if (cudaPeekAtLastError() != cudaSuccess) goto fail;
  }
  return TQ_OK;
fail:
  return cuda_fail(cudaPeekAtLastError());
}

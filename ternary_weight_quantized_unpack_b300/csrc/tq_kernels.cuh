// Internal launchers shared between libtq translation units (not part of the ABI).
#pragma once

#include "tq_internal.cuh"

namespace tq {

// Block FWHT (block 128) of bf16 rows; apply = 0 copies (bf16 -> fp32/fp16) without transforming.
cudaError_t launch_fwht_bf16(const uint16_t* x, void* out, int out_fp16, int rows, int K, int apply,
                             cudaStream_t s);
// Block FWHT (block 128) of fp32 rows into fp32.
cudaError_t launch_fwht_f32(const float* x, float* out, int rows, int K, cudaStream_t s);

// Decode GEMV (activation prep kernel + mma.sync decode kernel); workspace from gemv_workspace_bytes.
size_t gemv_workspace_bytes(const tq_desc* d, int batch);
cudaError_t launch_gemv(const tq_desc* d, const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                        int batch, float* y, void* ws, cudaStream_t s);

// Kernels one launch_gemv call launches for this shape on the current device (-1: CUDA error).
int gemv_kernel_count(const tq_desc* d, int batch);

// Decode GEMV over chunks of routed tokens (expert layer).  chunks[0] = number of records (at most
// max_chunks); record c = chunks[1 + c * (2 + B)] = {expert, count, rows[B]}.  For slot b < count the
// input is, mode 1: row rows[b] / topk of x (bf16, K wide); mode 2: silu(gate) * up of row rows[b] of
// gu (float, gate then up, 2K wide), copied to h_out (K wide) when h_out is not null.  Output row
// rows[b] of y (N wide) receives the expert's product.  Codes / scales of expert e start
// e * codes_estride / e * scales_estride elements in.
// combine (may be null): after a CTA has stored its output rows it counts, per token t = rows[b] /
// topk, one more finished slot in combine->count[t * row_tiles + row tile]; the CTA that completes a
// token's topk slots writes combine->y[t][rows of the tile] = sum_j gate[t][j] * y[t * topk + j][rows]
// (slots in order j = 0..topk-1, so the sum does not depend on which CTA forms it) and sets the count
// back to 0.  The counts must be zero before the launch; row_tiles_out receives the tile count.
struct ChunkCombine {
  int* count;
  const float* gate;
  float* y;
};
size_t gemv_chunks_workspace_bytes(const tq_desc* d, int B, int max_chunks);
// Row tiles (CTAs along N) of the chunked GEMV for this shape and batch, or -1.
int gemv_chunks_row_tiles(const tq_desc* d, int B);
cudaError_t launch_gemv_chunks(const tq_desc* d, const uint32_t* codes, const uint16_t* scales, size_t codes_estride,
                               size_t scales_estride, int mode, const uint16_t* x, const float* gu, float* h_out,
                               int topk, const int* chunks, int B, int max_chunks, float* y, void* ws,
                               cudaStream_t s, const ChunkCombine* combine = nullptr);

// Prefill GEMM (weights decoded to FP16 once per call, tcgen05 tensor cores); workspace from
// gemm_workspace_bytes.
size_t gemm_workspace_bytes(const tq_desc* d, int M);
cudaError_t launch_gemm(const tq_desc* d, const uint32_t* codes, const uint16_t* scales, const uint16_t* x, int M,
                        uint16_t* y, void* ws, cudaStream_t s);

// Grouped prefill GEMM (expert layer): one persistent tcgen05 launch over a device-written tile list;
// tiles[4 i .. 4 i + 3] = {A row, valid rows, B row, output column}, *count tiles (at most max_tiles).
// xa: FP16 [a_rows][K]; wa: FP16 [w_rows][K]; y: fp32, row r at y + r * ldy.
cudaError_t launch_gemm_grouped(const uint16_t* xa, int a_rows, const uint16_t* wa, int w_rows, int K, const int* tiles,
                                const int* count, int max_tiles, float* y, int ldy, cudaStream_t s);
// Prefill GEMM with FP8 E4M3 operands (per-row power-of-two factors; tcgen05 kind::f8f6f4).
size_t gemm_fp8_workspace_bytes(const tq_desc* d, int M);
cudaError_t launch_gemm_fp8(const tq_desc* d, const uint32_t* codes, const uint16_t* scales, const uint16_t* x, int M,
                            uint16_t* y, void* ws, cudaStream_t s);
// Weights of one matrix (or of stacked experts viewed as one matrix) decoded to FP16 s * t [N][K].
cudaError_t launch_decode(const tq_desc* d, const uint32_t* codes, const uint16_t* scales, uint16_t* w, cudaStream_t s);

// Host-side descriptor checks shared by the contraction entry points.
tq_status check_linear_desc(const tq_desc* d);
// check_linear_desc, also accepting 3-bit codes (the decode GEMV takes them)
tq_status check_gemv_desc(const tq_desc* d);

// Round up to a multiple of 256 bytes (workspace sub-buffer alignment).
inline size_t align256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

}  // namespace tq

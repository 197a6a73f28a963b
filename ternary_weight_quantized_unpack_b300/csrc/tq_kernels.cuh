// Internal launchers shared between libtq translation units (not part of the ABI).
#pragma once

#include "tq_internal.cuh"

namespace tq {

// Block FWHT (block 128) of bf16 rows; apply = 0 copies (bf16 -> fp32/fp16) without transforming.
cudaError_t launch_fwht_bf16(const uint16_t* x, void* out, int out_fp16, int rows, int K, int apply,
                             cudaStream_t s);
// Block FWHT (block 128) of fp32 rows into fp32.
cudaError_t launch_fwht_f32(const float* x, float* out, int rows, int K, cudaStream_t s);

// Tensor-core decode GEMV (preparation kernel + tcgen05 kernel); workspace from gemv_tc_workspace_bytes.
size_t gemv_tc_workspace_bytes(const tq_desc* d, int batch);
// Largest K the decode GEMV handles: 64 stages of 32 words per row (40960 base-3, 32768 2-bit).
inline int gemv_tc_max_k(int packing) { return 64 * (packing == TQ_PACK_B3 ? 640 : 512); }
cudaError_t launch_gemv_tc(const tq_desc* d, const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                           int batch, float* y, void* ws, cudaStream_t s);

// Host-side descriptor checks shared by the contraction entry points.
tq_status check_linear_desc(const tq_desc* d);

// Round up to a multiple of 256 bytes (workspace sub-buffer alignment).
inline size_t align256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

}  // namespace tq

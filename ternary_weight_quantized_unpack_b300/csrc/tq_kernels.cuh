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

// Prefill GEMM (weights decoded to FP16 once per call, tcgen05 tensor cores); workspace from
// gemm_workspace_bytes.
size_t gemm_workspace_bytes(const tq_desc* d, int M);
cudaError_t launch_gemm(const tq_desc* d, const uint32_t* codes, const uint16_t* scales, const uint16_t* x, int M,
                        uint16_t* y, void* ws, cudaStream_t s);

// Host-side descriptor checks shared by the contraction entry points.
tq_status check_linear_desc(const tq_desc* d);

// Round up to a multiple of 256 bytes (workspace sub-buffer alignment).
inline size_t align256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

}  // namespace tq

/*
 * tq.h - C ABI of libtq, the ternary-weight linear layer for NVIDIA B300 (sm_103a).
 *
 * The method (sources cited by page title and section):
 *   - Weights are ternary t in {-1, 0, +1} times a scale; one FP16 scale per group of weights
 *     ("27B 大模型塞进 5.9GB：三值量化，凭什么「不崩」？", section 一 and section 二 ②:
 *     128 weights per group; the TurboQuant-MLX 1.58-bit Qwen3.6-35B-A3B page, install command: the MoE build uses "g64").
 *   - Trits are stored packed: base-3, 20 trits per 32-bit integer, about 1.6 bits per weight
 *     (the TurboQuant-MLX 1.58-bit Qwen3.6-35B-A3B page, section "为什么 1.58bit 没变成乱码", point 3), or 2 bits per trit.
 *   - Weights were Hadamard-rotated offline; at inference the matching fast transform, O(n log n),
 *     is applied to the activations ("27B 大模型塞进 5.9GB", section 二 ①).
 *   - Kernels compute directly on the packed format; decompressing to floats in memory would give
 *     back the savings ("27B 大模型塞进 5.9GB", section 二 ③).
 *   - MoE: 256 routed experts, 8 active per token, router gate in full precision
 *     (the TurboQuant-MLX 1.58-bit Qwen3.6-35B-A3B page, section "为什么 1.58bit 没变成乱码", point 1).
 *
 * Conventions for every entry point:
 *   - Data pointers are DEVICE pointers owned by the caller.  The library allocates nothing and
 *     frees nothing; scratch space is a caller-provided workspace of at least *_workspace_bytes()
 *     bytes, 256-byte aligned.
 *   - Work is enqueued asynchronously on ``stream`` (a cudaStream_t passed as void*; NULL = the
 *     legacy default stream).  No entry point synchronizes.
 *   - Argument errors are detected on the host before anything is launched and returned
 *     synchronously (TQ_ERR_INVALID_ARG / TQ_ERR_UNSUPPORTED / TQ_ERR_MISALIGNED /
 *     TQ_ERR_WORKSPACE).  A failed launch returns TQ_ERR_CUDA.  Data errors found on the device
 *     (a non-canonical code word, a trit outside {-1,0,1}, a bounded wait that ran out) are
 *     recorded in a device status word read by tq_device_status().
 *   - Layouts are row-major.  codes [N][P] uint32 with P = tq_row_pitch_words();
 *     scales [N][ceil(K/group)] FP16; activations [rows][K] bf16; MoE weights stacked per expert.
 *   - bf16 and FP16 values are passed as their 16-bit patterns (uint16_t).
 *   - Single GPU.  There is no CPU fallback: without a CUDA device every compute call returns
 *     TQ_ERR_CUDA.
 */
#ifndef TQ_H_
#define TQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TQ_OK = 0,
  TQ_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, inconsistent descriptor */
  TQ_ERR_UNSUPPORTED = 2,   /* valid but not implemented: group not 64/128, K not a multiple of 128, ... */
  TQ_ERR_MISALIGNED = 3,    /* a pointer is not 16-byte aligned (workspace: 256-byte) */
  TQ_ERR_INVALID_CODE = 4,  /* device-reported: code word not canonical, or trit outside {-1,0,1} */
  TQ_ERR_CUDA = 5,          /* a CUDA runtime call or launch failed */
  TQ_ERR_TIMEOUT = 6,       /* device-reported: a bounded wait inside a kernel ran out */
  TQ_ERR_WORKSPACE = 7,     /* workspace smaller than the matching *_workspace_bytes() */
  TQ_ERR_RANGE = 8          /* device-reported: a transformed activation is outside the FP16 range */
} tq_status;

typedef enum {
  TQ_PACK_B3 = 1,   /* base-3: word = sum_{i<20} (t[20j+i]+1) * 3^i; pad trits t=0; row pitch multiple of 4 words */
  TQ_PACK_2BIT = 2, /* 2-bit : word = sum_{i<16} (t[16j+i]+1) << 2i;  field 3 invalid; pad trits t=0 */
  TQ_PACK_3BIT = 3  /* 3-bit codes q in -4..3 (the non-expert linears; see below) */
} tq_packing;
/* TQ_PACK_3BIT (the TurboQuant-MLX 1.58-bit Qwen3.6-35B-A3B page, "为什么 1.58bit 没变成乱码", point 1:
 * attention, GDN projections and lm_head stay at 3 bits; the page gives no format, this is the
 * library's): W = s * q with q in {-4..3}, digit d = q + 4.  A word has ten 3-bit slots, five per
 * 16-bit half: slot j < 5 at bits 3j, slot j >= 5 at bits 16 + 3(j - 5); bits 15 and 31 are zero (a
 * word with either set is invalid).  Each block of 64 codes takes 7 words: word i < 6 holds codes
 * 10i..10i+9 of the block in slots 0..9; word 6 holds codes 60, 61 in slots 0, 1 and 62, 63 in slots
 * 5, 6, digit 4 (q = 0) elsewhere; so no word straddles a group.  Row pitch ceil(K/64) * 7 words,
 * rounded up to a multiple of 4.  Supported by the size functions, tq_pack / tq_unpack (trits hold
 * q), tq_gemv and tq_gemv_noalloc (batch 1..16, tensor-core decode as for base-3); the other
 * contractions (tq_gemm, tq_seq_*, tq_moe_*) return TQ_ERR_UNSUPPORTED. */

/* One ternary weight matrix W [N][K] (y = W x~). */
typedef struct {
  int32_t N;          /* output features: rows of W, >= 1 */
  int32_t K;          /* input features (reduction dim), >= 1 */
  int32_t group;      /* weights per FP16 scale along K: 64 or 128 */
  int32_t packing;    /* tq_packing */
  int32_t fwht_block; /* 128: apply the block Walsh-Hadamard transform to the input; 0: input used as given */
  int32_t flags;      /* 0, or TQ_STATIC_WEIGHTS (tq_gemv and tq_gemv_noalloc only; other entry points ignore it) */
} tq_desc;

/* Promise that no kernel still running on the stream when tq_gemv is called writes this matrix's
 * codes or scales.  The GEMV kernel is launched as a programmatic dependent of the preceding kernel
 * and may then begin streaming the weights before that kernel has finished; without the flag it
 * reads nothing written by earlier work until the preceding kernel has completed. */
#define TQ_STATIC_WEIGHTS 1

/* ---- format sizes (host only, no device access) ------------------------------------------------
 * Row pitch in uint32 words: base-3 roundup(ceil(K/20), 4), 2-bit roundup(ceil(K/16), 4).
 * (the TurboQuant-MLX 1.58-bit Qwen3.6-35B-A3B page, point 3: 20 trits per 32-bit word.)  Return 0 for an invalid descriptor. */
size_t tq_row_pitch_words(const tq_desc* d);
size_t tq_packed_bytes(const tq_desc* d);      /* N * pitch * 4 */
size_t tq_scale_bytes(const tq_desc* d);       /* N * ceil(K/group) * 2 ("27B 大模型塞进 5.9GB", section 二 ②) */

/* ---- tq_pack: int8 trits [N][K] -> codes [N][P] --------------------------------------------------
 * Packs row-contiguous trits across group boundaries; trits past K and whole padding words hold
 * t = 0.  A trit outside {-1,0,1} records TQ_ERR_INVALID_CODE in the device status (its word is
 * written as if the trit were 0).  trits: device, 1-byte aligned; codes: device, 16-byte aligned. */
tq_status tq_pack(const tq_desc* d, const int8_t* trits, uint32_t* codes, void* stream);

/* ---- tq_unpack: codes [N][P] -> int8 trits [N][K] ------------------------------------------------
 * Digit i of a base-3 word v is (v / 3^i) mod 3, t = digit - 1; field i of a 2-bit word is
 * (v >> 2i) & 3.  invalid_words (device int32, may be NULL) receives the number of words in the
 * whole pitch that are not valid encodings (base-3: v > 3^20 - 1; 2-bit: a field equal to 3); it is
 * overwritten, not accumulated.  Invalid words are decoded as written (digits taken mod 3 / field 3
 * -> t = 2 is clamped to 0).  A non-zero count is also recorded as TQ_ERR_INVALID_CODE. */
tq_status tq_unpack(const tq_desc* d, const uint32_t* codes, int8_t* trits, int32_t* invalid_words,
                    void* stream);

/* ---- tq_quantize: offline, dense bf16 W [N][K] -> codes [N][P] + FP16 scales [N][K/group] -----------
 * The steps "27B 大模型塞进 5.9GB" puts before compression (section 二 ①: Hadamard rotation of the
 * weights; section 二 ②: one FP16 scale per group; section 一: three levels).  The pages give no
 * rounding rule; this uses absmean (BitNet b1.58):
 *   u = H_128 w per 128-block of each row (unnormalised Sylvester; fwht_block = 0: u = w),
 *   S = fp16_rn(mean_{group} |u| * c), c = 2^-3.5 (1 without the transform),
 *   t = sign(u) if |u| * c > S / 2 else 0,
 * all in fp64.  With fwht_block = 128 the result is the matrix tq_gemv / tq_gemm expect for the same
 * x: W x ~= sum s t x~.  The sums are exact (and the result therefore bit-reproducible by any exact
 * evaluation) when the magnitudes within each 128-block span less than 2^31.  A non-finite weight or
 * a scale beyond the FP16 range records TQ_ERR_RANGE.  Requires K a multiple of 128, K <= 196608,
 * group 64 or 128, flags 0.  w: device bf16, 16-byte aligned; codes: device, 16-byte aligned, the
 * layout of tq_pack; scales: device. */
tq_status tq_quantize(const tq_desc* d, const uint16_t* w, uint32_t* codes, uint16_t* scales, void* stream);

/* ---- tq_fwht: x~[r, 128b + i] = sum_c H[i][c] x[r, 128b + c] / sqrt(block) -----------------------
 * Block Walsh-Hadamard transform (Sylvester order) of each row of x (bf16 [rows][K]); block must be
 * 128 and K a multiple of it ("27B 大模型塞进 5.9GB", section 二 ①).  out_fp16 = 0: out is float [rows][K];
 * out_fp16 = 1: out is FP16 [rows][K] (values beyond the FP16 range record TQ_ERR_RANGE). */
tq_status tq_fwht(const uint16_t* x, void* out, int out_fp16, int rows, int K, int block, void* stream);

/* ---- tq_gemv: decode GEMV, y[b][n] = sum_k s[n][k/group] * t[n][k] * x~[b][k] ----------------------
 * x: bf16 [batch][K], 1 <= batch <= 16; x~ = block FWHT of x (or x itself when fwht_block = 0).
 * y: float [batch][N].  Requires K a multiple of 128.  Streams each code word from HBM once per call.
 * workspace >= tq_gemv_workspace_bytes(d, batch).  Calls on one stream are ordered; two calls that
 * share a workspace must not overlap in time. */
size_t tq_gemv_workspace_bytes(const tq_desc* d, int batch);
tq_status tq_gemv(const tq_desc* d, const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                  int batch, float* y, void* workspace, size_t workspace_bytes, void* stream);

/* Number of CUDA kernels one tq_gemv call with this descriptor and batch launches on the current
 * device (1: the activation transform runs inside the decode kernel; 2: a prep kernel precedes it),
 * or -1 for an invalid descriptor / batch or a CUDA error.  No counterpart on the pages: it lets a
 * caller count launches, e.g. per CUDA-graph step. */
int tq_gemv_kernel_count(const tq_desc* d, int batch);

/* ---- tq_gemv_noalloc: tq_gemv without a workspace -------------------------------------------------
 * No counterpart on the pages: a library convenience.  Same computation, arguments, layouts and
 * errors as tq_gemv, but the scratch lives in a fixed 1 MiB device array inside libtq, for callers
 * that cannot provide device memory (for example a decode loop that must not call an allocator,
 * which can synchronise the device, or a C caller without an allocator of its own).  Shapes whose
 * tq_gemv_workspace_bytes(d, batch) exceeds 1 MiB (at batch 16: K above 31488 for groups of 64, above
 * 32128 for groups of 128) return TQ_ERR_WORKSPACE before anything is launched.  The first call with a device current looks up that
 * device's array; make it before any stream capture.  Nothing has to be zeroed first.  All calls on a
 * device share the array: calls whose kernels overlap in time race on it, so serialise them.  The
 * looked-up address is kept for the life of the process: do not use the library across a
 * cudaDeviceReset() (the device copy of the array may move). */
tq_status tq_gemv_noalloc(const tq_desc* d, const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                          int batch, float* y, void* stream);

/* ---- tq_seq: a decode step (a chain of dependent GEMVs) as one launch ------------------------------
 * Decoding one token runs every linear of the model once, each on the previous one's output
 * ("27B 大模型塞进 5.9GB", section 三: single-stream decode of the whole model; section 二 ③: kernels
 * that compute on the packed ternary format).  tq_seq_run executes calls[0..ncalls-1] in order, with
 * the result of issuing tq_gemv for each on one stream (same arithmetic and tolerance), in ONE
 * cooperative kernel launch: every CTA streams its weight tiles continuously across the calls, and
 * calls are ordered by a grid-wide barrier, so HBM does not go idle between dependent calls.
 * The input of call j is selected by x_src:
 *   TQ_SEQ_X_BF16        x: bf16 [batch][K] in device memory (required for call 0);
 *   TQ_SEQ_X_PREV        the first K entries of each batch row of call j-1's y (needs N_{j-1} >= K);
 *   TQ_SEQ_X_SWIGLU_PREV silu(y_{j-1}[b][k]) * y_{j-1}[b][K + k] (needs N_{j-1} = 2K: a stacked
 *                        gate/up projection, gate rows first);
 *   TQ_SEQ_X_RMS_PREV    the TQ_SEQ_X_PREV input divided by sqrt(mean_k(input^2) + 1e-6) per batch
 *                        row (RMS normalisation with unit gain, as a pre-norm decoder applies it
 *                        before its attention and FFN projections).
 * Then x~ = block FWHT(input) if fwht_block = 128, y[b][n] = sum_k s t x~ (float [batch][N]).
 * Limits: one packing (TQ_PACK_2BIT or TQ_PACK_B3; 3-bit codes: TQ_ERR_UNSUPPORTED) and one group
 * size for all calls; 2-bit: K a multiple of 8 * group (each row of scales a multiple of 16 bytes:
 * they are fetched by TMA); N a multiple of 4; 1 <= batch <= 8; K * batch small enough for the
 * transformed activations of the widest call to sit in shared memory (2-bit: K up to about 40000 at
 * batch 1, 5120 at batch 8; base-3 leaves less room, TQ_ERR_UNSUPPORTED where it does not fit);
 * TQ_STATIC_WEIGHTS is implied (weights must not change
 * while the plan is in use).  A call's y must not be the x of any call, nor the y of the call before
 * it.  All pointers: device memory, 16-byte aligned.
 *
 * tq_seq_create checks the calls and builds a host-side plan (tensor maps of every weight matrix,
 * work split for the current device); it allocates host memory only.  The plan needs a caller-owned
 * device workspace of tq_seq_workspace_bytes(plan) bytes (256-byte aligned), filled once by
 * tq_seq_upload (synchronous: copies the call records, clears the barrier and handoff words) and
 * then used by every tq_seq_run with that plan; tq_seq_run only enqueues the launch (no allocation, no
 * synchronisation; capturable in a CUDA graph).  Two runs that share a workspace must not overlap.
 * A bounded wait that runs out records TQ_ERR_TIMEOUT in the device status and leaves the workspace's
 * barrier words dirty: call tq_seq_upload again before the next run.  The plan is tied to the device
 * that was current at creation. */
#define TQ_SEQ_X_BF16 0
#define TQ_SEQ_X_PREV 1
#define TQ_SEQ_X_SWIGLU_PREV 2
#define TQ_SEQ_X_RMS_PREV 3

typedef struct {
  tq_desc d;               /* N, K, group, packing (TQ_PACK_2BIT or TQ_PACK_B3), fwht_block; flags ignored */
  const uint32_t* codes;   /* [N][P] */
  const uint16_t* scales;  /* [N][K / group] FP16 */
  int32_t x_src;           /* TQ_SEQ_X_* */
  const uint16_t* x;       /* bf16 [batch][K] for TQ_SEQ_X_BF16, else ignored */
  float* y;                /* [batch][N] */
} tq_seq_call;

typedef struct tq_seq tq_seq;

tq_status tq_seq_create(const tq_seq_call* calls, int ncalls, int batch, tq_seq** plan);
size_t tq_seq_workspace_bytes(const tq_seq* plan);
tq_status tq_seq_upload(const tq_seq* plan, void* workspace, size_t workspace_bytes);
tq_status tq_seq_run(const tq_seq* plan, void* workspace, void* stream);
int tq_seq_kernel_count(const tq_seq* plan);   /* kernels one tq_seq_run launches (1), -1 for NULL */
void tq_seq_destroy(tq_seq* plan);

/* ---- tq_moe_route: top-k experts per token --------------------------------------------------------
 * logits: float [T][E] (router at full precision, the TurboQuant-MLX 1.58-bit Qwen3.6-35B-A3B page, point 1).  idx: int32 [T][topk]
 * in the order (logit descending, expert index ascending); gate: float [T][topk] =
 * softmax over the topk chosen logits.  E <= 256, topk <= 8 (the pages' top-8 of 256). */
tq_status tq_moe_route(const float* logits, int T, int E, int topk, int32_t* idx, float* gate, void* stream);

/* ---- tq_moe_gemv: routed SwiGLU expert layer at decode time ----------------------------------------
 * For each token: route (as tq_moe_route); x~ = FWHT(x); for each chosen expert e:
 * g = Wg[e] x~, u = Wu[e] x~ (gate_up rows 0..F-1 then F..2F-1), h = silu(g) * u,
 * y_e = Wd[e] FWHT(h); y = sum_j gate_j y_{e_j} in slot order j = 0..topk-1 (deterministic).
 * gate_up: desc with N = 2F, K = H; down: desc with N = H, K = F (same packing/group/fwht).
 * gu_codes [E][2F][P_H], gu_scales [E][2F][H/group], d_codes [E][H][P_F], d_scales [E][H][F/group].
 * x: bf16 [T][H]; idx/gate as tq_moe_route; h_out: float [T][topk][F] or NULL; y: float [T][H].
 * Three launches: routing and the chunk table (one CTA), the gate/up GEMV, the down GEMV with the
 * combine fused into it.  The tokens routed to an expert are processed in chunks of 1 (T = 1) or 2
 * tokens; each chunk streams its expert's codes once, so an expert with n routed tokens is read
 * ceil(n / 2) times per call. */
size_t tq_moe_workspace_bytes(int T, int E, int topk, int H, int F);
tq_status tq_moe_gemv(const tq_desc* gate_up, const tq_desc* down, int E, int topk,
                      const uint32_t* gu_codes, const uint16_t* gu_scales,
                      const uint32_t* d_codes, const uint16_t* d_scales,
                      const float* router_logits, const uint16_t* x, int T,
                      int32_t* topk_idx, float* topk_gate, float* h_out, float* y,
                      void* workspace, size_t workspace_bytes, void* stream);

/* ---- tq_moe_gemm: the same expert layer at prefill sizes (many tokens per expert) -------------------
 * Same computation, arguments and layouts as tq_moe_gemv (the TurboQuant-MLX 1.58-bit Qwen3.6-35B-A3B
 * page, "为什么 1.58bit 没变成乱码", points 1-2), organised as a grouped tensor-core GEMM: the (token, slot) assignments are sorted by
 * expert, the tokens' block-transformed inputs are gathered in that order as FP16 (|x~| below 65504,
 * else TQ_ERR_RANGE), every expert's weights are decoded to FP16 s * t, one persistent tcgen05 launch
 * per projection walks a tile list over (expert, 128 sorted rows, 256 weight rows), silu(gate) * up
 * and its transform go to FP16 for the down projection, and the combine adds the slots in slot order
 * (deterministic).  Nine launches.  Requires H and 2F multiples of 256 and T * topk < 2^24.
 * workspace >= tq_moe_gemm_workspace_bytes(T, E, topk, H, F): it holds every expert's decoded
 * weights (E * 3 * H * F * 2 bytes) besides per-assignment rows. */
size_t tq_moe_gemm_workspace_bytes(int T, int E, int topk, int H, int F);
tq_status tq_moe_gemm(const tq_desc* gate_up, const tq_desc* down, int E, int topk,
                      const uint32_t* gu_codes, const uint16_t* gu_scales,
                      const uint32_t* d_codes, const uint16_t* d_scales,
                      const float* router_logits, const uint16_t* x, int T,
                      int32_t* topk_idx, float* topk_gate, float* h_out, float* y,
                      void* workspace, size_t workspace_bytes, void* stream);

/* ---- tq_gemm: batched prefill, Y[m][n] = bf16( sum_k s[n][k/group] t[n][k] x~[m][k] ) -------------
 * x: bf16 [M][K]; y: bf16 [M][N]; fp32 accumulation.  x~ is held as FP16 (|x~| must stay below
 * 65504, else TQ_ERR_RANGE is recorded).  Requires K a multiple of 128.
 * workspace >= tq_gemm_workspace_bytes(d, M). */
size_t tq_gemm_workspace_bytes(const tq_desc* d, int M);
tq_status tq_gemm(const tq_desc* d, const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                  int M, uint16_t* y, void* workspace, size_t workspace_bytes, void* stream);

/* ---- tq_gemm_fp8: tq_gemm with FP8 E4M3 operands ----------------------------------------------------
 * No page states this variant; it is the library's: the batched contraction on the packed codes
 * ("27B 大模型塞进 5.9GB", section 二 ③) with both operands in FP8 E4M3 for the tensor cores' FP8 rate
 * (tcgen05.mma kind::f8f6f4).  Each token row is scaled by 2^-ea[m], each weight row by 2^-eb[n],
 * ea[m] = floor(log2 max_k |x~[m][k]|) - 7, eb[n] = floor(log2 max_g |s[n][g]|) - 7 (0 for an all-zero
 * row), and rounded to E4M3 to nearest even:
 *   Y[m][n] = bf16( 2^(ea[m] + eb[n]) * sum_k e4m3(x~[m][k] 2^-ea[m]) e4m3(s[n][k/group] t[n][k] 2^-eb[n]) ).
 * t is exact in E4M3; s and x~ keep 4 significant bits, so |Y - exact| <= (2^-3 + 2^-8) sum_k |s t x~|
 * plus a subnormal term of 2^-10 times the row factors (and fp32 accumulation, bf16 output rounding).
 * Inf / NaN in a row of x~ or of the scales records TQ_ERR_RANGE.  x, y, requirements as tq_gemm
 * (no FP16 range limit on x~).  workspace >= tq_gemm_fp8_workspace_bytes(d, M): the E4M3 operands
 * (M * K and N * K bytes) and the row exponents. */
size_t tq_gemm_fp8_workspace_bytes(const tq_desc* d, int M);
tq_status tq_gemm_fp8(const tq_desc* d, const uint32_t* codes, const uint16_t* scales, const uint16_t* x,
                      int M, uint16_t* y, void* workspace, size_t workspace_bytes, void* stream);

/* ---- tq_selftest_wait: the bounded-wait path, made to run out on purpose ------------------------------
 * Launches one CTA that waits on something nothing completes, with a wait limit of limit_ns
 * (1 .. 1e9 ns) instead of the kernels' 4 s: kind 0 an mbarrier that is never arrived on (the
 * TMA-ring wait of the decode and prefill kernels), kind 1 the grid barrier of tq_seq on a counter
 * that no CTA arrives at (workspace: >= 4 bytes of device memory, 256-byte aligned, zeroed by this
 * call; NULL allowed for kind 0).  The wait gives up, the kernel records TQ_ERR_TIMEOUT in the device
 * status word (read it with tq_device_status) and returns; the context stays usable.  Diagnostic
 * only: no result is computed. */
tq_status tq_selftest_wait(int kind, long long limit_ns, void* workspace, void* stream);

/* ---- status ---------------------------------------------------------------------------------------
 * The address of each device's status word is looked up once per process; do not use the library
 * across a cudaDeviceReset().
 * Reads the device status word of the current device (the first error any kernel recorded since the
 * last read), stores it in *status (TQ_OK if none) and clears it.  This call synchronizes the device. */
tq_status tq_device_status(int32_t* status);
const char* tq_status_str(tq_status s);
/* The cudaError_t code of the last CUDA call that made an entry point of this library return
 * TQ_ERR_CUDA in the calling host thread (0 if none), then clears it.  No device access. */
int tq_last_cuda_error(void);
int tq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H_ */

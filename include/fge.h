/*
 * fge.h -- C ABI of libfge: W4A8 grouped-expert MoE prefill and dense per-tensor W8A8
 * projections on one NVIDIA GB300 (sm_103a).
 *
 * Source of the method: "FP8 grouped-expert prefill with on-chip int4-to-e4m3 dequant"
 * (section 1, Contribution): activations quantized on the fly to e4m3, packed int4 expert
 * weights dequantized to e4m3 on chip without unpacking the resident bank, one grouped
 * expert GEMM per layer in place of one dispatch per routed token, and per-(token, group)
 * activation scales folded into the accumulator path.  The per-tensor W8A8 projection and
 * the "all device work in one call, no host sync" boundary follow "feat(qwen4_exp):
 * load-time per-tensor FP8 dense projections (W8A8 via _scaled_mm)" (section "What this
 * adds") and "Module fp8_ffi" (module documentation and struct Fp8Scratch).
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers unless a parameter says "host".  Every tensor is dense
 *    row-major with the shape given; every pointer must be 16-byte aligned.
 *  - Ownership: the caller allocates all buffers, including the workspace whose size the
 *    matching fge_workspace_bytes() query returns.  The library allocates no device memory
 *    and keeps no per-call state; it only caches per-device properties in fge_init().
 *  - Streams: all work is enqueued on `stream` (a cudaStream_t; 0 = legacy default) in
 *    order, with no host synchronisation and no branch on tensor values (shapes only).
 *  - Errors: argument, shape and alignment problems return a status before anything is
 *    enqueued.  A launch failure returns FGE_ERR_CUDA.  Problems detected on the device
 *    (a pipeline wait that ran out of its time budget: FGE_ERR_DEVICE_TIMEOUT; an
 *    activation to quantize that is an infinity or a NaN: FGE_ERR_NONFINITE) are written to
 *    the status word at the start of the workspace -- the first problem wins -- and the
 *    kernels finish without trapping; read the word with fge_read_device_status().
 *  - Sizes: K, H and I are multiples of 128 (the scale group); N is a multiple of 128.
 */
#ifndef FGE_H_
#define FGE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fge_stream_t; /* same type as cudaStream_t */

typedef enum {
  FGE_OK = 0,
  FGE_ERR_INVALID_ARG = 1,        /* null pointer, bad enum, k > E, ... */
  FGE_ERR_BAD_SHAPE = 2,          /* a size is not a multiple of 128 or out of range */
  FGE_ERR_MISALIGNED = 3,         /* a pointer is not 16-byte aligned */
  FGE_ERR_WORKSPACE_TOO_SMALL = 4,
  FGE_ERR_UNSUPPORTED_DEVICE = 5, /* not sm_103 / kernel resources unavailable */
  FGE_ERR_CUDA = 6,               /* a CUDA runtime call or launch failed */
  FGE_ERR_DEVICE_TIMEOUT = 7,     /* device status only: a pipeline wait ran out */
  FGE_ERR_NOT_INITIALIZED = 8,    /* fge_init() was not called for the current device */
  FGE_ERR_EXCEEDS_STATIC_SCRATCH = 9, /* fge_linear_w8a8_noalloc: M*K beyond its fixed scratch */
  FGE_ERR_NONFINITE = 10          /* device status only: an activation the call quantized was an
                                     infinity or a NaN (its scale and codes are meaningless) */
} fge_status;

typedef enum {
  FGE_SCALE_PER_TENSOR = 0,     /* one amax over the whole [M, K] tensor */
  FGE_SCALE_PER_TOKEN_G128 = 1, /* one scale per (row, 128-element K group) */
  FGE_SCALE_PER_ROW = 2         /* one scale per row (token) over its K elements */
} fge_scale_mode;

typedef enum { FGE_DTYPE_BF16 = 0, FGE_DTYPE_F32 = 1 } fge_dtype;

typedef enum {
  FGE_EPI_STORE = 0,          /* write the GEMM result in out_dtype */
  FGE_EPI_SWIGLU_REQUANT = 1  /* h = silu(gate) * up, then e4m3 per (row, 128 group) */
} fge_epilogue;

/* Resident int4 bank formats produced by fge_w4_prepack.  Both hold two int4 values per
 * byte; they differ in how the kernel turns a nibble into an e4m3 tensor-core operand:
 *  FGE_W4_LUT:       the e4m3 code of the integer itself (byte-permute table lookup);
 *  FGE_W4_SUBNORMAL: the e4m3 code of q * 2^-9 (the subnormal/normal code whose bits are
 *                    the integer in sign-magnitude form), with 2^9 folded into the
 *                    prepacked weight scales.  Both are exact. */
typedef enum { FGE_W4_LUT = 0, FGE_W4_SUBNORMAL = 1 } fge_w4_format;

typedef enum {
  FGE_OP_QUANT_PER_TENSOR = 0, /* args: (M, K) */
  FGE_OP_PERMUTE = 1,          /* args: (T, H, -, E, k) */
  FGE_OP_GROUPED_GEMM = 2,     /* args: unused */
  FGE_OP_LINEAR_W8A8 = 3,      /* args: (M, K, N); N = 0: no K-split scratch */
  FGE_OP_MOE_LAYER = 4,        /* args: (T, H, I, E, k) */
  FGE_OP_DISPATCH_BASELINE = 5, /* args: (T, H, I, E, k) */
  FGE_OP_LINEAR_W8A8_ROWS = 6   /* args: (M, K) */
} fge_op;

/* Library version (major*10000 + minor*100 + patch). */
int fge_version(void);

/* Checks that `device` is an sm_103 GPU and caches its SM count.  Idempotent and safe to
 * call from several host threads; call once per device before any other call on it.  Each
 * kernel's shared-memory limit is set on its first launch on a device (per device, under a
 * lock), so a process may drive several GPUs. */
fge_status fge_init(int device);

/* Human-readable name of a status code (static string). */
const char* fge_status_string(fge_status status);

/* Workspace bytes an operation needs for the given sizes (0 for a bad op). */
size_t fge_workspace_bytes(fge_op op, int64_t a, int64_t b, int64_t c, int E, int k);

/* Host-side ledger of this process's calls into the library (counted from library load
 * or the last fge_reset_ledger; thread-safe; no device access):
 *   calls              compute entry-point calls;
 *   refused            of those, calls refused before anything was enqueued (bad argument,
 *                      shape, alignment, workspace size, device not initialised, ...);
 *   layers             fge_moe_layer_forward calls that enqueued their kernels;
 *   grouped_gemms      grouped W4A8 GEMM launches (stand-alone or inside a layer);
 *   dense_decode_tile  dense W8A8 projections run at decode sizes (M <= 16: the weight-
 *                      streaming decode kernel; otherwise the 16-token decode tile);
 *   dense_row_tile     dense W8A8 GEMMs run with 128-row tiles. */
typedef struct {
  uint64_t calls;
  uint64_t refused;
  uint64_t layers;
  uint64_t grouped_gemms;
  uint64_t dense_decode_tile;
  uint64_t dense_row_tile;
} fge_ledger;
fge_status fge_read_ledger(fge_ledger* out);
fge_status fge_reset_ledger(void);

/* Zero the device status word of a workspace (enqueued on `stream`). */
fge_status fge_clear_device_status(void* workspace, fge_stream_t stream);

/* Synchronises `stream`, then copies the workspace's device status word to *out (host). */
fge_status fge_read_device_status(const void* workspace, fge_stream_t stream, int32_t* out);

/* fp8_quant_act -- dynamic e4m3 activation quantization.
 * Per "FP8 grouped-expert prefill ..." section 1 (per-(token, group) scale) and "Module
 * fp8_ffi" (amax reduce, scale finalize, e4m3 quantize, one stream, no host sync):
 *   amax = max|x| over the group (G128) or the whole tensor (PER_TENSOR);
 *   s = amax / 448 (IEEE float division; s = 1 when amax = 0; s >= 2^-126);
 *   q = e4m3(x / s), round to nearest even, saturating at +-448, where x / s is the IEEE
 *   float32 quotient (formed from one rounded reciprocal of s and an exact-residual
 *   correction, which equals the division for every bf16 x).
 * PER_ROW takes the amax over each row's K elements (the row-wise activation scales that
 * "feat(qwen4_exp) ..." measures against per-tensor, section "Limits").
 * x_bf16: [M, K] bf16.  xq: [M, K] e4m3 codes (out).  xs: [M, K/128] float (G128), [M] float
 * (PER_ROW) or one float (PER_TENSOR) (out).  PER_TENSOR needs a workspace of
 * fge_workspace_bytes(FGE_OP_QUANT_PER_TENSOR, M, K, ...); G128 and PER_ROW need none (may
 * be NULL), but given one of at least 256 bytes they report a non-finite input
 * (FGE_ERR_NONFINITE) in its status word, as PER_TENSOR always does.
 * M may be 0. */
fge_status fge_fp8_quant_act(const void* x_bf16, int64_t M, int64_t K, fge_scale_mode mode,
                             uint8_t* xq, float* xs, void* workspace, size_t workspace_bytes,
                             fge_stream_t stream);

/* mx_quant_e2m1 -- FP4 (E2M1) activations with one power-of-two scale per 32 values
 * (MXFP4).  "[RFC] Support FP4 (E2M1) activation dispatch in MegaMoE" proposes E2M1
 * activations for the expert dispatch buffer (half the bytes of e4m3) feeding an MXF4
 * main loop; the block size and scale format are the MX convention it names:
 *   E = max(floor(log2(amax)) - 2, -127) over each block of 32 consecutive values of a row
 *   (-127 for an all-zero block), stored as the E8M0 code E + 127 (scale 2^E);
 *   q = E2M1(x * 2^-E), round to nearest even, saturating at 6; a zero keeps its sign.
 * x_bf16: [M, K] bf16, 16-byte aligned.  xq: [M, K/2] bytes (out), 16-byte aligned: byte b
 * of a row holds the codes of elements 2b (low nibble) and 2b + 1 (high nibble).
 * xs: [M, K/32] E8M0 codes (out), any alignment.  K % 32 == 0; M may be 0.
 * FGE_ERR_BAD_SHAPE, FGE_ERR_INVALID_ARG (NULL pointer) or FGE_ERR_MISALIGNED before any
 * launch; no workspace, no host sync. */
fge_status fge_mx_quant_e2m1(const void* x_bf16, int64_t M, int64_t K, uint8_t* xq,
                             uint8_t* xs, fge_stream_t stream);

/* moe_topk_gate -- top-k experts per token and their gates.
 * The pages route tokens to experts without fixing the rule ("FP8 grouped-expert prefill
 * ..." section 1); this is standard top-k routing: experts in descending logit order (ties
 * to the lower id), gate_j = exp(l_j - l_max) / sum over the chosen k of exp(l - l_max).
 * logits: [T, E] float.  ids: [T, k] int32 (out).  gates: [T, k] float (out).
 * 1 <= k <= min(E, 32), E <= 1024. */
fge_status fge_moe_topk_gate(const float* logits, int64_t T, int E, int k, int32_t* ids,
                             float* gates, fge_stream_t stream);

/* moe_permute -- expert-contiguous rows for the single grouped GEMM ("FP8 grouped-expert
 * prefill ..." section 1: one grouped expert GEMM per layer instead of one dispatch per
 * routed token).  Histogram of ids, exclusive scan, stable scatter ordered by (expert,
 * token, slot), then a copy of each token's e4m3 row and group scales to its k rows.
 * ids: [T, k] int32 in [0, E) (distinct within a row).  xq: [T, H] codes; xs: [T, H/128].
 * offsets: [E+1] (out); row_token: [T*k] (out); token_row: [T, k] (out);
 * aq: [T*k, H] (out); as: [T*k, H/128] (out).  With aq and as both NULL the call is
 * index-only (offsets, row_token and token_row; xq and xs may then be NULL too), for
 * fge_grouped_gemm_w4a8_gather.  Workspace: FGE_OP_PERMUTE. */
fge_status fge_moe_permute(const int32_t* ids, int64_t T, int k, int E, const uint8_t* xq,
                           const float* xs, int64_t H, int32_t* offsets, int32_t* row_token,
                           int32_t* token_row, uint8_t* aq, float* as, void* workspace,
                           size_t workspace_bytes, fge_stream_t stream);

/* moe_permute_quant -- fge_moe_permute with the G128 activation quantization of
 * fge_fp8_quant_act folded into the row copy: each token's bf16 row is read once and its
 * e4m3 codes and scales are written straight to its k expert rows (same codes and scales as
 * quantizing first, bit for bit).  x_bf16: [T, H] bf16; other arguments as fge_moe_permute.
 * Workspace: FGE_OP_PERMUTE. */
fge_status fge_moe_permute_quant(const int32_t* ids, int64_t T, int k, int E,
                                 const void* x_bf16, int64_t H, int32_t* offsets,
                                 int32_t* row_token, int32_t* token_row, uint8_t* aq, float* as,
                                 void* workspace, size_t workspace_bytes, fge_stream_t stream);

/* w4_prepack -- load-time layout of a resident int4 expert bank for the grouped GEMM.
 * Input (canonical): w [E, N, K/2] bytes, two's-complement nibbles, byte b of a row holds
 * element 2b in the low nibble and 2b+1 in the high nibble; w_scale [E, N, K/128] float.
 * Output: w_dev [E, N, K/2] in `format` (nibbles regrouped within each 8-element word for
 * FGE_W4_SUBNORMAL) and w_scale_dev [E, K/128, N] (transposed; times 2^9 for
 * FGE_W4_SUBNORMAL).  gate_up_interleave = 1 reorders rows in blocks of 128: 64 gate rows
 * then the 64 matching up rows (gate = rows [0, N/2), up = rows [N/2, N) of the input);
 * required by FGE_EPI_SWIGLU_REQUANT.  Not part of the timed path. */
fge_status fge_w4_prepack(const uint8_t* w, const float* w_scale, int E, int64_t N, int64_t K,
                          int gate_up_interleave, fge_w4_format format, uint8_t* w_dev,
                          float* w_scale_dev, fge_stream_t stream);

/* grouped_gemm_w4a8 -- one grouped expert GEMM over all routed rows ("FP8 grouped-expert
 * prefill ..." section 1).  For expert e and rows r in [offsets[e], offsets[e+1]):
 *   C[r, n] = sum_g as[r, g] * sw[e, n, g] * sum_{k in group g} aq[r, k] * q[e, n, k]
 * computed with tcgen05 kind::f8f6f4 MMAs (int4 dequantized to e4m3 in shared memory) and
 * fp32 promotion per K group.  aq: [R, K] e4m3; as: [R, K/128]; offsets: [E+1] on device
 * (offsets[E] <= R; the host never reads them); w_dev / w_scale_dev from fge_w4_prepack.
 * FGE_EPI_STORE: out [R, N] in out_dtype (rows past offsets[E] untouched).
 * FGE_EPI_SWIGLU_REQUANT (needs N % 256 == 0 and an interleaved bank): out = hq [R, N/2]
 * e4m3, out_scales = hs [R, N/256].  E <= 512.  Workspace: FGE_OP_GROUPED_GEMM. */
fge_status fge_grouped_gemm_w4a8(const uint8_t* aq, const float* as, const int32_t* offsets,
                                 int64_t R, const uint8_t* w_dev, const float* w_scale_dev,
                                 int E, int64_t N, int64_t K, fge_w4_format format,
                                 fge_epilogue epilogue, fge_dtype out_dtype, void* out,
                                 float* out_scales, void* workspace, size_t workspace_bytes,
                                 fge_stream_t stream);

/* grouped_gemm_mxf4_w4 -- the grouped expert GEMM with MXFP4 activations: E2M1 codes with
 * one power-of-two (UE8M0) scale per 32 values along K, the format fge_mx_quant_e2m1 writes
 * ("[RFC] Support FP4 (E2M1) activation dispatch in MegaMoE": E2M1 dispatch halves the
 * activation bytes; the expert GEMM consumes them in its MX main loop).  For expert e and
 * rows r in [offsets[e], offsets[e+1]):
 *   C[r, n] = sum_g sw[e, n, g] * sum_{k in group g} a[r, k] * q[e, n, k],
 *   a[r, k] = e2m1(code[r, k]) * 2^(scale[r, k/32] - 127)
 * computed with tcgen05 block-scaled MMAs (kind::mxf8f6f4, scale_vec::1X: the activation
 * scales are applied inside the tensor core, one per K = 32 step, from TMEM), the int4 bank
 * dequantized to e4m3 in shared memory and the weight scale promoted per 128-K group in fp32.
 * a_codes: [R, K/2] packed E2M1 (element 2b in the low nibble of byte b), 32-byte aligned;
 * a_scales: [R, K/32] UE8M0 codes; offsets, w_dev, w_scale_dev as fge_grouped_gemm_w4a8
 * (FGE_W4_SUBNORMAL bank only).  out: [R, N] in out_dtype (BF16 or F32; rows past
 * offsets[E] untouched).  N % 128 == 0, K % 128 == 0.  Workspace: FGE_OP_GROUPED_GEMM.
 * Errors: FGE_ERR_INVALID_ARG (null pointer, other bank format or dtype), FGE_ERR_BAD_SHAPE,
 * FGE_ERR_MISALIGNED, FGE_ERR_WORKSPACE_TOO_SMALL; device waits that run out are reported
 * through fge_read_device_status. */
fge_status fge_grouped_gemm_mxf4_w4(const uint8_t* a_codes, const uint8_t* a_scales,
                                   const int32_t* offsets, int64_t R, const uint8_t* w_dev,
                                   const float* w_scale_dev, int E, int64_t N, int64_t K,
                                   fge_w4_format format, fge_dtype out_dtype, void* out,
                                   void* workspace, size_t workspace_bytes, fge_stream_t stream);

/* grouped_gemm_w4a8_gather -- the same GEMM with the permutation folded into the A load: the
 * A rows are gathered from the token-ordered activations by TMA row gathers (4 rows a copy)
 * instead of being read from a permuted copy, so the permute's row copy disappears.
 * Routed row r uses row row_token[r] of xq [T, K] and of xs [T, K/128] (row_token: [R] from
 * fge_moe_permute, values in [0, T)).  Other arguments and the output as
 * fge_grouped_gemm_w4a8 (out rows stay in routed order). */
fge_status fge_grouped_gemm_w4a8_gather(const uint8_t* xq, const float* xs, int64_t T,
                                        const int32_t* row_token, const int32_t* offsets,
                                        int64_t R, const uint8_t* w_dev,
                                        const float* w_scale_dev, int E, int64_t N, int64_t K,
                                        fge_w4_format format, fge_epilogue epilogue,
                                        fge_dtype out_dtype, void* out, float* out_scales,
                                        void* workspace, size_t workspace_bytes,
                                        fge_stream_t stream);

/* swiglu_quant -- unfused SwiGLU + requant (parity/ablation of the fused epilogue):
 * h = silu(c[:, i]) * c[:, I + i], silu(g) = g / (1 + exp(-g)), then e4m3 per (row, 128
 * group) as fp8_quant_act.  c: [R, 2I] float.  hq: [R, I]; hs: [R, I/128]. */
fge_status fge_swiglu_quant(const float* c, int64_t R, int64_t I, uint8_t* hq, float* hs,
                            fge_stream_t stream);

/* moe_combine -- out[t] = sum_{j=0..k-1} gates[t, j] * y[token_row[t, j]], accumulated in
 * fp32 in slot order (deterministic; no atomics).  y: [T*k, H] in y_dtype; token_row,
 * gates: [T, k]; out: [T, H] in out_dtype. */
fge_status fge_moe_combine(const void* y, fge_dtype y_dtype, const int32_t* token_row,
                           const float* gates, int64_t T, int k, int64_t H,
                           fge_dtype out_dtype, void* out, fge_stream_t stream);

/* moe_combine_staged -- the same sums, bit for bit, as the MoE layer computes them for a
 * bf16 y: each (token, 2048-column block) gathers its k slot rows' blocks into shared memory
 * with bulk copies (no per-thread loads in flight), then sums them in slot order.
 * y_bf16: [T*k, H] bf16, k <= 8, H % 2048 == 0; token_row, gates, out as moe_combine.
 * workspace: at least 256 bytes (its status word receives FGE_ERR_DEVICE_TIMEOUT if a
 * copy never lands; read with fge_read_device_status).  Errors: FGE_ERR_BAD_SHAPE outside
 * those sizes, FGE_ERR_MISALIGNED, FGE_ERR_WORKSPACE_TOO_SMALL. */
fge_status fge_moe_combine_staged(const void* y_bf16, const int32_t* token_row,
                                  const float* gates, int64_t T, int k, int64_t H,
                                  fge_dtype out_dtype, void* out, void* workspace,
                                  size_t workspace_bytes, fge_stream_t stream);

/* gemm_w8a8 -- dense per-tensor W8A8 GEMM, the grouped kernel run with one expert
 * ("feat(qwen4_exp) ..." section "What this adds"; "Module fp8_ffi": activation scale
 * folded with the weight scale into one device scalar):  y = (sa * sw) * aq @ wq^T.
 * aq: [M, K] e4m3; sa, sw: device float scalars; wq: [N, K] e4m3; y: [M, N] in out_dtype.
 * At decode sizes (M <= 16; also in fge_gemm_w8a8_rows, fge_linear_w8a8* and the
 * allocation-free call) with K <= 2560, a weight-streaming kernel runs instead: each block
 * copies 16 weight rows into shared memory with bulk copies and eight warps split K with
 * warp-level e4m3 MMAs, the partial sums added in warp order (deterministic); it is launched
 * as a programmatic dependent of the kernel before it, so its weight stream overlaps that
 * kernel's end.  With a larger K the grouped kernel swaps its operands: the weights fill the
 * 128-row side of the MMA and the activations one 16-row tile, y written transposed back.
 * Workspace: FGE_OP_GROUPED_GEMM. */
fge_status fge_gemm_w8a8(const uint8_t* aq, const float* sa, int64_t M, int64_t K,
                         const uint8_t* wq, const float* sw, int64_t N, fge_dtype out_dtype,
                         void* y, void* workspace, size_t workspace_bytes,
                         fge_stream_t stream);

/* linear_w8a8 -- the whole dense projection in one call, as the "Module fp8_ffi" prefill
 * call does it: per-tensor amax, scale, e4m3 cast, then the W8A8 GEMM, one stream, no host
 * sync.  x_bf16: [M, K]; wq: [N, K] e4m3 with device scalar w_scale; y_bf16: [M, N].
 * Workspace: FGE_OP_LINEAR_W8A8 (holds the quantized activation and the scale block).  At
 * decode sizes (M <= 16) the GEMM is the decode kernel described at fge_gemm_w8a8 when
 * K <= 2560; with a larger K it splits K over several CTAs per 128-feature tile (as many as
 * fill the SMs in one wave, each at least two 128-wide K groups); the last of them to finish
 * adds the fp32 partials in split order, so the result does not depend on timing.  That needs
 * scratch for the partials: size the workspace with N
 * (fge_workspace_bytes(FGE_OP_LINEAR_W8A8, M, K, N)); a workspace sized without it runs the
 * GEMM unsplit. */
fge_status fge_linear_w8a8(const void* x_bf16, int64_t M, int64_t K, const uint8_t* wq,
                           const float* w_scale, int64_t N, void* y_bf16, void* workspace,
                           size_t workspace_bytes, fge_stream_t stream);

/* gemm_w8a8_rows -- the one-group W8A8 GEMM with one activation scale per row instead of one
 * per tensor (row-wise scales, "feat(qwen4_exp) ..." section "Limits"):
 *   y[m, n] = (sa[m] * sw) * sum_k aq[m, k] * wq[n, k].
 * aq: [M, K] e4m3; sa: [M] device floats; wq: [N, K] e4m3; sw: device float scalar;
 * y: [M, N] in out_dtype.  Workspace: FGE_OP_GROUPED_GEMM. */
fge_status fge_gemm_w8a8_rows(const uint8_t* aq, const float* sa, int64_t M, int64_t K,
                              const uint8_t* wq, const float* sw, int64_t N, fge_dtype out_dtype,
                              void* y, void* workspace, size_t workspace_bytes,
                              fge_stream_t stream);

/* linear_w8a8_rows -- the dense projection with row-wise activation scales in one call:
 * per-row amax and e4m3 cast (FGE_SCALE_PER_ROW), then fge_gemm_w8a8_rows.  Arguments as
 * fge_linear_w8a8.  Workspace: FGE_OP_LINEAR_W8A8_ROWS (quantized rows and their scales). */
fge_status fge_linear_w8a8_rows(const void* x_bf16, int64_t M, int64_t K, const uint8_t* wq,
                                const float* w_scale, int64_t N, void* y_bf16, void* workspace,
                                size_t workspace_bytes, fge_stream_t stream);

/* moe_layer_per_token_dispatch -- the baseline the grouped GEMM replaces ("FP8
 * grouped-expert prefill ..." section 1: one dispatch per routed token per layer): one CTA
 * per routed (token, slot) runs that expert's FFN on the token with int4 weights
 * dequantized in registers (q * per-group scale), bf16 activations in fp32, SwiGLU in fp32
 * and no activation quantization; then the combine.  Same routing as
 * fge_moe_layer_forward.  Weights in the canonical layout of fge_w4_prepack's input
 * (w_gu [E, 2I, H/2] with gate rows then up rows, s_gu [E, 2I, H/128], w_dn [E, H, I/2],
 * s_dn [E, H, I/128]).  Workspace: FGE_OP_DISPATCH_BASELINE with (T, H, I, E, k). */
fge_status fge_moe_layer_per_token_dispatch(const float* logits, const void* x_bf16, int64_t T,
                                            int64_t H, int E, int k, int64_t I,
                                            const uint8_t* w_gu, const float* s_gu,
                                            const uint8_t* w_dn, const float* s_dn,
                                            fge_dtype out_dtype, void* out, void* workspace,
                                            size_t workspace_bytes, fge_stream_t stream);

/* linear_w8a8_noalloc -- the same projection as fge_linear_w8a8 for callers that cannot
 * allocate device memory: hosts that own all device memory through their own pool and forbid
 * other allocations while serving, latency-critical paths where a cudaMalloc (which may
 * synchronise the device) is not allowed, and foreign-language hosts that can pass device
 * pointers for inputs and outputs but have no device allocator for a workspace.  The pages
 * have no counterpart of this call; it is an addition of this library.
 * Scratch: a fixed 16 MiB device array inside libfge (held by every GPU that loads the
 * library until the process exits), so M*K must not exceed 16 MiB - 256 bytes (for example
 * M <= 6553 at K = 2560); larger sizes return FGE_ERR_EXCEEDS_STATIC_SCRATCH.  The call
 * allocates nothing and needs no fge_init().  Its first call on a device looks up the
 * array's device address on that device (make that first call before any stream capture).
 * All calls share the one array and it keeps the last call's contents (the call clears what
 * must start at zero itself), so calls whose GPU work overlaps -- on different streams, or
 * from several host threads -- race on it; issue them on one stream or serialise them.
 * Arguments as fge_linear_w8a8: x_bf16 [M, K], wq [N, K] e4m3, w_scale device scalar,
 * y_bf16 [M, N].  M may be 0: nothing is read or written then (any pointer may be NULL).
 * A device-side problem of the last call (see fge_linear_w8a8_noalloc_status) leaves y
 * incomplete. */
fge_status fge_linear_w8a8_noalloc(const void* x_bf16, int64_t M, int64_t K, const uint8_t* wq,
                                   const float* w_scale, int64_t N, void* y_bf16,
                                   fge_stream_t stream);

/* linear_w8a8_noalloc_status -- the device status word of fge_linear_w8a8_noalloc's scratch:
 * FGE_ERR_DEVICE_TIMEOUT if a pipeline wait of its last call ran out of its time budget
 * (the output is then incomplete), else 0.  Waits for `stream`, then copies the word to *out
 * (host).  The word is shared by all calls on the current device, like the rest of the
 * scratch, and each call clears it before its kernels run.  Allocates nothing. */
fge_status fge_linear_w8a8_noalloc_status(fge_stream_t stream, int32_t* out);

/* moe_layer_forward -- one MoE FFN prefill layer in one call: top-k gate -> G128 quant ->
 * permute -> gate_up grouped GEMM with fused SwiGLU + requant -> down grouped GEMM ->
 * combine.  logits: [T, E] float; x_bf16: [T, H]; w_gu_dev / s_gu_dev: prepacked gate_up
 * bank ([E, 2I, H/2], interleaved) and scales; w_dn_dev / s_dn_dev: prepacked down bank
 * ([E, H, I/2]) and scales; out: [T, H] in out_dtype (expert outputs are kept in the same
 * dtype before the combine).  Workspace: FGE_OP_MOE_LAYER with (T, H, I, E, k). */
fge_status fge_moe_layer_forward(const float* logits, const void* x_bf16, int64_t T, int64_t H,
                                 int E, int k, int64_t I, const uint8_t* w_gu_dev,
                                 const float* s_gu_dev, const uint8_t* w_dn_dev,
                                 const float* s_dn_dev, fge_w4_format format,
                                 fge_dtype out_dtype, void* out, void* workspace,
                                 size_t workspace_bytes, fge_stream_t stream);

/* moe_layer_forward_fused_combine -- fge_moe_layer_forward with the combine folded into the
 * down GEMM's epilogue (the "fuse the edges" step of "FP8 grouped-expert prefill ...":
 * gate_up -> SwiGLU -> down -> combine with no combine kernel of its own).  Every routed
 * row's 128-column chunk is stored to the workspace's expert-output buffer as usual, then
 * counted per (token, chunk) with a device-scope atomic; the k-th arrival -- whichever slot
 * row lands last -- sums the token's k slot rows of that chunk, gate-weighted, in slot order
 * with float32 fmaf, exactly as the combine kernel does.  The output is therefore
 * bit-identical to fge_moe_layer_forward with out_dtype BF16, whatever order the tiles run
 * in: no float atomics.  out: [T, H] bf16.  Same arguments, workspace (FGE_OP_MOE_LAYER) and
 * errors as fge_moe_layer_forward; the arrival counters live in the workspace and are
 * cleared on the stream by each call. */
fge_status fge_moe_layer_forward_fused_combine(const float* logits, const void* x_bf16,
                                               int64_t T, int64_t H, int E, int k, int64_t I,
                                               const uint8_t* w_gu_dev, const float* s_gu_dev,
                                               const uint8_t* w_dn_dev, const float* s_dn_dev,
                                               fge_w4_format format, void* out, void* workspace,
                                               size_t workspace_bytes, fge_stream_t stream);

/* selftest_wait_timeout -- exercises the device failure path without faulting anything: a
 * one-warp kernel waits on an mbarrier that is never arrived on, with a budget of
 * budget_cycles (1 .. 2^32) SM clock cycles; the wait gives up, writes
 * FGE_ERR_DEVICE_TIMEOUT into the workspace status word and the kernel returns.  Read the
 * result with fge_read_device_status.  The pipeline kernels use the same bounded wait with
 * a budget of about one second. */
fge_status fge_selftest_wait_timeout(void* workspace, int64_t budget_cycles,
                                     fge_stream_t stream);

/* Glue of the stacked prefill (not page steps; RMSNorm, router, attention stand-in).
 * rmsnorm: out_bf16[t] = h[t] / sqrt(mean(h[t]^2) + eps), h float [T, H].
 * router_logits: logits[t, e] = sum_h xn[t, h] * w[e, h] in fp32 (lane l of a warp sums the
 *   products at h = 256 i + 8 l + c, c < 8, in order, then the warp adds its 32 lane sums);
 *   xn bf16 [T, H], w float [E, H]; H a multiple of 256, at most 7168; E at most 65536.
 * identity_attention: attn[t, h*128 + d] = v[t, (h / (n_heads / n_kv_heads))*128 + d];
 *   v bf16 [T, n_kv_heads*128], attn bf16 [T, n_heads*128].
 * residual_add: h[i] += y[i] for i < n, h float, y in y_dtype.
 * residual_rmsnorm: residual_add over [T, H] followed by rmsnorm of the updated h into
 *   out_bf16, in one pass per row; the same bits as the two calls in turn.  H % 8 == 0;
 *   h, y, out 16-byte aligned. */
fge_status fge_rmsnorm(const float* h, int64_t T, int64_t H, float eps, void* out_bf16,
                       fge_stream_t stream);
fge_status fge_router_logits(const void* xn_bf16, const float* w_router, int64_t T, int64_t H,
                             int E, float* logits, fge_stream_t stream);
fge_status fge_identity_attention(const void* v_bf16, int64_t T, int n_heads, int n_kv_heads,
                                  void* attn_bf16, fge_stream_t stream);
fge_status fge_residual_add(float* h, const void* y, fge_dtype y_dtype, int64_t n,
                            fge_stream_t stream);
fge_status fge_residual_rmsnorm(float* h, const void* y, fge_dtype y_dtype, int64_t T,
                                int64_t H, float eps, void* out_bf16, fge_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FGE_H_ */

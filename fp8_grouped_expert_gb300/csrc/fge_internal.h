// Internal declarations shared by the CUDA translation units of libfge (not installed).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/fge.h"

namespace fge {

constexpr int kGroup = 128;          // K-group of the per-group scales
constexpr int kMaxExperts = 512;     // grouped GEMM keeps offsets in shared memory
constexpr size_t kWsHeaderBytes = 256;

// Workspace header (first 256 bytes of every workspace):
//   int32  status       device-detected error code (0 = none)
//   uint32 amax_bits    per-tensor amax as float bits (non-negative floats order as uints)
//   float  scale        per-tensor activation scale written by the cast pass
struct WsHeader {
  int32_t status;
  uint32_t amax_bits;
  float scale;
  int32_t pad[61];
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Weight-bank formats of the int4 path (see include/fge.h).
enum BankFormat { kBankLut = 0, kBankSubnormal = 1 };

// Launchers (return a cudaError_t from the launch; argument checks happen in the API layer).
// status (may be null): a device status word that receives FGE_ERR_NONFINITE when an input
// value is an infinity or a NaN.
cudaError_t launch_quant_g128(const uint16_t* x, int64_t M, int64_t K, uint8_t* xq, float* xs,
                              int32_t* status, cudaStream_t s);
cudaError_t launch_quant_rows(const uint16_t* x, int64_t M, int64_t K, uint8_t* xq, float* xs,
                              int32_t* status, cudaStream_t s);
cudaError_t launch_mx_quant_e2m1(const uint16_t* x, int64_t M, int64_t K, uint8_t* xq,
                                 uint8_t* xs, cudaStream_t s);
// zero / n_zero: words the call also sets to 0 before it returns (the K-split counters of
// the GEMM that follows), or null / 0.
cudaError_t launch_quant_per_tensor(const uint16_t* x, int64_t M, int64_t K, uint8_t* xq,
                                    float* xs, WsHeader* hdr, cudaStream_t s,
                                    int32_t* zero = nullptr, int n_zero = 0);
cudaError_t launch_topk_gate(const float* logits, int64_t T, int E, int k, int32_t* ids,
                             float* gates, cudaStream_t s);
size_t permute_scratch_bytes(int64_t T, int E);
cudaError_t launch_permute(const int32_t* ids, int64_t T, int k, int E, const uint8_t* xq,
                           const float* xs, int64_t H, int32_t* offsets, int32_t* row_token,
                           int32_t* token_row, uint8_t* aq, float* as, void* scratch,
                           cudaStream_t s);
// Permutation with the G128 activation quantization fused into the row copy (x: bf16 [T, H]).
cudaError_t launch_permute_quant(const int32_t* ids, int64_t T, int k, int E,
                                 const uint16_t* x, int64_t H, int32_t* offsets,
                                 int32_t* row_token, int32_t* token_row, uint8_t* aq, float* as,
                                 void* scratch, int32_t* status, cudaStream_t s);
// status (may be null): with a status word, the bf16 case with k <= 8 and H % 2048 == 0
// runs the bulk-copy combine, whose bounded waits report there; otherwise the plain kernel.
cudaError_t launch_combine(const void* y, int y_f32, const int32_t* token_row,
                           const float* gates, int64_t T, int k, int64_t H, int out_f32,
                           void* out, cudaStream_t s, int32_t* status = nullptr);
cudaError_t launch_swiglu_quant(const float* c, int64_t R, int64_t I, uint8_t* hq, float* hs,
                                cudaStream_t s);
cudaError_t launch_w4_prepack(const uint8_t* w, const float* sw, int E, int64_t N, int64_t K,
                              int interleave, int fmt, uint8_t* w_dev, float* sw_dev,
                              cudaStream_t s);

// Grouped GEMM.  mode: 0 = int4 bank with per-group scales, 1 = e4m3 weights, per-tensor.
// The combine folded into the down GEMM's bf16 epilogue: every routed row's 128-column
// chunk counts its arrival per (token, chunk); the k-th arrival sums the token's k slot rows
// of that chunk, gate-weighted in slot order, into out.
struct FusedCombine {
  void* out;                  // [T, N] bf16, or null (no fused combine)
  const int32_t* row_token;   // [R] token of routed row r
  const int32_t* token_row;   // [T, k] routed row of (token, slot)
  const float* gates;         // [T, k]
  int32_t* count;             // [T, N/128] arrival counters, zero before the launch
  int k;
};

struct GroupedGemmArgs {
  const uint8_t* aq;        // [R, K] e4m3 codes (MXFP4: [R, K/2] packed E2M1 codes)
  const uint8_t* a_sf;      // MXFP4 activations: [R, K/32] UE8M0 block scales, else null
  const float* as;          // [R, K/128] (group mode)
  const float* sa_tensor;   // device scalar (per-tensor mode)
  const float* sa_rows;     // [R] per-row activation scales (per-tensor mode), or null
  const int32_t* offsets;   // [E+1]
  const int32_t* row_token; // gather mode: routed row r reads A row row_token[r] of aq
                            // ([rows_a, K], token order) and its scales; else null
  int64_t rows_a;           // gather mode: rows of aq / as
  const uint8_t* w;         // int4 bank [E, N, K/2] (prepacked) or e4m3 [N, K]
  const float* sw;          // [E, K/128, N] prepacked group scales, or device scalar
  int E;
  int64_t N, K, R;
  int bank_format;          // BankFormat (int4 mode)
  int per_tensor;           // 0: int4 + group scales; 1: e4m3 + per-tensor scales
  int epilogue;             // 0 store f32, 1 store bf16, 2 SwiGLU + e4m3 requant
  void* out;
  float* out_scales;
  int32_t* status;
  const FusedCombine* comb;  // down GEMM, bf16 store: the combine folded in (device memory,
                            // written by launch_combine_setup), or null
  // per-tensor (one-group) mode: K split over ksplit CTAs per output tile (0 or 1: none);
  // partials [tiles, ksplit, 128, BN] fp32 and split_count [tiles, epilogue warps] int32,
  // zero before the launch (the kernel leaves it zero again)
  int ksplit;
  float* partials;
  int32_t* split_count;
};
// K split of a per-tensor (one-group) W8A8 GEMM with M activation rows, N outputs and K
// inputs: how many CTAs share each output tile (1: no split), chosen to fill the SMs, and
// the scratch it needs (partials and counters, bytes).
int dense_ksplit(int64_t M, int64_t N, int64_t K);
// Scratch of a K split: the counters (*counter_bytes, first) then the partials.
size_t dense_split_bytes(int64_t M, int64_t N, int ksplit, size_t* counter_bytes);
// Zeroes the arrival counters (n of them) and writes c to dst (device memory) for the down
// GEMM's folded combine; one launch, stream-ordered.
cudaError_t launch_combine_setup(const FusedCombine& c, int64_t n, FusedCombine* dst,
                                 cudaStream_t s);
cudaError_t launch_grouped_gemm(const GroupedGemmArgs& a, cudaStream_t s, fge_status* st);
// launch_grouped_gemm, except that a one-group (dense W8A8) GEMM of at most 16 rows with
// N % 16 == 0, K % 64 == 0 and K <= 2560 runs the decode kernel of decode.cu instead
// (weights streamed once by bulk copies, warp-level MMAs; a programmatic dependent launch),
// which needs no K-split scratch.
cudaError_t launch_one_group_gemm(const GroupedGemmArgs& a, cudaStream_t s, fge_status* st);

cudaError_t launch_rmsnorm(const float* h, int64_t T, int64_t H, float eps, uint16_t* out,
                           cudaStream_t s);
cudaError_t launch_router(const uint16_t* xn, const float* wr, int64_t T, int64_t H, int E,
                          float* logits, cudaStream_t s);
cudaError_t launch_identity_attention(const uint16_t* v, int64_t T, int n_heads, int n_kv,
                                      uint16_t* attn, cudaStream_t s);
cudaError_t launch_residual_add(float* h, const void* y, int y_f32, int64_t n, cudaStream_t s);
cudaError_t launch_residual_rmsnorm(float* h, const void* y, int y_f32, int64_t T, int64_t H,
                                    float eps, uint16_t* out, cudaStream_t s);

cudaError_t launch_per_token_dispatch(const uint16_t* x, const int32_t* ids, int64_t T, int k,
                                      int64_t H, int64_t I, const uint8_t* w_gu,
                                      const float* s_gu, const uint8_t* w_dn, const float* s_dn,
                                      float* y, int32_t* token_row, cudaStream_t s);

// Host-side ledger of the library's calls (see fge_read_ledger in include/fge.h).
enum LedgerField {
  kLedCalls = 0,
  kLedRefused,
  kLedLayers,
  kLedGroupedGemms,
  kLedDenseDecodeTile,
  kLedDenseRowTile,
  kLedFields
};
void ledger_note(LedgerField f);

// SM count of the current device (cached per device; queried on first use, which allocates
// nothing, so calls that need no fge_init still size their grids from the real count).
int num_sms();

// Per-device set-up of one kernel, done once per (device, kernel) with that device current
// and guarded by a mutex: sets the dynamic shared-memory limit to smem_bytes and checks that
// the kernel was compiled with at least min_regs registers per thread (kernels that split
// their registers with setmaxnreg need the whole launch allotment).  False if either fails.
bool device_kernel_ready(int dev, const void* kernel, int smem_bytes, int min_regs);

}  // namespace fge

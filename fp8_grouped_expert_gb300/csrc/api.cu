// C ABI of libfge: argument validation, workspace carving and stream-ordered launches.
// No entry point allocates device memory or synchronises the host (except
// fge_read_device_status, which exists to read a result back).
#include <atomic>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "fge_internal.h"

namespace fge {

namespace {
constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices] = {0};
bool g_init[kMaxDevices] = {false};
std::mutex g_mu;

std::atomic<uint64_t> g_ledger[kLedFields];

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Every compute entry point starts here: counts the call, and the call as refused when the
// current device was not initialised.
inline fge_status cur_device_ok() {
  g_ledger[kLedCalls].fetch_add(1, std::memory_order_relaxed);
  int dev = 0;
  fge_status st = FGE_OK;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) st = FGE_ERR_CUDA;
  else if (!g_init[dev]) st = FGE_ERR_NOT_INITIALIZED;
  if (st != FGE_OK) g_ledger[kLedRefused].fetch_add(1, std::memory_order_relaxed);
  return st;
}

// Enqueue-side NVTX range (a profiler shows each layer stage by name; free without one).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

inline fge_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FGE_OK : FGE_ERR_CUDA; }

#define FGE_CHECK(expr)                 \
  do {                                  \
    const fge_status st_ = (expr);      \
    if (st_ != FGE_OK) return st_;      \
  } while (0)

#define FGE_REQUIRE(cond, code)                                           \
  do {                                                                    \
    if (!(cond)) {                                                        \
      fge::g_ledger[fge::kLedRefused].fetch_add(1, std::memory_order_relaxed); \
      return (code);                                                      \
    }                                                                     \
  } while (0)

// Workspace layout of a full MoE layer.
struct LayerWs {
  WsHeader* hdr;
  uint8_t* xq;
  float* xs;
  int32_t* ids;
  float* gates;
  void* perm;
  int32_t* offsets;
  int32_t* row_token;
  int32_t* token_row;
  uint8_t* aq;
  float* as;
  uint8_t* hq;
  float* hs;
  void* y;
  int32_t* comb_count;
  FusedCombine* comb_args;
  size_t bytes;
};

LayerWs carve_layer(void* base, int64_t T, int64_t H, int64_t I, int E, int k) {
  LayerWs w{};
  const int64_t R = T * k;
  size_t off = 0;
  auto take = [&](size_t n) {
    void* p = base ? static_cast<uint8_t*>(base) + off : nullptr;
    off += align_up(n, 256);
    return p;
  };
  w.hdr = static_cast<WsHeader*>(take(kWsHeaderBytes));
  w.xq = static_cast<uint8_t*>(take(T * H));
  w.xs = static_cast<float*>(take(T * (H / 128) * 4));
  w.ids = static_cast<int32_t*>(take(R * 4));
  w.gates = static_cast<float*>(take(R * 4));
  w.perm = take(permute_scratch_bytes(T, E));
  w.offsets = static_cast<int32_t*>(take((E + 1) * 4));
  w.row_token = static_cast<int32_t*>(take(R * 4));
  w.token_row = static_cast<int32_t*>(take(R * 4));
  w.aq = static_cast<uint8_t*>(take(R * H));
  w.as = static_cast<float*>(take(R * (H / 128) * 4));
  w.hq = static_cast<uint8_t*>(take(R * I));
  w.hs = static_cast<float*>(take(R * (I / 128) * 4));
  w.y = take(R * H * 4);
  w.comb_count = static_cast<int32_t*>(take(T * (H / 128) * 4));
  w.comb_args = static_cast<FusedCombine*>(take(sizeof(FusedCombine)));
  w.bytes = off;
  return w;
}

}  // namespace

void ledger_note(LedgerField f) { g_ledger[f].fetch_add(1, std::memory_order_relaxed); }

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_sms[dev] > 0) return g_sms[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 1;
  g_sms[dev] = n;
  return n;
}

namespace {
struct KernelSetup {
  int dev;
  const void* kernel;
  bool ok;
};
constexpr int kMaxKernelSetups = 512;
std::mutex g_kernel_mu;
KernelSetup g_kernel_setup[kMaxKernelSetups];
int g_kernel_setups = 0;
}  // namespace

bool device_kernel_ready(int dev, const void* kernel, int smem_bytes, int min_regs) {
  std::lock_guard<std::mutex> lock(g_kernel_mu);
  for (int i = 0; i < g_kernel_setups; ++i)
    if (g_kernel_setup[i].dev == dev && g_kernel_setup[i].kernel == kernel)
      return g_kernel_setup[i].ok;
  bool ok = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem_bytes) == cudaSuccess;
  cudaFuncAttributes attr;
  if (ok) ok = cudaFuncGetAttributes(&attr, kernel) == cudaSuccess && attr.numRegs >= min_regs;
  if (g_kernel_setups < kMaxKernelSetups)
    g_kernel_setup[g_kernel_setups++] = KernelSetup{dev, kernel, ok};
  return ok;
}

}  // namespace fge

using namespace fge;

extern "C" {

int fge_version(void) { return 100; }

const char* fge_status_string(fge_status s) {
  switch (s) {
    case FGE_OK: return "ok";
    case FGE_ERR_INVALID_ARG: return "invalid argument";
    case FGE_ERR_BAD_SHAPE: return "bad shape";
    case FGE_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case FGE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case FGE_ERR_UNSUPPORTED_DEVICE: return "unsupported device or kernel resources";
    case FGE_ERR_CUDA: return "CUDA error";
    case FGE_ERR_DEVICE_TIMEOUT: return "device pipeline wait timed out";
    case FGE_ERR_NOT_INITIALIZED: return "fge_init not called for this device";
    case FGE_ERR_EXCEEDS_STATIC_SCRATCH: return "size exceeds the fixed scratch of the no-alloc call";
    case FGE_ERR_NONFINITE: return "an activation to quantize is an infinity or a NaN";
  }
  return "unknown status";
}

fge_status fge_init(int device) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (device < 0 || device >= kMaxDevices) return FGE_ERR_INVALID_ARG;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return FGE_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return FGE_ERR_UNSUPPORTED_DEVICE;
  g_sms[device] = prop.multiProcessorCount;
  g_init[device] = true;
  return FGE_OK;
}

size_t fge_workspace_bytes(fge_op op, int64_t a, int64_t b, int64_t c, int E, int k) {
  switch (op) {
    case FGE_OP_QUANT_PER_TENSOR: return kWsHeaderBytes;
    case FGE_OP_PERMUTE: return kWsHeaderBytes + permute_scratch_bytes(a, E);
    case FGE_OP_GROUPED_GEMM: return kWsHeaderBytes;
    case FGE_OP_LINEAR_W8A8: {
      // with N (c > 0): also the scratch of a K split at small M
      size_t counters = 0;
      const size_t split = c > 0 ? dense_split_bytes(a, c, dense_ksplit(a, c, b), &counters) : 0;
      return kWsHeaderBytes + align_up(static_cast<size_t>(a * b), 256) + split;
    }
    case FGE_OP_MOE_LAYER: return carve_layer(nullptr, a, b, c, E, k).bytes;
    case FGE_OP_LINEAR_W8A8_ROWS:
      return kWsHeaderBytes + align_up(static_cast<size_t>(a * b), 256) +
             align_up(static_cast<size_t>(a) * 4, 256);
    case FGE_OP_DISPATCH_BASELINE: {
      const size_t r = static_cast<size_t>(a) * k;
      return kWsHeaderBytes + 3 * align_up(r * 4, 256) + align_up(r * b * 4, 256);
    }
  }
  return 0;
}

fge_status fge_read_ledger(fge_ledger* out) {
  if (!out) return FGE_ERR_INVALID_ARG;
  out->calls = g_ledger[kLedCalls].load();
  out->refused = g_ledger[kLedRefused].load();
  out->layers = g_ledger[kLedLayers].load();
  out->grouped_gemms = g_ledger[kLedGroupedGemms].load();
  out->dense_decode_tile = g_ledger[kLedDenseDecodeTile].load();
  out->dense_row_tile = g_ledger[kLedDenseRowTile].load();
  return FGE_OK;
}

fge_status fge_reset_ledger(void) {
  for (int i = 0; i < kLedFields; ++i) g_ledger[i].store(0);
  return FGE_OK;
}

fge_status fge_clear_device_status(void* ws, fge_stream_t stream) {
  FGE_REQUIRE(ws, FGE_ERR_INVALID_ARG);
  return from_cuda(cudaMemsetAsync(ws, 0, sizeof(int32_t), stream));
}

fge_status fge_read_device_status(const void* ws, fge_stream_t stream, int32_t* out) {
  FGE_REQUIRE(ws && out, FGE_ERR_INVALID_ARG);
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FGE_ERR_CUDA;
  return from_cuda(cudaMemcpy(out, ws, sizeof(int32_t), cudaMemcpyDeviceToHost));
}

fge_status fge_fp8_quant_act(const void* x, int64_t M, int64_t K, fge_scale_mode mode,
                             uint8_t* xq, float* xs, void* ws, size_t ws_bytes,
                             fge_stream_t stream) {
  FGE_CHECK(cur_device_ok());
  FGE_REQUIRE(M >= 0 && K > 0 && K % 128 == 0, FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(x && xq && xs, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(al16(x) && al16(xq), FGE_ERR_MISALIGNED);
  // G128 and per-row take no workspace; with one (>= its 256-byte header) a non-finite input
  // is reported in its status word
  int32_t* status = (ws && ws_bytes >= kWsHeaderBytes && al16(ws))
                        ? &static_cast<WsHeader*>(ws)->status : nullptr;
  if (mode == FGE_SCALE_PER_TOKEN_G128) {
    return from_cuda(launch_quant_g128(static_cast<const uint16_t*>(x), M, K, xq, xs, status,
                                       stream));
  }
  if (mode == FGE_SCALE_PER_ROW) {
    return from_cuda(launch_quant_rows(static_cast<const uint16_t*>(x), M, K, xq, xs, status,
                                       stream));
  }
  FGE_REQUIRE(mode == FGE_SCALE_PER_TENSOR, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(ws, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(al16(ws), FGE_ERR_MISALIGNED);
  FGE_REQUIRE(ws_bytes >= kWsHeaderBytes, FGE_ERR_WORKSPACE_TOO_SMALL);
  return from_cuda(launch_quant_per_tensor(static_cast<const uint16_t*>(x), M, K, xq, xs,
                                           static_cast<WsHeader*>(ws), stream));
}

fge_status fge_mx_quant_e2m1(const void* x, int64_t M, int64_t K, uint8_t* xq, uint8_t* xs,
                             fge_stream_t stream) {
  FGE_CHECK(cur_device_ok());
  FGE_REQUIRE(M >= 0 && K > 0 && K % 32 == 0, FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(x && xq && xs, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(al16(x) && al16(xq), FGE_ERR_MISALIGNED);
  return from_cuda(launch_mx_quant_e2m1(static_cast<const uint16_t*>(x), M, K, xq, xs, stream));
}

fge_status fge_moe_topk_gate(const float* logits, int64_t T, int E, int k, int32_t* ids,
                             float* gates, fge_stream_t stream) {
  FGE_CHECK(cur_device_ok());
  FGE_REQUIRE(logits && ids && gates, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(T >= 0 && E >= 1 && E <= 1024 && k >= 1 && k <= E && k <= 32, FGE_ERR_BAD_SHAPE);
  return from_cuda(launch_topk_gate(logits, T, E, k, ids, gates, stream));
}

fge_status fge_moe_permute(const int32_t* ids, int64_t T, int k, int E, const uint8_t* xq,
                           const float* xs, int64_t H, int32_t* offsets, int32_t* row_token,
                           int32_t* token_row, uint8_t* aq, float* as, void* ws,
                           size_t ws_bytes, fge_stream_t stream) {
  FGE_CHECK(cur_device_ok());
  // aq and as both null: index-only (offsets, row_token, token_row), no row copy
  FGE_REQUIRE(ids && offsets && row_token && token_row && ws && ((aq == nullptr) == (as == nullptr)),
              FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(aq == nullptr || (xq && xs), FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(T >= 0 && E >= 1 && E <= 1024 && k >= 1 && k <= E && k <= 32, FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(H > 0 && H % 128 == 0 && T * k < (1LL << 31), FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(aq == nullptr || (al16(xq) && al16(aq)), FGE_ERR_MISALIGNED);
  FGE_REQUIRE(al16(ws), FGE_ERR_MISALIGNED);
  FGE_REQUIRE(ws_bytes >= fge_workspace_bytes(FGE_OP_PERMUTE, T, H, 0, E, k),
              FGE_ERR_WORKSPACE_TOO_SMALL);
  return from_cuda(launch_permute(ids, T, k, E, xq, xs, H, offsets, row_token, token_row, aq, as,
                                  static_cast<uint8_t*>(ws) + kWsHeaderBytes, stream));
}

fge_status fge_moe_permute_quant(const int32_t* ids, int64_t T, int k, int E, const void* x,
                                 int64_t H, int32_t* offsets, int32_t* row_token,
                                 int32_t* token_row, uint8_t* aq, float* as, void* ws,
                                 size_t ws_bytes, fge_stream_t stream) {
  FGE_CHECK(cur_device_ok());
  FGE_REQUIRE(ids && x && offsets && row_token && token_row && aq && as && ws,
              FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(T >= 0 && E >= 1 && E <= 1024 && k >= 1 && k <= E && k <= 32, FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(H > 0 && H % 128 == 0 && T * k < (1LL << 31), FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(al16(x) && al16(aq) && al16(ws), FGE_ERR_MISALIGNED);
  FGE_REQUIRE(ws_bytes >= fge_workspace_bytes(FGE_OP_PERMUTE, T, H, 0, E, k),
              FGE_ERR_WORKSPACE_TOO_SMALL);
  return from_cuda(launch_permute_quant(ids, T, k, E, static_cast<const uint16_t*>(x), H, offsets,
                                        row_token, token_row, aq, as,
                                        static_cast<uint8_t*>(ws) + kWsHeaderBytes,
                                        &static_cast<WsHeader*>(ws)->status, stream));
}

fge_status fge_w4_prepack(const uint8_t* w, const float* w_scale, int E, int64_t N, int64_t K,
                          int gate_up_interleave, fge_w4_format format, uint8_t* w_dev,
                          float* w_scale_dev, fge_stream_t stream) {
  FGE_CHECK(cur_device_ok());
  FGE_REQUIRE(w && w_scale && w_dev && w_scale_dev, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(format == FGE_W4_LUT || format == FGE_W4_SUBNORMAL, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(E >= 1 && N > 0 && N % 128 == 0 && K > 0 && K % 128 == 0, FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(!gate_up_interleave || N % 256 == 0, FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(al16(w) && al16(w_dev) && al16(w_scale_dev), FGE_ERR_MISALIGNED);
  return from_cuda(launch_w4_prepack(w, w_scale, E, N, K, gate_up_interleave ? 1 : 0,
                                     static_cast<int>(format), w_dev, w_scale_dev, stream));
}

static fge_status grouped_common(const uint8_t* aq, const float* as, const int32_t* offsets,
                                 int64_t R, const uint8_t* w, const float* sw, int E, int64_t N,
                                 int64_t K, int format, int per_tensor, const float* sa_t,
                                 int epilogue, void* out, float* out_scales, void* ws,
                                 size_t ws_bytes, fge_stream_t stream,
                                 const float* sa_rows = nullptr,
                                 const int32_t* row_token = nullptr, int64_t rows_a = 0,
                                 const FusedCombine* comb = nullptr) {
  FGE_REQUIRE(R >= 0 && R < (1LL << 31) && N > 0 && N % 128 == 0 && N < (1LL << 24) && K > 0 &&
                  K % 128 == 0 && K < (1LL << 24),
              FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(E >= 1 && E <= kMaxExperts, FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(ws && out && aq && w && sw, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(al16(aq) && al16(w) && al16(out) && al16(ws) && (per_tensor || al16(sw)),
              FGE_ERR_MISALIGNED);
  FGE_REQUIRE(ws_bytes >= kWsHeaderBytes, FGE_ERR_WORKSPACE_TOO_SMALL);
  if (R == 0) return FGE_OK;
  GroupedGemmArgs a{};
  a.aq = aq;
  a.as = as;
  a.sa_tensor = sa_t;
  a.sa_rows = sa_rows;
  a.row_token = row_token;
  a.rows_a = rows_a;
  a.offsets = offsets;
  a.w = w;
  a.sw = sw;
  a.E = E;
  a.N = N;
  a.K = K;
  a.R = R;
  a.bank_format = format;
  a.per_tensor = per_tensor;
  a.epilogue = epilogue;
  a.out = out;
  a.out_scales = out_scales;
  a.status = &static_cast<WsHeader*>(ws)->status;
  a.comb = comb;
  fge_status st = FGE_OK;
  const cudaError_t e = launch_one_group_gemm(a, stream, &st);
  if (e != cudaSuccess) return FGE_ERR_CUDA;
  return st;
}

fge_status fge_grouped_gemm_w4a8(const uint8_t* aq, const float* as, const int32_t* offsets,
                                 int64_t R, const uint8_t* w_dev, const float* w_scale_dev,
                                 int E, int64_t N, int64_t K, fge_w4_format format,
                                 fge_epilogue epilogue, fge_dtype out_dtype, void* out,
                                 float* out_scales, void* ws, size_t ws_bytes,
                                 fge_stream_t stream) {
  FGE_CHECK(cur_device_ok());
  FGE_REQUIRE(as && offsets, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(format == FGE_W4_LUT || format == FGE_W4_SUBNORMAL, FGE_ERR_INVALID_ARG);
  int epi;
  if (epilogue == FGE_EPI_SWIGLU_REQUANT) {
    FGE_REQUIRE(out_scales, FGE_ERR_INVALID_ARG);
    FGE_REQUIRE(N % 256 == 0, FGE_ERR_BAD_SHAPE);
    epi = 2;
  } else {
    FGE_REQUIRE(epilogue == FGE_EPI_STORE, FGE_ERR_INVALID_ARG);
    FGE_REQUIRE(out_dtype == FGE_DTYPE_BF16 || out_dtype == FGE_DTYPE_F32, FGE_ERR_INVALID_ARG);
    epi = out_dtype == FGE_DTYPE_F32 ? 0 : 1;
  }
  return grouped_common(aq, as, offsets, R, w_dev, w_scale_dev, E, N, K, format, 0, nullptr, epi,
                        out, out_scales, ws, ws_bytes, stream);
}

fge_status fge_grouped_gemm_mxf4_w4(const uint8_t* a_codes, const uint8_t* a_scales,
                                   const int32_t* offsets, int64_t R, const uint8_t* w_dev,
                                   const float* w_scale_dev, int E, int64_t N, int64_t K,
                                   fge_w4_format format, fge_dtype out_dtype, void* out,
                                   void* ws, size_t ws_bytes, fge_stream_t stream) {
  FGE_CHECK(cur_device_ok());
  FGE_REQUIRE(a_codes && a_scales && offsets && w_dev && w_scale_dev && out && ws,
              FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(format == FGE_W4_SUBNORMAL, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(out_dtype == FGE_DTYPE_BF16 || out_dtype == FGE_DTYPE_F32, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(R >= 0 && R < (1LL << 31) && N > 0 && N % 128 == 0 && N < (1LL << 24) && K > 0 &&
                  K % 128 == 0 && K < (1LL << 24),
              FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(E >= 1 && E <= kMaxExperts, FGE_ERR_BAD_SHAPE);
  // the padded-E2M1 TMA wants a 32-byte aligned base (its row stride K/2 is a multiple of 64)
  FGE_REQUIRE((reinterpret_cast<uintptr_t>(a_codes) & 31u) == 0 && al16(a_scales) &&
                  al16(w_dev) && al16(w_scale_dev) && al16(out) && al16(ws),
              FGE_ERR_MISALIGNED);
  FGE_REQUIRE(ws_bytes >= kWsHeaderBytes, FGE_ERR_WORKSPACE_TOO_SMALL);
  if (R == 0) return FGE_OK;
  GroupedGemmArgs a{};
  a.aq = a_codes;
  a.a_sf = a_scales;
  a.offsets = offsets;
  a.w = w_dev;
  a.sw = w_scale_dev;
  a.E = E;
  a.N = N;
  a.K = K;
  a.R = R;
  a.bank_format = format;
  a.epilogue = out_dtype == FGE_DTYPE_F32 ? 0 : 1;
  a.out = out;
  a.status = &static_cast<WsHeader*>(ws)->status;
  fge_status st = FGE_OK;
  if (launch_one_group_gemm(a, static_cast<cudaStream_t>(stream), &st) != cudaSuccess)
    return FGE_ERR_CUDA;
  return st;
}

fge_status fge_grouped_gemm_w4a8_gather(const uint8_t* xq, const float* xs, int64_t T,
                                        const int32_t* row_token, const int32_t* offsets,
                                        int64_t R, const uint8_t* w_dev,
                                        const float* w_scale_dev, int E, int64_t N, int64_t K,
                                        fge_w4_format format, fge_epilogue epilogue,
                                        fge_dtype out_dtype, void* out, float* out_scales,
                                        void* ws, size_t ws_bytes, fge_stream_t stream) {
  FGE_CHECK(cur_device_ok());
  FGE_REQUIRE(xs && offsets && row_token, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(T > 0 && T < (1LL << 31), FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(format == FGE_W4_LUT || format == FGE_W4_SUBNORMAL, FGE_ERR_INVALID_ARG);
  int epi;
  if (epilogue == FGE_EPI_SWIGLU_REQUANT) {
    FGE_REQUIRE(out_scales, FGE_ERR_INVALID_ARG);
    FGE_REQUIRE(N % 256 == 0, FGE_ERR_BAD_SHAPE);
    epi = 2;
  } else {
    FGE_REQUIRE(epilogue == FGE_EPI_STORE, FGE_ERR_INVALID_ARG);
    FGE_REQUIRE(out_dtype == FGE_DTYPE_BF16 || out_dtype == FGE_DTYPE_F32, FGE_ERR_INVALID_ARG);
    epi = out_dtype == FGE_DTYPE_F32 ? 0 : 1;
  }
  return grouped_common(xq, xs, offsets, R, w_dev, w_scale_dev, E, N, K, format, 0, nullptr, epi,
                        out, out_scales, ws, ws_bytes, stream, nullptr, row_token, T);
}

fge_status fge_swiglu_quant(const float* c, int64_t R, int64_t I, uint8_t* hq, float* hs,
                            fge_stream_t stream) {
  FGE_CHECK(cur_device_ok());
  FGE_REQUIRE(c && hq && hs, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(R >= 0 && I > 0 && I % 128 == 0, FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(al16(c) && al16(hq), FGE_ERR_MISALIGNED);
  return from_cuda(launch_swiglu_quant(c, R, I, hq, hs, stream));
}

fge_status fge_moe_combine(const void* y, fge_dtype y_dtype, const int32_t* token_row,
                           const float* gates, int64_t T, int k, int64_t H,
                           fge_dtype out_dtype, void* out, fge_stream_t stream) {
  FGE_CHECK(cur_device_ok());
  FGE_REQUIRE(y && token_row && gates && out, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE((y_dtype == FGE_DTYPE_BF16 || y_dtype == FGE_DTYPE_F32) &&
                  (out_dtype == FGE_DTYPE_BF16 || out_dtype == FGE_DTYPE_F32),
              FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(T >= 0 && k >= 1 && k <= 32 && H > 0 && H % 128 == 0, FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(al16(y) && al16(out), FGE_ERR_MISALIGNED);
  return from_cuda(launch_combine(y, y_dtype == FGE_DTYPE_F32, token_row, gates, T, k, H,
                                  out_dtype == FGE_DTYPE_F32, out, stream));
}

fge_status fge_moe_combine_staged(const void* y_bf16, const int32_t* token_row,
                                  const float* gates, int64_t T, int k, int64_t H,
                                  fge_dtype out_dtype, void* out, void* ws, size_t ws_bytes,
                                  fge_stream_t stream) {
  FGE_CHECK(cur_device_ok());
  FGE_REQUIRE(y_bf16 && token_row && gates && out && ws, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(out_dtype == FGE_DTYPE_BF16 || out_dtype == FGE_DTYPE_F32, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(T >= 0 && k >= 1 && k <= 8 && H > 0 && H % 2048 == 0, FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(al16(y_bf16) && al16(out) && al16(ws), FGE_ERR_MISALIGNED);
  FGE_REQUIRE(ws_bytes >= sizeof(WsHeader), FGE_ERR_WORKSPACE_TOO_SMALL);
  return from_cuda(launch_combine(y_bf16, 0, token_row, gates, T, k, H,
                                  out_dtype == FGE_DTYPE_F32, out, stream,
                                  &static_cast<WsHeader*>(ws)->status));
}

fge_status fge_gemm_w8a8(const uint8_t* aq, const float* sa, int64_t M, int64_t K,
                         const uint8_t* wq, const float* sw, int64_t N, fge_dtype out_dtype,
                         void* y, void* ws, size_t ws_bytes, fge_stream_t stream) {
  FGE_CHECK(cur_device_ok());
  FGE_REQUIRE(sa, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(out_dtype == FGE_DTYPE_BF16 || out_dtype == FGE_DTYPE_F32, FGE_ERR_INVALID_ARG);
  return grouped_common(aq, nullptr, nullptr, M, wq, sw, 1, N, K, 0, 1, sa,
                        out_dtype == FGE_DTYPE_F32 ? 0 : 1, y, nullptr, ws, ws_bytes, stream);
}

// The per-tensor W8A8 GEMM of the dense projection, optionally with K split over ks CTAs
// per output tile (partials and zeroed counters in the caller's scratch).
static fge_status dense_gemm(const uint8_t* xq, int64_t M, const uint8_t* wq,
                             const float* w_scale, int64_t N, int64_t K, const float* sa,
                             void* y, void* ws, size_t ws_bytes, fge_stream_t stream, int ks,
                             float* partials, int32_t* counters) {
  FGE_REQUIRE(M >= 0 && M < (1LL << 31) && N > 0 && N % 128 == 0 && N < (1LL << 24) && K > 0 &&
                  K % 128 == 0 && K < (1LL << 24),
              FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(al16(xq) && al16(wq) && al16(y) && al16(ws), FGE_ERR_MISALIGNED);
  FGE_REQUIRE(ws_bytes >= kWsHeaderBytes, FGE_ERR_WORKSPACE_TOO_SMALL);
  if (M == 0) return FGE_OK;
  GroupedGemmArgs a{};
  a.aq = xq;
  a.sa_tensor = sa;
  a.w = wq;
  a.sw = w_scale;
  a.E = 1;
  a.N = N;
  a.K = K;
  a.R = M;
  a.per_tensor = 1;
  a.epilogue = 1;
  a.out = y;
  a.status = &static_cast<WsHeader*>(ws)->status;
  a.ksplit = ks;
  a.partials = partials;
  a.split_count = counters;
  fge_status st = FGE_OK;
  if (launch_one_group_gemm(a, static_cast<cudaStream_t>(stream), &st) != cudaSuccess)
    return FGE_ERR_CUDA;
  return st;
}

fge_status fge_linear_w8a8(const void* x, int64_t M, int64_t K, const uint8_t* wq,
                           const float* w_scale, int64_t N, void* y, void* ws, size_t ws_bytes,
                           fge_stream_t stream) {
  FGE_CHECK(cur_device_ok());
  FGE_REQUIRE(x && wq && w_scale && y && ws, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(M >= 0 && K > 0 && K % 128 == 0 && N > 0 && N % 128 == 0, FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(al16(x) && al16(ws), FGE_ERR_MISALIGNED);
  FGE_REQUIRE(ws_bytes >= fge_workspace_bytes(FGE_OP_LINEAR_W8A8, M, K, 0, 0, 0),
              FGE_ERR_WORKSPACE_TOO_SMALL);
  NvtxRange range("fge.linear_w8a8");
  WsHeader* hdr = static_cast<WsHeader*>(ws);
  // layout: header | K-split counters | xq | K-split partials; the split (small M: several
  // CTAs per output tile) is used when the workspace was sized with N
  int ks = dense_ksplit(M, N, K);
  size_t counter_bytes = 0;
  size_t split_bytes = dense_split_bytes(M, N, ks, &counter_bytes);
  const size_t xq_bytes = align_up(static_cast<size_t>(M * K), 256);
  if (ws_bytes < kWsHeaderBytes + xq_bytes + split_bytes) {
    ks = 1;
    counter_bytes = split_bytes = 0;
  }
  uint8_t* base = static_cast<uint8_t*>(ws) + kWsHeaderBytes;
  int32_t* counters = reinterpret_cast<int32_t*>(base);
  uint8_t* xq = base + counter_bytes;
  float* partials = reinterpret_cast<float*>(xq + xq_bytes);
  FGE_CHECK(from_cuda(launch_quant_per_tensor(static_cast<const uint16_t*>(x), M, K, xq,
                                              &hdr->scale, hdr, stream, counters,
                                              static_cast<int>(counter_bytes / 4))));
  return dense_gemm(xq, M, wq, w_scale, N, K, &hdr->scale, y, ws, ws_bytes, stream, ks,
                    partials, counters);
}

fge_status fge_gemm_w8a8_rows(const uint8_t* aq, const float* sa, int64_t M, int64_t K,
                              const uint8_t* wq, const float* sw, int64_t N, fge_dtype out_dtype,
                              void* y, void* ws, size_t ws_bytes, fge_stream_t stream) {
  FGE_CHECK(cur_device_ok());
  FGE_REQUIRE(sa, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(out_dtype == FGE_DTYPE_BF16 || out_dtype == FGE_DTYPE_F32, FGE_ERR_INVALID_ARG);
  return grouped_common(aq, nullptr, nullptr, M, wq, sw, 1, N, K, 0, 1, nullptr,
                        out_dtype == FGE_DTYPE_F32 ? 0 : 1, y, nullptr, ws, ws_bytes, stream, sa);
}

fge_status fge_linear_w8a8_rows(const void* x, int64_t M, int64_t K, const uint8_t* wq,
                                const float* w_scale, int64_t N, void* y, void* ws,
                                size_t ws_bytes, fge_stream_t stream) {
  FGE_CHECK(cur_device_ok());
  FGE_REQUIRE(x && wq && w_scale && y && ws, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(M >= 0 && K > 0 && K % 128 == 0 && N > 0 && N % 128 == 0, FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(al16(x) && al16(ws), FGE_ERR_MISALIGNED);
  FGE_REQUIRE(ws_bytes >= fge_workspace_bytes(FGE_OP_LINEAR_W8A8_ROWS, M, K, 0, 0, 0),
              FGE_ERR_WORKSPACE_TOO_SMALL);
  uint8_t* xq = static_cast<uint8_t*>(ws) + kWsHeaderBytes;
  float* xs = reinterpret_cast<float*>(xq + align_up(static_cast<size_t>(M * K), 256));
  FGE_CHECK(from_cuda(launch_quant_rows(static_cast<const uint16_t*>(x), M, K, xq, xs,
                                        &static_cast<WsHeader*>(ws)->status, stream)));
  return grouped_common(xq, nullptr, nullptr, M, wq, w_scale, 1, N, K, 0, 1, nullptr, 1, y,
                        nullptr, ws, ws_bytes, stream, xs);
}

// One MoE FFN layer: top-k gate, permutation with the G128 quantization in the row copy,
// gate_up GEMM with the fused SwiGLU requant, down GEMM, combine.  fused_combine: the
// combine runs inside the down GEMM's epilogue (bf16 output only) instead of as a kernel.
static fge_status layer_forward(const float* logits, const void* x, int64_t T, int64_t H, int E,
                                int k, int64_t I, const uint8_t* w_gu, const float* s_gu,
                                const uint8_t* w_dn, const float* s_dn, fge_w4_format format,
                                fge_dtype out_dtype, void* out, void* ws, size_t ws_bytes,
                                fge_stream_t stream, bool fused_combine) {
  FGE_CHECK(cur_device_ok());
  FGE_REQUIRE(logits && x && w_gu && s_gu && w_dn && s_dn && out && ws, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(format == FGE_W4_LUT || format == FGE_W4_SUBNORMAL, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(out_dtype == FGE_DTYPE_BF16 || (out_dtype == FGE_DTYPE_F32 && !fused_combine),
              FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(T >= 0 && H > 0 && H % 128 == 0 && I > 0 && I % 128 == 0, FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(E >= 1 && E <= kMaxExperts && k >= 1 && k <= E && k <= 32, FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(T * k < (1LL << 31) && (2 * I) % 256 == 0, FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(al16(x) && al16(ws) && al16(out) && al16(w_gu) && al16(w_dn) && al16(s_gu) &&
                  al16(s_dn),
              FGE_ERR_MISALIGNED);
  const LayerWs w = carve_layer(ws, T, H, I, E, k);
  FGE_REQUIRE(ws_bytes >= w.bytes, FGE_ERR_WORKSPACE_TOO_SMALL);
  if (T == 0) return FGE_OK;
  const int64_t R = T * k;
  const int out_f32 = out_dtype == FGE_DTYPE_F32;
  NvtxRange layer_range("fge.moe_layer");
  {
    NvtxRange r("fge.topk_gate");
    FGE_CHECK(from_cuda(launch_topk_gate(logits, T, E, k, w.ids, w.gates, stream)));
  }

  // The permuted copy of the activation rows plus a tiled A load beats gathering the rows
  // in the GEMM (fge_grouped_gemm_w4a8_gather): 32 four-row TMA gathers per K group cost
  // more than the copy kernel saves.
  // the G128 activation quantization runs inside the permutation's row copy: each token's
  // bf16 row is read once and its codes and scales go straight to its k expert rows
  {
    NvtxRange r("fge.permute_quant");
    FGE_CHECK(from_cuda(launch_permute_quant(w.ids, T, k, E, static_cast<const uint16_t*>(x), H,
                                             w.offsets, w.row_token, w.token_row, w.aq, w.as,
                                             w.perm, &w.hdr->status, stream)));
  }
  {
    NvtxRange r("fge.gate_up_gemm");
    FGE_CHECK(grouped_common(w.aq, w.as, w.offsets, R, w_gu, s_gu, E, 2 * I, H, format, 0,
                             nullptr, 2, w.hq, w.hs, ws, ws_bytes, stream));
  }
  if (fused_combine) {
    NvtxRange r("fge.down_gemm_combine");
    const FusedCombine comb{out, w.row_token, w.token_row, w.gates, w.comb_count, k};
    FGE_CHECK(from_cuda(launch_combine_setup(comb, T * (H / 128), w.comb_args, stream)));
    const fge_status st = grouped_common(w.hq, w.hs, w.offsets, R, w_dn, s_dn, E, H, I, format,
                                         0, nullptr, 1, w.y, nullptr, ws, ws_bytes, stream,
                                         nullptr, nullptr, 0, w.comb_args);
    if (st == FGE_OK) ledger_note(kLedLayers);
    return st;
  }
  {
    NvtxRange r("fge.down_gemm");
    FGE_CHECK(grouped_common(w.hq, w.hs, w.offsets, R, w_dn, s_dn, E, H, I, format, 0, nullptr,
                             out_f32 ? 0 : 1, w.y, nullptr, ws, ws_bytes, stream));
  }
  NvtxRange r("fge.combine");
  const fge_status st = from_cuda(launch_combine(w.y, out_f32, w.token_row, w.gates, T, k, H,
                                                 out_f32, out, stream, &w.hdr->status));
  if (st == FGE_OK) ledger_note(kLedLayers);
  return st;
}

fge_status fge_moe_layer_forward(const float* logits, const void* x, int64_t T, int64_t H, int E,
                                 int k, int64_t I, const uint8_t* w_gu, const float* s_gu,
                                 const uint8_t* w_dn, const float* s_dn, fge_w4_format format,
                                 fge_dtype out_dtype, void* out, void* ws, size_t ws_bytes,
                                 fge_stream_t stream) {
  return layer_forward(logits, x, T, H, E, k, I, w_gu, s_gu, w_dn, s_dn, format, out_dtype, out,
                       ws, ws_bytes, stream, false);
}

fge_status fge_moe_layer_forward_fused_combine(const float* logits, const void* x, int64_t T,
                                               int64_t H, int E, int k, int64_t I,
                                               const uint8_t* w_gu, const float* s_gu,
                                               const uint8_t* w_dn, const float* s_dn,
                                               fge_w4_format format, void* out, void* ws,
                                               size_t ws_bytes, fge_stream_t stream) {
  return layer_forward(logits, x, T, H, E, k, I, w_gu, s_gu, w_dn, s_dn, format, FGE_DTYPE_BF16,
                       out, ws, ws_bytes, stream, true);
}

fge_status fge_moe_layer_per_token_dispatch(const float* logits, const void* x, int64_t T,
                                            int64_t H, int E, int k, int64_t I,
                                            const uint8_t* w_gu, const float* s_gu,
                                            const uint8_t* w_dn, const float* s_dn,
                                            fge_dtype out_dtype, void* out, void* ws,
                                            size_t ws_bytes, fge_stream_t stream) {
  FGE_CHECK(cur_device_ok());
  FGE_REQUIRE(logits && x && w_gu && s_gu && w_dn && s_dn && out && ws, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(out_dtype == FGE_DTYPE_BF16 || out_dtype == FGE_DTYPE_F32, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(T >= 0 && H > 0 && H % 128 == 0 && H <= 8192 && I > 0 && I % 128 == 0 &&
                  I <= 8192,
              FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(E >= 1 && E <= 1024 && k >= 1 && k <= E && k <= 32 && T * k < (1LL << 31),
              FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(al16(x) && al16(ws) && al16(out) && al16(w_gu) && al16(w_dn), FGE_ERR_MISALIGNED);
  FGE_REQUIRE(ws_bytes >= fge_workspace_bytes(FGE_OP_DISPATCH_BASELINE, T, H, I, E, k),
              FGE_ERR_WORKSPACE_TOO_SMALL);
  if (T == 0) return FGE_OK;
  const size_t r = static_cast<size_t>(T) * k;
  uint8_t* base = static_cast<uint8_t*>(ws) + kWsHeaderBytes;
  int32_t* ids = reinterpret_cast<int32_t*>(base);
  float* gates = reinterpret_cast<float*>(base + align_up(r * 4, 256));
  int32_t* token_row = reinterpret_cast<int32_t*>(base + 2 * align_up(r * 4, 256));
  float* y = reinterpret_cast<float*>(base + 3 * align_up(r * 4, 256));
  FGE_CHECK(from_cuda(launch_topk_gate(logits, T, E, k, ids, gates, stream)));
  FGE_CHECK(from_cuda(launch_per_token_dispatch(static_cast<const uint16_t*>(x), ids, T, k, H, I,
                                                w_gu, s_gu, w_dn, s_dn, y, token_row, stream)));
  return from_cuda(launch_combine(y, 1, token_row, gates, T, k, H,
                                  out_dtype == FGE_DTYPE_F32, out, stream));
}

fge_status fge_rmsnorm(const float* h, int64_t T, int64_t H, float eps, void* out,
                       fge_stream_t stream) {
  FGE_CHECK(cur_device_ok());
  FGE_REQUIRE(h && out, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(T >= 0 && H > 0 && H % 8 == 0, FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(al16(h) && al16(out), FGE_ERR_MISALIGNED);
  return from_cuda(launch_rmsnorm(h, T, H, eps, static_cast<uint16_t*>(out), stream));
}

fge_status fge_router_logits(const void* xn, const float* w, int64_t T, int64_t H, int E,
                             float* logits, fge_stream_t stream) {
  FGE_CHECK(cur_device_ok());
  FGE_REQUIRE(xn && w && logits, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(T >= 0 && H > 0 && H % 256 == 0 && H <= 7168 && E >= 1 && E <= 65536,
              FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(al16(xn) && al16(w), FGE_ERR_MISALIGNED);
  return from_cuda(launch_router(static_cast<const uint16_t*>(xn), w, T, H, E, logits, stream));
}

fge_status fge_identity_attention(const void* v, int64_t T, int n_heads, int n_kv,
                                  void* attn, fge_stream_t stream) {
  FGE_CHECK(cur_device_ok());
  FGE_REQUIRE(v && attn, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(T >= 0 && n_kv >= 1 && n_heads >= n_kv && n_heads % n_kv == 0, FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(al16(v) && al16(attn), FGE_ERR_MISALIGNED);
  return from_cuda(launch_identity_attention(static_cast<const uint16_t*>(v), T, n_heads, n_kv,
                                             static_cast<uint16_t*>(attn), stream));
}

fge_status fge_residual_add(float* h, const void* y, fge_dtype y_dtype, int64_t n,
                            fge_stream_t stream) {
  FGE_CHECK(cur_device_ok());
  FGE_REQUIRE(h && y, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(y_dtype == FGE_DTYPE_BF16 || y_dtype == FGE_DTYPE_F32, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(n >= 0 && n % 4 == 0, FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(al16(h) && al16(y), FGE_ERR_MISALIGNED);
  return from_cuda(launch_residual_add(h, y, y_dtype == FGE_DTYPE_F32, n, stream));
}

fge_status fge_residual_rmsnorm(float* h, const void* y, fge_dtype y_dtype, int64_t T,
                                int64_t H, float eps, void* out, fge_stream_t stream) {
  FGE_CHECK(cur_device_ok());
  FGE_REQUIRE(h && y && out, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(y_dtype == FGE_DTYPE_BF16 || y_dtype == FGE_DTYPE_F32, FGE_ERR_INVALID_ARG);
  FGE_REQUIRE(T >= 0 && H > 0 && H % 8 == 0, FGE_ERR_BAD_SHAPE);
  FGE_REQUIRE(al16(h) && al16(y) && al16(out), FGE_ERR_MISALIGNED);
  return from_cuda(launch_residual_rmsnorm(h, y, y_dtype == FGE_DTYPE_F32, T, H, eps,
                                           static_cast<uint16_t*>(out), stream));
}

}  // extern "C"

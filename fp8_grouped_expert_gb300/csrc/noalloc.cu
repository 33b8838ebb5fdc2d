// fge_linear_w8a8_noalloc: the dense W8A8 projection (per-tensor quant + one-expert GEMM)
// with its scratch in a fixed device array of this library instead of a caller workspace.
//
// Why it exists: some callers cannot allocate device memory at the point where they run a
// projection -- hosts that hand out all device memory through their own pool and forbid
// any other allocation while serving, latency-critical paths where a cudaMalloc (which may
// synchronise the device) is not acceptable, and foreign-language hosts that can pass
// device pointers for inputs and outputs but have no device allocator to make a workspace.
// This entry point needs only x, the weights and y from the caller.
#include <mutex>

#include "fge_internal.h"

namespace fge {
namespace {

// Scratch: a 256-byte header (status word, amax word, activation scale), the counters of a K
// split, the e4m3 copy of the activations and the K split's partials.  Every GPU that loads the library holds this array until
// the process exits.
constexpr size_t kNoallocScratchBytes = size_t(16) << 20;  // 16 MiB
constexpr size_t kNoallocMaxActBytes = kNoallocScratchBytes - kWsHeaderBytes;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDev = 64;
void* g_scratch_ptr[kMaxDev] = {nullptr};
std::mutex g_scratch_mu;

// Device address of the array on the current device.  In host code the array's name is a
// host-side stand-in, not a device address, so the address is looked up once per device
// (with that device current) and cached.
fge_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return FGE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return FGE_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FGE_OK;
}

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Argument checks of fge_linear_w8a8_noalloc, before anything is enqueued.
fge_status noalloc_checks(const void* x, int64_t M, int64_t K, const uint8_t* wq,
                          const float* w_scale, int64_t N, void* y) {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return FGE_ERR_CUDA;
  if (major != 10 || minor != 3) return FGE_ERR_UNSUPPORTED_DEVICE;
  if (M < 0 || K <= 0 || K % 128 != 0 || N <= 0 || N % 128 != 0 || N >= (1LL << 24) ||
      K >= (1LL << 24) || M >= (1LL << 31))
    return FGE_ERR_BAD_SHAPE;
  if (M == 0) return FGE_OK;  // nothing is read or written: x and y may be NULL
  if (!x || !wq || !w_scale || !y) return FGE_ERR_INVALID_ARG;
  if (static_cast<uint64_t>(M) * static_cast<uint64_t>(K) > kNoallocMaxActBytes)
    return FGE_ERR_EXCEEDS_STATIC_SCRATCH;
  if (!al16(x) || !al16(wq) || !al16(y)) return FGE_ERR_MISALIGNED;
  return FGE_OK;
}

// The projection itself: per-tensor quantization into the scratch, then the one-expert GEMM.
fge_status noalloc_run(const void* x, int64_t M, int64_t K, const uint8_t* wq,
                       const float* w_scale, int64_t N, void* y, fge_stream_t stream) {
  void* scratch = nullptr;
  const fge_status st = scratch_for_current_device(&scratch);
  if (st != FGE_OK) return st;
  WsHeader* hdr = static_cast<WsHeader*>(scratch);
  // Layout as fge_linear_w8a8's workspace: header | K-split counters | xq | K-split partials.
  // The K split is the one fge_linear_w8a8 takes (so the two agree bit for bit) whenever its
  // scratch fits beside the activations; otherwise the GEMM runs unsplit.
  int ks = dense_ksplit(M, N, K);
  size_t counter_bytes = 0;
  size_t split_bytes = dense_split_bytes(M, N, ks, &counter_bytes);
  const size_t xq_bytes = align_up(static_cast<size_t>(M * K), 256);
  if (kWsHeaderBytes + xq_bytes + split_bytes > kNoallocScratchBytes) {
    ks = 1;
    counter_bytes = split_bytes = 0;
  }
  uint8_t* base = static_cast<uint8_t*>(scratch) + kWsHeaderBytes;
  int32_t* counters = reinterpret_cast<int32_t*>(base);
  uint8_t* xq = base + counter_bytes;
  float* partials = reinterpret_cast<float*>(xq + xq_bytes);

  // The array keeps the previous call's contents: the status word is cleared here, the amax
  // word and the split counters by the quantization launcher, before anything reads them.
  if (cudaMemsetAsync(&hdr->status, 0, sizeof(int32_t), stream) != cudaSuccess)
    return FGE_ERR_CUDA;
  if (launch_quant_per_tensor(static_cast<const uint16_t*>(x), M, K, xq, &hdr->scale, hdr,
                              stream, counters, static_cast<int>(counter_bytes / 4)) !=
      cudaSuccess)
    return FGE_ERR_CUDA;

  GroupedGemmArgs a{};
  a.aq = xq;
  a.as = nullptr;
  a.sa_tensor = &hdr->scale;
  a.offsets = nullptr;
  a.w = wq;
  a.sw = w_scale;
  a.E = 1;
  a.N = N;
  a.K = K;
  a.R = M;
  a.bank_format = 0;
  a.per_tensor = 1;
  a.epilogue = 1;  // bf16 store
  a.out = y;
  a.out_scales = nullptr;
  a.status = &hdr->status;
  a.ksplit = ks;
  a.partials = partials;
  a.split_count = counters;
  fge_status gst = FGE_OK;
  if (launch_one_group_gemm(a, stream, &gst) != cudaSuccess) return FGE_ERR_CUDA;
  return gst;
}

}  // namespace
}  // namespace fge

using namespace fge;

extern "C" fge_status fge_linear_w8a8_noalloc(const void* x, int64_t M, int64_t K,
                                              const uint8_t* wq, const float* w_scale,
                                              int64_t N, void* y, fge_stream_t stream) {
  ledger_note(kLedCalls);
  const fge_status st = noalloc_checks(x, M, K, wq, w_scale, N, y);
  if (st != FGE_OK) {
    ledger_note(kLedRefused);
    return st;
  }
  if (M == 0) return FGE_OK;
  return noalloc_run(x, M, K, wq, w_scale, N, y, stream);
}

// Device status word of the no-alloc call's scratch (the same header layout as a workspace):
// non-zero when a pipeline wait of one of its kernels ran out of its time budget, or when an
// activation was an infinity or a NaN.  Waits for `stream`, then copies the word to *out
// (host).  Like the rest of the scratch it is shared by every call on the device and cleared
// at the start of each call.
extern "C" fge_status fge_linear_w8a8_noalloc_status(fge_stream_t stream, int32_t* out) {
  if (!out) return FGE_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const fge_status st = scratch_for_current_device(&scratch);
  if (st != FGE_OK) return st;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FGE_ERR_CUDA;
  if (cudaMemcpy(out, &static_cast<WsHeader*>(scratch)->status, sizeof(int32_t),
                 cudaMemcpyDeviceToHost) != cudaSuccess)
    return FGE_ERR_CUDA;
  return FGE_OK;
}

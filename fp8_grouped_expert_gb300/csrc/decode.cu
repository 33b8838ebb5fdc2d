// Dense W8A8 projection at decode sizes (at most 16 activation rows): y[m, n] = s(m) *
// sum_k a[m, k] w[n, k], s(m) = sa * sw (per-tensor activation scale) or sa[m] * sw (one
// scale per row) ("feat(qwen4_exp): load-time per-tensor FP8 dense projections", section
// "Why": the small-M projections are bound by reading the weights).  Each weight byte is
// read once from HBM and used for at most 16 products, so the kernel is organised around
// the weight stream: a block takes 16 output features, a producer warp copies their weight
// rows into shared memory with one bulk copy per row, all at once, and eight warps split K
// and multiply with warp-level mma.sync (m16n8k32, e4m3 x e4m3, fp32 accumulate) against the
// activation rows, which stay in L2.  The eight partial sums of each output are added in
// warp order through shared memory, scaled and stored.
//
// K is walked in 64-byte chunks; within a chunk lane q of a quad reads bytes [16 q, 16 q +
// 16) of every weight row and activation row, and the two MMAs of the chunk take the first
// and the second 8 of those bytes.  A weight row and an activation row are split the same
// way, so each MMA multiplies matching k and every product of the dot product is taken
// once.  A K too large for the weight rows to fit in shared memory goes to the grouped
// kernel's 16-token decode tile.
#include "fge_device.cuh"
#include "fge_internal.h"

namespace fge {

constexpr int kDecWarps = 8;   // warps per block; warp w takes K chunks w, w + 8, ...
constexpr int kDecChunk = 64;  // bytes of K per chunk (two MMAs of K = 32)

__device__ __forceinline__ void mma_e4m3_16832(float (&c)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The block's 16 weight rows (K bytes each, contiguous) land in shared memory through one
// bulk copy per row, so the whole weight stream is in flight from the start without
// registers; meanwhile the eight consumer warps load the activation fragments of all their
// chunks from L2.  Warp w then multiplies chunks w, w + 8, ... from shared memory.  A row
// pitch of K + 64 bytes puts the MMA operand reads of a quarter warp on distinct banks.
constexpr int kBkFeat = 16;                   // two MMA column tiles of 8
constexpr int kBkMaxK = 2560;
constexpr int kBkMaxChunks = kBkMaxK / (kDecChunk * kDecWarps);  // per warp
constexpr int kBkSmem = kBkFeat * (kBkMaxK + 64) + 16;

__device__ __forceinline__ void bk_bulk_load(uint32_t smem_dst, const void* src, uint32_t bytes,
                                             uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

template <bool OF32>
__global__ void __launch_bounds__(288, 3)
    decode_gemv_bulk_kernel(const uint8_t* __restrict__ aq, int M, const uint8_t* __restrict__ w,
                            int64_t N, int64_t K, const float* __restrict__ sa_tensor,
                            const float* __restrict__ sa_rows, const float* __restrict__ sw,
                            int32_t* status, void* __restrict__ out) {
  extern __shared__ __align__(128) uint8_t bsm[];
  __shared__ float part[kDecWarps][16][kBkFeat];
  __shared__ int s_abort;
  const int64_t pitch = K + 64;
  const uint32_t w_full = smem_u32(bsm + kBkFeat * pitch);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kBkFeat;
  if (threadIdx.x == 0) {
    mbar_init(w_full, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == kDecWarps) {
    // producer: lane r < 16 copies weight row n0 + r
    if (lane == 0) mbar_arrive_expect_tx(w_full, static_cast<uint32_t>(kBkFeat * K));
    __syncwarp();
    if (lane < kBkFeat)
      bk_bulk_load(smem_u32(bsm + lane * pitch), w + (n0 + lane) * K, static_cast<uint32_t>(K),
                   w_full);
    return;
  }
  const int g = lane >> 2, q = lane & 3;
  const bool live0 = g < M, live1 = g + 8 < M;
  const int64_t chunks = K / kDecChunk;
  // launched as a programmatic dependent of the quantization: the weights (above) do not
  // depend on it, the activations and their scale do
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the activation fragments of this warp's chunks (warp, warp + 8, ...), all in flight
  uint4 a0v[kBkMaxChunks], a1v[kBkMaxChunks];
#pragma unroll
  for (int u = 0; u < kBkMaxChunks; ++u) {
    const int64_t ch = warp + static_cast<int64_t>(u) * kDecWarps;
    const int64_t off = ch * kDecChunk + q * 16;
    a0v[u] = (ch < chunks && live0)
                 ? __ldg(reinterpret_cast<const uint4*>(aq + static_cast<int64_t>(g) * K + off))
                 : make_uint4(0, 0, 0, 0);
    a1v[u] = (ch < chunks && live1)
                 ? __ldg(reinterpret_cast<const uint4*>(aq + static_cast<int64_t>(g + 8) * K + off))
                 : make_uint4(0, 0, 0, 0);
  }
  float c[2][4];
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) c[j][i] = 0.0f;
  const bool ok = mbar_wait(w_full, 0, &s_abort, status);
  if (ok) {
#pragma unroll
    for (int u = 0; u < kBkMaxChunks; ++u) {
      const int64_t ch = warp + static_cast<int64_t>(u) * kDecWarps;
      if (ch < chunks) {
        const uint32_t a_lo[4] = {a0v[u].x, a1v[u].x, a0v[u].y, a1v[u].y};
        const uint32_t a_hi[4] = {a0v[u].z, a1v[u].z, a0v[u].w, a1v[u].w};
        const uint8_t* base = bsm + g * pitch + ch * kDecChunk + q * 16;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const uint4 wv = *reinterpret_cast<const uint4*>(base + j * 8 * pitch);
          mma_e4m3_16832(c[j], a_lo, wv.x, wv.y);
          mma_e4m3_16832(c[j], a_hi, wv.z, wv.w);
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    part[warp][g][8 * j + 2 * q] = c[j][0];
    part[warp][g][8 * j + 2 * q + 1] = c[j][1];
    part[warp][g + 8][8 * j + 2 * q] = c[j][2];
    part[warp][g + 8][8 * j + 2 * q + 1] = c[j][3];
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kDecWarps * 32) : "memory");
  if (!ok || s_abort) return;
  const float sw_t = __ldg(sw);
  const float st = sa_rows ? sw_t : __ldg(sa_tensor) * sw_t;
  for (int i = threadIdx.x; i < 16 * kBkFeat; i += kDecWarps * 32) {
    const int m = i / kBkFeat, f = i - m * kBkFeat;
    if (m >= M) continue;
    float acc = 0.0f;
#pragma unroll
    for (int ww = 0; ww < kDecWarps; ++ww) acc += part[ww][m][f];
    const float sc = sa_rows ? __ldg(sa_rows + m) * st : st;
    const float yv = sc * acc;
    if constexpr (OF32)
      reinterpret_cast<float*>(out)[m * N + n0 + f] = yv;
    else
      reinterpret_cast<__nv_bfloat16*>(out)[m * N + n0 + f] = __float2bfloat16_rn(yv);
  }
}

cudaError_t launch_one_group_gemm(const GroupedGemmArgs& a, cudaStream_t s, fge_status* st) {
  if (a.per_tensor && a.E == 1 && a.offsets == nullptr && a.row_token == nullptr &&
      a.comb == nullptr && a.a_sf == nullptr && (a.epilogue == 0 || a.epilogue == 1) &&
      a.R >= 1 && a.R <= 16 && a.N % kBkFeat == 0 && a.K % kDecChunk == 0 && a.K <= kBkMaxK) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const void* kern = a.epilogue == 0
                           ? reinterpret_cast<const void*>(decode_gemv_bulk_kernel<true>)
                           : reinterpret_cast<const void*>(decode_gemv_bulk_kernel<false>);
    if (device_kernel_ready(dev, kern, kBkSmem, 0)) {
      ledger_note(kLedDenseDecodeTile);
      // a programmatic dependent launch: the kernel may start while the kernel before it
      // (the quantization) finishes, and its weight copies overlap that kernel's tail
      cudaLaunchConfig_t cfg{};
      cfg.gridDim = dim3(static_cast<unsigned>(a.N / kBkFeat));
      cfg.blockDim = dim3(288);
      cfg.dynamicSmemBytes = kBkSmem;
      cfg.stream = s;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      const int m = static_cast<int>(a.R);
      if (a.epilogue == 0)
        return cudaLaunchKernelEx(&cfg, decode_gemv_bulk_kernel<true>, a.aq, m, a.w, a.N, a.K,
                                  a.sa_tensor, a.sa_rows, a.sw, a.status, a.out);
      return cudaLaunchKernelEx(&cfg, decode_gemv_bulk_kernel<false>, a.aq, m, a.w, a.N, a.K,
                                a.sa_tensor, a.sa_rows, a.sw, a.status, a.out);
    }
  }
  return launch_grouped_gemm(a, s, st);
}

}  // namespace fge

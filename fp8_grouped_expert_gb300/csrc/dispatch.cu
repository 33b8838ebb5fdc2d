// Per-token int4 expert dispatch: the baseline that the grouped expert GEMM replaces ("FP8
// grouped-expert prefill with on-chip int4-to-e4m3 dequant", section 1: one dispatch per
// routed token per layer).  One CTA per routed (token, slot) pair runs that expert's FFN
// on the single token: int4 weights dequantized in registers (q * per-group scale), bf16
// activations widened to fp32, fp32 accumulation, SwiGLU in fp32, no activation
// quantization.  Every pair re-reads its expert's whole weight bank, which is the cost the
// grouped GEMM removes.  The expert outputs go to y [T*k, H] (fp32, row t*k + j) and are
// combined by the combine kernel.
#include <algorithm>

#include "fge_device.cuh"

namespace fge {

constexpr int kDispatchThreads = 256;

// dot(x[0..K), dequant(row)) for a canonical int4 row (two's complement, low nibble = even
// element) with one scale per 128 elements; one warp, 16-byte chunks (32 values) per lane.
// A nibble becomes a float exactly through the exponent trick: for u = nibble ^ 8 in 0..15,
// float(2^23 + u) - (2^23 + 8) = q, two integer ops and one add instead of a conversion.
__device__ __forceinline__ float warp_dot_int4(const uint8_t* __restrict__ row,
                                               const float* __restrict__ scales,
                                               const float* __restrict__ x, int K, int lane) {
  float acc = 0.0f;
  for (int c = lane; c < K / 32; c += 32) {
    const uint4 p = __ldg(reinterpret_cast<const uint4*>(row) + c);
    const uint32_t w[4] = {p.x ^ 0x88888888u, p.y ^ 0x88888888u, p.z ^ 0x88888888u,
                           p.w ^ 0x88888888u};
    const float4* xc = reinterpret_cast<const float4*>(x + c * 32);
    float part = 0.0f;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float4 x0 = xc[2 * b], x1 = xc[2 * b + 1];
      const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const float q = __uint_as_float(0x4B000000u | ((w[b] >> (4 * n)) & 0xFu)) - 8388616.0f;
        part = fmaf(q, xv[n], part);
      }
    }
    acc = fmaf(__ldg(scales + (c * 32) / 128), part, acc);
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, d);
  return acc;
}

__global__ void __launch_bounds__(kDispatchThreads)
    per_token_dispatch_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ ids,
                              int64_t T, int k, int H, int I, const uint8_t* __restrict__ w_gu,
                              const float* __restrict__ s_gu, const uint8_t* __restrict__ w_dn,
                              const float* __restrict__ s_dn, float* __restrict__ y) {
  extern __shared__ float sm[];
  float* xs = sm;           // [H]
  float* cg = xs + H;       // [2I] gate_up output, then h in [0, I)
  const int64_t pair = blockIdx.x;  // t * k + j
  const int64_t t = pair / k;
  const int e = ids[pair];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = kDispatchThreads / 32;
  for (int i = threadIdx.x; i < H; i += kDispatchThreads)
    xs[i] = __uint_as_float(static_cast<uint32_t>(x[t * H + i]) << 16);
  __syncthreads();
  const int n_gu = 2 * I;
  const uint8_t* wg = w_gu + static_cast<size_t>(e) * n_gu * (H / 2);
  const float* sg = s_gu + static_cast<size_t>(e) * n_gu * (H / 128);
  for (int n = warp; n < n_gu; n += nwarps) {
    const float v = warp_dot_int4(wg + static_cast<size_t>(n) * (H / 2),
                                  sg + static_cast<size_t>(n) * (H / 128), xs, H, lane);
    if (lane == 0) cg[n] = v;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < I; i += kDispatchThreads) {
    const float g = cg[i];
    cg[i] = __fdiv_rn(g, 1.0f + expf(-g)) * cg[I + i];
  }
  __syncthreads();
  const uint8_t* wd = w_dn + static_cast<size_t>(e) * H * (I / 2);
  const float* sd = s_dn + static_cast<size_t>(e) * H * (I / 128);
  for (int m = warp; m < H; m += nwarps) {
    const float v = warp_dot_int4(wd + static_cast<size_t>(m) * (I / 2),
                                  sd + static_cast<size_t>(m) * (I / 128), cg, I, lane);
    if (lane == 0) y[pair * H + m] = v;
  }
}

__global__ void identity_rows_kernel(int32_t* __restrict__ rows, int64_t n) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    rows[i] = static_cast<int32_t>(i);
}

cudaError_t launch_per_token_dispatch(const uint16_t* x, const int32_t* ids, int64_t T, int k,
                                      int64_t H, int64_t I, const uint8_t* w_gu,
                                      const float* s_gu, const uint8_t* w_dn, const float* s_dn,
                                      float* y, int32_t* token_row, cudaStream_t s) {
  const int64_t pairs = T * k;
  if (pairs == 0) return cudaSuccess;
  const size_t smem = static_cast<size_t>(H + 2 * I) * sizeof(float);
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return ce;
  if (!device_kernel_ready(dev, reinterpret_cast<const void*>(per_token_dispatch_kernel),
                           96 * 1024, 0))
    return cudaErrorInvalidConfiguration;
  per_token_dispatch_kernel<<<static_cast<unsigned>(pairs), kDispatchThreads, smem, s>>>(
      x, ids, T, k, static_cast<int>(H), static_cast<int>(I), w_gu, s_gu, w_dn, s_dn, y);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  identity_rows_kernel<<<static_cast<int>(std::min<int64_t>((pairs + 255) / 256, num_sms() * 4)),
                         256, 0, s>>>(token_row, pairs);
  return cudaGetLastError();
}

}  // namespace fge

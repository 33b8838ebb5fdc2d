// fp8_quant_act: dynamic e4m3 activation quantization, per (row, 128-element group), per row
// or per tensor ("FP8 grouped-expert prefill with on-chip int4-to-e4m3 dequant", section 1;
// "Module fp8_ffi": amax reduce -> scale finalize -> e4m3 quantize on one stream).
// HBM-bound: 16-byte vector loads and stores, warp-shuffle amax, grids sized to the SMs.
#include <algorithm>

#include <cuda_fp4.h>

#include "fge_device.cuh"
#include "quotient.cuh"

namespace fge {

// 16-byte loads each lane keeps in flight per trip in the flat-array kernels below.
constexpr int kQuantUnroll = 4;

// Per-tensor pass 1: amax over the tensor, combined across blocks with atomicMax on the
// float bits (|x| >= 0, so the unsigned order of the bits is the float order).
// Folds the 8 bf16 values of v into the running amax m and the non-finite detector bad.
__device__ __forceinline__ void amax_fold8(const uint4& v, float& m, float& bad) {
  m = fmaxf(m, fmaxf(fmaxf(fabsf(bf16_lo(v.x)), fabsf(bf16_hi(v.x))),
                     fmaxf(fabsf(bf16_lo(v.y)), fabsf(bf16_hi(v.y)))));
  m = fmaxf(m, fmaxf(fmaxf(fabsf(bf16_lo(v.z)), fabsf(bf16_hi(v.z))),
                     fmaxf(fabsf(bf16_lo(v.w)), fabsf(bf16_hi(v.w)))));
  bad = nonfinite_fold(nonfinite_fold(nonfinite_fold(nonfinite_fold(bad, bf16_lo(v.x)),
                                                     bf16_hi(v.x)),
                                      bf16_lo(v.y)),
                       bf16_hi(v.y));
  bad = nonfinite_fold(nonfinite_fold(nonfinite_fold(nonfinite_fold(bad, bf16_lo(v.z)),
                                                     bf16_hi(v.z)),
                                      bf16_lo(v.w)),
                       bf16_hi(v.w));
}

__global__ void amax_kernel(const uint4* __restrict__ x, int64_t n8, uint32_t* __restrict__ amax_bits,
                            int32_t* status) {
  float m = 0.0f, bad = 0.0f;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  // kQuantUnroll independent 16-byte loads in flight per thread and trip
  for (int64_t i0 = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i0 < n8;
       i0 += stride * kQuantUnroll) {
    uint4 v[kQuantUnroll];
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      const int64_t i = i0 + u * stride;
      v[u] = i < n8 ? __ldg(x + i) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) amax_fold8(v[u], m, bad);
  }
  report_nonfinite(status, bad);
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
  __shared__ float red[32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
    if (threadIdx.x == 0) atomicMax(amax_bits, __float_as_uint(m));
  }
}

// Per-tensor pass 2: every thread derives the same scale from the amax word and casts.
__global__ void cast_per_tensor_kernel(const uint4* __restrict__ x, int64_t n8,
                                       const uint32_t* __restrict__ amax_bits,
                                       uint2* __restrict__ xq, float* __restrict__ xs,
                                       float* __restrict__ scale_out) {
  const float s = scale_from_amax(__uint_as_float(*amax_bits));
  const float y = __frcp_rn(s);
  const bool fast = quot_fast_ok(s);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    xs[0] = s;
    if (scale_out) *scale_out = s;
  }
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i0 = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i0 < n8;
       i0 += stride * kQuantUnroll) {
    uint4 v[kQuantUnroll];
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      const int64_t i = i0 + u * stride;
      v[u] = i < n8 ? __ldg(x + i) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < n8) xq[i] = cast8(v[u], s, y, fast);
    }
  }
}

// One scale per row (token): one warp per row, two passes over the row (amax, then the
// cast; the second pass reads the row back from L1/L2).
__global__ void quant_row_kernel(const uint4* __restrict__ x, int64_t M, int64_t n8_row,
                                 uint2* __restrict__ xq, float* __restrict__ xs,
                                 int32_t* status) {
  // a decode-size projection's GEMM may launch now (see quant_tensor_small_kernel)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int64_t wid = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t r = wid; r < M; r += nw) {
    const uint4* xr = x + r * n8_row;
    float amax = 0.0f, bad = 0.0f;
    for (int64_t i0 = lane; i0 < n8_row; i0 += 32 * kQuantUnroll) {
      uint4 v[kQuantUnroll];
#pragma unroll
      for (int u = 0; u < kQuantUnroll; ++u) {
        const int64_t i = i0 + 32 * u;
        v[u] = i < n8_row ? __ldg(xr + i) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kQuantUnroll; ++u) amax_fold8(v[u], amax, bad);
    }
    report_nonfinite(status, bad);
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
    const float s = scale_from_amax(amax);
    const float y = __frcp_rn(s);
    const bool fast = quot_fast_ok(s);
    uint2* qr = xq + r * n8_row;
    for (int64_t i0 = lane; i0 < n8_row; i0 += 32 * kQuantUnroll) {
      uint4 v[kQuantUnroll];
#pragma unroll
      for (int u = 0; u < kQuantUnroll; ++u) {
        const int64_t i = i0 + 32 * u;
        v[u] = i < n8_row ? __ldg(xr + i) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kQuantUnroll; ++u) {
        const int64_t i = i0 + 32 * u;
        if (i < n8_row) qr[i] = cast8(v[u], s, y, fast);
      }
    }
    if (lane == 0) xs[r] = s;
  }
}

// MXFP4 activations ("[RFC] Support FP4 (E2M1) activation dispatch in MegaMoE": E2M1 codes
// halve the dispatch bytes of e4m3).  One power-of-two scale per 32 consecutive values:
// E = max(floor(log2(amax)) - 2, -127), stored as the E8M0 code E + 127, so the block's
// largest magnitude lands in [4, 8); each value is cast to E2M1 from x * 2^-E (exact: a
// power-of-two multiply) with round to nearest even, saturating at 6.  Rows never split a
// block (K % 32 == 0), so the tensor is walked as one flat array: 8 values per lane, four
// lanes per block, one 4-byte store of codes per lane.
__global__ void mx_e2m1_kernel(const uint4* __restrict__ x, int64_t n8, uint32_t* __restrict__ xq,
                               uint8_t* __restrict__ xs) {
  const int lane = threadIdx.x & 31;
  const int64_t t0 = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  // warp-uniform trip count; kQuantUnroll independent 16-byte loads per lane per trip
  for (int64_t w0 = t0 - lane; w0 < n8; w0 += stride * kQuantUnroll) {
    uint4 v[kQuantUnroll];
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      const int64_t c = w0 + u * stride + lane;
      v[u] = c < n8 ? __ldcs(x + c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      const int64_t c = w0 + u * stride + lane;
      const float f[8] = {bf16_lo(v[u].x), bf16_hi(v[u].x), bf16_lo(v[u].y), bf16_hi(v[u].y),
                          bf16_lo(v[u].z), bf16_hi(v[u].z), bf16_lo(v[u].w), bf16_hi(v[u].w)};
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      // floor(log2(amax)) is the exponent field minus 127 for a normal amax; a zero or
      // subnormal amax lands on the clamp
      const int ef = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
      const int e = max(ef - 129, -127);
      const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-E
      uint32_t q = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        q |= (static_cast<uint32_t>(__nv_cvt_float_to_fp4(f[i] * inv, __NV_E2M1,
                                                          cudaRoundNearest)) & 0xFu) << (4 * i);
      if (c < n8) {
        xq[c] = q;
        if ((lane & 3) == 0) xs[c >> 2] = static_cast<uint8_t>(e + 127);
      }
    }
  }
}

cudaError_t launch_mx_quant_e2m1(const uint16_t* x, int64_t M, int64_t K, uint8_t* xq,
                                 uint8_t* xs, cudaStream_t s) {
  const int64_t n8 = M * (K / 8);
  if (n8 == 0) return cudaSuccess;
  const int grid = static_cast<int>(
      std::min<int64_t>((n8 + 256 * kQuantUnroll - 1) / (256 * kQuantUnroll), num_sms() * 8));
  mx_e2m1_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const uint4*>(x), n8,
                                      reinterpret_cast<uint32_t*>(xq), xs);
  return cudaGetLastError();
}

cudaError_t launch_quant_rows(const uint16_t* x, int64_t M, int64_t K, uint8_t* xq, float* xs,
                              int32_t* status, cudaStream_t s) {
  if (M == 0) return cudaSuccess;
  const int grid = static_cast<int>(std::min<int64_t>((M + 7) / 8, num_sms() * 8));
  quant_row_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const uint4*>(x), M, K / 8,
                                        reinterpret_cast<uint2*>(xq), xs, status);
  return cudaGetLastError();
}

// Per-tensor quantization of a small tensor (decode sizes) in one launch: a cluster of
// kSmallCtas CTAs, each thread holding its kSmallPer 16-byte chunks in registers; every CTA
// reduces its amax, the cluster exchanges the CTA maxima through distributed shared memory,
// and the same registers are cast -- one read, no atomics, no second launch.  The amax and
// the codes are those of the two-pass kernels (a max does not depend on the order of its
// operands).  Chunk i belongs to thread i % (kSmallCtas * kSmallThreads) of the cluster.
constexpr int kSmallCtas = 8, kSmallThreads = 128, kSmallPer = 8;

__global__ void __cluster_dims__(kSmallCtas, 1, 1) __launch_bounds__(kSmallThreads)
    quant_tensor_small_kernel(const uint4* __restrict__ x, int64_t n8, uint2* __restrict__ xq,
                              float* __restrict__ xs, float* __restrict__ scale_out,
                              int32_t* status, int32_t* zero, int n_zero) {
  // a decode-size projection's GEMM may launch now and start streaming its weights; it
  // waits for this kernel's results before reading them
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ float red[kSmallThreads / 32];
  __shared__ float cta_amax;
  const int gt = blockIdx.x * kSmallThreads + threadIdx.x;
  constexpr int kAll = kSmallCtas * kSmallThreads;
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < n_zero; i += kSmallThreads) zero[i] = 0;
  uint4 v[kSmallPer];
  float m = 0.0f, bad = 0.0f;
#pragma unroll
  for (int u = 0; u < kSmallPer; ++u) {
    const int64_t i = gt + static_cast<int64_t>(u) * kAll;
    v[u] = i < n8 ? __ldg(x + i) : make_uint4(0, 0, 0, 0);
    amax_fold8(v[u], m, bad);
  }
  report_nonfinite(status, bad);
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float c = red[0];
#pragma unroll
    for (int w = 1; w < kSmallThreads / 32; ++w) c = fmaxf(c, red[w]);
    cta_amax = c;
  }
  // every CTA's maximum is published before any CTA reads them
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
  m = 0.0f;
  const uint32_t local = smem_u32(&cta_amax);
#pragma unroll
  for (int r = 0; r < kSmallCtas; ++r) {
    uint32_t remote;
    float c;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(r));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(c) : "r"(remote) : "memory");
    m = fmaxf(m, c);
  }
  // no CTA leaves (and gives up its shared memory) while another may still read it
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
  const float sc = scale_from_amax(m);
  const float y = __frcp_rn(sc);
  const bool fast = quot_fast_ok(sc);
  if (gt == 0) {
    xs[0] = sc;
    if (scale_out) *scale_out = sc;
  }
#pragma unroll
  for (int u = 0; u < kSmallPer; ++u) {
    const int64_t i = gt + static_cast<int64_t>(u) * kAll;
    if (i < n8) xq[i] = cast8(v[u], sc, y, fast);
  }
}

cudaError_t launch_quant_per_tensor(const uint16_t* x, int64_t M, int64_t K, uint8_t* xq,
                                    float* xs, WsHeader* hdr, cudaStream_t s, int32_t* zero,
                                    int n_zero) {
  const int64_t n8 = M * K / 8;
  if (n8 <= static_cast<int64_t>(kSmallCtas) * kSmallThreads * kSmallPer) {
    quant_tensor_small_kernel<<<kSmallCtas, kSmallThreads, 0, s>>>(
        reinterpret_cast<const uint4*>(x), n8, reinterpret_cast<uint2*>(xq), xs, &hdr->scale,
        &hdr->status, zero, n_zero);
    return cudaGetLastError();
  }
  // the amax word, and the words to clear when they follow the header directly (one memset)
  uint8_t* hdr_end = reinterpret_cast<uint8_t*>(hdr) + sizeof(WsHeader);
  const bool adjacent = n_zero > 0 && reinterpret_cast<uint8_t*>(zero) == hdr_end;
  cudaError_t e = cudaMemsetAsync(&hdr->amax_bits, 0,
                                  adjacent ? static_cast<size_t>(hdr_end - reinterpret_cast<uint8_t*>(
                                                                               &hdr->amax_bits)) +
                                                 static_cast<size_t>(n_zero) * 4
                                           : sizeof(uint32_t),
                                  s);
  if (e != cudaSuccess) return e;
  if (n_zero > 0 && !adjacent) {
    e = cudaMemsetAsync(zero, 0, static_cast<size_t>(n_zero) * 4, s);
    if (e != cudaSuccess) return e;
  }
  const int grid = static_cast<int>(
      std::max<int64_t>(1, std::min<int64_t>((n8 + 255) / 256, num_sms() * 8)));
  if (n8 > 0) {
    amax_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const uint4*>(x), n8, &hdr->amax_bits,
                                     &hdr->status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  cast_per_tensor_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const uint4*>(x), n8,
                                              &hdr->amax_bits, reinterpret_cast<uint2*>(xq), xs,
                                              &hdr->scale);
  return cudaGetLastError();
}

}  // namespace fge

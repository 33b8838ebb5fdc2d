// Glue of the stacked prefill workload (not steps of the method): RMSNorm, fp32 router
// logits, the identity stand-in for the attention core, and the fp32 residual add.
#include <algorithm>

#include "chain.cuh"
#include "fge_device.cuh"

namespace fge {

// One block per row: sum of squares in fp32, then h / sqrt(mean + eps) rounded to bf16.
// ADD: the residual add first, h[t] += y[t] (y bf16 or float, YF32), the updated row written
// back; each thread adds and squares the same elements in the same order as the separate
// residual add followed by the plain norm, so the two give the same bits.
template <bool ADD, bool YF32>
__global__ void rmsnorm_kernel(float* __restrict__ h, const void* __restrict__ y, int64_t H,
                               float eps, uint16_t* __restrict__ out) {
  chain_enter();
  float* row = h + blockIdx.x * H;
  float ss = 0.0f;
  for (int64_t i = threadIdx.x * 4; i < H; i += blockDim.x * 4) {
    float4 v = *reinterpret_cast<const float4*>(row + i);
    if constexpr (ADD) {
      if constexpr (YF32) {
        const float4 b =
            *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(y) + blockIdx.x * H + i);
        v.x += b.x; v.y += b.y; v.z += b.z; v.w += b.w;
      } else {
        const uint2 b = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(y) +
                                                        blockIdx.x * H + i);
        v.x += bf16_lo(b.x); v.y += bf16_hi(b.x); v.z += bf16_lo(b.y); v.w += bf16_hi(b.y);
      }
      *reinterpret_cast<float4*>(row + i) = v;
    }
    ss = fmaf(v.x, v.x, ss);
    ss = fmaf(v.y, v.y, ss);
    ss = fmaf(v.z, v.z, ss);
    ss = fmaf(v.w, v.w, ss);
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, d);
  __shared__ float red[32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    ss = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, d);
    if (threadIdx.x == 0) red[0] = ss;
  }
  __syncthreads();
  const float denom = __fsqrt_rn(__fdiv_rn(red[0], static_cast<float>(H)) + eps);
  uint16_t* orow = out + blockIdx.x * H;
  // each thread reads back only the elements it wrote itself
  for (int64_t i = threadIdx.x * 4; i < H; i += blockDim.x * 4) {
    const float4 v = *reinterpret_cast<const float4*>(row + i);
    uint2 o;
    o.x = pack_bf16x2(__fdiv_rn(v.x, denom), __fdiv_rn(v.y, denom));
    o.y = pack_bf16x2(__fdiv_rn(v.z, denom), __fdiv_rn(v.w, denom));
    *reinterpret_cast<uint2*>(orow + i) = o;
  }
}

// Router logits, logits[t, e] = sum_k xn[t, k] * wr[e, k] in fp32.  One block per kRouterTok
// tokens and 32 experts: the tokens' bf16 rows stay in shared memory.  Each warp takes
// kRouterExp experts at a time; lane l accumulates the products at k = 8 l + 256 i for every
// token of the block and each of those experts, so a row chunk read from shared memory serves
// kRouterExp experts and a router chunk read from L2 serves every token.  The warp then adds
// its lanes' sums.
constexpr int kRouterTok = 16, kRouterExp = 4;

__global__ void __launch_bounds__(256)
    router_kernel(const uint16_t* __restrict__ xn, const float* __restrict__ wr, int64_t T,
                  int64_t H, int E, float* __restrict__ logits) {
  chain_enter();
  extern __shared__ uint4 sx[];  // [kRouterTok][H / 8], 8 bf16 each
  const int64_t t0 = blockIdx.x * static_cast<int64_t>(kRouterTok);
  const int nt = static_cast<int>(T - t0 < kRouterTok ? T - t0 : kRouterTok);
  const int64_t row8 = H / 8;
  for (int64_t i0 = threadIdx.x; i0 < kRouterTok * row8; i0 += 4 * blockDim.x) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {  // four loads in flight per thread
      const int64_t i = i0 + u * blockDim.x;
      const int r = static_cast<int>(i / row8);
      v[u] = (i < kRouterTok * row8 && r < nt)
                 ? __ldg(reinterpret_cast<const uint4*>(xn + (t0 + r) * H) + (i - r * row8))
                 : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = i0 + u * blockDim.x;
      if (i < kRouterTok * row8) sx[i] = v[u];
    }
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int e_end = min(E, static_cast<int>(blockIdx.y + 1) * nwarps * kRouterExp);
  for (int e0 = static_cast<int>(blockIdx.y) * nwarps * kRouterExp + warp * kRouterExp;
       e0 < e_end; e0 += nwarps * kRouterExp) {
    float acc[kRouterExp][kRouterTok];
#pragma unroll
    for (int j = 0; j < kRouterExp; ++j)
#pragma unroll
      for (int r = 0; r < kRouterTok; ++r) acc[j][r] = 0.0f;
    for (int64_t i = lane * 8; i < H; i += 256) {
      float wv[kRouterExp][8];
#pragma unroll
      for (int j = 0; j < kRouterExp; ++j) {
        const int e = min(e0 + j, E - 1);  // experts past E repeat the last; never stored
        const float4 w0 = __ldg(reinterpret_cast<const float4*>(wr + e * H + i));
        const float4 w1 = __ldg(reinterpret_cast<const float4*>(wr + e * H + i + 4));
        wv[j][0] = w0.x; wv[j][1] = w0.y; wv[j][2] = w0.z; wv[j][3] = w0.w;
        wv[j][4] = w1.x; wv[j][5] = w1.y; wv[j][6] = w1.z; wv[j][7] = w1.w;
      }
#pragma unroll
      for (int r = 0; r < kRouterTok; ++r) {
        const uint4 xv = sx[r * row8 + i / 8];
        const float x[8] = {bf16_lo(xv.x), bf16_hi(xv.x), bf16_lo(xv.y), bf16_hi(xv.y),
                            bf16_lo(xv.z), bf16_hi(xv.z), bf16_lo(xv.w), bf16_hi(xv.w)};
#pragma unroll
        for (int j = 0; j < kRouterExp; ++j) {
          float a = acc[j][r];
#pragma unroll
          for (int c = 0; c < 8; ++c) a = fmaf(x[c], wv[j][c], a);
          acc[j][r] = a;
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kRouterExp; ++j)
#pragma unroll
      for (int r = 0; r < kRouterTok; ++r)
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) acc[j][r] += __shfl_xor_sync(0xffffffffu, acc[j][r], d);
#pragma unroll
    for (int j = 0; j < kRouterExp; ++j)
#pragma unroll
      for (int r = 0; r < kRouterTok; ++r)
        if (lane == (j * kRouterTok + r) % 32 && r < nt && e0 + j < E)
          logits[(t0 + r) * E + e0 + j] = acc[j][r];
  }
}

// attn[t, h*128 + d] = v[t, (h / rep)*128 + d], 16-byte copies.
__global__ void identity_attention_kernel(const uint4* __restrict__ v, int64_t T, int n_heads,
                                          int n_kv, uint4* __restrict__ attn) {
  chain_enter();
  const int rep = n_heads / n_kv;
  const int64_t per_row = static_cast<int64_t>(n_heads) * 16;  // 128 bf16 = 16 uint4 per head
  const int64_t total = T * per_row;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i / per_row, c = i % per_row;
    const int64_t head = c / 16, d = c % 16;
    attn[i] = __ldg(v + t * n_kv * 16 + (head / rep) * 16 + d);
  }
}

template <bool YF32>
__global__ void residual_add_kernel(float* __restrict__ h, const void* __restrict__ y, int64_t n) {
  chain_enter();
  for (int64_t i = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) * 4; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x * 4) {
    float4 a = *reinterpret_cast<float4*>(h + i);
    if constexpr (YF32) {
      const float4 b = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(y) + i);
      a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
    } else {
      const uint2 b = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(y) + i);
      a.x += bf16_lo(b.x); a.y += bf16_hi(b.x); a.z += bf16_lo(b.y); a.w += bf16_hi(b.y);
    }
    *reinterpret_cast<float4*>(h + i) = a;
  }
}

cudaError_t launch_rmsnorm(const float* h, int64_t T, int64_t H, float eps, uint16_t* out,
                           cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  return launch_chained(rmsnorm_kernel<false, false>, dim3(static_cast<unsigned>(T)), dim3(256), 0,
                        s, const_cast<float*>(h), static_cast<const void*>(nullptr), H, eps, out);
}

cudaError_t launch_residual_rmsnorm(float* h, const void* y, int y_f32, int64_t T, int64_t H,
                                    float eps, uint16_t* out, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(T)), block(256);
  if (y_f32)
    return launch_chained(rmsnorm_kernel<true, true>, grid, block, 0, s, h, y, H, eps, out);
  return launch_chained(rmsnorm_kernel<true, false>, grid, block, 0, s, h, y, H, eps, out);
}

cudaError_t launch_router(const uint16_t* xn, const float* wr, int64_t T, int64_t H, int E,
                          float* logits, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int smem = static_cast<int>(kRouterTok * H * 2);  // H <= 7168: at most 224 KB
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return ce;
  // the limit is raised once per device to the largest row the call accepts
  if (!device_kernel_ready(dev, reinterpret_cast<const void*>(router_kernel),
                           kRouterTok * 7168 * 2, 0))
    return cudaErrorInvalidConfiguration;
  // blocks split the experts too (32 per block), so that a small T still fills the SMs
  const dim3 grid(static_cast<unsigned>((T + kRouterTok - 1) / kRouterTok),
                  static_cast<unsigned>((E + 8 * kRouterExp - 1) / (8 * kRouterExp)));
  return launch_chained(router_kernel, grid, dim3(256), static_cast<size_t>(smem), s, xn, wr, T,
                        H, E, logits);
}

cudaError_t launch_identity_attention(const uint16_t* v, int64_t T, int n_heads, int n_kv,
                                      uint16_t* attn, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int grid = num_sms() * 8;
  return launch_chained(identity_attention_kernel, dim3(grid), dim3(256), 0, s,
                        reinterpret_cast<const uint4*>(v), T, n_heads, n_kv,
                        reinterpret_cast<uint4*>(attn));
}

cudaError_t launch_residual_add(float* h, const void* y, int y_f32, int64_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int grid = static_cast<int>(std::min<int64_t>((n / 4 + 255) / 256, num_sms() * 8));
  if (y_f32) return launch_chained(residual_add_kernel<true>, dim3(grid), dim3(256), 0, s, h, y, n);
  return launch_chained(residual_add_kernel<false>, dim3(grid), dim3(256), 0, s, h, y, n);
}

}  // namespace fge

// Glue of the stacked prefill workload (not steps of the method): RMSNorm, fp32 router
// logits, the identity stand-in for the attention core, and the fp32 residual add.
#include <algorithm>

#include "fge_device.cuh"

namespace fge {

// One block per row: sum of squares in fp32, then h / sqrt(mean + eps) rounded to bf16.
__global__ void rmsnorm_kernel(const float* __restrict__ h, int64_t H, float eps,
                               uint16_t* __restrict__ out) {
  const float* row = h + blockIdx.x * H;
  float ss = 0.0f;
  for (int64_t i = threadIdx.x * 4; i < H; i += blockDim.x * 4) {
    const float4 v = *reinterpret_cast<const float4*>(row + i);
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
  for (int64_t i = threadIdx.x * 4; i < H; i += blockDim.x * 4) {
    const float4 v = *reinterpret_cast<const float4*>(row + i);
    uint2 o;
    o.x = pack_bf16x2(__fdiv_rn(v.x, denom), __fdiv_rn(v.y, denom));
    o.y = pack_bf16x2(__fdiv_rn(v.z, denom), __fdiv_rn(v.w, denom));
    *reinterpret_cast<uint2*>(orow + i) = o;
  }
}

// One warp per (token, expert): fp32 dot product over H in a fixed lane-strided order.
__global__ void router_kernel(const uint16_t* __restrict__ xn, const float* __restrict__ wr,
                              int64_t T, int64_t H, int E, float* __restrict__ logits) {
  const int lane = threadIdx.x & 31;
  const int64_t wid = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t item = wid; item < T * E; item += nw) {
    const int64_t t = item / E, e = item % E;
    const uint16_t* x = xn + t * H;
    const float* w = wr + e * H;
    float acc = 0.0f;
    for (int64_t i = lane * 8; i < H; i += 256) {
      const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x + i));
      const float4 w0 = __ldg(reinterpret_cast<const float4*>(w + i));
      const float4 w1 = __ldg(reinterpret_cast<const float4*>(w + i + 4));
      acc = fmaf(bf16_lo(xv.x), w0.x, acc);
      acc = fmaf(bf16_hi(xv.x), w0.y, acc);
      acc = fmaf(bf16_lo(xv.y), w0.z, acc);
      acc = fmaf(bf16_hi(xv.y), w0.w, acc);
      acc = fmaf(bf16_lo(xv.z), w1.x, acc);
      acc = fmaf(bf16_hi(xv.z), w1.y, acc);
      acc = fmaf(bf16_lo(xv.w), w1.z, acc);
      acc = fmaf(bf16_hi(xv.w), w1.w, acc);
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, d);
    if (lane == 0) logits[item] = acc;
  }
}

// attn[t, h*128 + d] = v[t, (h / rep)*128 + d], 16-byte copies.
__global__ void identity_attention_kernel(const uint4* __restrict__ v, int64_t T, int n_heads,
                                          int n_kv, uint4* __restrict__ attn) {
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
  rmsnorm_kernel<<<static_cast<unsigned>(T), 256, 0, s>>>(h, H, eps, out);
  return cudaGetLastError();
}

cudaError_t launch_router(const uint16_t* xn, const float* wr, int64_t T, int64_t H, int E,
                          float* logits, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int grid = static_cast<int>(std::min<int64_t>((T * E + 7) / 8, num_sms() * 16));
  router_kernel<<<grid, 256, 0, s>>>(xn, wr, T, H, E, logits);
  return cudaGetLastError();
}

cudaError_t launch_identity_attention(const uint16_t* v, int64_t T, int n_heads, int n_kv,
                                      uint16_t* attn, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int grid = num_sms() * 8;
  identity_attention_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const uint4*>(v), T, n_heads,
                                                 n_kv, reinterpret_cast<uint4*>(attn));
  return cudaGetLastError();
}

cudaError_t launch_residual_add(float* h, const void* y, int y_f32, int64_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int grid = static_cast<int>(std::min<int64_t>((n / 4 + 255) / 256, num_sms() * 8));
  if (y_f32) residual_add_kernel<true><<<grid, 256, 0, s>>>(h, y, n);
  else residual_add_kernel<false><<<grid, 256, 0, s>>>(h, y, n);
  return cudaGetLastError();
}

}  // namespace fge

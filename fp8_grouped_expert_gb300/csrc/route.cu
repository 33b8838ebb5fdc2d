// Routing kernels around the grouped GEMM: top-k gate, the expert permutation (histogram ->
// exclusive scan -> stable rank -> row copy) and the gate-weighted combine.  The pages
// replace per-token expert dispatch by one grouped GEMM ("FP8 grouped-expert prefill with
// on-chip int4-to-e4m3 dequant", section 1); these kernels make the routed rows of each
// expert contiguous and bring the expert outputs back to token order.  All are
// deterministic: ranks come from warp-synchronous scans, never from atomic order.
#include <algorithm>
#include <cfloat>

#include "fge_device.cuh"
#include "chain.cuh"
#include "quotient.cuh"

namespace fge {

constexpr int kChunkTokens = 128;  // tokens per permutation chunk
constexpr int kQuantQuads = 2;     // group quads whose loads a warp keeps in flight
constexpr int kQuantBlocks = 4;    // resident 256-thread blocks per SM (launch bounds)


// ------------------------------------------------------------------------------ top-k
// Float bits mapped to an unsigned key with the same order (negative values reversed).
// -0 and +0 compare equal as floats, so both take the key of +0.
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = f == 0.0f ? 0u : __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The float a key stands for (the inverse of order_key; -0 comes back as +0).
__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// One warp per token: lane l holds the keys of logits l, l + 32, ...; k rounds, each taking
// the largest untaken key (ties to the lower expert id) with two warp reductions: the maximum
// key, then the lowest id among the lanes offering it.  The chosen logit is read back from
// the key.  Up to four keys a lane (E <= 128) are sorted once, by key descending and id
// ascending, so a lane always offers its first entry and the winner shifts its list by one;
// with more keys a lane rescans its untaken keys every round.
template <int PER>
__global__ void topk_kernel(const float* __restrict__ logits, int64_t T, int E, int k,
                            int32_t* __restrict__ ids, float* __restrict__ gates) {
  chain_enter();
  constexpr uint32_t kNone = 0x7fffffffu;
  const int lane = threadIdx.x & 31;
  const int64_t wid = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t t = wid; t < T; t += nw) {
    uint32_t key[PER], id[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane + 32 * i;
      key[i] = e < E ? order_key(__ldg(logits + t * E + e)) : 0u;
      id[i] = e < E ? static_cast<uint32_t>(e) : kNone;  // slots past E: offered last, never won
    }
    float my_val = 0.0f;
    int my_id = 0;
    if constexpr (PER <= 4) {
      // sorting network on (key descending, id ascending): a total order, so the result is
      // the same whatever the network
      auto cswap = [&](int a, int b) {
        const bool sw = key[b] > key[a] || (key[b] == key[a] && id[b] < id[a]);
        const uint32_t ka = key[a], ia = id[a];
        key[a] = sw ? key[b] : ka;
        id[a] = sw ? id[b] : ia;
        key[b] = sw ? ka : key[b];
        id[b] = sw ? ia : id[b];
      };
      if constexpr (PER >= 2) cswap(0, 1);
      if constexpr (PER == 3) {
        cswap(1, 2);
        cswap(0, 1);
      }
      if constexpr (PER == 4) {
        cswap(2, 3);
        cswap(0, 2);
        cswap(1, 3);
        cswap(1, 2);
      }
      for (int j = 0; j < k; ++j) {
        const uint32_t top = __reduce_max_sync(0xffffffffu, key[0]);
        const uint32_t win = __reduce_min_sync(0xffffffffu, key[0] == top ? id[0] : kNone);
        if (id[0] == win) {
#pragma unroll
          for (int i = 0; i + 1 < PER; ++i) {
            key[i] = key[i + 1];
            id[i] = id[i + 1];
          }
          key[PER - 1] = 0u;
          id[PER - 1] = kNone;
        }
        if (lane == j) {
          my_id = static_cast<int>(win);
          my_val = key_value(top);
        }
      }
    } else {
      uint32_t taken = 0;
      for (int j = 0; j < k; ++j) {
        // this lane's best untaken key (the lowest id among equal ones: i ascending)
        uint32_t best = 0u, bid = kNone;
        int bi = -1;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
          const bool better = !((taken >> i) & 1u) && id[i] != kNone && (bi < 0 || key[i] > best);
          best = better ? key[i] : best;
          bid = better ? id[i] : bid;
          bi = better ? i : bi;
        }
        const uint32_t top = __reduce_max_sync(0xffffffffu, best);
        const uint32_t win = __reduce_min_sync(0xffffffffu, best == top ? bid : kNone);
        if (bi >= 0 && bid == win) taken |= 1u << bi;
        if (lane == j) {
          my_id = static_cast<int>(win);
          my_val = key_value(top);
        }
      }
    }
    const float m = __shfl_sync(0xffffffffu, my_val, 0);
    const float ex = lane < k ? expf(my_val - m) : 0.0f;
    float sum = ex;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, d);
    if (lane < k) {
      ids[t * k + lane] = my_id;
      gates[t * k + lane] = __fdiv_rn(ex, sum);
    }
  }
}

cudaError_t launch_topk_gate(const float* logits, int64_t T, int E, int k, int32_t* ids,
                             float* gates, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int grid = static_cast<int>(std::min<int64_t>((T + 7) / 8, num_sms() * 16));
  const int per = (E + 31) / 32;
  const dim3 g(grid), b(256);
  if (per <= 1) return launch_chained(topk_kernel<1>, g, b, 0, s, logits, T, E, k, ids, gates);
  if (per <= 2) return launch_chained(topk_kernel<2>, g, b, 0, s, logits, T, E, k, ids, gates);
  if (per <= 4) return launch_chained(topk_kernel<4>, g, b, 0, s, logits, T, E, k, ids, gates);
  if (per <= 8) return launch_chained(topk_kernel<8>, g, b, 0, s, logits, T, E, k, ids, gates);
  if (per <= 16) return launch_chained(topk_kernel<16>, g, b, 0, s, logits, T, E, k, ids, gates);
  return launch_chained(topk_kernel<32>, g, b, 0, s, logits, T, E, k, ids, gates);
}

// ------------------------------------------------------------------------ permutation
size_t permute_scratch_bytes(int64_t T, int E) {
  const int64_t chunks = (T + kChunkTokens - 1) / kChunkTokens;
  return align_up(static_cast<size_t>(chunks) * E * sizeof(int32_t), 256);
}

// (1) per-chunk expert histogram
__global__ void permute_count_kernel(const int32_t* __restrict__ ids, int64_t T, int k, int E,
                                     int32_t* __restrict__ chunk_counts) {
  chain_enter();
  extern __shared__ int hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kChunkTokens;
  const int64_t n = (T - t0 < kChunkTokens ? T - t0 : static_cast<int64_t>(kChunkTokens)) * k;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) atomicAdd(&hist[ids[t0 * k + i]], 1);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    chunk_counts[static_cast<int64_t>(blockIdx.x) * E + e] = hist[e];
}

// (2) exclusive scan: offsets[e] and, in place, the first row of (chunk, expert).  The 1024
// threads split as P = 1024 / E' threads per expert (E' = E rounded up to a power of two),
// thread j of an expert owning a contiguous slice of the chunks, so that the chain of
// dependent loads per thread is chunks / P long instead of chunks.
__global__ void permute_scan_kernel(int32_t* __restrict__ chunk_counts, int64_t chunks, int E,
                                    int32_t* __restrict__ offsets) {
  chain_enter();
  __shared__ int part_sum[1024];   // slice sums, then slice bases within the expert
  __shared__ int totals[1024];     // per expert: total, then the expert's first row
  __shared__ int warp_sums[32];
  int ep2 = 1;
  while (ep2 < E) ep2 <<= 1;
  const int P = static_cast<int>(blockDim.x) / ep2;  // >= 1 (E <= 1024)
  const int t = threadIdx.x;
  const int e = t / P, j = t - (t / P) * P;
  const int64_t per = (chunks + P - 1) / P;
  const int64_t c0 = j * per < chunks ? j * per : chunks;
  const int64_t c1 = c0 + per < chunks ? c0 + per : chunks;
  // pass 1: this slice's count
  int run = 0;
  if (e < E) {
    for (int64_t c = c0; c < c1; c += 8) {
      int cnt[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) cnt[i] = c + i < c1 ? chunk_counts[(c + i) * E + e] : 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) run += cnt[i];
    }
  }
  part_sum[t] = run;
  __syncthreads();
  // slice bases within the expert, and the expert's total
  int base = 0, total = 0;
  if (e < E) {
    for (int i = 0; i < P; ++i) {
      const int v = part_sum[e * P + i];
      if (i < j) base += v;
      total += v;
    }
  }
  __syncthreads();
  part_sum[t] = base;
  if (e < E && j == 0) totals[e] = total;
  __syncthreads();
  // block-wide exclusive scan of the per-expert totals (thread x holds expert x)
  const int lane = t & 31, w = t >> 5;
  const int my_total = t < E ? totals[t] : 0;
  int incl = my_total;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) warp_sums[w] = incl;
  __syncthreads();
  if (w == 0) {
    const int ws = lane < static_cast<int>(blockDim.x >> 5) ? warp_sums[lane] : 0;
    int wi = ws;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, wi, d);
      if (lane >= d) wi += v;
    }
    warp_sums[lane] = wi - ws;
  }
  __syncthreads();
  const int excl = warp_sums[w] + incl - my_total;
  __syncthreads();
  if (t < E) {
    totals[t] = excl;
    offsets[t] = excl;
    if (t == E - 1) offsets[E] = excl + my_total;
  }
  __syncthreads();
  // pass 2: each slice writes the first row of (chunk, expert) for its chunks
  if (e < E) {
    int row = totals[e] + part_sum[t];
    for (int64_t c = c0; c < c1; c += 8) {
      int cnt[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) cnt[i] = c + i < c1 ? chunk_counts[(c + i) * E + e] : 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (c + i < c1) chunk_counts[(c + i) * E + e] = row;
        row += cnt[i];
      }
    }
  }
}

// (3) stable rank.  A block of kRankWarps warps takes one chunk; warp w owns a contiguous
// slice of its tokens.  Pass 1: each warp counts its slice per expert.  Then every warp's
// base per expert is the chunk's base plus the counts of the slices before it.  Pass 2:
// each warp walks its slice in (token, slot) order.  Lanes hold consecutive entries; a
// token's k experts are distinct, so lanes sharing an expert belong to different tokens and
// their lane order is the token order.  The result equals a serial walk of the chunk.
constexpr int kRankWarps = 8;

__global__ void permute_rank_kernel(const int32_t* __restrict__ ids, int64_t T, int k, int E,
                                    const int32_t* __restrict__ chunk_base,
                                    int32_t* __restrict__ row_token,
                                    int32_t* __restrict__ token_row) {
  chain_enter();
  extern __shared__ int sm[];
  int* cnt = sm;                          // [kRankWarps][E]: slice counts, then slice bases
  int* sid = sm + kRankWarps * E;         // the chunk's ids
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t chunk = blockIdx.x;
  const int64_t t0 = chunk * kChunkTokens;
  const int64_t nt = T - t0 < kChunkTokens ? T - t0 : static_cast<int64_t>(kChunkTokens);
  const int64_t n = nt * k;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) sid[i] = ids[t0 * k + i];
  for (int i = threadIdx.x; i < kRankWarps * E; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  // this warp's slice: tokens [w * tps, (w + 1) * tps) of the chunk
  const int64_t tps = (kChunkTokens + kRankWarps - 1) / kRankWarps;
  const int64_t lo = (w * tps < nt ? w * tps : nt) * k;
  const int64_t hi = ((w + 1) * tps < nt ? (w + 1) * tps : nt) * k;
  const int per = (32 / k) * k;  // lanes used per step: whole tokens only
  const uint32_t lt_mask = (1u << lane) - 1u;
  int* my = cnt + w * E;
  for (int64_t base = lo; base < hi; base += per) {       // pass 1: counts
    const int64_t i = base + lane;
    const bool active = lane < per && i < hi;
    const int e = active ? sid[i] : -1 - lane;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (active && (peers >> lane) == 1u) my[e] += __popc(peers);  // highest lane of the group
    __syncwarp();
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {     // slice bases
    int run = chunk_base[chunk * E + e];
#pragma unroll
    for (int ww = 0; ww < kRankWarps; ++ww) {
      const int c = cnt[ww * E + e];
      cnt[ww * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  for (int64_t base = lo; base < hi; base += per) {       // pass 2: ranks
    const int64_t i = base + lane;
    const bool active = lane < per && i < hi;
    const int e = active ? sid[i] : -1 - lane;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    int r = 0;
    if (active) r = my[e] + __popc(peers & lt_mask);
    __syncwarp();
    if (active && (peers >> lane) == 1u) my[e] += __popc(peers);
    __syncwarp();
    if (active) {
      row_token[r] = static_cast<int32_t>(t0 + i / k);
      token_row[t0 * k + i] = r;
    }
  }
}

// (4) copy each token's e4m3 row and scales to its k expert rows: one warp per token,
// each 512-byte slice read once and written k times.
__global__ void permute_copy_kernel(const uint8_t* __restrict__ xq, const float* __restrict__ xs,
                                    int64_t T, int k, int64_t H,
                                    const int32_t* __restrict__ token_row,
                                    uint8_t* __restrict__ aq, float* __restrict__ as) {
  chain_enter();
  const int lane = threadIdx.x & 31;
  const int64_t wid = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t G = H / 128;
  for (int64_t t = wid; t < T; t += nw) {
    const int my_row = lane < k ? __ldg(token_row + t * k + lane) : 0;
    const uint4* src = reinterpret_cast<const uint4*>(xq + t * H);
    for (int64_t c0 = 0; c0 < H / 16; c0 += 32) {  // all lanes iterate; shuffles stay full
      const int64_t c = c0 + lane;
      const bool in = c < H / 16;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (in) v = __ldcs(src + c);
      for (int j = 0; j < k; ++j) {
        const int r = __shfl_sync(0xffffffffu, my_row, j);
        if (in) reinterpret_cast<uint4*>(aq + static_cast<int64_t>(r) * H)[c] = v;
      }
    }
    for (int64_t g0 = 0; g0 < G; g0 += 32) {
      const int64_t g = g0 + lane;
      const bool in = g < G;
      const float sv = in ? __ldg(xs + t * G + g) : 0.0f;
      for (int j = 0; j < k; ++j) {
        const int r = __shfl_sync(0xffffffffu, my_row, j);
        if (in) as[static_cast<int64_t>(r) * G + g] = sv;
      }
    }
  }
}

// The magnitudes of a lane's 8 bfloat16 values, pairwise maxima packed two per word: the
// low 15 bits of a bfloat16 order like its absolute value, so an unsigned maximum of
// (w & 0x7fff) over values is the pattern of their largest |x|.  A pattern at or above 0x7f80
// is an infinity or a NaN.
__device__ __forceinline__ uint32_t mag_bits_pack(const uint4& v) {
  return __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                  __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
}

// amax of each 128-value group for U groups per lane group of a warp: a group's values are
// spread over 16 / W adjacent lanes, W x 8 per lane, lane's share v[u W .. u W + W) for its
// u-th group.  While every value the warp holds is finite, amax comes from the bit patterns.
// Otherwise the whole warp takes the float path (the maximum over the finite values, as the
// division-based quantizer defines it), and each lane holding an infinity or a NaN reports
// it to status; the scale and codes of such a group are meaningless (an infinite amax
// becomes a NaN scale in g128_scale).  All 32 lanes call it (the shuffles and the vote are
// warp-wide); the U reductions are interleaved.
template <int U, int W>
__device__ __forceinline__ void g128_amax(const uint4 (&v)[U * W], float (&amax)[U],
                                          int32_t* status) {
  uint32_t mb[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    uint32_t m = mag_bits_pack(v[u * W]);
#pragma unroll
    for (int w = 1; w < W; ++w) m = __vmaxu2(m, mag_bits_pack(v[u * W + w]));
    mb[u] = max(m & 0xFFFFu, m >> 16);
  }
#pragma unroll
  for (int d = 8 / W; d > 0; d >>= 1)
#pragma unroll
    for (int u = 0; u < U; ++u) mb[u] = max(mb[u], __shfl_xor_sync(0xffffffffu, mb[u], d));
  uint32_t top = 0;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    top = max(top, mb[u]);
    amax[u] = __uint_as_float(mb[u] << 16);
  }
  if (!__any_sync(0xffffffffu, top >= 0x7F80u)) return;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    float a = 0.0f, b = 0.0f;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      const uint4& x = v[u * W + w];
      const float f[8] = {bf16_lo(x.x), bf16_hi(x.x), bf16_lo(x.y), bf16_hi(x.y),
                          bf16_lo(x.z), bf16_hi(x.z), bf16_lo(x.w), bf16_hi(x.w)};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        a = fmaxf(a, fabsf(f[i]));
        b = nonfinite_fold(b, f[i]);
      }
    }
    report_nonfinite(status, b);
#pragma unroll
    for (int d = 8 / W; d > 0; d >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, d));
    amax[u] = a;
  }
}

// The group's scale s = max(RN(amax / 448), 2^-126), 1 for an all-zero group: the quotient
// by the correction step of quotient.cuh from the constant RN(1/448) = 0x1.24924ap-9.  The
// product q0 * 448 = 7 q0 * 64 is a multiple of 64 ulp(q0), so the residual is exact for
// every amax, and the result equals the division for every finite bfloat16 amax (all 2^15
// magnitudes checked on the host).  An infinite amax gives NaN.
__device__ __forceinline__ float g128_scale(float amax) {
  float s = quot_rn(amax, 448.0f, 0x1.24924ap-9f);
  if (amax == 0.0f) s = 1.0f;
  if (s < 0x1p-126f) s = 0x1p-126f;
  return s;
}

// (4') quantize and copy in one pass: one warp per token reads its bf16 row once, quantizes
// each 128-value group as quant_g128_kernel does (shuffle amax, s = amax / 448, the IEEE
// quotient x / s, e4m3 round to nearest even; here 16 lanes x 8 values a group) and writes
// the codes and the scale to the token's k expert rows.  Two groups per warp step.
__global__ void permute_quant_copy_kernel(const uint4* __restrict__ x, int64_t T, int k,
                                          int64_t H, const int32_t* __restrict__ token_row,
                                          uint8_t* __restrict__ aq, float* __restrict__ as,
                                          int32_t* status) {
  chain_enter();
  const int lane = threadIdx.x & 31;
  const int half = lane >> 4, hl = lane & 15;
  const int64_t wid = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t G = H / 128;
  constexpr int U = 4;  // group pairs per trip: their loads are issued together
  for (int64_t t = wid; t < T; t += nw) {
    const int my_row = lane < k ? __ldg(token_row + t * k + lane) : 0;
    for (int64_t g0 = 0; g0 < G; g0 += 2 * U) {  // all lanes iterate; shuffles stay full
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t g = g0 + 2 * u + half;
        v[u] = g < G ? __ldcs(x + (t * G + g) * 16 + hl) : make_uint4(0, 0, 0, 0);
      }
      float amax[U];
      g128_amax<U, 1>(v, amax, status);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t g = g0 + 2 * u + half;
        const bool in = g < G;
        const float sc = g128_scale(amax[u]);
        const uint2 q = cast8(v[u], sc, __frcp_rn(sc), quot_fast_ok(sc));
        for (int j = 0; j < k; ++j) {
          const int64_t r = __shfl_sync(0xffffffffu, my_row, j);
          if (in) {
            reinterpret_cast<uint2*>(aq + r * H)[g * 16 + hl] = q;
            if (hl == 0) as[r * G + g] = sc;
          }
        }
      }
    }
  }
}

cudaError_t launch_permute_quant(const int32_t* ids, int64_t T, int k, int E,
                                 const uint16_t* x, int64_t H, int32_t* offsets,
                                 int32_t* row_token, int32_t* token_row, uint8_t* aq, float* as,
                                 void* scratch, int32_t* status, cudaStream_t s) {
  cudaError_t e = launch_permute(ids, T, k, E, nullptr, nullptr, H, offsets, row_token,
                                 token_row, nullptr, nullptr, scratch, s);
  if (e != cudaSuccess || T == 0) return e;
  const int grid = static_cast<int>(std::min<int64_t>((T + 7) / 8, num_sms() * 8));
  return launch_chained(permute_quant_copy_kernel, dim3(grid), dim3(256), 0, s,
                        reinterpret_cast<const uint4*>(x), T, k, H, token_row, aq, as, status);
}

cudaError_t launch_permute(const int32_t* ids, int64_t T, int k, int E, const uint8_t* xq,
                           const float* xs, int64_t H, int32_t* offsets, int32_t* row_token,
                           int32_t* token_row, uint8_t* aq, float* as, void* scratch,
                           cudaStream_t s) {
  const int64_t chunks = (T + kChunkTokens - 1) / kChunkTokens;
  int32_t* cc = reinterpret_cast<int32_t*>(scratch);
  if (chunks > 0) {
    const cudaError_t e = launch_chained(permute_count_kernel, dim3(static_cast<int>(chunks)),
                                         dim3(256), E * sizeof(int), s, ids, T, k, E, cc);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = launch_chained(permute_scan_kernel, dim3(1), dim3(1024), 0, s, cc, chunks, E,
                                 offsets);
  if (e != cudaSuccess || chunks == 0) return e;
  e = launch_chained(permute_rank_kernel, dim3(static_cast<int>(chunks)), dim3(32 * kRankWarps),
                     (kRankWarps * E + kChunkTokens * k) * sizeof(int), s, ids, T, k, E, cc,
                     row_token, token_row);
  if (e != cudaSuccess) return e;
  if (aq == nullptr) return cudaSuccess;  // index-only: the GEMM gathers rows by row_token
  const int grid = static_cast<int>(std::min<int64_t>((T + 7) / 8, num_sms() * 8));
  return launch_chained(permute_copy_kernel, dim3(grid), dim3(256), 0, s, xq, xs, T, k, H,
                        token_row, aq, as);
}

// ----------------------------------------------------------------------------- combine
template <bool YF32, bool OF32>
__global__ void combine_kernel(const void* __restrict__ y, const int32_t* __restrict__ token_row,
                               const float* __restrict__ gates, int64_t T, int k, int64_t H,
                               void* __restrict__ out) {
  // one warp per token and per 2048-column block; lane l owns columns l*8 + 256*c (c < 8).
  // Each slot's row block (4 KB in bf16) is read as 8 independent 16-byte loads per lane
  // and summed in slot order.
  const int lane = threadIdx.x & 31;
  const int64_t wid = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t nb = (H + 2047) / 2048;
  for (int64_t item = wid; item < T * nb; item += nw) {
    const int64_t t = item / nb;
    const int64_t c0 = (item - t * nb) * 2048;
    const int my_row = lane < k ? __ldg(token_row + t * k + lane) : 0;
    const float my_gate = lane < k ? __ldg(gates + t * k + lane) : 0.0f;
    float acc[8][8];
#pragma unroll
    for (int c = 0; c < 8; ++c)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[c][i] = 0.0f;
    for (int j = 0; j < k; ++j) {
      const int64_t r = __shfl_sync(0xffffffffu, my_row, j);
      const float g = __shfl_sync(0xffffffffu, my_gate, j);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int64_t col = c0 + 256 * c + lane * 8;
        if (col >= H) continue;
        float v[8];
        if constexpr (YF32) {
          const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(y) + r * H + col);
          const float4 a = __ldcs(p), b = __ldcs(p + 1);
          v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        } else {
          const uint4 a = __ldcs(reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(y) + r * H + col));
          v[0] = bf16_lo(a.x); v[1] = bf16_hi(a.x); v[2] = bf16_lo(a.y); v[3] = bf16_hi(a.y);
          v[4] = bf16_lo(a.z); v[5] = bf16_hi(a.z); v[6] = bf16_lo(a.w); v[7] = bf16_hi(a.w);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[c][i] = fmaf(g, v[i], acc[c][i]);
      }
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int64_t col = c0 + 256 * c + lane * 8;
      if (col >= H) continue;
      if constexpr (OF32) {
        float4* o = reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + t * H + col);
        o[0] = make_float4(acc[c][0], acc[c][1], acc[c][2], acc[c][3]);
        o[1] = make_float4(acc[c][4], acc[c][5], acc[c][6], acc[c][7]);
      } else {
        *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(out) + t * H + col) =
            make_uint4(pack_bf16x2(acc[c][0], acc[c][1]), pack_bf16x2(acc[c][2], acc[c][3]),
                       pack_bf16x2(acc[c][4], acc[c][5]), pack_bf16x2(acc[c][6], acc[c][7]));
      }
    }
  }
}

// The layer's combine (bf16 y, k <= 8, H a multiple of 2048) through bulk copies.  An item
// is (token t, 2048-column block); its k slot rows' blocks of y are 4 KB each and
// contiguous, so a producer warp copies them into a shared-memory stage with k
// cp.async.bulk copies counted on the stage's mbarrier, and eight consumer warps sum them in
// slot order with the same fmaf chain as combine_kernel (thread i owns columns 8 i .. 8 i + 7
// of the block), so the results are the same bits.  Three stages keep three items' 96 KB in
// flight per CTA, two CTAs per SM, without holding the rows in registers.  Every wait is
// bounded: one that runs out records FGE_ERR_DEVICE_TIMEOUT in *status and the CTA stops.
constexpr int kCombCols = 2048, kCombStages = 3, kCombMaxK = 8;
constexpr int kCombStageBytes = kCombMaxK * kCombCols * 2;
constexpr int kCombSmem = kCombStages * kCombStageBytes + 2 * kCombStages * 8;

__device__ __forceinline__ void comb_bulk_load(uint32_t smem_dst, const void* src, uint32_t bytes,
                                               uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

template <bool OF32>
__global__ void __launch_bounds__(288)
    combine_bulk_kernel(const uint16_t* __restrict__ y, const int32_t* __restrict__ token_row,
                        const float* __restrict__ gates, int64_t T, int k, int64_t H,
                        void* __restrict__ out, int32_t* status) {
  extern __shared__ __align__(128) uint8_t csm[];
  __shared__ int s_abort;
  const uint32_t stage0 = smem_u32(csm);
  const uint32_t full0 = stage0 + kCombStages * kCombStageBytes;
  const uint32_t empty0 = full0 + 8 * kCombStages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kCombStages; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, 8);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int64_t nb = H / kCombCols;
  const int64_t items = T * nb;
  uint32_t it = 0;
  if (warp == 8) {
    // producer: lane j < k copies slot row j's block of the item
    for (int64_t item = blockIdx.x; item < items; item += gridDim.x, ++it) {
      const uint32_t st = it % kCombStages;
      if (!mbar_wait(empty0 + 8 * st, ((it / kCombStages) & 1) ^ 1, &s_abort, status)) break;
      const int64_t t = item / nb;
      const int64_t c0 = (item - t * nb) * kCombCols;
      if (lane == 0) mbar_arrive_expect_tx(full0 + 8 * st, static_cast<uint32_t>(k) * kCombCols * 2);
      __syncwarp();
      if (lane < k) {
        const int64_t r = __ldg(token_row + t * k + lane);
        comb_bulk_load(stage0 + st * kCombStageBytes + lane * (kCombCols * 2), y + r * H + c0,
                       kCombCols * 2, full0 + 8 * st);
      }
    }
  } else {
    for (int64_t item = blockIdx.x; item < items; item += gridDim.x, ++it) {
      const uint32_t st = it % kCombStages;
      const int64_t t = item / nb;
      const int64_t c0 = (item - t * nb) * kCombCols;
      const float my_gate = lane < k ? __ldg(gates + t * k + lane) : 0.0f;
      if (!mbar_wait(full0 + 8 * st, (it / kCombStages) & 1, &s_abort, status)) break;
      const uint8_t* src = csm + st * kCombStageBytes + threadIdx.x * 16;
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
      for (int j = 0; j < k; ++j) {
        const float g = __shfl_sync(0xffffffffu, my_gate, j);
        const uint4 a = *reinterpret_cast<const uint4*>(src + j * (kCombCols * 2));
        const float v[8] = {bf16_lo(a.x), bf16_hi(a.x), bf16_lo(a.y), bf16_hi(a.y),
                            bf16_lo(a.z), bf16_hi(a.z), bf16_lo(a.w), bf16_hi(a.w)};
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(g, v[i], acc[i]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * st);
      const int64_t col = c0 + threadIdx.x * 8;
      if constexpr (OF32) {
        float4* o = reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + t * H + col);
        o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
      } else {
        *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(out) + t * H + col) =
            make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                       pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
      }
    }
  }
}

// Arrival counters of the combine folded into the down GEMM set to zero, and the combine's
// arguments written where the GEMM reads them.
__global__ void combine_setup_kernel(FusedCombine c, int64_t n, FusedCombine* dst) {
  if (blockIdx.x == 0 && threadIdx.x == 0) *dst = c;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    c.count[i] = 0;
}

cudaError_t launch_combine_setup(const FusedCombine& c, int64_t n, FusedCombine* dst,
                                 cudaStream_t s) {
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, 4L * num_sms());
  combine_setup_kernel<<<static_cast<int>(std::max<int64_t>(blocks, 1)), 256, 0, s>>>(c, n, dst);
  return cudaGetLastError();
}

cudaError_t launch_combine(const void* y, int y_f32, const int32_t* token_row,
                           const float* gates, int64_t T, int k, int64_t H, int out_f32,
                           void* out, cudaStream_t s, int32_t* status) {
  if (T == 0) return cudaSuccess;
  if (status && !y_f32 && k <= kCombMaxK && H % kCombCols == 0) {
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return ce;
    const void* kern = out_f32 ? reinterpret_cast<const void*>(combine_bulk_kernel<true>)
                               : reinterpret_cast<const void*>(combine_bulk_kernel<false>);
    if (device_kernel_ready(dev, kern, kCombSmem, 0)) {
      const int64_t items = T * (H / kCombCols);
      const int grid = static_cast<int>(std::min<int64_t>(items, 2LL * num_sms()));
      const uint16_t* yb = static_cast<const uint16_t*>(y);
      if (out_f32)
        combine_bulk_kernel<true><<<grid, 288, kCombSmem, s>>>(yb, token_row, gates, T, k, H,
                                                               out, status);
      else
        combine_bulk_kernel<false><<<grid, 288, kCombSmem, s>>>(yb, token_row, gates, T, k, H,
                                                                out, status);
      return cudaGetLastError();
    }
  }
  const int64_t items = T * ((H + 2047) / 2048);
  const int grid = static_cast<int>(std::min<int64_t>((items + 7) / 8, num_sms() * 8));
  if (y_f32 && out_f32) combine_kernel<true, true><<<grid, 256, 0, s>>>(y, token_row, gates, T, k, H, out);
  else if (y_f32) combine_kernel<true, false><<<grid, 256, 0, s>>>(y, token_row, gates, T, k, H, out);
  else if (out_f32) combine_kernel<false, true><<<grid, 256, 0, s>>>(y, token_row, gates, T, k, H, out);
  else combine_kernel<false, false><<<grid, 256, 0, s>>>(y, token_row, gates, T, k, H, out);
  return cudaGetLastError();
}

// The stand-alone G128 activation quantization.  Rows hold whole groups (K % 128 == 0), so
// the tensor is a flat array of M * K / 128 groups whose scales are stored in the same order.
// Each quarter-warp (8 lanes) quantizes one group, 16 values a lane (bytes [32 j, 32 j + 32)
// of the group for lane j, and 16 code bytes out), so the per-group work -- the scale, its
// reciprocal, the range test -- is spread over 16 values instead of the quantizing copy's 8,
// with the same codes and scales.  The warps stride over group quads with kQuantQuads quads'
// loads in flight, so every warp gets the same share of the tensor whatever M and K are.
__global__ void __launch_bounds__(256, kQuantBlocks)
    quant_g128_kernel(const uint4* __restrict__ x, int64_t ngroups,
                      uint4* __restrict__ xq, float* __restrict__ xs, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int quarter = lane >> 3, ql = lane & 7;
  const int64_t wid = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t nquads = (ngroups + 3) / 4;
  for (int64_t p0 = wid; p0 < nquads; p0 += nw * kQuantQuads) {  // warp-uniform trips
    uint4 v[2 * kQuantQuads];
#pragma unroll
    for (int u = 0; u < kQuantQuads; ++u) {
      const int64_t g = 4 * (p0 + u * nw) + quarter;
      const bool in = g < ngroups;
      v[2 * u] = in ? __ldcs(x + g * 16 + 2 * ql) : make_uint4(0, 0, 0, 0);
      v[2 * u + 1] = in ? __ldcs(x + g * 16 + 2 * ql + 1) : make_uint4(0, 0, 0, 0);
    }
    float amax[kQuantQuads];
    g128_amax<kQuantQuads, 2>(v, amax, status);
#pragma unroll
    for (int u = 0; u < kQuantQuads; ++u) {
      const int64_t g = 4 * (p0 + u * nw) + quarter;
      const float sc = g128_scale(amax[u]);
      const float y = __frcp_rn(sc);
      const bool fast = quot_fast_ok(sc);
      if (g < ngroups) {
        const uint2 lo = cast8(v[2 * u], sc, y, fast), hi = cast8(v[2 * u + 1], sc, y, fast);
        __stcs(xq + g * 8 + ql, make_uint4(lo.x, lo.y, hi.x, hi.y));
        if (ql == 0) xs[g] = sc;
      }
    }
  }
}

cudaError_t launch_quant_g128(const uint16_t* x, int64_t M, int64_t K, uint8_t* xq, float* xs,
                              int32_t* status, cudaStream_t s) {
  const int64_t ngroups = M * (K / 128);
  if (ngroups == 0) return cudaSuccess;
  const int64_t quads = (ngroups + 3) / 4;
  // kQuantBlocks blocks of 256 threads are resident per SM (launch bounds): one wave
  const int grid = static_cast<int>(std::min<int64_t>(
      (quads + 8 * kQuantQuads - 1) / (8 * kQuantQuads), num_sms() * kQuantBlocks));
  quant_g128_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const uint4*>(x), ngroups,
                                         reinterpret_cast<uint4*>(xq), xs, status);
  return cudaGetLastError();
}

}  // namespace fge

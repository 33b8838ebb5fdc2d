// Grouped expert GEMM for sm_103a: one persistent, warp-specialised kernel that runs the
// W4A8 expert GEMMs of an MoE layer ("FP8 grouped-expert prefill with on-chip
// int4-to-e4m3 dequant", section 1) and, run with one expert and per-tensor scales, the
// dense W8A8 projection ("feat(qwen4_exp): load-time per-tensor FP8 dense projections").
//
// Per CTA (one per SM), warp roles:
//   warps 0-3   unpack: int4 tile (shared memory) -> e4m3 in the 128-byte swizzle layout;
//               with MXFP4 activations also the K group's block scales into TMEM
//   warp  6     TMA producer: A tile [128 rows x 128 K] + B tile per K group
//   warp  7     TMEM allocator and single-thread tcgen05.mma issuer (kind::f8f6f4, or the
//               block-scaled kind::mxf8f6f4 for MXFP4 activations)
//   warps 4-5   idle
//   warps 8..   epilogue warpgroups: per-group fp32 promotion acc += as*sw*P from TMEM,
//               then the store / SwiGLU + requant epilogue (optionally the folded combine)
// A K group (128 values) is exactly one 128-byte swizzle atom row, so each pipeline
// stage carries one group and each group is 4 MMAs of K = 32 into a fresh TMEM buffer.
// Two TMEM buffers (2 x BN columns) let the MMA run one group ahead of the promotion.
// Run with one group (per-tensor scales) the whole K accumulates in TMEM; at decode sizes
// K may be split over several CTAs per output tile (SplitArgs).
#include <algorithm>
#include <mutex>
#include <cudaTypedefs.h>

#include "fge_device.cuh"

namespace fge {

enum { kBfmtInt4Lut = 0, kBfmtInt4Sub = 1, kBfmtE4m3 = 2 };
enum { kEpiF32 = 0, kEpiBf16 = 1, kEpiSwiglu = 2 };
// activation (A) operand: e4m3 codes, or MXFP4 (E2M1 codes, one UE8M0 scale per 32 values)
enum { kAfmtE4m3 = 0, kAfmtMxf4 = 1 };
// control warps (warpgroup 1); epilogue warps 8..15 keep their lane quarters
constexpr int kProducerWarp = 6, kMmaWarp = 7;

struct GemmParams {
  const float* as;         // [R, G] activation group scales
  const float* sw;         // [E, G, N] prepacked weight group scales
  const float* sa_tensor;  // per-tensor activation scale (device scalar)
  const float* sa_rows;    // per-row activation scales [rows] (one-group path), or null
  const float* sw_tensor;  // per-tensor weight scale (device scalar)
  const int32_t* offsets;  // [E+1]
  const int32_t* row_token;  // gather mode: A row of routed row r is row_token[r], else null
  void* out;
  float* out_scales;
  int32_t* status;
  int E, N, K, G;
  int dense_rows;          // offsets == nullptr: one expert owning rows [0, dense_rows)
  int swap_m;              // BN = 16 (decode sizes): tokens in the B tile; out is [swap_m, out_ld]
  int out_ld;
  const uint8_t* sf_a;     // MXFP4 activations: [R, K/32] UE8M0 block scales
  const FusedCombine* comb; // bf16 group-mode store: the combine folded into the epilogue
                           // (device memory; null: plain store)
};

// K split of the one-group (per-tensor) GEMM, a kernel argument of its own.
struct SplitArgs {
  float* partials;         // [tiles, ksplit, 128, BN] fp32 partials
  int32_t* split_count;    // [tiles, epilogue warps] arrival counters (start at 0)
  int ksplit;              // CTAs per tile, each a contiguous range of K groups (1: none)
};

constexpr int align16(int x) { return (x + 15) / 16 * 16; }

template <int BN, int BFMT, int EPI, int AFMT = kAfmtE4m3>
struct Cfg {
  static constexpr bool kInt4 = BFMT != kBfmtE4m3;
  // MXFP4 activations: the TMA expands the packed E2M1 rows into the 16-byte-padded layout
  // the MMA reads (16 values in the low 8 bytes of every 16), so an A stage is the same
  // 128 rows x 128 bytes as for e4m3; the block scales go to TMEM beside the accumulators
  static constexpr bool kMxA = AFMT == kAfmtMxf4;
  static constexpr bool kGroupScale = kInt4;  // int4 path: per-group; e4m3 path: per-tensor
  static constexpr int kABytes = 128 * 128;
  static constexpr int kBLoadBytes = kInt4 ? BN * 64 : BN * 128;
  static constexpr int kBUBytes = BN * 128;
  static constexpr int kNU = kInt4 ? 2 : 0;
  static constexpr int kStageBytes = kABytes + kBLoadBytes;
  // bytes the TMA reports per stage: the padded E2M1 copy writes only the 8 data bytes of
  // every 16-byte chunk, half of the A tile's footprint
  static constexpr int kStageTx = (AFMT == 1 ? kABytes / 2 : kABytes) + kBLoadBytes;
  static constexpr int kPipeBytes = 192 * 1024;
  static constexpr int kNS = (kPipeBytes - kNU * kBUBytes) / kStageBytes;
  // one warpgroup per 128 columns; the 16-column decode tile still needs all 128 lanes
  static constexpr int kEpiWarps = BN >= 128 ? BN / 32 : 4;
  static constexpr int kEpiThreads = kEpiWarps * 32;
  static constexpr int kThreads = 256 + kEpiThreads;
  static constexpr int kTmemCols = kMxA ? 512 : 2 * BN;
  // MXFP4: TMEM columns of the activation scale ring (4 per unpack slot: lane l of every
  // lane quarter, column j, byte b = the scale of tile row l + 32 j, K step b) and of the
  // weight-side scales (all 2^0)
  static constexpr int kSfaCol = 2 * BN;
  static constexpr int kSfbCol = 2 * BN + 4 * kNU;
  // group mode: each epilogue warpgroup owns 128 columns ("half") of every TMEM buffer with
  // its own full/empty barriers, so the halves pipeline independently of each other
  static constexpr int kHalves = 1;  // one hand-off per buffer: N = BN per MMA instruction
  // register split (group mode only): the unpack warpgroup keeps a working set for 16
  // units in flight, the producer/MMA warpgroup needs few, the epilogue holds 128 fp32
  // accumulators per thread plus two TMEM chunks in flight.
  static constexpr int kLaunchRegs = (65536 / kThreads) / 8 * 8;
  static constexpr int kRegsUnpack = 64;
  static constexpr int kRegsCtrl = 32;
  static constexpr int kRegsHigh0 =
      (kLaunchRegs * kThreads - 128 * kRegsUnpack - 128 * kRegsCtrl) / kEpiThreads / 8 * 8;
  static constexpr int kRegsHigh = kRegsHigh0 > 240 ? 240 : kRegsHigh0;
  // shared memory layout (offsets from a 1024-aligned base)
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kNS * kABytes;
  static constexpr int kOffBU = kOffB + kNS * kBLoadBytes;
  static constexpr int kNSW = kGroupScale ? 4 : 0;  // weight-scale ring (one K group each)
  static constexpr int kSWBytes = BN * 4;
  static constexpr int kOffSW = kOffBU + kNU * kBUBytes;
  static constexpr int kOffBar = kOffSW + kNSW * kSWBytes;
  static constexpr int kNumBars = 2 * kNS + 2 * kNU + 4 * kHalves + 1 + 2 * kNSW;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kOffOffs = align16(kOffMisc + 16);
  static constexpr int kOffMtp = kOffOffs + (kMaxExperts + 1) * 4;
  static constexpr int kOffRed = align16(kOffMtp + (kMaxExperts + 1) * 4);
  static constexpr int kOffRT = align16(kOffRed + 2 * 2 * 128 * 4);  // gather: tile row ids
  // bf16 and SwiGLU store epilogues (group mode): per warpgroup one 8 KB buffer, a 2 KB
  // slice per warp staging that warp's 32 rows for its own TMA tile stores
  static constexpr bool kStageOut = kGroupScale && (EPI == kEpiBf16 || EPI == kEpiSwiglu);
  static constexpr int kOffST = (kOffRT + 128 * 4 + 1023) / 1024 * 1024;
  static constexpr int kSTBytes = kStageOut ? 2 * 8192 : 0;
  static constexpr int kSmemBytes = kOffST + kSTBytes + 1024;  // + alignment slack
  static_assert(kNS >= 2, "pipeline needs at least two stages");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// 1-D bulk copy global -> shared, completion counted on an mbarrier (16-byte multiples).
__device__ __forceinline__ void bulk_load(uint32_t smem_dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  return static_cast<uint64_t>(__float_as_uint(lo)) |
         (static_cast<uint64_t>(__float_as_uint(hi)) << 32);
}

// acc2 (two fp32 in a 64-bit register) += (sa2 * w2) * (p0, p1), packed f32x2 math.
__device__ __forceinline__ void fma2_pair(uint64_t& acc2, uint64_t sa2, uint64_t w2, uint32_t p0,
                                          uint32_t p1) {
  asm("{\n\t.reg .b64 pp, ss;\n\t"
      "mov.b64 pp, {%1, %2};\n\t"
      "mul.rn.f32x2 ss, %3, %4;\n\t"
      "fma.rn.f32x2 %0, ss, pp, %0;\n\t}"
      : "+l"(acc2)
      : "r"(p0), "r"(p1), "l"(sa2), "l"(w2));
}

__device__ __forceinline__ float lo_f32(uint64_t v) {
  return __uint_as_float(static_cast<uint32_t>(v));
}
__device__ __forceinline__ float hi_f32(uint64_t v) {
  return __uint_as_float(static_cast<uint32_t>(v >> 32));
}

// Values loaded from TMEM may only be used after tcgen05.wait::ld; this empty volatile asm,
// ordered after the wait, makes every later use depend on it.
__device__ __forceinline__ void reg_fence16(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]));
}

__device__ __forceinline__ void reg_fence32(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31]));
}

// 8 int4 values (two's complement, nibble i = element i) -> e4m3 codes of the integers.
// Two 8-entry byte-permute tables (codes of 0..7 and of -8..-1) and a per-byte select.
__device__ __forceinline__ uint2 w4_to_e4m3_lut(uint32_t w) {
  const uint32_t idx = w & 0x77777777u;
  const uint32_t t = w & 0x88888888u;
  const uint32_t msel = t | (t >> 3);  // nibble 0x9 (sign of byte 1 = 0xFF) when negative
  const uint32_t pl = prmt(0x44403800u, 0x4E4C4A48u, idx);
  const uint32_t ph = prmt(0x44403800u, 0x4E4C4A48u, idx >> 16);
  const uint32_t nl = prmt(0xCACCCED0u, 0xB8C0C4C8u, idx);
  const uint32_t nh = prmt(0xCACCCED0u, 0xB8C0C4C8u, idx >> 16);
  const uint32_t ml = prmt(0x00008000u, 0u, msel);
  const uint32_t mh = prmt(0x00008000u, 0u, msel >> 16);
  return make_uint2((pl & ~ml) | (nl & ml), (ph & ~mh) | (nh & mh));
}

// 8 int4 values in the subnormal bank order (byte b: low nibble = element b, high nibble =
// element b+4) -> e4m3 codes of q * 2^-9.  Those codes are the integer in sign-magnitude
// form: q >= 0 -> q; q < 0 -> 0x80 | -q (for the nibble x = q + 16: 0x90 - x).
__device__ __forceinline__ uint2 w4_to_e4m3_sub(uint32_t w) {
  const uint32_t lo = w & 0x0F0F0F0Fu;
  const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;
  const uint32_t ml = prmt(w << 4, 0u, 0xBA98u);  // 0xFF per negative element 0..3
  const uint32_t mh = prmt(w, 0u, 0xBA98u);       // 0xFF per negative element 4..7
  const uint32_t dl = 0x90909090u - lo;
  const uint32_t dh = 0x90909090u - hi;
  return make_uint2((lo & ~ml) | (dl & ml), (hi & ~mh) | (dh & mh));
}

struct TileInfo {
  int e, row0, rows, n0;
};

__device__ __forceinline__ TileInfo decode_tile(int t, int nt_count, int bn, const int* s_off,
                                                const int* s_mtp, int E) {
  const int mt = t / nt_count;
  const int nt = t - mt * nt_count;
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_mtp[mid] <= mt) lo = mid; else hi = mid;
  }
  TileInfo ti;
  ti.e = lo;
  ti.row0 = s_off[lo] + (mt - s_mtp[lo]) * 128;
  ti.rows = min(128, s_off[lo + 1] - ti.row0);
  ti.n0 = nt * bn;
  return ti;
}

// K split over ks CTAs: after this warp has written its partial rows, publishes them and
// counts its arrival for (tile, epilogue warp).  True in every lane of the ks-th warp to
// arrive, for which every split's partials are then visible; the counter wraps back to 0.
__device__ __forceinline__ bool split_arrive_last(int32_t* count, int ks, int lane) {
  __threadfence();
  __syncwarp();
  unsigned last = 0;
  if (lane == 0)
    last = atomicInc(reinterpret_cast<unsigned*>(count), static_cast<unsigned>(ks - 1)) ==
           static_cast<unsigned>(ks - 1);
  last = __shfl_sync(0xffffffffu, last, 0);
  if (last) __threadfence();
  return last != 0u;
}

// Wait that ignores the abort flag (used to drain copies/MMAs already in flight).
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitBudgetCycles) return;
  }
}

template <int BN, int BFMT, int EPI, int AFMT = kAfmtE4m3>
__global__ void __launch_bounds__(Cfg<BN, BFMT, EPI, AFMT>::kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmY, const GemmParams p,
                        const SplitArgs sk) {
  using C = Cfg<BN, BFMT, EPI, AFMT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  const uint32_t bar_full = smem_u32(bars);
  const uint32_t bar_empty = bar_full + 8 * C::kNS;
  const uint32_t bar_ufull = bar_empty + 8 * C::kNS;
  const uint32_t bar_uempty = bar_ufull + 8 * C::kNU;
  const uint32_t bar_tfull = bar_uempty + 8 * C::kNU;
  const uint32_t bar_tempty = bar_tfull + 16 * C::kHalves;
  const uint32_t bar_drain = bar_tempty + 16 * C::kHalves;
  const uint32_t bar_swfull = bar_drain + 8;
  const uint32_t bar_swempty = bar_swfull + 8 * C::kNSW;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  int* s_off = reinterpret_cast<int*>(smem + C::kOffOffs);
  int* s_mtp = reinterpret_cast<int*>(smem + C::kOffMtp);
  float* s_red = reinterpret_cast<float*>(smem + C::kOffRed);

  const int E = p.E;
  const int G = p.G;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kNS; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, C::kInt4 ? 5 : 1);
    }
    for (int i = 0; i < C::kNU; ++i) {
      mbar_init(bar_ufull + 8 * i, 4);
      mbar_init(bar_uempty + 8 * i, 1);
    }
    for (int i = 0; i < 2 * C::kHalves; ++i) {
      mbar_init(bar_tfull + 8 * i, 1);
      mbar_init(bar_tempty + 8 * i, C::kEpiWarps / C::kHalves);
    }
    mbar_init(bar_drain, 1);
    for (int i = 0; i < C::kNSW; ++i) {
      mbar_init(bar_swfull + 8 * i, 1);
      mbar_init(bar_swempty + 8 * i, C::kEpiWarps);
    }
    *s_abort = 0;
    fence_mbar_init();
  }
  if (p.offsets) {
    for (int i = threadIdx.x; i <= E; i += blockDim.x) s_off[i] = p.offsets[i];
  } else if (threadIdx.x == 0) {
    s_off[0] = 0;
    s_off[1] = p.dense_rows;
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(s_tmem), C::kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 0) {
    // exclusive prefix of per-expert m-tile counts
    int carry = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      const int cnt = e < E ? (s_off[e + 1] - s_off[e] + 127) / 128 : 0;
      int incl = cnt;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
      }
      if (e < E) s_mtp[e] = carry + incl - cnt;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s_mtp[E] = carry;
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int nt_count = p.N / BN;
  const int base_tiles = s_mtp[E] * nt_count;
  // one-group mode may split K over ks CTAs per tile, each taking a contiguous range of K
  // groups; the last of them to finish adds the fp32 partials in split order
  const int ks = C::kGroupScale ? 1 : sk.ksplit;
  const int total_tiles = base_tiles * ks;

  if (warp < 4) {
    // ------------------------------------------------------------------ unpack (WG0)
    if constexpr (C::kGroupScale) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::kRegsUnpack));
    if constexpr (C::kInt4) {
      const int tid = threadIdx.x;  // 0..127
      uint32_t it = 0;
      bool ok = true;
      // MXFP4: this warp's TMEM lane quarter; the weight-side scales are all 2^0 (code 127)
      const uint32_t quarter = static_cast<uint32_t>(warp * 32) << 16;
      if constexpr (C::kMxA) {
        tmem_st_32x32b_x4(tmem_base + quarter + C::kSfbCol, 0x7F7F7F7Fu, 0x7F7F7F7Fu,
                          0x7F7F7F7Fu, 0x7F7F7F7Fu);
        tmem_wait_st();
      }
      for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
        TileInfo ti{};
        if constexpr (C::kMxA) ti = decode_tile(t, nt_count, BN, s_off, s_mtp, E);
        for (int g = 0; g < G; ++g, ++it) {
          // MXFP4: the four K-step scales of tile rows lane + 32 j of this group, one 32-bit
          // word per row (rows past the tile read as 2^0; their results are never stored)
          uint32_t sfw[4] = {0u, 0u, 0u, 0u};
          if constexpr (C::kMxA) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int rr = lane + 32 * j;
              sfw[j] = rr < ti.rows
                           ? __ldg(reinterpret_cast<const uint32_t*>(
                                       p.sf_a + static_cast<size_t>(ti.row0 + rr) * (p.K / 32)) +
                                   g)
                           : 0x7F7F7F7Fu;
            }
          }
          const uint32_t s = it % C::kNS, u = it % C::kNU;
          if (!mbar_wait(bar_full + 8 * s, (it / C::kNS) & 1, s_abort, p.status) ||
              !mbar_wait(bar_uempty + 8 * u, ((it / C::kNU) & 1) ^ 1, s_abort, p.status)) {
            ok = false;
            break;
          }
          // unit i of this thread: row (tid/8) + 16 i, 16-byte chunk j = tid%8.  Row & 7 and
          // j do not depend on i, so source and swizzled destination advance by constants.
          const uint8_t* src = smem + C::kOffB + s * C::kBLoadBytes + (tid >> 3) * 64 + (tid & 7) * 8;
          uint8_t* dst = smem + C::kOffBU + u * C::kBUBytes + (tid >> 3) * 128 +
                         (((tid & 7) ^ ((tid >> 3) & 7)) << 4);
          // loads are batched ahead of the stores: source and destination are both shared
          // memory, so a store in between would keep every later load waiting behind it
#pragma unroll
          for (int i0 = 0; i0 < BN / 16; i0 += 8) {
            uint2 wv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
              wv[i] = *reinterpret_cast<const uint2*>(src + (i0 + i) * 1024);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              uint2 a, b;
              if constexpr (BFMT == kBfmtInt4Sub) {
                a = w4_to_e4m3_sub(wv[i].x);
                b = w4_to_e4m3_sub(wv[i].y);
              } else {
                a = w4_to_e4m3_lut(wv[i].x);
                b = w4_to_e4m3_lut(wv[i].y);
              }
              *reinterpret_cast<uint4*>(dst + (i0 + i) * 2048) = make_uint4(a.x, a.y, b.x, b.y);
            }
          }
          if constexpr (C::kMxA) {
            // the group's activation scales into this slot's TMEM columns (every lane
            // quarter holds the same copy), complete before the MMA is told
            tmem_st_32x32b_x4(tmem_base + quarter + C::kSfaCol + u * 4, sfw[0], sfw[1], sfw[2],
                              sfw[3]);
            tmem_wait_st();
            tc_fence_before();
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(bar_ufull + 8 * u);
            mbar_arrive(bar_empty + 8 * s);
          }
        }
      }
    }
  } else if (warp < 8) {
    if constexpr (C::kGroupScale) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::kRegsCtrl));
    if (warp == kProducerWarp) {
      // ---------------------------------------------------------------- TMA producer
      // Lane 0 waits for free stages and issues the B tile, the weight scales and a plain A
      // tile.  In gather mode the warp first stages the tile's 128 source row ids (rows past
      // the expert's last repeat its last row; their results are never stored) and each of
      // the 32 lanes then issues one four-row gather of the A tile per K group.
      int32_t* s_rt = reinterpret_cast<int32_t*>(smem + C::kOffRT);
      const bool gather = p.row_token != nullptr;
      if (lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
      }
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
        const int tsplit = C::kGroupScale ? 0 : t / base_tiles;
        const TileInfo ti = decode_tile(C::kGroupScale ? t : t - tsplit * base_tiles, nt_count,
                                        BN, s_off, s_mtp, E);
        const int g0 = C::kGroupScale ? 0 : tsplit * G / ks;
        const int g1 = C::kGroupScale ? G : (tsplit + 1) * G / ks;
        if (gather) {
          for (int i = lane; i < 128; i += 32)
            s_rt[i] = __ldg(p.row_token + ti.row0 + (i < ti.rows ? i : ti.rows - 1));
          __syncwarp();
        }
        for (int g = g0; g < g1; ++g, ++it) {
          const uint32_t s = it % C::kNS;
          if (lane == 0) {
            if (!mbar_wait(bar_empty + 8 * s, ((it / C::kNS) & 1) ^ 1, s_abort, p.status)) {
              ok = false;
            } else {
              if constexpr (C::kGroupScale) {
                // the tile's weight scales of this K group: BN contiguous floats
                const uint32_t w = it % C::kNSW;
                if (!mbar_wait(bar_swempty + 8 * w, ((it / C::kNSW) & 1) ^ 1, s_abort,
                               p.status)) {
                  ok = false;
                } else {
                  mbar_arrive_expect_tx(bar_swfull + 8 * w, C::kSWBytes);
                  bulk_load(smem_u32(smem + C::kOffSW + w * C::kSWBytes),
                            p.sw + (static_cast<size_t>(ti.e) * G + g) * p.N + ti.n0,
                            C::kSWBytes, bar_swfull + 8 * w);
                }
              }
              if (ok) {
                mbar_arrive_expect_tx(bar_full + 8 * s, C::kStageTx);
                if (!gather)
                  tma_load_2d(smem_u32(smem + C::kOffA + s * C::kABytes), &tmA, bar_full + 8 * s,
                              g * 128, ti.row0);
                if constexpr (C::kInt4) {
                  tma_load_2d(smem_u32(smem + C::kOffB + s * C::kBLoadBytes), &tmB,
                              bar_full + 8 * s, g * 64, ti.e * p.N + ti.n0);
                } else {
                  tma_load_2d(smem_u32(smem + C::kOffB + s * C::kBLoadBytes), &tmB,
                              bar_full + 8 * s, g * 128, ti.n0);
                }
              }
            }
          }
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!ok) break;  // before ++it: the drain below counts issued stages only
          // gather mode: each lane copies 4 of the 128 rows (its stage slot is free: lane 0
          // waited for it above)
          if (gather)
            tma_gather4_2d(smem_u32(smem + C::kOffA + s * C::kABytes) + lane * 512, &tmA,
                           bar_full + 8 * s, g * 128,
                           *reinterpret_cast<const int4*>(s_rt + 4 * lane));
        }
        __syncwarp();  // every lane is done with s_rt before the next tile rewrites it
      }
      if (lane == 0) {
        // drain: every issued stage must have landed before the CTA can exit
        const uint32_t issued = it;
        const uint32_t first = issued > static_cast<uint32_t>(C::kNS) ? issued - C::kNS : 0;
        for (uint32_t i = first; i < issued; ++i)
          mbar_wait_drain(bar_full + 8 * (i % C::kNS), (i / C::kNS) & 1);
        if constexpr (C::kGroupScale) {
          const uint32_t first_w = issued > static_cast<uint32_t>(C::kNSW) ? issued - C::kNSW : 0;
          for (uint32_t i = first_w; i < issued; ++i)
            mbar_wait_drain(bar_swfull + 8 * (i % C::kNSW), (i / C::kNSW) & 1);
        }
      }
    } else if (warp == kMmaWarp && lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc = make_idesc_e4m3(128, BN);
      constexpr uint32_t idesc_half = make_idesc_e4m3(128, BN / C::kHalves);
      uint32_t it = 0, ait = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
        uint32_t a = ait & 1;
        const int tsplit = C::kGroupScale ? 0 : t / base_tiles;
        const int g0 = C::kGroupScale ? 0 : tsplit * G / ks;
        const int g1 = C::kGroupScale ? G : (tsplit + 1) * G / ks;
        if constexpr (!C::kGroupScale) {
          if (!mbar_wait(bar_tempty + 8 * a, ((ait >> 1) & 1) ^ 1, s_abort, p.status)) break;
          tc_fence_after();
        }
        for (int g = g0; g < g1; ++g, ++it) {
          const uint32_t s = it % C::kNS;
          if (!mbar_wait(bar_full + 8 * s, (it / C::kNS) & 1, s_abort, p.status)) {
            ok = false;
            break;
          }
          uint32_t b_base;
          const uint32_t u = it % (C::kNU ? C::kNU : 1);
          if constexpr (C::kInt4) {
            if (!mbar_wait(bar_ufull + 8 * u, (it / C::kNU) & 1, s_abort, p.status)) {
              ok = false;
              break;
            }
            b_base = smem_u32(smem + C::kOffBU + u * C::kBUBytes);
          } else {
            b_base = smem_u32(smem + C::kOffB + s * C::kBLoadBytes);
          }
          const uint32_t a_base = smem_u32(smem + C::kOffA + s * C::kABytes);
          if constexpr (C::kGroupScale) {
            // one fresh partial per K group, written half by half (N = 128 each), each half
            // handed to its epilogue warpgroup as soon as its 4 MMAs complete
            a = ait & 1;
            for (int h = 0; h < C::kHalves; ++h) {
              const uint32_t slot = a * C::kHalves + h;
              if (!mbar_wait(bar_tempty + 8 * slot, ((ait >> 1) & 1) ^ 1, s_abort, p.status)) {
                ok = false;
                break;
              }
              tc_fence_after();
              constexpr int kHalfN = BN / C::kHalves;
              const uint32_t d_tmem = tmem_base + a * BN + h * kHalfN;
              const uint32_t b_half = b_base + h * kHalfN * 128;
              if constexpr (C::kMxA) {
                const uint32_t sfa = tmem_base + C::kSfaCol + u * 4;
                const uint32_t sfb = tmem_base + C::kSfbCol;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  mma_mxf8f6f4(d_tmem, make_sdesc_sw128(a_base + kk * 32),
                               make_sdesc_sw128(b_half + kk * 32),
                               make_idesc_mxf4_e4m3(128, kHalfN, static_cast<uint32_t>(kk)), sfa,
                               sfb, kk > 0 ? 1u : 0u);
              } else {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  mma_f8f6f4(d_tmem, make_sdesc_sw128(a_base + kk * 32),
                             make_sdesc_sw128(b_half + kk * 32), idesc_half, kk > 0 ? 1u : 0u);
              }
              mma_commit(bar_tfull + 8 * slot);
            }
            if (!ok) break;
            ++ait;
          } else {
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + a * BN;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f8f6f4(d_tmem, make_sdesc_sw128(a_base + kk * 32),
                         make_sdesc_sw128(b_base + kk * 32), idesc, (kk > 0 || g > g0) ? 1u : 0u);
          }
          mma_commit(bar_empty + 8 * s);
          if constexpr (C::kInt4) mma_commit(bar_uempty + 8 * u);
        }
        if constexpr (!C::kGroupScale) {
          if (!ok) break;
          mma_commit(bar_tfull + 8 * a);
          ++ait;
        }
      }
      // drain: all MMAs issued by this thread complete before TMEM is released
      mma_commit(bar_drain);
      mbar_wait_drain(bar_drain, 0);
    }
  } else {
    // -------------------------------------------------------------------- epilogue
    if constexpr (C::kGroupScale) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::kRegsHigh));
    const int ewarp = warp - 8;
    const int wg = ewarp >> 2;
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int r_in = q * 32 + lane;
    // warpgroup wg owns columns [wg*128, wg*128 + 128) of the tile: col_a.. and col_b..
    const int col_a = wg * 128, col_b = wg * 128 + 64;
    const uint32_t half_slot = C::kHalves > 1 ? static_cast<uint32_t>(wg) : 0u;
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    float tensor_scale = 1.0f;
    if constexpr (!C::kGroupScale)
      tensor_scale = p.sa_rows ? __ldg(p.sw_tensor) : __ldg(p.sa_tensor) * __ldg(p.sw_tensor);
    uint32_t ait = 0;
    int tile_parity = 0;
    bool ok = true;
    float pf0 = 0.0f, pf1 = 0.0f;  // group mode: next tile's first two activation scales
    bool pf_ok = false;
    for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x, tile_parity ^= 1) {
      const int split = C::kGroupScale ? 0 : t / base_tiles;
      const int tix = C::kGroupScale ? t : t - split * base_tiles;  // output tile of this split
      const TileInfo ti = decode_tile(tix, nt_count, BN, s_off, s_mtp, E);
      const bool valid = r_in < ti.rows;
      const int row = ti.row0 + r_in;
      if constexpr (C::kGroupScale) {
        uint64_t acc2[64];  // acc2[j] holds columns 2j, 2j+1 of the thread's 128
#pragma unroll
        for (int i = 0; i < 64; ++i) acc2[i] = 0;
        // activation scales run two groups ahead of their use (global-load latency)
        // gather mode: the scales of routed row r are those of its source row row_token[r]
        const int src_row = p.row_token ? __ldg(p.row_token + (valid ? row : ti.row0))
                                        : (valid ? row : 0);
        // MXFP4: the activation scales are applied inside the MMA; here 1
        const float* as_row = C::kMxA ? nullptr : p.as + static_cast<size_t>(src_row) * G;
        // the first two scales of a tile were requested at the start of the previous tile
        float sa0 = C::kMxA ? 1.0f : (pf_ok ? pf0 : (valid ? __ldg(as_row) : 0.0f));
        float sa1 = C::kMxA ? 1.0f : (pf_ok ? pf1 : ((valid && G > 1) ? __ldg(as_row + 1) : 0.0f));
        pf_ok = false;
        if (!C::kMxA && t + static_cast<int>(gridDim.x) < total_tiles) {
          const TileInfo tn = decode_tile(t + gridDim.x, nt_count, BN, s_off, s_mtp, E);
          const bool vn = r_in < tn.rows;
          const int rn = p.row_token ? __ldg(p.row_token + (vn ? tn.row0 + r_in : tn.row0))
                                     : (vn ? tn.row0 + r_in : 0);
          pf0 = vn ? __ldg(p.as + static_cast<size_t>(rn) * G) : 0.0f;
          pf1 = (vn && G > 1) ? __ldg(p.as + static_cast<size_t>(rn) * G + 1) : 0.0f;
          pf_ok = true;
        }
        for (int g = 0; g < G; ++g) {
          const uint32_t a = ait & 1;
          const uint32_t w = ait % C::kNSW;
          const float sa2 = C::kMxA ? 1.0f : ((valid && g + 2 < G) ? __ldg(as_row + g + 2) : 0.0f);
          if (!mbar_wait(bar_swfull + 8 * w, (ait / C::kNSW) & 1, s_abort, p.status) ||
              !mbar_wait(bar_tfull + 8 * (a * C::kHalves + half_slot), (ait >> 1) & 1, s_abort,
                         p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float* sws = reinterpret_cast<const float*>(smem + C::kOffSW + w * C::kSWBytes);
          const uint32_t tb = tmem_base + lane_addr + a * BN;
          const uint64_t sa2x = pack_f32x2(sa0, sa0);
          // the warpgroup's 128 columns in 4 loads of 32, double-buffered: tcgen05.wait::ld
          // waits for every outstanding load, so fewer and larger loads expose less latency
          uint32_t v[2][32];
          tmem_ld_32x32b_x32(tb + col_a, v[0]);
          tmem_wait_ld();
          reg_fence32(v[0]);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            if (c + 1 < 4) tmem_ld_32x32b_x32(tb + col_a + (c + 1) * 32, v[(c + 1) & 1]);
            const ulonglong2* sw2 = reinterpret_cast<const ulonglong2*>(sws + col_a + c * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const ulonglong2 wv = sw2[i];  // 4 weight scales as two f32x2 pairs
              const uint32_t* vv = v[c & 1] + 4 * i;
              fma2_pair(acc2[c * 16 + 2 * i], sa2x, wv.x, vv[0], vv[1]);
              fma2_pair(acc2[c * 16 + 2 * i + 1], sa2x, wv.y, vv[2], vv[3]);
            }
            if (c + 1 < 4) {
              tmem_wait_ld();
              reg_fence32(v[(c + 1) & 1]);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(bar_tempty + 8 * (a * C::kHalves + half_slot));
            mbar_arrive(bar_swempty + 8 * w);
          }
          ++ait;
          sa0 = sa1;
          sa1 = sa2;
        }
        if (!ok) break;
        if constexpr (EPI == kEpiSwiglu) {
          // columns [col_a, col_a+64) are gate rows i = wg*64.., [col_b, col_b+64) the matching
          // up rows (the bank interleaves gate and up in blocks of 64 rows)
          float hv[64];
          float amax = 0.0f;
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            const float gt = (i & 1) ? hi_f32(acc2[i >> 1]) : lo_f32(acc2[i >> 1]);
            const float up = (i & 1) ? hi_f32(acc2[32 + (i >> 1)]) : lo_f32(acc2[32 + (i >> 1)]);
            const float h = __fdividef(gt, 1.0f + __expf(-gt)) * up;
            hv[i] = h;
            amax = fmaxf(amax, fabsf(h));
          }
          float* red = s_red + tile_parity * 256;
          red[wg * 128 + r_in] = amax;
          asm volatile("bar.sync 1, %0;" ::"n"(C::kEpiThreads) : "memory");
          const float amax_all = fmaxf(red[r_in], red[128 + r_in]);
          const float s = scale_from_amax(amax_all);
          const float inv_s = __frcp_rn(s);  // h * (1/s): same e4m3 code as h / s except
                                             // within 2^-23 of a rounding boundary
          const int inter = p.N / 2;
          uint4 o[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int i = 16 * c;
            o[c].x = cvt_e4m3x4(hv[i + 0] * inv_s, hv[i + 1] * inv_s,
                                hv[i + 2] * inv_s, hv[i + 3] * inv_s);
            o[c].y = cvt_e4m3x4(hv[i + 4] * inv_s, hv[i + 5] * inv_s,
                                hv[i + 6] * inv_s, hv[i + 7] * inv_s);
            o[c].z = cvt_e4m3x4(hv[i + 8] * inv_s, hv[i + 9] * inv_s,
                                hv[i + 10] * inv_s, hv[i + 11] * inv_s);
            o[c].w = cvt_e4m3x4(hv[i + 12] * inv_s, hv[i + 13] * inv_s,
                                hv[i + 14] * inv_s, hv[i + 15] * inv_s);
          }
          if (C::kStageOut && ti.rows == 128) {
            // full tile: each warp's 32 rows x 64 codes go out as one TMA tile store from
            // the warp's own 2 KB slice (64-byte swizzle), with no barrier across warps
            uint8_t* buf = smem + C::kOffST + wg * 8192 + q * 2048;
            if (lane == 0) bulk_wait_read0();  // this warp's previous store has left the slice
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 4; ++c)
              *reinterpret_cast<uint4*>(buf + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)) = o[c];
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmY, smem_u32(buf), ti.n0 / 2 + wg * 64, ti.row0 + q * 32);
              bulk_commit();
            }
          } else if (valid) {
            uint8_t* hq = reinterpret_cast<uint8_t*>(p.out) + static_cast<size_t>(row) * inter +
                          (ti.n0 / 2) + wg * 64;
#pragma unroll
            for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(hq + 16 * c) = o[c];
          }
          if (valid && wg == 0)
            p.out_scales[static_cast<size_t>(row) * (inter / 128) + ti.n0 / 256] = s;
        } else if (C::kStageOut && ti.rows == 128 && p.comb == nullptr) {
          // full tile, bf16: each warp stores its 32 rows in eight 16-column chunks from its
          // own 2 KB slice, two 1 KB halves used in turn (row r at r * 32 bytes, 16-byte
          // pieces swizzled by (r / 4) % 2 as the tensor map's 32-byte swizzle expects), so
          // a chunk is staged while the previous one is still being read; no barrier across
          // warps
          uint8_t* slice = smem + C::kOffST + wg * 8192 + q * 2048;
          const int swz = (lane >> 2) & 1;
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            uint8_t* buf = slice + (ch & 1) * 1024;
            if (lane == 0) bulk_wait_read1();  // the store two chunks back has left this half
            __syncwarp();
            const int j = ch * 8;  // acc2[j..j+7]: columns 16 ch .. 16 ch + 15
            const uint4 v0 = make_uint4(pack_bf16x2(lo_f32(acc2[j]), hi_f32(acc2[j])),
                                        pack_bf16x2(lo_f32(acc2[j + 1]), hi_f32(acc2[j + 1])),
                                        pack_bf16x2(lo_f32(acc2[j + 2]), hi_f32(acc2[j + 2])),
                                        pack_bf16x2(lo_f32(acc2[j + 3]), hi_f32(acc2[j + 3])));
            const uint4 v1 = make_uint4(pack_bf16x2(lo_f32(acc2[j + 4]), hi_f32(acc2[j + 4])),
                                        pack_bf16x2(lo_f32(acc2[j + 5]), hi_f32(acc2[j + 5])),
                                        pack_bf16x2(lo_f32(acc2[j + 6]), hi_f32(acc2[j + 6])),
                                        pack_bf16x2(lo_f32(acc2[j + 7]), hi_f32(acc2[j + 7])));
            *reinterpret_cast<uint4*>(buf + lane * 32 + (swz << 4)) = v0;
            *reinterpret_cast<uint4*>(buf + lane * 32 + ((swz ^ 1) << 4)) = v1;
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmY, smem_u32(buf), ti.n0 + col_a + ch * 16, ti.row0 + q * 32);
              bulk_commit();
            }
          }
        } else if (valid) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int col = (c < 2) ? col_a + c * 32 : col_b + (c - 2) * 32;
            if constexpr (EPI == kEpiF32) {
              float* o = reinterpret_cast<float*>(p.out) + static_cast<size_t>(row) * p.N + ti.n0 + col;
#pragma unroll
              for (int i = 0; i < 32; i += 4)
                *reinterpret_cast<float4*>(o + i) =
                    make_float4(lo_f32(acc2[(c * 32 + i) / 2]), hi_f32(acc2[(c * 32 + i) / 2]),
                                lo_f32(acc2[(c * 32 + i) / 2 + 1]), hi_f32(acc2[(c * 32 + i) / 2 + 1]));
            } else {
              __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(row) * p.N + ti.n0 + col;
#pragma unroll
              for (int i = 0; i < 32; i += 8)
                *reinterpret_cast<uint4*>(o + i) = make_uint4(
                    pack_bf16x2(lo_f32(acc2[(c * 32 + i) / 2]), hi_f32(acc2[(c * 32 + i) / 2])),
                    pack_bf16x2(lo_f32(acc2[(c * 32 + i) / 2 + 1]), hi_f32(acc2[(c * 32 + i) / 2 + 1])),
                    pack_bf16x2(lo_f32(acc2[(c * 32 + i) / 2 + 2]), hi_f32(acc2[(c * 32 + i) / 2 + 2])),
                    pack_bf16x2(lo_f32(acc2[(c * 32 + i) / 2 + 3]), hi_f32(acc2[(c * 32 + i) / 2 + 3])));
            }
          }
        }
        if constexpr (EPI == kEpiBf16) {
          if (p.comb != nullptr) {
            const FusedCombine cb = *p.comb;
            // Combine folded into the epilogue.  This thread's 128 columns of routed row `row`
            // are in y (plain stores above); after a fence it counts their arrival for
            // (token, chunk).  The k-th arrival, whichever slot row it is, combines the chunk:
            // the whole warp sums the token's k slot rows in slot order with the same fmaf
            // chain as the combine kernel, so the result is bit-identical to it.
            const int nchunk = p.N / 128;
            const int chunk = (ti.n0 + col_a) / 128;  // the same for every lane of the warp
            int64_t tok = 0;
            bool last = false;
            if (valid) {
              tok = __ldg(cb.row_token + row);
              __threadfence();
              last = atomicAdd(cb.count + tok * nchunk + chunk, 1) == cb.k - 1;
            }
            unsigned todo = __ballot_sync(0xffffffffu, last);
            if (todo) __threadfence();  // the other slot rows' stores, ordered by the counter
            const int64_t c = static_cast<int64_t>(chunk) * 128 + lane * 4;
            const uint16_t* yb = reinterpret_cast<const uint16_t*>(p.out);
            while (todo) {
              const int src = __ffs(todo) - 1;
              todo &= todo - 1;
              const int64_t t = __shfl_sync(0xffffffffu, tok, src);
              float acc0 = 0.0f, acc1 = 0.0f, acc2c = 0.0f, acc3 = 0.0f;
#pragma unroll 8
              for (int j = 0; j < cb.k; ++j) {
                const int64_t r = __ldg(cb.token_row + t * cb.k + j);
                const float g = __ldg(cb.gates + t * cb.k + j);
                const uint2 v = __ldcg(reinterpret_cast<const uint2*>(yb + r * p.N + c));
                acc0 = fmaf(g, bf16_lo(v.x), acc0);
                acc1 = fmaf(g, bf16_hi(v.x), acc1);
                acc2c = fmaf(g, bf16_lo(v.y), acc2c);
                acc3 = fmaf(g, bf16_hi(v.y), acc3);
              }
              *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(cb.out) + t * p.N + c) =
                  make_uint2(pack_bf16x2(acc0, acc1), pack_bf16x2(acc2c, acc3));
            }
          }
        }
      } else if constexpr (BN == 16) {
        // decode sizes, operands swapped: the 128 lanes are output features (A rows = weight
        // rows), the 16 columns are tokens; token j's value of feature `row` goes to
        // out[j * out_ld + row], so each store of a warp covers 32 consecutive features
        const uint32_t a = ait & 1;
        if (!mbar_wait(bar_tfull + 8 * a, (ait >> 1) & 1, s_abort, p.status)) break;
        tc_fence_after();
        uint32_t v[16];
        tmem_ld_32x32b_x16(tmem_base + lane_addr + a * BN, v);
        tmem_wait_ld();
        reg_fence16(v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_tempty + 8 * a);
        ++ait;
        float acc[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[j] = __uint_as_float(v[j]);
        bool store = valid;
        if (ks > 1) {
          // K split: this split's partial row goes out; the last split adds all of them
          float* part = sk.partials + ((static_cast<size_t>(tix) * ks + split) * 128 + r_in) * 16;
          if (valid) {
#pragma unroll
            for (int j = 0; j < 16; j += 4)
              *reinterpret_cast<float4*>(part + j) =
                  make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
          }
          store = split_arrive_last(sk.split_count + static_cast<size_t>(tix) * C::kEpiWarps +
                                        ewarp, ks, lane) &&
                  valid;
          if (store) {
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
            for (int s2 = 0; s2 < ks; ++s2) {
              const float* q =
                  sk.partials + ((static_cast<size_t>(tix) * ks + s2) * 128 + r_in) * 16;
#pragma unroll
              for (int j = 0; j < 16; j += 4) {
                const float4 f = __ldcg(reinterpret_cast<const float4*>(q + j));
                acc[j] += f.x;
                acc[j + 1] += f.y;
                acc[j + 2] += f.z;
                acc[j + 3] += f.w;
              }
            }
          }
        }
        if (store) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (j < p.swap_m) {
              // per-row activation scales belong to the tokens: one per column here
              const float rs = p.sa_rows ? __ldg(p.sa_rows + j) * tensor_scale : tensor_scale;
              const float yv = rs * acc[j];
              const size_t o = static_cast<size_t>(j) * p.out_ld + row;
              if constexpr (EPI == kEpiF32)
                reinterpret_cast<float*>(p.out)[o] = yv;
              else
                reinterpret_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(yv);
            }
          }
        }
      } else {
        // per-tensor scales: the whole K accumulated in TMEM; one scalar in the epilogue
        // (per-row activation scales: that row's scale times the weight scale)
        const float rs = p.sa_rows ? (valid ? __ldg(p.sa_rows + row) : 0.0f) * tensor_scale
                                   : tensor_scale;
        const uint32_t a = ait & 1;
        if (!mbar_wait(bar_tfull + 8 * a, (ait >> 1) & 1, s_abort, p.status)) break;
        tc_fence_after();
        const uint32_t tb = tmem_base + lane_addr + a * BN;
        uint32_t v[2][16];
        tmem_ld_32x32b_x16(tb + col_a, v[0]);
        tmem_wait_ld();
        reg_fence16(v[0]);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          if (c + 1 < 8) {
            const int coln = (c + 1 < 4) ? col_a + (c + 1) * 16 : col_b + (c - 3) * 16;
            tmem_ld_32x32b_x16(tb + coln, v[(c + 1) & 1]);
          }
          const int col = (c < 4) ? col_a + c * 16 : col_b + (c - 4) * 16;
          const uint32_t* vv = v[c & 1];
          if (valid && ks > 1) {
            // K split: this split's raw partial of the row goes out
            float* part = sk.partials +
                          ((static_cast<size_t>(tix) * ks + split) * 128 + r_in) * BN + col;
#pragma unroll
            for (int i = 0; i < 16; i += 4)
              *reinterpret_cast<float4*>(part + i) =
                  make_float4(__uint_as_float(vv[i]), __uint_as_float(vv[i + 1]),
                              __uint_as_float(vv[i + 2]), __uint_as_float(vv[i + 3]));
          } else if (valid) {
            if constexpr (EPI == kEpiF32) {
              float* o = reinterpret_cast<float*>(p.out) + static_cast<size_t>(row) * p.N + ti.n0 + col;
#pragma unroll
              for (int i = 0; i < 16; i += 4)
                *reinterpret_cast<float4*>(o + i) = make_float4(
                    rs * __uint_as_float(vv[i]), rs * __uint_as_float(vv[i + 1]),
                    rs * __uint_as_float(vv[i + 2]), rs * __uint_as_float(vv[i + 3]));
            } else {
              __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(row) * p.N + ti.n0 + col;
#pragma unroll
              for (int i = 0; i < 16; i += 8)
                *reinterpret_cast<uint4*>(o + i) = make_uint4(
                    pack_bf16x2(rs * __uint_as_float(vv[i]), rs * __uint_as_float(vv[i + 1])),
                    pack_bf16x2(rs * __uint_as_float(vv[i + 2]), rs * __uint_as_float(vv[i + 3])),
                    pack_bf16x2(rs * __uint_as_float(vv[i + 4]), rs * __uint_as_float(vv[i + 5])),
                    pack_bf16x2(rs * __uint_as_float(vv[i + 6]), rs * __uint_as_float(vv[i + 7])));
            }
          }
          if (c + 1 < 8) {
            tmem_wait_ld();
            reg_fence16(v[(c + 1) & 1]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_tempty + 8 * a);
        ++ait;
        if (ks > 1 &&
            split_arrive_last(sk.split_count + static_cast<size_t>(tix) * C::kEpiWarps + ewarp, ks,
                              lane) &&
            valid) {
          // the last split: every split's partial of the row added in split order, scaled
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            const int col = (c < 4) ? col_a + c * 16 : col_b + (c - 4) * 16;
            float acc[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
            for (int s2 = 0; s2 < ks; ++s2) {
              const float* q = sk.partials +
                               ((static_cast<size_t>(tix) * ks + s2) * 128 + r_in) * BN + col;
#pragma unroll
              for (int i = 0; i < 16; i += 4) {
                const float4 f = __ldcg(reinterpret_cast<const float4*>(q + i));
                acc[i] += f.x;
                acc[i + 1] += f.y;
                acc[i + 2] += f.z;
                acc[i + 3] += f.w;
              }
            }
            if constexpr (EPI == kEpiF32) {
              float* o = reinterpret_cast<float*>(p.out) + static_cast<size_t>(row) * p.N + ti.n0 + col;
#pragma unroll
              for (int i = 0; i < 16; i += 4)
                *reinterpret_cast<float4*>(o + i) =
                    make_float4(rs * acc[i], rs * acc[i + 1], rs * acc[i + 2], rs * acc[i + 3]);
            } else {
              __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(row) * p.N + ti.n0 + col;
#pragma unroll
              for (int i = 0; i < 16; i += 8)
                *reinterpret_cast<uint4*>(o + i) = make_uint4(
                    pack_bf16x2(rs * acc[i], rs * acc[i + 1]),
                    pack_bf16x2(rs * acc[i + 2], rs * acc[i + 3]),
                    pack_bf16x2(rs * acc[i + 4], rs * acc[i + 5]),
                    pack_bf16x2(rs * acc[i + 6], rs * acc[i + 7]));
            }
          }
        }
      }
    }
    if constexpr (C::kStageOut) {
      if (lane == 0) bulk_wait0();  // every tile store this warp issued has completed
    }
  }

  // ---------------------------------------------------------------------- teardown
  __syncwarp();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// -------------------------------------------------------------------------------------
// host side
// -------------------------------------------------------------------------------------
// The driver's tensor-map encoder, looked up once per process (thread-safe).
static PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

static bool make_map_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                        uint32_t box_inner, uint32_t box_outer, bool swizzle128) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// MXFP4 activations [rows, K] as packed E2M1 (K/2 bytes a row): boxes of 128 values x 128
// rows, each 16 values landing in the low 8 bytes of a 16-byte smem chunk (the padded layout
// kind::mxf8f6f4 reads), 128-byte swizzle.  Needs a 32-byte aligned base and K % 128 == 0.
static bool make_map_e2m1_padded(CUtensorMap* m, const void* base, uint64_t k, uint64_t rows) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {k, rows};
  cuuint64_t strides[1] = {k / 2};
  cuuint32_t box[2] = {128, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Output map of the staged SwiGLU store: [rows, inner] bytes, boxes of 64 bytes x 32 rows
// (one warp's rows) with the 64-byte swizzle.
static bool make_map_u8_swz64(CUtensorMap* m, void* base, uint64_t inner, uint64_t rows) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {64, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Output map of the staged bf16 store: [rows, N] bf16, boxes of 16 columns x 32 rows (one
// warp's chunk) with the 32-byte swizzle.
static bool make_map_bf16_out(CUtensorMap* m, void* base, uint64_t n, uint64_t rows) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {n, rows};
  cuuint64_t strides[1] = {n * 2};
  cuuint32_t box[2] = {16, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int BN, int BFMT, int EPI, int AFMT = kAfmtE4m3>
static cudaError_t run(const GroupedGemmArgs& a, cudaStream_t s, fge_status* st) {
  using C = Cfg<BN, BFMT, EPI, AFMT>;
  auto kern = grouped_gemm_kernel<BN, BFMT, EPI, AFMT>;
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return ce;
  // group mode: the register split must fit in what the CTA is launched with, or the growing
  // warpgroups would wait forever; the per-device set-up refuses a kernel with fewer
  const long need = C::kGroupScale ? 128L * C::kRegsUnpack + 128L * C::kRegsCtrl +
                                         static_cast<long>(C::kEpiThreads) * C::kRegsHigh
                                   : 0L;
  const int min_regs = static_cast<int>((need + C::kThreads - 1) / C::kThreads);
  if (!device_kernel_ready(dev, reinterpret_cast<const void*>(kern), C::kSmemBytes, min_regs)) {
    *st = FGE_ERR_UNSUPPORTED_DEVICE;
    return cudaSuccess;
  }
  CUtensorMap tmA, tmB;
  // gather mode: A is the token-ordered [rows_a, K] tensor read one row per box (4 per copy)
  const bool okA = C::kMxA      ? make_map_e2m1_padded(&tmA, a.aq, a.K, a.R)
                   : a.row_token ? make_map_u8(&tmA, a.aq, a.K, a.rows_a, 128, 1, true)
                                 : make_map_u8(&tmA, a.aq, a.K, a.R, 128, 128, true);
  if (!okA) {
    *st = FGE_ERR_CUDA;
    return cudaSuccess;
  }
  bool okB;
  if (C::kInt4)
    okB = make_map_u8(&tmB, a.w, a.K / 2, static_cast<uint64_t>(a.E) * a.N, 64, BN, false);
  else
    okB = make_map_u8(&tmB, a.w, a.K, a.N, 128, BN, true);
  if (!okB) {
    *st = FGE_ERR_CUDA;
    return cudaSuccess;
  }
  GemmParams p{};
  p.as = a.as;
  p.sf_a = a.a_sf;
  const SplitArgs sk{a.partials, a.split_count, std::max(1, a.ksplit)};
  p.sw = a.per_tensor ? nullptr : a.sw;
  p.sa_tensor = a.sa_tensor;
  p.sa_rows = a.sa_rows;
  p.sw_tensor = a.per_tensor ? a.sw : nullptr;
  p.offsets = a.offsets;
  p.row_token = a.row_token;
  p.out = a.out;
  p.out_scales = a.out_scales;
  p.status = a.status;
  p.comb = a.comb;
  p.E = a.E;
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.G = static_cast<int>(a.K / 128);
  p.dense_rows = static_cast<int>(a.R);
  const long tiles_bound = (a.R / 128 + a.E) * (a.N / BN) * std::max(1, a.ksplit);
  const int grid = static_cast<int>(std::max<long>(1, std::min<long>(num_sms(), tiles_bound)));
  CUtensorMap tmY = tmA;  // unused unless the store is staged
  bool okY = true;
  if constexpr (C::kStageOut) {
    if (EPI == kEpiSwiglu)  // hq: [rows, N/2] e4m3 codes, 64-byte x 32-row boxes (one warp)
      okY = make_map_u8_swz64(&tmY, a.out, a.N / 2, a.R);
    else
      okY = make_map_bf16_out(&tmY, a.out, a.N, a.R);
  }
  if (!okY) {
    *st = FGE_ERR_CUDA;
    return cudaSuccess;
  }
  kern<<<grid, C::kThreads, C::kSmemBytes, s>>>(tmA, tmB, tmY, p, sk);
  *st = FGE_OK;
  return cudaGetLastError();
}

// Decode sizes (at most 16 activation rows, one expert, per-tensor or per-row scales): the
// operands trade places so that the 128-row side of the MMA walks the weights.  A = the
// weight matrix [N, K] in 128-row tiles, B = the activations as one 16-row tile (rows past
// M read as zeros), N = 16 per MMA; one CTA per 128 output features streams its weight rows
// once, and the epilogue writes the result transposed back to [M, N].
template <int EPI>
static cudaError_t run_swapped(const GroupedGemmArgs& a, cudaStream_t s, fge_status* st) {
  using C = Cfg<16, kBfmtE4m3, EPI>;
  auto kern = grouped_gemm_kernel<16, kBfmtE4m3, EPI>;
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return ce;
  if (!device_kernel_ready(dev, reinterpret_cast<const void*>(kern), C::kSmemBytes, 0)) {
    *st = FGE_ERR_UNSUPPORTED_DEVICE;
    return cudaSuccess;
  }
  CUtensorMap tmA, tmB;
  if (!make_map_u8(&tmA, a.w, a.K, a.N, 128, 128, true) ||
      !make_map_u8(&tmB, a.aq, a.K, a.R, 128, 16, true)) {
    *st = FGE_ERR_CUDA;
    return cudaSuccess;
  }
  GemmParams p{};
  p.sa_tensor = a.sa_tensor;
  p.sa_rows = a.sa_rows;
  p.sw_tensor = a.sw;
  p.offsets = nullptr;
  p.row_token = nullptr;
  p.out = a.out;
  p.status = a.status;
  p.E = 1;
  p.N = 16;
  p.K = static_cast<int>(a.K);
  p.G = static_cast<int>(a.K / 128);
  p.dense_rows = static_cast<int>(a.N);
  p.swap_m = static_cast<int>(a.R);
  p.out_ld = static_cast<int>(a.N);
  const SplitArgs sk{a.partials, a.split_count, std::max(1, a.ksplit)};
  const int grid = static_cast<int>(std::max<long>(
      1, std::min<long>(num_sms(), (a.N + 127) / 128 * std::max(1, a.ksplit))));
  kern<<<grid, C::kThreads, C::kSmemBytes, s>>>(tmA, tmB, tmA, p, sk);
  *st = FGE_OK;
  return cudaGetLastError();
}

// Output tiles of the per-tensor GEMM and their width: the decode tile (M <= 16, 128 weight
// rows by 16 tokens) or 128-row tiles of BN = 256 (128 when N % 256 != 0) columns.
static void dense_tiles(int64_t M, int64_t N, int64_t* tiles, int64_t* bn, int64_t* warps) {
  if (M <= 16) {
    *tiles = (N + 127) / 128;
    *bn = 16;
    *warps = 4;
  } else {
    *bn = N % 256 == 0 ? 256 : 128;
    *tiles = (M + 127) / 128 * (N / *bn);
    *warps = *bn / 32;
  }
}

int dense_ksplit(int64_t M, int64_t N, int64_t K) {
  // only the decode tile splits: with 128-row tiles the last split's read-back of the others'
  // 128 x BN partials costs more than the shorter K walk saves (measured)
  if (M <= 0 || M > 16 || N <= 0 || K < 256) return 1;
  int64_t tiles, bn, warps;
  dense_tiles(M, N, &tiles, &bn, &warps);
  // as many CTAs per tile as fit on the SMs in one wave, each with at least 2 K groups
  int64_t ks = num_sms() / std::max<int64_t>(tiles, 1);
  ks = std::min<int64_t>(ks, (K / 128) / 2);
  ks = std::min<int64_t>(ks, 8);
  return static_cast<int>(std::max<int64_t>(ks, 1));
}

size_t dense_split_bytes(int64_t M, int64_t N, int ksplit, size_t* counter_bytes) {
  *counter_bytes = 0;
  if (ksplit <= 1) return 0;
  int64_t tiles, bn, warps;
  dense_tiles(M, N, &tiles, &bn, &warps);
  *counter_bytes = align_up(static_cast<size_t>(tiles * warps) * 4, 256);
  return *counter_bytes + static_cast<size_t>(tiles) * ksplit * 128 * bn * 4;
}

cudaError_t launch_grouped_gemm(const GroupedGemmArgs& a, cudaStream_t s, fge_status* st) {
  const bool bn256 = (a.N % 256) == 0;
  if (a.a_sf != nullptr) {
    // MXFP4 activations: 128-column tiles (the scale columns need TMEM beside the two
    // accumulators), subnormal int4 bank, plain store
    ledger_note(kLedGroupedGemms);
    return a.epilogue == 0 ? run<128, kBfmtInt4Sub, kEpiF32, kAfmtMxf4>(a, s, st)
                           : run<128, kBfmtInt4Sub, kEpiBf16, kAfmtMxf4>(a, s, st);
  }
  if (a.per_tensor && a.offsets == nullptr && a.row_token == nullptr && a.R <= 16) {
    ledger_note(kLedDenseDecodeTile);
    return a.epilogue == 0 ? run_swapped<kEpiF32>(a, s, st) : run_swapped<kEpiBf16>(a, s, st);
  }
  ledger_note(a.per_tensor ? kLedDenseRowTile : kLedGroupedGemms);
  if (a.per_tensor) {
    if (a.epilogue == 0) return bn256 ? run<256, kBfmtE4m3, kEpiF32>(a, s, st) : run<128, kBfmtE4m3, kEpiF32>(a, s, st);
    return bn256 ? run<256, kBfmtE4m3, kEpiBf16>(a, s, st) : run<128, kBfmtE4m3, kEpiBf16>(a, s, st);
  }
  if (a.bank_format == kBankSubnormal) {
    if (a.epilogue == 2) return run<256, kBfmtInt4Sub, kEpiSwiglu>(a, s, st);
    if (a.epilogue == 0) return bn256 ? run<256, kBfmtInt4Sub, kEpiF32>(a, s, st) : run<128, kBfmtInt4Sub, kEpiF32>(a, s, st);
    return bn256 ? run<256, kBfmtInt4Sub, kEpiBf16>(a, s, st) : run<128, kBfmtInt4Sub, kEpiBf16>(a, s, st);
  }
  if (a.epilogue == 2) return run<256, kBfmtInt4Lut, kEpiSwiglu>(a, s, st);
  if (a.epilogue == 0) return bn256 ? run<256, kBfmtInt4Lut, kEpiF32>(a, s, st) : run<128, kBfmtInt4Lut, kEpiF32>(a, s, st);
  return bn256 ? run<256, kBfmtInt4Lut, kEpiBf16>(a, s, st) : run<128, kBfmtInt4Lut, kEpiBf16>(a, s, st);
}

// -------------------------------------------------------------------------------------
// Load-time prepack of an int4 bank and its scales.
// -------------------------------------------------------------------------------------
// Row order of an interleaved gate_up bank: destination rows come in blocks of 128, each
// 64 gate rows followed by the 64 matching up rows (gate = source rows [0, N/2), up =
// [N/2, N)), so one 128-column half of a 256-column tile holds gate and up of 64 rows of I.
__device__ __forceinline__ int64_t interleaved_source_row(int64_t rd, int64_t N) {
  const int64_t blk = rd / 128, within = rd % 128;
  return within < 64 ? blk * 64 + within : N / 2 + blk * 64 + (within - 64);
}

__global__ void w4_prepack_kernel(const uint32_t* __restrict__ w, uint32_t* __restrict__ wd,
                                  int E, int64_t N, int64_t words_per_row, int interleave,
                                  int fmt) {
  const int64_t total = static_cast<int64_t>(E) * N * words_per_row;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t wi = i % words_per_row;
    const int64_t rd = (i / words_per_row) % N;  // destination row
    const int64_t e = i / (words_per_row * N);
    int64_t rs = rd;
    if (interleave) rs = interleaved_source_row(rd, N);
    uint32_t v = w[(e * N + rs) * words_per_row + wi];
    if (fmt == kBankSubnormal) {
      // nibble i holds element i; regroup so byte b holds elements b (low) and b+4 (high)
      uint32_t o = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        o |= ((v >> (4 * b)) & 0xFu) << (8 * b);
        o |= ((v >> (4 * (b + 4))) & 0xFu) << (8 * b + 4);
      }
      v = o;
    }
    wd[i] = v;
  }
}

__global__ void w4_prepack_scale_kernel(const float* __restrict__ sw, float* __restrict__ sd,
                                        int E, int64_t N, int G, int interleave, float mult) {
  const int64_t total = static_cast<int64_t>(E) * N * G;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t nd = i % N;  // destination layout [E, G, N]
    const int64_t g = (i / N) % G;
    const int64_t e = i / (N * G);
    int64_t rs = nd;
    if (interleave) rs = interleaved_source_row(nd, N);
    sd[i] = sw[(e * N + rs) * G + g] * mult;
  }
}

cudaError_t launch_w4_prepack(const uint8_t* w, const float* sw, int E, int64_t N, int64_t K,
                              int interleave, int fmt, uint8_t* w_dev, float* sw_dev,
                              cudaStream_t s) {
  const int grid = num_sms() * 4;
  w4_prepack_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const uint32_t*>(w),
                                         reinterpret_cast<uint32_t*>(w_dev), E, N, K / 8,
                                         interleave, fmt);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  w4_prepack_scale_kernel<<<grid, 256, 0, s>>>(sw, sw_dev, E, N, static_cast<int>(K / 128),
                                               interleave,
                                               fmt == kBankSubnormal ? 512.0f : 1.0f);
  return cudaGetLastError();
}

// -------------------------------------------------------------------------------------
// Unfused SwiGLU + requant (parity and ablation of the fused epilogue): one warp per
// (row, 128-group of I), four values per lane.
// -------------------------------------------------------------------------------------
__global__ void swiglu_quant_kernel(const float* __restrict__ c, int64_t R, int64_t I,
                                    uint8_t* __restrict__ hq, float* __restrict__ hs) {
  const int lane = threadIdx.x & 31;
  const int64_t groups = I / 128;
  const int64_t total = R * groups;
  const int64_t wid = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t item = wid; item < total; item += nw) {
    const int64_t r = item / groups, g = item % groups;
    const float* gate = c + r * 2 * I + g * 128 + lane * 4;
    const float4 gv = *reinterpret_cast<const float4*>(gate);
    const float4 uv = *reinterpret_cast<const float4*>(gate + I);
    float h[4] = {__fdiv_rn(gv.x, 1.0f + expf(-gv.x)) * uv.x, __fdiv_rn(gv.y, 1.0f + expf(-gv.y)) * uv.y,
                  __fdiv_rn(gv.z, 1.0f + expf(-gv.z)) * uv.z, __fdiv_rn(gv.w, 1.0f + expf(-gv.w)) * uv.w};
    float amax = fmaxf(fmaxf(fabsf(h[0]), fabsf(h[1])), fmaxf(fabsf(h[2]), fabsf(h[3])));
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
    const float s = scale_from_amax(amax);
    *reinterpret_cast<uint32_t*>(hq + r * I + g * 128 + lane * 4) =
        cvt_e4m3x4(__fdiv_rn(h[0], s), __fdiv_rn(h[1], s), __fdiv_rn(h[2], s), __fdiv_rn(h[3], s));
    if (lane == 0) hs[r * groups + g] = s;
  }
}

cudaError_t launch_swiglu_quant(const float* c, int64_t R, int64_t I, uint8_t* hq, float* hs,
                                cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  const int64_t warps = R * (I / 128);
  const int grid = static_cast<int>(std::min<int64_t>((warps + 7) / 8, num_sms() * 16));
  swiglu_quant_kernel<<<grid, 256, 0, s>>>(c, R, I, hq, hs);
  return cudaGetLastError();
}

}  // namespace fge

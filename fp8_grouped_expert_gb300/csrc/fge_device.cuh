// Device-side building blocks for sm_103a: mbarrier with bounded waits, TMA tiled loads,
// tcgen05 (TMEM allocation, MMA issue, commit, TMEM loads) and the e4m3 conversions.
// Everything is hand-written inline PTX; no CUTLASS/CuTe.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fge_internal.h"

namespace fge {

// ---------------------------------------------------------------------------------------
// Status word.  A device-detected failure (a wait that ran out) is recorded in a caller
// visible int32 and the kernel winds down instead of hanging.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void set_device_error(int32_t* status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

// Non-finite input probe: folding every value x of a group into acc = fma(x, 0, acc) leaves
// acc at 0 for finite values and makes it NaN as soon as one x is an infinity or a NaN
// (fmaxf-based amax reductions skip NaN, so the amax alone cannot tell).
__device__ __forceinline__ float nonfinite_fold(float acc, float x) { return fmaf(x, 0.0f, acc); }
__device__ __forceinline__ void report_nonfinite(int32_t* status, float acc) {
  if (status && acc != acc) set_device_error(status, FGE_ERR_NONFINITE);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
// Blocking probe: the thread is suspended until the phase completes or the time hint
// (nanoseconds) runs out, so waiting warps take no issue slots from working ones.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}

// Cycle budget of one wait: about one second at the GB300 clock range.  A correct
// pipeline never comes near it; it exists so that a protocol bug reports an error code
// instead of hanging a shared GPU.
constexpr long long kWaitBudgetCycles = 2000000000LL;

// Bounded wait.  Returns false when the budget ran out or another role raised the CTA's
// abort flag; the caller then stops issuing work and proceeds to the teardown.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int32_t* status, long long budget = kWaitBudgetCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  uint32_t spins = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++spins & 3u) == 0) {
      if (*abort_flag) return false;
      if (clock64() - t0 > budget) {
        *abort_flag = 1;
        set_device_error(status, FGE_ERR_DEVICE_TIMEOUT);
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor), 2-D tiled load into this CTA's shared memory.
// x is the innermost coordinate in elements; callers keep x * elem_size % 16 == 0.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t smem_dst, const CUtensorMap* map,
                                            uint32_t bar, int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
// Row gather: 4 rows (y0..y3) of a 2-D tensor, each the map's one-row box at column x,
// land as 4 consecutive box rows at smem_dst (the map's swizzle applies as for a 4-row box).
__device__ __forceinline__ void tma_gather4_2d(uint32_t smem_dst, const CUtensorMap* map,
                                               uint32_t bar, int32_t x, int4 y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y.x), "r"(y.y), "r"(y.z),
      "r"(y.w)
      : "memory");
}
// Shared -> global tile store through a tensor map (bulk-group completion).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t smem_src,
                                             int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_src), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until this thread's committed bulk stores have read their shared-memory source.
__device__ __forceinline__ void bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until all but the most recent of this thread's committed bulk stores have read their
// shared-memory source.
__device__ __forceinline__ void bulk_wait_read1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// Wait until this thread's committed bulk stores are complete.
__device__ __forceinline__ void bulk_wait0() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Generic-proxy writes to shared memory become visible to the async proxy (tcgen05.mma
// operand reads) after this fence.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------------------
// tcgen05
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t smem_result, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_result),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f8f6f4 (e4m3 x e4m3 -> f32).
__device__ __forceinline__ void mma_f8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The mbarrier receives one arrive when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// Instruction descriptor, kind::f8f6f4: D f32, A and B e4m3, both K-major, M x N.
__host__ __device__ constexpr uint32_t make_idesc_e4m3(int m, int n) {
  return (1u << 4)                                // D format: f32
         | (0u << 7) | (0u << 10)                 // A, B format: e4m3
         | (0u << 15) | (0u << 16)                // A, B K-major
         | (static_cast<uint32_t>(n >> 3) << 17)  // N / 8
         | (static_cast<uint32_t>(m >> 4) << 24); // M / 16
}

// Block-scaled MMA, kind::mxf8f6f4 with one power-of-two (UE8M0) scale per 32 K values
// (scale_vec::1X): D[tmem] (+)= (A * 2^sfa) * (B * 2^sfb)^T.  The scale factors are read from
// TMEM at sfa / sfb; the instruction descriptor's scale-factor IDs pick the byte of each
// 32-bit TMEM cell (one byte per K = 32 step).
__device__ __forceinline__ void mma_mxf8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                             uint32_t idesc, uint32_t sfa_tmem,
                                             uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of the block-scaled kind::mxf8f6f4 MMA: A E2M1 (format 5), B e4m3
// (format 0), both K-major, D f32 (implied), UE8M0 scales (bit 23), M x N, and the byte
// sf_id of the A and B scale cells (bits 29-30 and 4-5).
__host__ __device__ constexpr uint32_t make_idesc_mxf4_e4m3(int m, int n, uint32_t sf_id) {
  return (sf_id << 4)                             // B scale-factor byte
         | (5u << 7) | (0u << 10)                 // A E2M1, B e4m3
         | (0u << 15) | (0u << 16)                // A, B K-major
         | (static_cast<uint32_t>(n >> 3) << 17)  // N / 8
         | (1u << 23)                             // scale type UE8M0
         | (static_cast<uint32_t>(m >> 4) << 24)  // M / 16
         | (sf_id << 29);                         // A scale-factor byte
}

// Shared-memory matrix descriptor for a K-major operand in the 128-byte swizzle layout:
// rows of 128 bytes, 8-row atoms of 1024 bytes stacked at a 1024-byte stride.  The start
// address advances by 32 bytes per K=32 step inside the atom.
__device__ __forceinline__ uint64_t make_sdesc_sw128(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu);        // start address
  d |= static_cast<uint64_t>(0) << 16;                          // LBO (unused for SW128 K-major)
  d |= static_cast<uint64_t>((1024u >> 4) & 0x3FFFu) << 32;     // SBO: 8 rows * 128 B
  d |= static_cast<uint64_t>(1) << 46;                          // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                          // swizzle: 128 B
  return d;
}

// 32 lanes x 32 consecutive 32-bit columns from TMEM into registers (one warp).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Registers into TMEM: lane i of the warp writes 4 consecutive 32-bit columns of TMEM lane
// (its quarter's first lane + i) at taddr.
__device__ __forceinline__ void tmem_st_32x32b_x4(uint32_t taddr, uint32_t v0, uint32_t v1,
                                                  uint32_t v2, uint32_t v3) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
               "r"(v0), "r"(v1), "r"(v2), "r"(v3)
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------------------
// e4m3 helpers
// ---------------------------------------------------------------------------------------
// Two floats -> two e4m3 codes (round to nearest even, saturating); lo in the low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  return static_cast<uint32_t>(
      __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ uint32_t cvt_e4m3x4(float a, float b, float c, float d) {
  return cvt_e4m3x2(a, b) | (cvt_e4m3x2(c, d) << 16);
}

// Scale of a quantization group: s = amax / 448 (IEEE division), 1 for an all-zero group,
// raised to the smallest normal float for a tiny group.
__device__ __forceinline__ float scale_from_amax(float amax) {
  float s = __fdiv_rn(amax, 448.0f);
  if (amax == 0.0f) s = 1.0f;
  if (s < 1.17549435e-38f) s = 1.17549435e-38f;
  return s;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

}  // namespace fge

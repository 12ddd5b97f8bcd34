// tcgen05 (5th-generation tensor core) helpers for sm_103a: TMEM allocation, shared-memory matrix
// descriptors, the f16 MMA with fp32 accumulation in TMEM, commit to an mbarrier, TMEM loads.
//
// Operands live in shared memory in the K-major, 128-byte-swizzled layout: a tile of R rows x 64
// fp16 (one Q2_0 k-block) is R/8 atoms of 8 rows x 128 bytes (1024 bytes, 1024-aligned); inside an
// atom, the 16-byte chunk c of row r sits at chunk position c ^ (r % 8).
#pragma once
#include "device_common.cuh"

namespace strata {
namespace tc {

// byte offset of 16-byte chunk c (0..7) of row r in a 128B-swizzled K-major tile of 64 fp16 per row
__host__ __device__ __forceinline__ uint32_t swz_off(uint32_t r, uint32_t c) {
  return (r >> 3) * 1024u + (r & 7u) * 128u + ((c ^ (r & 7u)) << 4);
}

// Shared-memory matrix descriptor: start address, leading byte offset (unused for swizzled K-major
// tiles that are one swizzle atom wide), stride byte offset between 8-row atoms (1024), descriptor
// version 1, base offset 0 (atoms are 1024-byte aligned), layout SWIZZLE_128B.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1u << 16;                // LBO (ignored here)
  d |= (uint64_t)(1024u >> 4) << 32;      // SBO
  d |= (uint64_t)1u << 46;                // version
  d |= (uint64_t)2u << 61;                // SWIZZLE_128B
  return d;
}

// Instruction descriptor of kind::f16 with fp16 A and B, fp32 accumulator, both K-major.
__host__ __device__ __forceinline__ uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4)                        // D format fp32
         | ((uint32_t)(N >> 3) << 17)     // N / 8
         | ((uint32_t)(M >> 4) << 24);    // M / 16
}

// One warp allocates ncols TMEM columns (power of two >= 32); the base address is written to *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, M x N x 16, issued by one thread.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One 64-wide k-block of MMAs (K = 16 each; descriptors advance 32 bytes per step) into accumulator d0
// from a0 against b; the first step accumulates only if acc_first != 0.  The mbarrier at next_bar is
// tested (non-blocking) for phase parity next_par before the MMAs and its result read after them, so
// the test's latency hides behind their issue; returns 1 if that phase had completed.
__device__ __forceinline__ uint32_t mma_kblock_test_next(uint32_t d0, uint64_t a0, uint64_t b, uint32_t idesc,
                                                         uint32_t acc_first, uint32_t next_bar, uint32_t next_par) {
  uint32_t ready;
  asm volatile(
      "{\n\t.reg .pred pr, pa, pt;\n\t.reg .b64 ta, tb;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 pr, [%6], %7;\n\t"
      "setp.ne.b32 pa, %5, 0;\n\t"
      "setp.eq.b32 pt, %4, %4;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], %2, %3, %4, pa;\n\t"
      "add.s64 ta, %2, 2;\n\tadd.s64 tb, %3, 2;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], ta, tb, %4, pt;\n\t"
      "add.s64 ta, %2, 4;\n\tadd.s64 tb, %3, 4;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], ta, tb, %4, pt;\n\t"
      "add.s64 ta, %2, 6;\n\tadd.s64 tb, %3, 6;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], ta, tb, %4, pt;\n\t"
      "selp.u32 %0, 1, 0, pr;\n\t}"
      : "=r"(ready)
      : "r"(d0), "l"(a0), "l"(b), "r"(idesc), "r"(acc_first), "r"(next_bar), "r"(next_par)
      : "memory");
  return ready;
}

// Four consecutive fp32 reductions (16-byte aligned address) with an L2 eviction-policy hint.
__device__ __forceinline__ void red_add_v4_f32_hint(float* p, float a, float b, float c, float d, uint64_t policy) {
  asm volatile("red.global.add.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "f"(a), "f"(b), "f"(c),
               "f"(d), "l"(policy)
               : "memory");
}

// 4 x 4 transpose across the lanes 4g .. 4g + 3 of a warp (j = lane & 3): lane j holds row j of the
// block in v[0..3] on entry and column j (rows 0..3) on return.  Two butterfly steps, lane distance 2
// then 1, each exchanging one half of the lane's values.
__device__ __forceinline__ void transpose4_lanes(uint32_t (&v)[4], int j) {
  const bool a2 = (j & 2) != 0, a1 = (j & 1) != 0;
  uint32_t r0 = __shfl_xor_sync(0xffffffffu, a2 ? v[0] : v[2], 2);
  uint32_t r1 = __shfl_xor_sync(0xffffffffu, a2 ? v[1] : v[3], 2);
  if (a2) { v[0] = r0; v[1] = r1; } else { v[2] = r0; v[3] = r1; }
  r0 = __shfl_xor_sync(0xffffffffu, a1 ? v[0] : v[1], 1);
  r1 = __shfl_xor_sync(0xffffffffu, a1 ? v[2] : v[3], 1);
  if (a1) { v[0] = r0; v[2] = r1; } else { v[1] = r0; v[3] = r1; }
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// The fp16 token copy the tensor-core expert path reads its token tiles from: X16[kb][t][128 bytes] =
// x[t][64 kb .. 64 kb + 63] times sc, as fp16, each 16-weight group in the order 0,8,1,9,..,7,15 (the
// order one LOP3 per half2 gives the dequantised weights), chunk c (16 bytes) of a row holding
// weights {4(c&1) .. +3} interleaved with {8 + 4(c&1) .. +3} of group c / 2.  Called by a whole warp for
// token t with a = x[t][4 (lane + 32 i) .. +3]: the float4 8 weights further is two lanes up, so lanes
// 4j and 4j + 1 each assemble and store one chunk.
__device__ __forceinline__ void x16_store_chunk(const float4 a, int i, float sc, int t, int T, uint8_t* x16) {
  const int lane = threadIdx.x & 31;
  float4 b;
  b.x = __shfl_down_sync(0xffffffffu, a.x, 2);
  b.y = __shfl_down_sync(0xffffffffu, a.y, 2);
  b.z = __shfl_down_sync(0xffffffffu, a.z, 2);
  b.w = __shfl_down_sync(0xffffffffu, a.w, 2);
  if ((lane & 2) == 0) {
    const int m = lane + 32 * i;  // float4 index: 16-group m >> 2, half m & 1
    const int kb = m >> 4, c = 2 * ((m >> 2) & 3) + (m & 1);
    const __half2 h0 = __floats2half2_rn(a.x * sc, b.x * sc), h1 = __floats2half2_rn(a.y * sc, b.y * sc);
    const __half2 h2 = __floats2half2_rn(a.z * sc, b.z * sc), h3 = __floats2half2_rn(a.w * sc, b.w * sc);
    *reinterpret_cast<uint4*>(x16 + ((size_t)kb * T + t) * 128 + c * 16) =
        make_uint4(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1),
                   *reinterpret_cast<const uint32_t*>(&h2), *reinterpret_cast<const uint32_t*>(&h3));
  }
}

// Arrive (once) on an mbarrier when every MMA issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// generic-proxy shared-memory writes -> visible to the tensor core (async proxy)
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }


// 32 lanes x 32 bits x 16 columns into registers without waiting: thread t of the warp gets lane
// (quadrant*32 + t), 16 consecutive columns; tmem_wait_ld() makes every such load issued so far complete.
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
      "[%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 bits x 16 columns: thread t of the warp gets lane (quadrant*32 + t), 16 consecutive columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
      "[%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace tc
}  // namespace strata

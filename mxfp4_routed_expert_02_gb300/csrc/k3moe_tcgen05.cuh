// k3moe_tcgen05.cuh -- device helpers of the 5th-generation tensor-core path shared by
// the grouped GEMM (k3moe_tc.cu), its encoders (k3moe_prefill.cu) and the single-token
// tensor-core gate/up (k3moe_gateup_tc.cu): tensor-memory allocation and access,
// shared-memory matrix descriptors, block-scaled MMA issue, tiled TMA loads, and the
// MXFP4 multi-term encoding of an activation group.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>

#include "k3moe_tc.cuh"

namespace k3 {

constexpr int kTcTile = kTcRows;          // A rows and B rows per tile
constexpr int kTcChunkBytes = kTcChunk;   // K bytes per stage (one swizzle atom)
constexpr uint32_t kTcBox = kTcTile * kTcChunkBytes;  // bytes of one A box (16 KB)
constexpr int kSfB = 2 * kTcSteps;        // scale bytes per row per stage (2 per K step)
constexpr int kSfW = 4 * kTcSteps;        // TMEM columns of one operand's scales per stage
static_assert(kTcChunkBytes == 64 || kTcChunkBytes == 128, "64- or 128-byte swizzle");

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, int cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, int cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Shared-memory matrix descriptors (K-major, swizzled: 8-row atoms of kTcChunkBytes-byte
// rows).  The MMAs take a descriptor as its low word (start address >> 4; leading byte
// offset 1, unused for swizzled K-major) plus this constant high word (stride byte offset
// = one 8-row atom, descriptor version 1, swizzle mode 4 = 64 B or 2 = 128 B); offsets
// within shared memory change only the address field of the low word, which cannot carry
// out of it below 256 KB.  A K step inside the atom moves the start address by 32 bytes.
constexpr uint32_t kDescHi = ((8u * kTcChunkBytes) >> 4) | (1u << 14) |
                             ((kTcChunkBytes == 64 ? 4u : 2u) << 29);
__device__ __forceinline__ uint32_t sw_desc_lo(uint32_t saddr) {
  return ((saddr & 0x3FFFFu) >> 4) | (1u << 16);
}
__device__ __forceinline__ void mma_mxf4_el_lo(uint32_t d, uint32_t alo, uint32_t blo, uint32_t hi,
                                               uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                               uint32_t acc) {
  asm volatile(
      "{ .reg .pred p, e; .reg .b32 r; .reg .b64 da, db; elect.sync r|e, 0xffffffff;\n"
      "  setp.ne.b32 p, %7, 0; mov.b64 da, {%1, %3}; mov.b64 db, {%2, %3};\n"
      "  @e tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], da, db, %4, "
      "[%5], [%6], p; }" ::"r"(d),
      "r"(alo), "r"(blo), "r"(hi), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_f16_el_lo(uint32_t d, uint32_t alo, uint32_t blo, uint32_t hi,
                                              uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p, e; .reg .b32 r; .reg .b64 da, db; elect.sync r|e, 0xffffffff;\n"
      "  setp.ne.b32 p, %5, 0; mov.b64 da, {%1, %3}; mov.b64 db, {%2, %3};\n"
      "  @e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, p; }" ::"r"(d),
      "r"(alo), "r"(blo), "r"(hi), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void tc_commit_el(uint64_t *bar) {
  asm volatile(
      "{ .reg .pred e; .reg .b32 r; elect.sync r|e, 0xffffffff;\n"
      "  @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0]; }" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 3-D tiled TMA load (x = K byte, y = row, z = group or term) completing on `bar`.
__device__ __forceinline__ void tma_load3d(void *dst, const CUtensorMap *map, int x, int y, int z,
                                           uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// The same with an L2 eviction policy.
__device__ __forceinline__ void tma_load3d_pol(void *dst, const CUtensorMap *map, int x, int y,
                                               int z, uint64_t *bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ void tma_load4d_pol(void *dst, const CUtensorMap *map, int x, int y,
                                               int z, int w, uint64_t *bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar)),
      "l"(pol)
      : "memory");
}
__device__ __forceinline__ void tma_load4d(void *dst, const CUtensorMap *map, int x, int y, int z,
                                           int w, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_st_x1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v)
               : "memory");
}
__device__ __forceinline__ void tmem_st_x16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_x8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
      : "memory");
}
// One operand's scale columns of a stage (x8 or x16 by the array's size).
__device__ __forceinline__ void tmem_st_sf(uint32_t taddr, const uint32_t (&v)[8]) {
  tmem_st_x8(taddr, v);
}
[[maybe_unused]] __device__ __forceinline__ void tmem_st_sf(uint32_t taddr,
                                                            const uint32_t (&v)[16]) {
  tmem_st_x16(taddr, v);
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}
// Waits for this thread's outstanding tcgen05.ld; the registers are passed through so the
// compiler cannot read them before the wait.
__device__ __forceinline__ void tmem_wait_ld2(uint32_t (&v)[16], uint32_t (&w)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]),
                 "+r"(v[6]), "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]),
                 "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15]), "+r"(w[0]), "+r"(w[1]),
                 "+r"(w[2]), "+r"(w[3]), "+r"(w[4]), "+r"(w[5]), "+r"(w[6]), "+r"(w[7]),
                 "+r"(w[8]), "+r"(w[9]), "+r"(w[10]), "+r"(w[11]), "+r"(w[12]), "+r"(w[13]),
                 "+r"(w[14]), "+r"(w[15])
               :
               : "memory");
}
// The kSfB scale bytes of one row for K chunk c (groups kSfB*c ..), fewer at the row's end;
// bytes past the row read 0.  Returned in .x (and .y for 8 bytes).
__device__ __forceinline__ uint2 load_scales(const uint8_t *row, int G, int c) {
  const int g0 = kSfB * c;
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int j = 0; j < kSfB; j++) {
    const uint32_t b = (g0 + j < G) ? (uint32_t)__ldg(row + g0 + j) : 0u;
    w[j >> 2] |= b << (8 * (j & 3));
  }
  return make_uint2(w[0], w[1]);
}
// kSfB staged scale bytes at p (kSfB-aligned) as a uint2 (.y = 0 for 4 bytes).
__device__ __forceinline__ uint2 ld_staged_scales(const uint8_t *p) {
  if (kSfB == 8) return *reinterpret_cast<const uint2 *>(p);
  return make_uint2(*reinterpret_cast<const uint32_t *>(p), 0u);
}
__device__ __forceinline__ void st_staged_scales(uint8_t *p, uint2 v) {
  if (kSfB == 8)
    *reinterpret_cast<uint2 *>(p) = v;
  else
    *reinterpret_cast<uint32_t *>(p) = v.x;
}
// The two scale bytes of K step i (groups 2i, 2i+1 of the chunk), in bytes 0 and 1.
__device__ __forceinline__ uint32_t step_scales(uint2 s, int i) {
  const uint32_t w = (i < 2) ? s.x : s.y;
  return (w >> (16 * (i & 1))) & 0xffffu;
}


// Four consecutive accumulator columns of this warp's lane quarter, and the wait for two
// such loads (registers passed through, so they cannot be read before it).
__device__ __forceinline__ void tmem_ld4_nowait(uint32_t taddr, uint32_t (&v)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_wait_ld4(uint32_t (&v)[4], uint32_t (&w)[4]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(w[0]), "+r"(w[1]),
                 "+r"(w[2]), "+r"(w[3])
               :
               : "memory");
}

// One group of 32 values -> NT MXFP4 terms: term i takes the residual left by terms
// 0..i-1, with the E8M0 scale 2^e chosen so that max|r| <= 6 * 2^e and each value rounded
// to the nearest E2M1 code (hardware conversion, round to nearest even); residuals are
// exact in float.  Codes packed two per byte, the even element in the low nibble.
template <int NT>
__device__ __forceinline__ void encode_terms(float (&r)[32], uint4 (&q)[NT], uint8_t (&sb)[NT]) {
#pragma unroll
  for (int t = 0; t < NT; t++) {
    float m = 0.f;
#pragma unroll
    for (int k = 0; k < 32; k++) m = fmaxf(m, fabsf(r[k]));
    int e = -127;
    if (m > 0.f) {
      e = exponent_of(m) - 2;
      if (m > 6.f * pow2i(e)) e++;
      e = e < -127 ? -127 : (e > 127 ? 127 : e);
    }
    sb[t] = (uint8_t)(e + 127);
    const float inv_s = pow2i(-e), s = pow2i(e);
    uint32_t w[4];
#pragma unroll
    for (int wq = 0; wq < 4; wq++) {
      uint32_t word = 0;
#pragma unroll
      for (int bb = 0; bb < 4; bb++) {
        const int k = 8 * wq + 2 * bb;
        uint32_t byte;
        asm("{ .reg .b8 t8; cvt.rn.satfinite.e2m1x2.f32 t8, %1, %2; cvt.u32.u8 %0, t8; }"
            : "=r"(byte)
            : "f"(r[k + 1] * inv_s), "f"(r[k] * inv_s));
        word |= byte << (8 * bb);
        // residual: subtract the decoded value (exact)
        const uint32_t h2 = e2m1x2_to_f16x2(byte);
        const __half2 hv = *reinterpret_cast<const __half2 *>(&h2);
        r[k] = __fsub_rn(r[k], __low2float(hv) * s);
        r[k + 1] = __fsub_rn(r[k + 1], __high2float(hv) * s);
      }
      w[wq] = word;
    }
    q[t] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace k3

// k3moe_device.cuh -- device helpers shared by the k3moe kernels (sm_103a).
//
// Number formats follow the README of FareedKhan-dev/kimi-k3-in-c, section 4
// "Reduction one: the experts already ship at half a byte": a weight is an E2M1 code
// (sign, two exponent bits, one mantissa bit) times an E8M0 scale 2^(s-127) shared by
// 32 consecutive weights of a row; scale byte 255 reads as 0; in a packed byte the low
// nibble is the even column.  bf16 widening is a 16-bit shift (section 5).
#pragma once
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "k3moe.h"

namespace k3 {

constexpr int kGroup = 32;  // MXFP4 block size

// First error wins; later errors leave the word alone.
__device__ __forceinline__ void set_status(int32_t *st, int code) {
  if (st) atomicCAS(st, 0, code);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// float -> bf16 bits, round to nearest even (NaN kept quiet).
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return (uint16_t)((u >> 16) | 0x40);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

// 2^e as a float: exact for -149 <= e <= 127, 0 below, +inf above.
__device__ __forceinline__ float pow2i(int e) {
  if (e >= -126 && e <= 127) return __int_as_float((e + 127) << 23);
  if (e > 127) return __int_as_float(0x7f800000);
  if (e >= -149) return __int_as_float(1 << (e + 149));
  return 0.f;
}

// Unbiased exponent of a finite nonzero float's magnitude (floor(log2|v|)); the
// subnormal range reports -127 (callers clamp).
__device__ __forceinline__ int exponent_of(float v) {
  return (int)((__float_as_uint(v) >> 23) & 0xff) - 127;
}

// One packed MXFP4 byte (two E2M1 codes) -> f16x2 with the low nibble (even column)
// in the low half.  Hardware conversion, exact (every E2M1 value is an f16).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte_in_low_bits) {
  uint32_t h;
  asm("{ .reg .b8 b; cvt.u8.u32 b, %1; cvt.rn.f16x2.e2m1x2 %0, b; }"
      : "=r"(h)
      : "r"(byte_in_low_bits));
  return h;
}

// Four packed bytes (eight E2M1 codes, columns 0..7 of the word) -> four f16x2.
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t q, uint32_t &h0, uint32_t &h1,
                                                  uint32_t &h2, uint32_t &h3) {
  asm("{ .reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %4;\n"
      "  cvt.rn.f16x2.e2m1x2 %0, b0; cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      "  cvt.rn.f16x2.e2m1x2 %2, b2; cvt.rn.f16x2.e2m1x2 %3, b3; }"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
      : "r"(q));
}

// c + x.lo * w.lo + x.hi * w.hi with f16 operands and an f32 accumulator: each product
// is exact (f16 x f16 fits in f32) and each add rounds once to f32.
__device__ __forceinline__ float fma2_f16_f32(uint32_t x2, uint32_t w2, float c) {
  float d;
  asm("{ .reg .b16 xl, xh, wl, wh; mov.b32 {xl, xh}, %1; mov.b32 {wl, wh}, %2;\n"
      "  fma.rn.f32.f16 %0, xl, wl, %3; fma.rn.f32.f16 %0, xh, wh, %0; }"
      : "=f"(d)
      : "r"(x2), "r"(w2), "f"(c));
  return d;
}

// c + x.lo * w.lo + x.hi * w.hi with bf16 operands and an f32 accumulator (mixed-precision
// FMA: each bf16 x bf16 product is exact in f32, each add rounds once) -- the same result
// as widening both to f32 first, without the widening instructions.
__device__ __forceinline__ float fma2_bf16_f32(uint32_t x2, uint32_t w2, float c) {
  float d;
  asm("{ .reg .b16 xl, xh, wl, wh; mov.b32 {xl, xh}, %1; mov.b32 {wl, wh}, %2;\n"
      "  fma.rn.f32.bf16 %0, xl, wl, %3; fma.rn.f32.bf16 %0, xh, wh, %0; }"
      : "=f"(d)
      : "r"(x2), "r"(w2), "f"(c));
  return d;
}

// The two exact products x.lo * w.lo and x.hi * w.hi of bf16 pairs, as floats (an FMA
// with -0 added keeps the sign of a zero product).
__device__ __forceinline__ void mul2_bf16_f32(uint32_t x2, uint32_t w2, float &p0, float &p1) {
  asm("{ .reg .b16 xl, xh, wl, wh; mov.b32 {xl, xh}, %2; mov.b32 {wl, wh}, %3;\n"
      "  fma.rn.f32.bf16 %0, xl, wl, 0f80000000; fma.rn.f32.bf16 %1, xh, wh, 0f80000000; }"
      : "=f"(p0), "=f"(p1)
      : "r"(x2), "r"(w2));
}

// Sum over the 32 columns of one MXFP4 group: sum_k x'[k] * e2m1[k] (unscaled), with
// x' given as 16 f16x2 registers (pair p = columns 2p, 2p+1) and the weights as the 16
// packed bytes of the group (4 words).  Two accumulators for latency.
__device__ __forceinline__ float group_dot(const uint32_t (&x)[16], uint4 w) {
  float a = 0.f, b = 0.f, c = 0.f, d = 0.f;  // four chains for latency
  uint32_t h0, h1, h2, h3;
  e2m1x8_to_f16x2x4(w.x, h0, h1, h2, h3);
  a = fma2_f16_f32(x[0], h0, a); b = fma2_f16_f32(x[1], h1, b);
  c = fma2_f16_f32(x[2], h2, c); d = fma2_f16_f32(x[3], h3, d);
  e2m1x8_to_f16x2x4(w.y, h0, h1, h2, h3);
  a = fma2_f16_f32(x[4], h0, a); b = fma2_f16_f32(x[5], h1, b);
  c = fma2_f16_f32(x[6], h2, c); d = fma2_f16_f32(x[7], h3, d);
  e2m1x8_to_f16x2x4(w.z, h0, h1, h2, h3);
  a = fma2_f16_f32(x[8], h0, a); b = fma2_f16_f32(x[9], h1, b);
  c = fma2_f16_f32(x[10], h2, c); d = fma2_f16_f32(x[11], h3, d);
  e2m1x8_to_f16x2x4(w.w, h0, h1, h2, h3);
  a = fma2_f16_f32(x[12], h0, a); b = fma2_f16_f32(x[13], h1, b);
  c = fma2_f16_f32(x[14], h2, c); d = fma2_f16_f32(x[15], h3, d);
  return (a + b) + (c + d);
}

// Same with x' = hi + lo (two f16 terms per column): sum_k (hi[k] + lo[k]) * e2m1[k].
// The hi products go through the exact f16 x f16 -> f32 path; the lo term (at most 2^-11
// of hi) is accumulated in packed f16 (HFMA2), whose rounding is ~2^-11 of a term that is
// itself ~2^-11 of the result, i.e. ~2^-22 relative -- far below f32 accumulation noise of
// a 1536-term sum.  |lo| <= 2^4 after prescaling, so the f16 sums cannot overflow.
__device__ __forceinline__ float group_dot2(const uint32_t (&xh)[16], const uint32_t (&xl)[16],
                                            uint4 w) {
  float a = 0.f, b = 0.f;
  __half2 l2 = __float2half2_rn(0.f);
  uint32_t h[4];
  const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int q = 0; q < 4; q++) {
    e2m1x8_to_f16x2x4(ww[q], h[0], h[1], h[2], h[3]);
#pragma unroll
    for (int p = 0; p < 4; p++) {
      if (p & 1)
        b = fma2_f16_f32(xh[4 * q + p], h[p], b);
      else
        a = fma2_f16_f32(xh[4 * q + p], h[p], a);
      l2 = __hfma2(*reinterpret_cast<const __half2 *>(&xl[4 * q + p]),
                   *reinterpret_cast<const __half2 *>(&h[p]), l2);
    }
  }
  return (a + b) + (__low2float(l2) + __high2float(l2));
}

// Layout of the routed activations handed from gate/up to down, per (token, slot) pair
// i: element k of input group gg lives at  i*I + ((k / 8) * (I/32) + gg) * 8 + k % 8,
// i.e. [pair][chunk of 8][group][8]: lanes that take consecutive groups read consecutive
// 16-byte chunks.
__host__ __device__ __forceinline__ size_t act_index(int i, int I, int gg, int k) {
  return (size_t)i * I + ((size_t)(k >> 3) * (I / 32) + gg) * 8 + (k & 7);
}

// Factor turning an unscaled group sum into its contribution: 2^(s - 127 + ex) where s
// is the E8M0 scale byte and ex the exponent the activation group was scaled by; a
// scale byte of 255 contributes nothing.
__device__ __forceinline__ float group_factor(uint32_t s, int ex) {
  // normal results (biased exponent s + ex in 1..254) are the exponent bits themselves;
  // subnormal, overflowing and s = 255 cases take the general path
  const uint32_t b = (uint32_t)((int)s + ex);
  if (s != 255u && b - 1u < 254u) return __uint_as_float(b << 23);
  return (s == 255u) ? 0.f : pow2i((int)s - 127 + ex);
}

// Prescale a group of 32 activations to f16: x' = x * 2^-ex with ex chosen so that
// max|x'| lies in [2^14, 2^15) (every bf16 value then converts to f16 exactly, bar
// values more than 2^28 below the group maximum).  Returns ex.
__device__ __forceinline__ int prescale_group_f16(const float (&v)[32], uint32_t (&out)[16]) {
  float m = 0.f;
#pragma unroll
  for (int k = 0; k < 32; k++) m = fmaxf(m, fabsf(v[k]));
  int ex = 0;
  if (m > 0.f) {
    ex = exponent_of(m) - 14;
    ex = ex < -110 ? -110 : ex;
  }
  const float s = pow2i(-ex);
#pragma unroll
  for (int p = 0; p < 16; p++) {
    __half2 h = __floats2half2_rn(v[2 * p] * s, v[2 * p + 1] * s);
    out[p] = *reinterpret_cast<uint32_t *>(&h);
  }
  return ex;
}

// The group prescaled as prescale_group_f16 does, as two f16 terms: hi = f16(x'), lo =
// f16(x' - hi) (the residual is exact in float), about 22 significant bits for float
// inputs.  Returns the exponent ex (x' = x 2^-ex).
__device__ __forceinline__ int prescale_group_f16_hilo(const float (&v)[32], uint32_t (&hi)[16],
                                                       uint32_t (&lo)[16]) {
  const int ex = prescale_group_f16(v, hi);
  const float s = pow2i(-ex);
#pragma unroll
  for (int p = 0; p < 16; p++) {
    const float2 h = __half22float2(*reinterpret_cast<const __half2 *>(&hi[p]));
    __half2 l = __floats2half2_rn(v[2 * p] * s - h.x, v[2 * p + 1] * s - h.y);
    lo[p] = *reinterpret_cast<uint32_t *>(&l);
  }
  return ex;
}

// SiTU-GLU (kimi-k3-in-c, section 9): the sigmoid takes the uncapped gate.
__device__ __forceinline__ float situ(float g, float u, float b1, float b2) {
  const float a = b1 * tanhf(g / b1) * (1.f / (1.f + expf(-g)));
  const float v = b2 * tanhf(u / b2);
  return a * v;
}

// Error-free sum (Knuth's TwoSum): s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// (hi, lo) += (bh, bl) for float-float pairs, renormalised.
__device__ __forceinline__ void ff_add(float &hi, float &lo, float bh, float bl) {
  float s, e;
  two_sum(hi, bh, s, e);
  e = __fadd_rn(e, __fadd_rn(lo, bl));
  hi = __fadd_rn(s, e);
  lo = __fsub_rn(e, __fsub_rn(hi, s));
}


// Transpose-reduce V values (V = 8, 16 or 32) over the 32 lanes of a warp: afterwards lane
// l holds the warp total of value (l % V).  Fixed shuffle tree: deterministic.
template <int V>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[V]) {
  const int lane = threadIdx.x & 31;
  // halving steps over lane bits log2(V)-1 .. 0
#pragma unroll
  for (int half = V / 2; half >= 1; half >>= 1) {
    const bool upper = (lane & half) != 0;
#pragma unroll
    for (int i = 0; i < half; i++) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, half);
    }
  }
  float r = v[0];
#pragma unroll
  for (int o = V; o < 32; o <<= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
  return r;
}

}  // namespace k3

// ---------------------------------------------------------------------------------
// Bulk async copies (TMA, non-tensor form) and mbarriers, sm_90+ PTX.
// ---------------------------------------------------------------------------------
namespace k3 {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
// Invalidate an mbarrier no thread uses any more, before its memory is initialised again.
__device__ __forceinline__ void mbar_inval(uint64_t *bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
      "selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Gives up after about
// `budget` SM clock cycles and returns false (the caller reports K3MOE_ERR_TIMEOUT).
constexpr long long kWaitBudget = 4000000000LL;  // ~2 s at 2 GHz
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          long long budget = kWaitBudget) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > budget) return false;
  }
  return true;
}

// global -> shared bulk copy completing on an mbarrier (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Bulk prefetch of global memory into L2 (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// L2 eviction policy "evict first" (for every access that carries it): bytes read once.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// bulk_prefetch_l2 with an L2 eviction policy.
__device__ __forceinline__ void bulk_prefetch_l2_pol(const void *src, uint32_t bytes,
                                                     uint64_t pol) {
  asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(src),
               "r"(bytes), "l"(pol)
               : "memory");
}
// bulk_g2s with an L2 eviction policy.
__device__ __forceinline__ void bulk_g2s_pol(void *dst, const void *src, uint32_t bytes,
                                             uint64_t *bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
      "[%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// Programmatic dependent launch: wait for the previous kernel's writes / let the next
// kernel start its prologue.  Both are no-ops when the launch is not programmatic.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace k3

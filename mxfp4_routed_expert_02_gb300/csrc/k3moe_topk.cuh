// k3moe_topk.cuh -- top-k selection of one token by one CTA (shared by the router's top-k
// kernel and the single-token gate/up kernel).
//
// The selection is the page's repeated strict maximum over the selection scores
// (README of FareedKhan-dev/kimi-k3-in-c, section 9 "Picking 16 experts of 896"): the K
// largest by (selection score desc, expert index asc), in that order.  Every expert
// becomes one 64-bit key whose unsigned order is exactly that order -- high word: the
// selection score's bits mapped to an unsigned integer that increases with the float
// value; low word: the complement of the index, so a lower index ranks higher.  Keys are
// distinct, so the K largest keys, in descending order, are the page's selection.
//
// Method: warps sort chunks of 64 keys (two per lane, a bitonic network in registers)
// and keep each chunk's K largest; the candidate set shrinks by 64/K per level until one
// chunk is left.  The K largest of a set are always among the K largest of the chunk
// that holds them, so nothing is lost.
#pragma once
#include "k3moe_device.cuh"

namespace k3 {

// Unsigned image of a float that increases with the float (negative values reversed).
__device__ __forceinline__ uint32_t float_order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Sort the 64 keys a warp holds (a at position lane, b at position lane + 32) into
// descending order in place.
__device__ __forceinline__ void warp_sort64_desc(unsigned long long &a, unsigned long long &b) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 64; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride == 32) {  // partners a <-> b of the same lane (size 64: descending block)
        const unsigned long long hi = a > b ? a : b, lo = a > b ? b : a;
        a = hi;
        b = lo;
      } else {
        const unsigned long long wa = __shfl_xor_sync(0xffffffffu, a, stride);
        const unsigned long long wb = __shfl_xor_sync(0xffffffffu, b, stride);
        const bool lower = (lane & stride) == 0;
        const bool desc_a = (lane & size) == 0, desc_b = ((lane + 32) & size) == 0;
        a = (lower == desc_a) ? (a > wa ? a : wa) : (a < wa ? a : wa);
        b = (lower == desc_b) ? (b > wb ? b : wb) : (b < wb ? b : wb);
      }
    }
  }
}

// Shared scratch (uint64) cta_topk needs: two candidate buffers of ceil(E/64)*K keys.
__host__ __device__ inline int topk_scratch_keys(int E, int K) { return 2 * ((E + 63) / 64) * K; }

// g_sc / g_ch: the token's E unbiased / selection scores (global).  cand: shared scratch of
// topk_scratch_keys(E, K) uint64.  Writes sel[K] (expert ids in selection order) and
// wsel[K] (the unbiased scores, renormalised by their float sum in that order when
// positive, times routed_scale) to shared memory; every thread returns after a
// __syncthreads.  K <= 32.
__device__ __forceinline__ void cta_topk(const float *__restrict__ g_sc,
                                         const float *__restrict__ g_ch, int E, int K,
                                         int renorm, float routed_scale,
                                         unsigned long long *cand, int *sel, float *wsel) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int NW = blockDim.x >> 5;
  auto key_of = [&](int e) -> unsigned long long {
    if (e >= E) return 0ull;  // below every real key
    float c = __fadd_rn(g_ch[e], 0.f);            // -0 -> +0: equal scores compare equal
    if (c != c) c = -__int_as_float(0x7f800000);  // a NaN never wins (it is reported)
    return ((unsigned long long)float_order_key(c) << 32) |
           (unsigned long long)(0xffffffffu - (uint32_t)e);
  };
  unsigned long long *src = cand, *dst = cand + ((E + 63) / 64) * K;
  // level 0: chunks of the E keys -> src
  int chunks = (E + 63) / 64;
  for (int c = warp; c < chunks; c += NW) {
    unsigned long long a = key_of(64 * c + lane), b = key_of(64 * c + 32 + lane);
    warp_sort64_desc(a, b);
    if (lane < K) src[c * K + lane] = a;  // K <= 32: the top K sit in a
  }
  int m = chunks * K;  // candidates in src
  __syncthreads();
  // further levels: chunks of 64 candidates, src -> dst, until one chunk's top K is left
  while (chunks > 1) {
    chunks = (m + 63) / 64;
    for (int c = warp; c < chunks; c += NW) {
      unsigned long long a = (64 * c + lane < m) ? src[64 * c + lane] : 0ull;
      unsigned long long b = (64 * c + 32 + lane < m) ? src[64 * c + 32 + lane] : 0ull;
      warp_sort64_desc(a, b);
      if (lane < K) dst[c * K + lane] = a;
    }
    m = chunks * K;
    unsigned long long *t = src;
    src = dst;
    dst = t;
    __syncthreads();
  }
  cand = src;
  if (warp == 0) {
    int e = 0;
    float s = 0.f;
    if (lane < K) {
      const unsigned long long key = cand[lane];
      e = (key == 0ull) ? 0 : (int)(0xffffffffu - (uint32_t)(key & 0xffffffffull));
      s = g_sc[e];
    }
    // float sum of the chosen scores in selection order
    float wsum = 0.f;
    for (int j = 0; j < K; j++) wsum = __fadd_rn(wsum, __shfl_sync(0xffffffffu, s, j));
    if (lane < K) {
      float w = s;
      if (renorm && wsum > 0.f) w = __fdiv_rn(w, wsum);
      sel[lane] = e;
      wsel[lane] = __fmul_rn(w, routed_scale);
    }
  }
  __syncthreads();
}

}  // namespace k3

// k3moe_topk.cuh -- top-k selection of one token by one CTA (shared by the router's top-k
// kernel and the single-token gate/up kernel).
#pragma once
#include "k3moe_device.cuh"

namespace k3 {

// ------------------------------------------------------------------------------------
// Top-k of one token by one CTA of 8+ warps (kimi-k3-in-c, section 9): each of the first
// 8 warps takes the top K of a contiguous slice of the experts by K rounds of a warp-wide
// maximum of (selection score desc, index asc); warp 0 merges the eight sorted lists with
// the same key.  Weights: the unbiased scores of the chosen experts, renormalised by their
// float sum (router order) when positive, times routed_scale.  Results in sel/wsel
// (shared); every thread returns after a __syncthreads.
// ------------------------------------------------------------------------------------
__device__ __forceinline__ bool topk_better(float ach, int ae, float bch, int be) {
  if (ae < 0) return false;
  if (be < 0) return true;
  if (ach > bch) return true;
  if (ach == bch) return ae < be;
  return (bch != bch) && (ach == ach);
}

__device__ __forceinline__ void topk_warp_best(float &ch, int &e) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float och = __shfl_xor_sync(0xffffffffu, ch, o);
    const int oe = __shfl_xor_sync(0xffffffffu, e, o);
    if (topk_better(och, oe, ch, e)) {
      ch = och;
      e = oe;
    }
  }
}

__device__ __forceinline__ void cta_topk(const float *__restrict__ g_sc,
                                         const float *__restrict__ g_ch, int E, int K,
                                         int renorm, float routed_scale,
                                         float *s_sc /* [E] smem */, float *s_ch /* [E] smem */,
                                         int *lst /* [8][32] smem */, int *sel /* [32] smem */,
                                         float *wsel /* [32] smem */) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // one coalesced pass over the scores into shared memory; the K selection rounds then
  // read shared memory only
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    s_sc[e] = g_sc[e];
    s_ch[e] = g_ch[e];
  }
  __syncthreads();
  const float *sc = s_sc, *ch = s_ch;
  const int NW = min(8, (int)(blockDim.x >> 5));  // slices; each <= 64 experts per lane
  if (warp < NW) {
    const int per = (E + NW - 1) / NW;
    const int lo = warp * per, hi = min(E, lo + per);
    unsigned long long taken = 0ull;
    for (int k = 0; k < K; k++) {
      float bc = 0.f;
      int be = -1;
      int i = 0;
      for (int e = lo + lane; e < hi; e += 32, i++) {
        if (taken & (1ull << i)) continue;
        const float c = ch[e];
        if (topk_better(c, e, bc, be)) {
          bc = c;
          be = e;
        }
      }
      topk_warp_best(bc, be);
      if (be >= 0 && ((be - lo) & 31) == lane) taken |= 1ull << ((be - lo) >> 5);
      if (lane == 0) lst[warp * 32 + k] = be;
    }
  }
  __syncthreads();
  if (warp == 0) {
    int head = 0;
    float wsum = 0.f, myw = 0.f;
    int mye = -1;
    for (int k = 0; k < K; k++) {
      int e = -1;
      float c = 0.f;
      if (lane < NW && head < K) {
        e = lst[lane * 32 + head];
        if (e >= 0) c = ch[e];
      }
      const int cand = e;
      topk_warp_best(c, e);
      if (lane < NW && e >= 0 && cand == e) head++;
      const float s = (e >= 0) ? sc[e] : 0.f;
      wsum = __fadd_rn(wsum, s);
      if (lane == k) {
        mye = e;
        myw = s;
      }
    }
    if (lane < K) {
      float v = myw;
      if (renorm && wsum > 0.f) v = __fdiv_rn(v, wsum);
      sel[lane] = mye < 0 ? 0 : mye;
      wsel[lane] = __fmul_rn(v, routed_scale);
    }
  }
  __syncthreads();
}

}  // namespace k3

// k3moe_router.cu -- router logits, shared-expert gate/up, top-k selection.
//
// The router follows the README of FareedKhan-dev/kimi-k3-in-c, section 9 "Picking 16
// experts of 896": a logit per expert (a bf16 dot product accumulated far wider than
// float, then rounded to float), an unbiased sigmoid score, a selection score with the
// correction bias added, top-k by repeated strict maximum (an equal selection score goes
// to the lower expert index), weights from the unbiased scores, renormalised by their
// float sum when it is positive, times routed_scale.  "Three invariants", item 3: the
// bias steers the selection only.
//
// The shared expert's gate and up rows (section 9, LatentMoE listing step 6) are bf16
// rows over the same input, so they share this kernel: a warp owns one router row, or
// one (gate, up) row pair of the shared expert, and streams it once per token chunk.
#include "k3moe_kernels.cuh"

namespace k3 {

// Rows [0, E) are router rows, rows [E, E + SI) shared-expert row pairs.
// x: bf16 [T][H]; logits: float [T][E]; act_s: float [T][SI].
// Dynamic shared memory: tc_max * H bf16 (one chunk of tokens).
__global__ void __launch_bounds__(256) k_router_shared(
    const uint16_t *__restrict__ x, int T, int H, const uint16_t *__restrict__ wr, int E,
    const uint16_t *__restrict__ sh_gate, const uint16_t *__restrict__ sh_up, int SI,
    float b1, float b2, float *__restrict__ logits, float *__restrict__ act_s, int tc_max) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint16_t *xs = reinterpret_cast<uint16_t *>(smem_raw);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const int nrows = E + SI;
  const int nchunk = H >> 3;  // 8 bf16 per 16-byte chunk
  const uint4 *xs4 = reinterpret_cast<const uint4 *>(xs);

  for (int t0 = 0; t0 < T; t0 += tc_max) {
    const int tc = min(tc_max, T - t0);
    __syncthreads();
    {
      const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)t0 * H);
      uint4 *dst = reinterpret_cast<uint4 *>(xs);
      for (int i = threadIdx.x; i < tc * nchunk; i += blockDim.x) dst[i] = src[i];
    }
    __syncthreads();
    for (int row = blockIdx.x * nwarps + warp; row < nrows; row += gridDim.x * nwarps) {
      if (row < E) {
        const uint4 *w4 = reinterpret_cast<const uint4 *>(wr + (size_t)row * H);
        float hi[kTokChunk], lo[kTokChunk];
#pragma unroll
        for (int t = 0; t < kTokChunk; t++) hi[t] = lo[t] = 0.f;
#pragma unroll 4
        for (int c = lane; c < nchunk; c += 32) {
          const uint4 wv = __ldg(w4 + c);
          const uint32_t wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
          for (int t = 0; t < kTokChunk; t++) {
            if (t < tc) {
              const uint4 xv = xs4[t * nchunk + c];
              const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
              for (int q = 0; q < 4; q++) {
                // bf16 x bf16 is exact in float; carry the sum as a float-float pair.
                float p = __fmul_rn(bf16_lo(wa[q]), bf16_lo(xa[q]));
                float s, e;
                two_sum(hi[t], p, s, e);
                hi[t] = s;
                lo[t] = __fadd_rn(lo[t], e);
                p = __fmul_rn(bf16_hi(wa[q]), bf16_hi(xa[q]));
                two_sum(hi[t], p, s, e);
                hi[t] = s;
                lo[t] = __fadd_rn(lo[t], e);
              }
            }
          }
        }
#pragma unroll
        for (int t = 0; t < kTokChunk; t++) {
          if (t < tc) {
            // normalise, then reduce the pairs across the warp in a fixed tree
            float h = hi[t], l = lo[t];
            {
              const float s = __fadd_rn(h, l);
              l = __fsub_rn(l, __fsub_rn(s, h));
              h = s;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
              const float oh = __shfl_xor_sync(0xffffffffu, h, o);
              const float ol = __shfl_xor_sync(0xffffffffu, l, o);
              ff_add(h, l, oh, ol);
            }
            if (lane == 0) logits[(size_t)(t0 + t) * E + row] = h;
          }
        }
      } else {
        const int r = row - E;
        const uint4 *g4 = reinterpret_cast<const uint4 *>(sh_gate + (size_t)r * H);
        const uint4 *u4 = reinterpret_cast<const uint4 *>(sh_up + (size_t)r * H);
        float ga[kTokChunk], ua[kTokChunk];
#pragma unroll
        for (int t = 0; t < kTokChunk; t++) ga[t] = ua[t] = 0.f;
#pragma unroll 4
        for (int c = lane; c < nchunk; c += 32) {
          const uint4 gv = __ldg(g4 + c);
          const uint4 uv = __ldg(u4 + c);
          const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
          const uint32_t uw[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
          for (int t = 0; t < kTokChunk; t++) {
            if (t < tc) {
              const uint4 xv = xs4[t * nchunk + c];
              const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
              for (int q = 0; q < 4; q++) {
                const float x0 = bf16_lo(xa[q]), x1 = bf16_hi(xa[q]);
                ga[t] = fmaf(bf16_lo(gw[q]), x0, ga[t]);
                ga[t] = fmaf(bf16_hi(gw[q]), x1, ga[t]);
                ua[t] = fmaf(bf16_lo(uw[q]), x0, ua[t]);
                ua[t] = fmaf(bf16_hi(uw[q]), x1, ua[t]);
              }
            }
          }
        }
#pragma unroll
        for (int t = 0; t < kTokChunk; t++) {
          if (t < tc) {
            float g = ga[t], u = ua[t];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
              g += __shfl_xor_sync(0xffffffffu, g, o);
              u += __shfl_xor_sync(0xffffffffu, u, o);
            }
            if (lane == 0) act_s[(size_t)(t0 + t) * SI + r] = situ(g, u, b1, b2);
          }
        }
      }
    }
  }
}

// Larger selection score first; an equal score goes to the lower expert index.  A NaN
// never wins against a number (the NaN itself is reported through the status word).
__device__ __forceinline__ bool better(float ach, int ae, float bch, int be) {
  if (ae < 0) return false;
  if (be < 0) return true;
  if (ach > bch) return true;
  if (ach == bch) return ae < be;
  return (bch != bch) && (ach == ach);
}

__device__ __forceinline__ void warp_best(float &ch, int &e) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float och = __shfl_xor_sync(0xffffffffu, ch, o);
    const int oe = __shfl_xor_sync(0xffffffffu, e, o);
    if (better(och, oe, ch, e)) {
      ch = och;
      e = oe;
    }
  }
}

// One CTA (256 threads = 8 warps) per token.  Scores and selection scores go to shared
// memory; each warp takes the top K of its contiguous slice of experts by K rounds of a
// warp-wide maximum, then warp 0 merges the eight sorted lists (same key), which equals
// the page's repeated maximum over all experts.
__global__ void __launch_bounds__(256) k_topk(const float *__restrict__ logits,
                                              const float *__restrict__ bias, int T, int E,
                                              int K, int renorm, float routed_scale,
                                              int32_t *__restrict__ idx, float *__restrict__ w,
                                              int32_t *status) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  float *sc = reinterpret_cast<float *>(smem_raw);  // [E]
  float *ch = sc + E;                                // [E]
  int *lst = reinterpret_cast<int *>(ch + E);        // [8][K]
  const int t = blockIdx.x;
  if (t >= T) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const float lg = logits[(size_t)t * E + e];
    const float s = (float)(1.0 / (1.0 + exp(-(double)lg)));
    const float c = __fadd_rn(s, bias ? bias[e] : 0.f);
    sc[e] = s;
    ch[e] = c;
    if (!(fabsf(c) <= 3.402823466e38f) || !(fabsf(s) <= 3.402823466e38f))
      set_status(status, K3MOE_ERR_NONFINITE);
  }
  __syncthreads();

  // per-warp slice [lo, hi)
  const int per = (E + 7) / 8;
  const int lo = warp * per, hi = min(E, lo + per);
  unsigned taken = 0u;  // bit i: expert lo + lane + 32 i already chosen (slice <= 32*32)
  for (int k = 0; k < K; k++) {
    float bc = 0.f;
    int be = -1;
    int i = 0;
    for (int e = lo + lane; e < hi; e += 32, i++) {
      if (taken & (1u << i)) continue;
      const float c = ch[e];
      if (better(c, e, bc, be)) {
        bc = c;
        be = e;
      }
    }
    warp_best(bc, be);
    if (be >= 0 && ((be - lo) & 31) == lane) taken |= 1u << ((be - lo) >> 5);
    if (lane == 0) lst[warp * K + k] = be;
  }
  __syncthreads();

  if (warp == 0) {
    int head = 0;  // lanes 0..7 walk list `lane`
    float wsum = 0.f;
    float myw = 0.f;
    int mye = -1;
    for (int k = 0; k < K; k++) {
      int e = -1;
      float c = 0.f;
      if (lane < 8 && head < K) {
        e = lst[lane * K + head];
        if (e >= 0) c = ch[e];
      }
      const int cand_e = e;
      warp_best(c, e);
      if (lane < 8 && e >= 0 && cand_e == e) head++;
      // e is the k-th choice (every lane agrees)
      const float s = (e >= 0) ? sc[e] : 0.f;
      wsum = __fadd_rn(wsum, s);  // float sum in router order
      if (lane == k) {
        mye = e;
        myw = s;
      }
    }
    if (lane < K) {
      float v = myw;
      if (renorm && wsum > 0.f) v = __fdiv_rn(v, wsum);
      v = __fmul_rn(v, routed_scale);
      idx[(size_t)t * K + lane] = mye < 0 ? 0 : mye;
      w[(size_t)t * K + lane] = v;
    }
  }
}

}  // namespace k3

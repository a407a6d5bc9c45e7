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
// x: bf16 [T][H]; sc/ch: float [T][E] (unbiased score, selection score); act_s: float
// [T][SI].  Dynamic shared memory: TC * H bf16 (one chunk of tokens).  TC = tokens per
// chunk held in registers (1 for a decode step, 8 for batches); tc_max <= TC.
template <int TC>
__global__ void __launch_bounds__(256) k_router_shared(
    const uint16_t *__restrict__ x, int T, int H, const uint16_t *__restrict__ wr, int E,
    const float *__restrict__ bias, const uint16_t *__restrict__ sh_gate,
    const uint16_t *__restrict__ sh_up, int SI, float b1, float b2, float *__restrict__ sc,
    float *__restrict__ ch, float *__restrict__ act_s, int tc_max, int32_t *status) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  pdl_wait();
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
        float hi[TC], lo[TC];
#pragma unroll
        for (int t = 0; t < TC; t++) hi[t] = lo[t] = 0.f;
#pragma unroll 7
        for (int c = lane; c < nchunk; c += 32) {
          const uint4 wv = __ldg(w4 + c);
          const uint32_t wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
          for (int t = 0; t < TC; t++) {
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
        for (int t = 0; t < TC; t++) {
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
            if (lane == 0) {
              // unbiased score: logistic of the float logit, in double, rounded once;
              // selection score: one float add of the correction bias
              const float sv = (float)(1.0 / (1.0 + exp(-(double)h)));
              const float cv = __fadd_rn(sv, bias ? bias[row] : 0.f);
              sc[(size_t)(t0 + t) * E + row] = sv;
              ch[(size_t)(t0 + t) * E + row] = cv;
              if (!(fabsf(cv) <= 3.402823466e38f)) set_status(status, K3MOE_ERR_NONFINITE);
            }
          }
        }
      } else {
        const int r = row - E;
        const uint4 *g4 = reinterpret_cast<const uint4 *>(sh_gate + (size_t)r * H);
        const uint4 *u4 = reinterpret_cast<const uint4 *>(sh_up + (size_t)r * H);
        float ga[TC], ua[TC];
#pragma unroll
        for (int t = 0; t < TC; t++) ga[t] = ua[t] = 0.f;
#pragma unroll 7
        for (int c = lane; c < nchunk; c += 32) {
          const uint4 gv = __ldg(g4 + c);
          const uint4 uv = __ldg(u4 + c);
          const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
          const uint32_t uw[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
          for (int t = 0; t < TC; t++) {
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
        for (int t = 0; t < TC; t++) {
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
  pdl_launch_dependents();
}

// One decode token.  Work units, one per warp, eight per CTA:
//   [0, E)                router row e (float-float dot, then score and selection score)
//   [Ep, Ep + 2 SI)       shared-expert rows: Ep + 2r = gate row r, Ep + 2r + 1 = up row r
// with Ep = E rounded up to even, so the gate and up rows of r are two warps of one CTA;
// the gate warp's lane 0 applies SiTU once both dots are in shared memory.  Each lane
// keeps 14 16-byte loads in flight.
__global__ void __launch_bounds__(256) k_router_t1(const uint16_t *__restrict__ x, int H,
                                                   const uint16_t *__restrict__ wr, int E,
                                                   const float *__restrict__ bias,
                                                   const uint16_t *__restrict__ sh_gate,
                                                   const uint16_t *__restrict__ sh_up, int SI,
                                                   float b1, float b2, float *__restrict__ sc,
                                                   float *__restrict__ ch,
                                                   float *__restrict__ act_s, int32_t *status) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ float dots[8];
  constexpr int kB = 14;  // loads in flight per lane
  uint16_t *xs = reinterpret_cast<uint16_t *>(smem_raw);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nchunk = H >> 3;
  const int Ep = E + (E & 1);
  pdl_wait();
  {
    const uint4 *src = reinterpret_cast<const uint4 *>(x);
    uint4 *dst = reinterpret_cast<uint4 *>(xs);
    for (int i = threadIdx.x; i < nchunk; i += blockDim.x) dst[i] = src[i];
  }
  __syncthreads();
  const uint4 *xs4 = reinterpret_cast<const uint4 *>(xs);
  const int unit = blockIdx.x * 8 + warp;
  const bool is_router = unit < E;
  const bool is_shared = unit >= Ep && unit < Ep + 2 * SI;
  if (is_router || is_shared) {
    const int r = is_router ? unit : (unit - Ep) >> 1;
    const bool up = is_shared && ((unit - Ep) & 1);
    const uint16_t *row = is_router ? wr + (size_t)r * H
                                    : (up ? sh_up : sh_gate) + (size_t)r * H;
    const uint4 *w4 = reinterpret_cast<const uint4 *>(row);
    float hi = 0.f, lo = 0.f, acc = 0.f;
    for (int c0 = lane; c0 < nchunk; c0 += 32 * kB) {
      uint4 wv[kB];
#pragma unroll
      for (int b = 0; b < kB; b++) {
        const int c = c0 + 32 * b;
        wv[b] = (c < nchunk) ? __ldg(w4 + c) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int b = 0; b < kB; b++) {
        const int c = c0 + 32 * b;
        if (c < nchunk) {
          const uint4 xv = xs4[c];
          const uint32_t wa[4] = {wv[b].x, wv[b].y, wv[b].z, wv[b].w};
          const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int q = 0; q < 4; q++) {
            if (is_router) {
              // bf16 x bf16 is exact in float; carry the sum as a float-float pair
              float p = __fmul_rn(bf16_lo(wa[q]), bf16_lo(xa[q]));
              float s, e;
              two_sum(hi, p, s, e);
              hi = s;
              lo = __fadd_rn(lo, e);
              p = __fmul_rn(bf16_hi(wa[q]), bf16_hi(xa[q]));
              two_sum(hi, p, s, e);
              hi = s;
              lo = __fadd_rn(lo, e);
            } else {
              acc = fmaf(bf16_lo(wa[q]), bf16_lo(xa[q]), acc);
              acc = fmaf(bf16_hi(wa[q]), bf16_hi(xa[q]), acc);
            }
          }
        }
      }
    }
    if (is_router) {
      {
        const float s = __fadd_rn(hi, lo);
        lo = __fsub_rn(lo, __fsub_rn(s, hi));
        hi = s;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float oh = __shfl_xor_sync(0xffffffffu, hi, o);
        const float ol = __shfl_xor_sync(0xffffffffu, lo, o);
        ff_add(hi, lo, oh, ol);
      }
      if (lane == 0) {
        // unbiased score: logistic of the float logit, in double, rounded once;
        // selection score: one float add of the correction bias
        const float sv = (float)(1.0 / (1.0 + exp(-(double)hi)));
        const float cv = __fadd_rn(sv, bias ? bias[r] : 0.f);
        sc[r] = sv;
        ch[r] = cv;
        if (!(fabsf(cv) <= 3.402823466e38f)) set_status(status, K3MOE_ERR_NONFINITE);
      }
    } else {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) dots[warp] = acc;
    }
  }
  __syncthreads();
  if (is_shared && !(((unit - Ep) & 1)) && lane == 0) {
    const int r = (unit - Ep) >> 1;
    act_s[r] = situ(dots[warp], dots[warp + 1], b1, b2);
  }
  pdl_launch_dependents();
}

cudaError_t launch_router_t1(cudaStream_t st, const uint16_t *x, int H, const uint16_t *wr,
                             int E, const float *bias, const uint16_t *sh_gate,
                             const uint16_t *sh_up, int SI, float b1, float b2, float *sc,
                             float *ch, float *act_s, int32_t *status, bool pdl) {
  const int Ep = E + (E & 1);
  const int units = Ep + 2 * SI;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((units + 7) / 8);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = (size_t)H * 2;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_router_t1, x, H, wr, E, bias, sh_gate, sh_up, SI, b1, b2, sc,
                            ch, act_s, status);
}

cudaError_t launch_router_shared(int tc, int grid, size_t smem, cudaStream_t st, const uint16_t *x,
                                 int T, int H, const uint16_t *wr, int E, const float *bias,
                                 const uint16_t *sh_gate, const uint16_t *sh_up, int SI, float b1,
                                 float b2, float *sc, float *ch, float *act_s, int32_t *status) {
  if (tc == 1)
    k_router_shared<1><<<grid, 256, smem, st>>>(x, T, H, wr, E, bias, sh_gate, sh_up, SI, b1, b2,
                                                sc, ch, act_s, 1, status);
  else
    k_router_shared<kTokChunk><<<grid, 256, smem, st>>>(x, T, H, wr, E, bias, sh_gate, sh_up, SI,
                                                        b1, b2, sc, ch, act_s, tc, status);
  return cudaGetLastError();
}

cudaError_t set_router_smem_limits(int bytes) {
  cudaError_t e = cudaFuncSetAttribute(k_router_shared<1>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_router_t1, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k_router_shared<kTokChunk>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

// One CTA (256 threads) per token: the top-k of its selection scores (cta_topk).
__global__ void __launch_bounds__(512) k_topk(const float *__restrict__ scores,
                                              const float *__restrict__ choice, int T, int E,
                                              int K, int renorm, float routed_scale,
                                              int32_t *__restrict__ idx, float *__restrict__ w,
                                              int32_t *status) {
  __shared__ int sel[32];
  __shared__ float wsel[32];
  extern __shared__ __align__(16) unsigned long long s_keys[];  // top-k scratch
  pdl_wait();
  const int t = blockIdx.x;
  if (t >= T) return;
  cta_topk(scores + (size_t)t * E, choice + (size_t)t * E, E, K, renorm, routed_scale, s_keys,
           sel, wsel);
  if (threadIdx.x < K) {
    idx[(size_t)t * K + threadIdx.x] = sel[threadIdx.x];
    w[(size_t)t * K + threadIdx.x] = wsel[threadIdx.x];
  }
  (void)status;
}

}  // namespace k3

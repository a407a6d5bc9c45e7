// k3moe_latent.cu -- the pieces of the LatentMoE layer that the direct layer does not
// have (README of FareedKhan-dev/kimi-k3-in-c, section 9, LatentMoE listing steps 2, 4,
// 5 and 6; section 5 for RMSNorm and the bf16 weight products):
//   * k_proj: out = W in for a bf16 weight matrix and a few input rows (bf16 or float) --
//     the down-projection into the latent, the up-projection back to the full width, and
//     the shared experts' down projection, whose result is added to the up-projection and
//     written to the layer output; with a second matrix it computes the shared experts'
//     gate and up rows together and applies SiTU.
//   * k_rmsnorm_f32w: RMSNorm of the aggregated latent with its weight.
// These are GEMVs for decode-sized batches: one warp streams one weight row with 16-byte
// loads, four in flight per lane and matrix (more in flight leaves the loads waiting on
// the arithmetic: a standalone sweep of this row-per-warp pattern read 51 MB in 17.7 us at
// four, 18.7 at eight and 22.8 at sixteen).  Launched as
// programmatic dependents, each kernel asks for its first weight rows in L2 while the
// kernel before it drains, and reads no activation before that kernel has completed.
#include "k3moe_kernels.cuh"

namespace k3 {

namespace {

// A weight chunk read once: no L1 allocation, first out of L2 (policy from l2_evict_first).
__device__ __forceinline__ uint4 ld_stream16(const uint4 *p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}

// The 8 inputs of 16-byte weight chunk c of token row t, as floats.
template <bool IN_F32>
__device__ __forceinline__ void load_in8(const void *in, int C, int t, int c, float (&v)[8]) {
  if (IN_F32) {
    const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(in) +
                                                       (size_t)t * C) + 2 * c;
    const float4 a = __ldg(p), b = __ldg(p + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
    const uint4 q = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(in) +
                                                          (size_t)t * C) + c);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int k = 0; k < 4; k++) {
      v[2 * k] = bf16_lo(w[k]);
      v[2 * k + 1] = bf16_hi(w[k]);
    }
  }
}

__device__ __forceinline__ float dot8_bf16(uint4 w, const float (&v)[8], float acc) {
  const uint32_t a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int k = 0; k < 4; k++) {
    acc = fmaf(bf16_lo(a[k]), v[2 * k], acc);
    acc = fmaf(bf16_hi(a[k]), v[2 * k + 1], acc);
  }
  return acc;
}

// Error-free sum of two floats: s + e == a + b exactly (Knuth's TwoSum, no contraction).
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// 1 / sqrt(ss / n + eps) for the row x[0..n), ss its sum of squares (kimi-k3-in-c, section
// 5, where the sum is accumulated in double).  Here the sum is a float-float pair: every
// square is split exactly (product + its FMA residual), the thread's terms in index order,
// then a butterfly per warp and the warps in order, so the result is the same on every run
// and within a few float roundings of the double sum; the root is rounded once (__frsqrt_rn).
// All threads of the block call it; the value is returned in thread 0.  red: 16 floats of
// shared memory.
__device__ float block_inv_rms(const float *x, int n, float eps, float *red) {
  float hi = 0.f, lo = 0.f;
  const int bd = blockDim.x;
  for (int i0 = threadIdx.x; i0 < n; i0 += 8 * bd) {
    float v[8];  // eight loads in flight; the missing tail adds exact zeros
#pragma unroll
    for (int k = 0; k < 8; k++) v[k] = i0 + k * bd < n ? x[i0 + k * bd] : 0.f;
#pragma unroll
    for (int k = 0; k < 8; k++) {
      const float p = __fmul_rn(v[k], v[k]);
      const float pe = fmaf(v[k], v[k], -p);
      float s, e;
      two_sum(hi, p, s, e);
      hi = s;
      lo = __fadd_rn(lo, __fadd_rn(e, pe));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {  // both partners add the same two pairs
    const float oh = __shfl_xor_sync(0xffffffffu, hi, o);
    const float ol = __shfl_xor_sync(0xffffffffu, lo, o);
    float s, e;
    two_sum(hi, oh, s, e);
    hi = s;
    lo = __fadd_rn(e, __fadd_rn(lo, ol));
  }
  if ((threadIdx.x & 31) == 0) {
    red[2 * (threadIdx.x >> 5)] = hi;
    red[2 * (threadIdx.x >> 5) + 1] = lo;
  }
  __syncthreads();
  float inv = 0.f;
  if (threadIdx.x == 0) {
    float th = 0.f, tl = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); w++) {
      float s, e;
      two_sum(th, red[2 * w], s, e);
      th = s;
      tl = __fadd_rn(tl, __fadd_rn(e, red[2 * w + 1]));
    }
    const float ms = __fdiv_rn(__fadd_rn(th, tl), (float)n);
    inv = __frsqrt_rn(__fadd_rn(ms, eps));
  }
  __syncthreads();  // red may be reused
  return inv;
}

}  // namespace

constexpr int kProjT = kProjRows;  // token rows per pass over a weight row
constexpr int kProjU = 4;  // 16-byte weight chunks in flight per lane and matrix

// Rows r of W [R][C] (bf16, row-major) against T input rows in [T][C]:
//   s[t][r] = sum_c W[r][c] in[t][c]           (fp32 products and sums; the lanes' parts
//                                                reduced in a fixed butterfly, so results
//                                                are the same on every run)
// GU: W2 [R][C] is a second matrix and the output is SiTU(s, s2) (shared gate and up).
// NORM (float input, T <= kProjT): the input rows are RMS-normalised first, in[t][c] ->
// (in[t][c] * inv_t) * nw[c] (nw == nullptr: weight 1), inv_t computed by every block
// from the whole row -- the same values k_rmsnorm_f32w writes.
// Output: when y == nullptr, out[t][r] = value (float); else the final layer output
// y[t][r] (=|+=) addend[t][r] + value, float or bf16 (round to nearest even).
template <bool IN_F32, bool GU, bool NORM>
__global__ void __launch_bounds__(256) k_proj(const uint16_t *__restrict__ W,
                                              const uint16_t *__restrict__ W2, int R, int C,
                                              const void *__restrict__ in, int T,
                                              float *__restrict__ out,
                                              const float *__restrict__ addend, void *y, int ydt,
                                              int accumulate, float b1, float b2,
                                              const float *__restrict__ nw, float eps) {
  __shared__ float s_red[16];
  __shared__ float s_inv[kProjT];
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const int nch = C >> 3;
  const int r_first = blockIdx.x * wpb + (threadIdx.x >> 5);
  const int r_step = gridDim.x * wpb;
  // each warp keeps its next row on its way to L2 while it reads the current one (weights
  // only: nothing the previous kernel writes)
  if (lane == 0 && r_first < R) {
    bulk_prefetch_l2_pol(W + (size_t)r_first * C, (uint32_t)C * 2, l2_evict_first());
    if (GU) bulk_prefetch_l2_pol(W2 + (size_t)r_first * C, (uint32_t)C * 2, l2_evict_first());
  }
  pdl_wait();
  pdl_launch_dependents();
  if (NORM) {
    for (int t = 0; t < T; t++) {
      const float v = block_inv_rms(static_cast<const float *>(in) + (size_t)t * C, C, eps,
                                    s_red);
      if (threadIdx.x == 0) s_inv[t] = v;
    }
    __syncthreads();
  }
  const uint64_t pol = l2_evict_first();  // the weights are read once
  for (int r = r_first; r < R; r += r_step) {
    if (lane == 0 && r + r_step < R) {
      bulk_prefetch_l2_pol(W + (size_t)(r + r_step) * C, (uint32_t)C * 2, pol);
      if (GU) bulk_prefetch_l2_pol(W2 + (size_t)(r + r_step) * C, (uint32_t)C * 2, pol);
    }
    const uint4 *w4 = reinterpret_cast<const uint4 *>(W + (size_t)r * C);
    const uint4 *u4 = GU ? reinterpret_cast<const uint4 *>(W2 + (size_t)r * C) : nullptr;
    for (int t0 = 0; t0 < T; t0 += kProjT) {
      const int nt = T - t0 < kProjT ? T - t0 : kProjT;
      float acc[kProjT], acc2[kProjT];
#pragma unroll
      for (int m = 0; m < kProjT; m++) acc[m] = acc2[m] = 0.f;
      for (int c0 = lane; c0 < nch; c0 += 32 * kProjU) {
        uint4 wv[kProjU], uv[kProjU];
#pragma unroll
        for (int k = 0; k < kProjU; k++) {
          const int c = c0 + 32 * k;
          wv[k] = c < nch ? ld_stream16(w4 + c, pol) : make_uint4(0u, 0u, 0u, 0u);
          if (GU) uv[k] = c < nch ? ld_stream16(u4 + c, pol) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int k = 0; k < kProjU; k++) {
          const int c = c0 + 32 * k;
          if (c >= nch) break;
#pragma unroll
          for (int m = 0; m < kProjT; m++) {
            if (m < nt) {
              float v[8];
              load_in8<IN_F32>(in, C, t0 + m, c, v);
              if (NORM) {
                const float inv = s_inv[t0 + m];
                float wn[8] = {1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f};
                if (nw) load_in8<true>(nw, C, 0, c, wn);
#pragma unroll
                for (int j = 0; j < 8; j++) {
                  const float q = __fmul_rn(v[j], inv);
                  v[j] = nw ? __fmul_rn(q, wn[j]) : q;
                }
              }
              acc[m] = dot8_bf16(wv[k], v, acc[m]);
              if (GU) acc2[m] = dot8_bf16(uv[k], v, acc2[m]);
            }
          }
        }
      }
#pragma unroll
      for (int m = 0; m < kProjT; m++) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], o);
          if (GU) acc2[m] += __shfl_xor_sync(0xffffffffu, acc2[m], o);
        }
      }
      if (lane < nt) {  // every lane holds every sum: lane m writes token t0 + m
        float v = 0.f, v2 = 0.f;
#pragma unroll
        for (int m = 0; m < kProjT; m++)
          if (lane == m) {
            v = acc[m];
            v2 = acc2[m];
          }
        const int t = t0 + lane;
        const float val = GU ? situ(v, v2, b1, b2) : v;
        const size_t o = (size_t)t * R + r;
        if (y == nullptr) {
          out[o] = val;
        } else {
          const float s = addend ? __fadd_rn(addend[o], val) : val;
          if (ydt == K3MOE_F32) {
            float *yf = static_cast<float *>(y);
            yf[o] = accumulate ? __fadd_rn(yf[o], s) : s;
          } else {
            uint16_t *yb = static_cast<uint16_t *>(y);
            yb[o] = f32_to_bf16(accumulate ? __fadd_rn(bf16_lo(yb[o]), s) : s);
          }
        }
      }
    }
  }
}

// out[t] = (in[t] * inv) * w (float, left to right; w == nullptr: weight 1) with
// inv = 1 / sqrt(ss / n + eps) from block_inv_rms (kimi-k3-in-c, section 5).  One block per
// row; in and out may be the same array.
__global__ void __launch_bounds__(256) k_rmsnorm_f32w(const float *in, int n,
                                                      const float *__restrict__ w, float eps,
                                                      float *out) {
  __shared__ float red[16];
  __shared__ float inv_s;
  pdl_wait();
  pdl_launch_dependents();
  const float *x = in + (size_t)blockIdx.x * n;
  float *o = out + (size_t)blockIdx.x * n;
  const float v = block_inv_rms(x, n, eps, red);
  if (threadIdx.x == 0) inv_s = v;
  __syncthreads();
  const float inv = inv_s;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const float t = __fmul_rn(x[i], inv);
    o[i] = w ? __fmul_rn(t, w[i]) : t;
  }
}

// y[i] (=|+=) up[i] + ds[i] (ds == nullptr: up[i]), float or bf16 (round to nearest even):
// the layer output of a pass whose projections ran on the tensor cores.
__global__ void __launch_bounds__(256) k_add_out(const float *__restrict__ up,
                                                 const float *__restrict__ ds, void *y, int ydt,
                                                 int accumulate, long long n) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const float s = ds ? __fadd_rn(up[i], ds[i]) : up[i];
    if (ydt == K3MOE_F32) {
      float *yf = static_cast<float *>(y);
      yf[i] = accumulate ? __fadd_rn(yf[i], s) : s;
    } else {
      uint16_t *yb = static_cast<uint16_t *>(y);
      yb[i] = f32_to_bf16(accumulate ? __fadd_rn(bf16_lo(yb[i]), s) : s);
    }
  }
}

namespace {

cudaLaunchConfig_t proj_config(cudaStream_t st, int grid, int block, bool pdl,
                               cudaLaunchAttribute *attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

}  // namespace

cudaError_t launch_proj(cudaStream_t st, int sms, const uint16_t *W, const uint16_t *W2, int R,
                        int C, const void *in, bool in_f32, int T, float *out,
                        const float *addend, void *y, int ydt, int accumulate, float b1,
                        float b2, bool pdl, bool norm, const float *nw, float eps) {
  if (norm && (!in_f32 || W2 || T > kProjT)) return cudaErrorInvalidValue;
  using Fn = void (*)(const uint16_t *, const uint16_t *, int, int, const void *, int, float *,
                      const float *, void *, int, int, float, float, const float *, float);
  const Fn fn = norm ? k_proj<true, false, true>
                     : W2 ? (in_f32 ? k_proj<true, true, false> : k_proj<false, true, false>)
                          : (in_f32 ? k_proj<true, false, false> : k_proj<false, false, false>);
  // one wave of resident blocks, each warp taking every (grid x 8)-th row
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, 256, 0) != cudaSuccess || occ < 1)
    occ = 1;
  int grid = (R + 7) / 8;
  if (grid > occ * sms) grid = occ * sms;
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = proj_config(st, grid, 256, pdl, attr);
  return cudaLaunchKernelEx(&cfg, fn, W, W2, R, C, in, T, out, addend, y, ydt, accumulate, b1,
                            b2, nw, eps);
}

cudaError_t launch_rmsnorm_f32w(cudaStream_t st, const float *in, int T, int n, const float *w,
                                float eps, float *out, bool pdl) {
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = proj_config(st, T, 256, pdl, attr);
  return cudaLaunchKernelEx(&cfg, k_rmsnorm_f32w, in, n, w, eps, out);
}

cudaError_t launch_add_out(cudaStream_t st, int sms, const float *up, const float *ds, void *y,
                           int ydt, int accumulate, long long n) {
  long long g = (n + 255) / 256;
  if (g > 8LL * sms) g = 8LL * sms;
  k_add_out<<<(int)g, 256, 0, st>>>(up, ds, y, ydt, accumulate, n);
  return cudaGetLastError();
}

}  // namespace k3

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
// loads, several loads in flight per lane, so the kernels are bound by HBM.
#include "k3moe_kernels.cuh"

namespace k3 {

namespace {

__device__ __forceinline__ uint4 ld_stream16(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
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

}  // namespace

constexpr int kProjT = 4;   // token rows per pass over a weight row
constexpr int kProjU = 4;   // 16-byte weight chunks in flight per lane

// Rows r of W [R][C] (bf16, row-major) against T input rows in [T][C]:
//   s[t][r] = sum_c W[r][c] in[t][c]           (fp32 products and sums; the lanes' parts
//                                                reduced in a fixed butterfly, so results
//                                                are the same on every run)
// GU: W2 [R][C] is a second matrix and the output is SiTU(s, s2) (shared gate and up).
// Output: when y == nullptr, out[t][r] = value (float); else the final layer output
// y[t][r] (=|+=) addend[t][r] + value, float or bf16 (round to nearest even).
template <bool IN_F32, bool GU>
__global__ void __launch_bounds__(256) k_proj(const uint16_t *__restrict__ W,
                                              const uint16_t *__restrict__ W2, int R, int C,
                                              const void *__restrict__ in, int T,
                                              float *__restrict__ out,
                                              const float *__restrict__ addend, void *y, int ydt,
                                              int accumulate, float b1, float b2) {
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const int nch = C >> 3;
  for (int r = blockIdx.x * wpb + (threadIdx.x >> 5); r < R; r += gridDim.x * wpb) {
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
          wv[k] = c < nch ? ld_stream16(w4 + c) : make_uint4(0u, 0u, 0u, 0u);
          if (GU) uv[k] = c < nch ? ld_stream16(u4 + c) : make_uint4(0u, 0u, 0u, 0u);
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
// inv = (float)(1 / sqrt(ss / n + eps)), ss the row's sum of squares in double (kimi-k3-in-c,
// section 5).  One block per row; the double partial sums are added in a fixed order.
// in and out may be the same array.
__global__ void __launch_bounds__(256) k_rmsnorm_f32w(const float *in, int n,
                                                      const float *__restrict__ w, float eps,
                                                      float *out) {
  __shared__ double red[8];
  __shared__ float inv_s;
  const float *x = in + (size_t)blockIdx.x * n;
  float *o = out + (size_t)blockIdx.x * n;
  double ss = 0.0;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const double v = (double)x[i];
    ss = fma(v, v, ss);
  }
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, s);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    double tot = 0.0;
    for (int k = 0; k < (int)(blockDim.x >> 5); k++) tot += red[k];
    inv_s = (float)(1.0 / sqrt(tot / (double)n + (double)eps));
  }
  __syncthreads();
  const float inv = inv_s;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const float t = __fmul_rn(x[i], inv);
    o[i] = w ? __fmul_rn(t, w[i]) : t;
  }
}

cudaError_t launch_proj(cudaStream_t st, int sms, const uint16_t *W, const uint16_t *W2, int R,
                        int C, const void *in, bool in_f32, int T, float *out,
                        const float *addend, void *y, int ydt, int accumulate, float b1,
                        float b2) {
  int grid = (R + 7) / 8;
  if (grid > 16 * sms) grid = 16 * sms;
  if (W2) {
    if (in_f32)
      k_proj<true, true><<<grid, 256, 0, st>>>(W, W2, R, C, in, T, out, addend, y, ydt,
                                               accumulate, b1, b2);
    else
      k_proj<false, true><<<grid, 256, 0, st>>>(W, W2, R, C, in, T, out, addend, y, ydt,
                                                accumulate, b1, b2);
  } else {
    if (in_f32)
      k_proj<true, false><<<grid, 256, 0, st>>>(W, W2, R, C, in, T, out, addend, y, ydt,
                                                accumulate, b1, b2);
    else
      k_proj<false, false><<<grid, 256, 0, st>>>(W, W2, R, C, in, T, out, addend, y, ydt,
                                                 accumulate, b1, b2);
  }
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm_f32w(cudaStream_t st, const float *in, int T, int n, const float *w,
                                float eps, float *out) {
  k_rmsnorm_f32w<<<T, 256, 0, st>>>(in, n, w, eps, out);
  return cudaGetLastError();
}

}  // namespace k3

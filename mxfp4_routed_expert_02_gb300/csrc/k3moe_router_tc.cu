// k3moe_router_tc.cu -- the router of the multi-token path: tensor-core screening, then the
// exact computation for the experts that can matter.
//
// The selection is the page's (README of FareedKhan-dev/kimi-k3-in-c, section 9 "Picking
// 16 experts of 896"): logit = x . Wr[e] rounded to float, sc = logistic(logit), ch = sc +
// bias, the K largest ch with the lower index first on ties, weights from sc.
//
// 1. L~[t][e] = x . Wr[e] with bf16 operands and fp32 accumulation on the tensor cores.
//    Every bf16 product is exact in float, so the only error of L~ is the rounding of at
//    most H additions, each within 2^-23 of a partial sum bounded by
//    S = sum_k |x_k Wr[e][k]| <= |x|_2 |Wr[e]|_2 (Cauchy-Schwarz):
//    |L~ - logit| <= H * 2^-23 * |x|_2 |Wr[e]|_2.  The bound is taken with a factor 2 to
//    spare; the norms come from k_row_norms.  Under split K (small batches) L~ is the
//    range-order sum of KS partials over H / KS inputs each: a chain of at most H / KS
//    additions inside a partial and KS more between partials, every partial sum bounded
//    by S, so H can be replaced by H / KS + KS in the bound.
// 2. Per token, from those intervals, a lower and an upper bound of every expert's ch.
//    With tau the K-th largest lower bound, at least K experts have ch >= tau, so an
//    expert whose upper bound is below tau is not among the K largest.  The others (the
//    candidates, at least K) get their logit computed exactly as in the decode router (a
//    float-float sum of the exact products, rounded once), then sc and ch as the page
//    defines them; the rest get ch = -inf.
// 3. The usual top-k kernel then selects among the candidates: same result as selecting
//    among all experts with exact scores.
#include "k3moe_tc.cuh"

namespace k3 {

// Euclidean norms of the R0 bf16 rows of v0 and the R1 rows of v1 (width H, a multiple of
// 8), one 128-thread block per row, rounded up by a relative 2^-10 so that each bounds the
// exact norm.  The squares of bf16 values are exact in float (8-bit significands); a thread
// adds n = 8 * ceil(H / 1024) of them in order (all its loads issued first), then five
// shuffle levels and the four warps' sums in order follow, so the float sum S' has
// |S' - S| <= g S with g = m u / (1 - m u), m = n + 8 additions on any path, u = 2^-24.
// With the square root and the final product rounded up, the result is >= sqrt(S) whenever
// g < 2^-9, that is for H below 2^19 (hidden sizes are at most 8192 here).
__global__ void __launch_bounds__(128) k_row_norms(const uint16_t *__restrict__ v0, int R0,
                                                   float *__restrict__ out0,
                                                   const uint16_t *__restrict__ v1, int R1,
                                                   float *__restrict__ out1, int H) {
  __shared__ float wsum[4];
  const int b = blockIdx.x;
  if (b >= R0 + R1) return;
  const uint16_t *v = b < R0 ? v0 + (size_t)b * H : v1 + (size_t)(b - R0) * H;
  const uint4 *row = reinterpret_cast<const uint4 *>(v);
  const int nq = H / 8;
  float acc = 0.f;
  for (int q0 = threadIdx.x; q0 < nq; q0 += 128 * 8) {
    uint4 w[8];  // eight loads in flight; past the row's end zeros, whose squares add nothing
#pragma unroll
    for (int k = 0; k < 8; k++)
      w[k] = q0 + 128 * k < nq ? __ldg(row + q0 + 128 * k) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int k = 0; k < 8; k++) {
      const uint32_t a[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
#pragma unroll
      for (int e = 0; e < 4; e++) {
        const float lo = bf16_lo(a[e]), hi = bf16_hi(a[e]);
        acc = __fmaf_rn(lo, lo, acc);
        acc = __fmaf_rn(hi, hi, acc);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
  if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = wsum[0];
    for (int k = 1; k < 4; k++) t = __fadd_rn(t, wsum[k]);
    const float nv = __fmul_ru(__fsqrt_ru(t), 1.0009765625f);  // 1 + 2^-10
    if (b < R0)
      out0[b] = nv;
    else
      out1[b - R0] = nv;
  }
}

// Logistic in float for the bounds (a few ulp from the exact value; the slack covers it).
__device__ __forceinline__ float logistic_f(float v) { return 1.f / (1.f + expf(-v)); }

// gridDim.y blocks per token (blockIdx.x = token).  Lt [T][E] screening logits, xn [T] /
// wn [E] row norms of x / Wr; x [T][H], wr [E][H] bf16; nadd bounds the additions on any
// path of the screening sums (H, or H / KS + KS under split K).  Every block of a token computes
// all E bounds and the threshold (cheap, and identical in every block); block y then owns
// the experts e with e % gridDim.y == y: it computes the exact sc / ch of its candidates and
// writes sc 0, ch -inf for its other experts, so no two blocks write the same entry.
// Dynamic shared memory: H bf16 of x, the lower and upper bounds (2E floats), the
// block's candidate list (E ints) and the top-k scratch.
__global__ void __launch_bounds__(256) k_route_candidates(
    const float *__restrict__ Lt, const float *__restrict__ xn, const float *__restrict__ wn,
    const uint16_t *__restrict__ x,
    const uint16_t *__restrict__ wr, const float *__restrict__ bias, int H, int E, int K,
    int nadd, float *__restrict__ sc, float *__restrict__ ch, int32_t *__restrict__ ncand,
    int32_t *status) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint16_t *xs = reinterpret_cast<uint16_t *>(smem);
  float *blo = reinterpret_cast<float *>(smem + (size_t)H * 2);
  float *bhi = blo + E;
  int *clist = reinterpret_cast<int *>(bhi + E);
  unsigned long long *keys = reinterpret_cast<unsigned long long *>(
      smem + (((size_t)H * 2 + (size_t)E * 12 + 15) & ~size_t(15)));
  __shared__ int sel[32];
  __shared__ float wsel[32];
  __shared__ int count, total;
  __shared__ float tau;
  const int t = blockIdx.x, S = gridDim.y, y = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const float *Lrow = Lt + (size_t)t * E;
  const float xnorm = xn[t];
  float *scr = sc + (size_t)t * E;
  float *chr = ch + (size_t)t * E;
  const float nerr = (float)nadd * 2.384185791015625e-07f;  // nadd * 2^-22
  if (threadIdx.x == 0) {
    count = 0;
    total = 0;
  }
  {
    const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)t * H);
    uint4 *dst = reinterpret_cast<uint4 *>(xs);
    for (int i = threadIdx.x; i < H / 8; i += blockDim.x) dst[i] = __ldg(src + i);
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const float L = Lrow[e], Sn = xnorm * wn[e], b = bias ? bias[e] : 0.f;
    float lo, hi;
    if (isfinite(L) && isfinite(Sn) && isfinite(b)) {
      const float d = __fmaf_rn(nerr, Sn, 1e-30f);
      const float slack = 2e-6f + 9.5367431640625e-07f * (fabsf(L) + fabsf(b));  // 2^-20
      lo = logistic_f(__fsub_rn(L, d)) + b - slack;
      hi = logistic_f(__fadd_rn(L, d)) + b + slack;
    } else {  // decided exactly below (and reported there if not finite)
      lo = -INFINITY;
      hi = INFINITY;
    }
    blo[e] = lo;
    bhi[e] = hi;
  }
  __syncthreads();
  cta_topk(blo, blo, E, K, 0, 1.f, keys, sel, wsel);  // ends with __syncthreads
  if (threadIdx.x == 0) tau = blo[sel[K - 1]];
  __syncthreads();
  int mine = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    if (bhi[e] < tau) continue;
    mine++;
    if (e % S == y) clist[atomicAdd(&count, 1)] = e;
  }
  if (y == 0 && ncand) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
    if (lane == 0) atomicAdd(&total, mine);
  }
  // the block's non-candidates: out of the selection
  for (int e = y + S * threadIdx.x; e < E; e += S * blockDim.x) {
    if (!(bhi[e] < tau)) continue;
    scr[e] = 0.f;
    chr[e] = -INFINITY;
  }
  __syncthreads();
  const int C = count;
  if (y == 0 && threadIdx.x == 0 && ncand) ncand[t] = total;
  // candidates: exact logit (float-float sum of exact products, fixed reduction tree)
  const int nchunk = H >> 3;
  const uint4 *xs4 = reinterpret_cast<const uint4 *>(xs);
  for (int c = warp; c < C; c += nw) {
    const int e = clist[c];
    const uint4 *w4 = reinterpret_cast<const uint4 *>(wr + (size_t)e * H);
    float hi = 0.f, lo = 0.f;
    for (int q0 = lane; q0 < nchunk; q0 += 32 * 8) {
      uint4 wq[8];  // the row's loads eight at a time, then summed in the same order
#pragma unroll
      for (int b = 0; b < 8; b++)
        wq[b] = q0 + 32 * b < nchunk ? __ldg(w4 + q0 + 32 * b) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int b = 0; b < 8; b++) {
        const int q = q0 + 32 * b;
        if (q >= nchunk) break;
        const uint4 wv = wq[b], xv = xs4[q];
        const uint32_t wa[4] = {wv.x, wv.y, wv.z, wv.w}, xa[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int k = 0; k < 4; k++) {
          float p = __fmul_rn(bf16_lo(wa[k]), bf16_lo(xa[k]));
          float s, er;
          two_sum(hi, p, s, er);
          hi = s;
          lo = __fadd_rn(lo, er);
          p = __fmul_rn(bf16_hi(wa[k]), bf16_hi(xa[k]));
          two_sum(hi, p, s, er);
          hi = s;
          lo = __fadd_rn(lo, er);
        }
      }
    }
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
      const float sv = (float)(1.0 / (1.0 + exp(-(double)hi)));
      const float cv = __fadd_rn(sv, bias ? bias[e] : 0.f);
      scr[e] = sv;
      chr[e] = cv;
      if (!(fabsf(cv) <= 3.402823466e38f)) set_status(status, K3MOE_ERR_NONFINITE);
    }
  }
}

size_t route_candidates_smem(int H, int E, int K) {
  return (((size_t)H * 2 + (size_t)E * 12 + 15) & ~size_t(15)) + (size_t)topk_scratch_keys(E, K) * 8;
}

}  // namespace k3

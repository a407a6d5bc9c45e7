// k3moe_prefill.cu -- the kernels around the tensor-core grouped GEMM of the multi-token
// path: expert dispatch (a stable counting sort of the (token, slot) pairs by expert),
// activation encoding for the block-scaled MMA, and the router-order combine.
//
// The combine is the page's routed sum (README of FareedKhan-dev/kimi-k3-in-c, section 9,
// LatentMoE listing, steps 3 and 6): y_t = sum_j w[t,j] d_j in slot order j, in float,
// then the shared expert added unweighted; README of Maknee/Kimi-K3.cpp, "The
// consumer-memory idea" item 7, fixes the router order of that sum.
#include "k3moe_tcgen05.cuh"

namespace k3 {

// ------------------------------------------------------------------------------ dispatch
// A stable counting sort of the (token, slot) pairs by expert, in chunks of `chunk`
// pairs (route_chunk): per-chunk counts, per-expert totals and their prefix sums, then every chunk places
// its pairs after those of the earlier chunks, in pair order.

// counts[c][e]: pairs of chunk c routed to expert e.  Pairs whose expert index is outside
// [0, E) are counted nowhere, get inv = -1 (the combine skips them) and set
// K3MOE_ERR_BAD_EXPERT.
__global__ void k_route_count(const int32_t *__restrict__ idx, int P, int E, int chunk,
                              int32_t *__restrict__ counts, int32_t *inv, int32_t *status) {
  extern __shared__ int32_t cnt[];  // [E]
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int p0 = blockIdx.x * chunk, p1 = min(P, p0 + chunk);
  for (int p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
    const int e = idx[p];
    if (e >= 0 && e < E) {
      atomicAdd(&cnt[e], 1);
    } else {
      inv[p] = -1;
      set_status(status, K3MOE_ERR_BAD_EXPERT);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    counts[(size_t)blockIdx.x * E + e] = cnt[e];
}

// One block: per-expert totals over the nch chunks, their exclusive prefix off[E+1], the
// prefix of ntile-row tiles tile_off[E+1], and counts[c][e] replaced by the first position
// of expert e's pairs of chunk c: off[e] + the pairs of e in chunks 0 .. c-1.
__global__ void k_route_hist(int32_t *__restrict__ counts, int nch, int E, int ntile,
                             int32_t *off, int32_t *tile_off) {
  extern __shared__ int32_t cnt[];  // [E]
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int n = 0;
    for (int c = 0; c < nch; c++) n += counts[(size_t)c * E + e];
    cnt[e] = n;
  }
  __syncthreads();
  // exclusive scans of the counts and of the tile counts: thread i takes a run of
  // consecutive experts, the run totals are scanned across the block by warp shuffles
  __shared__ int wsum[2][32];
  const int nt = blockDim.x, per = (E + nt - 1) / nt;
  const int e0 = min(E, threadIdx.x * per), e1 = min(E, e0 + per);
  int c = 0, tl = 0;
  for (int e = e0; e < e1; e++) {
    c += cnt[e];
    tl += (cnt[e] + ntile - 1) / ntile;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = nt >> 5;
  int ic = c, it = tl;  // inclusive scans within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, ic, o), b = __shfl_up_sync(0xffffffffu, it, o);
    if (lane >= o) {
      ic += a;
      it += b;
    }
  }
  if (lane == 31) {
    wsum[0][warp] = ic;
    wsum[1][warp] = it;
  }
  __syncthreads();
  int o = ic - c, to = it - tl;
  for (int w = 0; w < warp; w++) {
    o += wsum[0][w];
    to += wsum[1][w];
  }
  for (int e = e0; e < e1; e++) {
    off[e] = o;
    tile_off[e] = to;
    o += cnt[e];
    to += (cnt[e] + ntile - 1) / ntile;
  }
  if (threadIdx.x == nt - 1) {
    int so = 0, st = 0;
    for (int w = 0; w < nw; w++) {
      so += wsum[0][w];
      st += wsum[1][w];
    }
    off[E] = so;
    tile_off[E] = st;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int pos = off[e];
    for (int c = 0; c < nch; c++) {
      const int n = counts[(size_t)c * E + e];
      counts[(size_t)c * E + e] = pos;
      pos += n;
    }
  }
}

// Block c places the pairs of chunk c: the next position of expert e starts at first[c][e]
// (k_route_hist); one warp walks the chunk (staged in shared memory) in pair order, 32 pairs
// at a time (lanes with the same expert ranked by lane), so perm[off[e] + r] = p and
// inv[p] = off[e] + r for the r-th pair routed to e overall.
__global__ void k_route_scatter(const int32_t *__restrict__ idx, int P, int E, int chunk,
                                const int32_t *__restrict__ first, int32_t *perm,
                                int32_t *inv) {
  extern __shared__ int32_t next[];  // [E], then the chunk's expert indices
  int32_t *ci = next + E;
  const int c = blockIdx.x;
  const int p0 = c * chunk, p1 = min(P, p0 + chunk);
  for (int e = threadIdx.x; e < E; e += blockDim.x) next[e] = first[(size_t)c * E + e];
  for (int p = p0 + threadIdx.x; p < p1; p += blockDim.x) ci[p - p0] = idx[p];
  __syncthreads();
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  for (int pb = p0; pb < p1; pb += 32) {
    const int p = pb + lane;
    const int e = p < p1 ? ci[p - p0] : -1;
    const bool ok = e >= 0 && e < E;
    const unsigned m = __match_any_sync(0xffffffffu, ok ? e : -1);
    const int rank = __popc(m & ((1u << lane) - 1u));
    const int base = ok ? next[e] : 0;
    __syncwarp();
    if (ok) {
      perm[base + rank] = p;
      inv[p] = base + rank;
      if (rank == 0) next[e] = base + __popc(m);  // the lowest lane of the group advances it
    }
    __syncwarp();
  }
}


// x [T][H] bf16 (or float: XF32, the LatentMoE's latent) -> the kTcTermsX-term encoding of
// every (token, slot) pair's row, written at the pair's sorted position: xq [term][P][H/2]
// and the scale bytes xs [term][K chunk][P][8] (chunk = 8 groups).  One thread per (token,
// group); the token's K slots receive the same bytes.
template <bool XF32>
__global__ void k_quant_x(const void *__restrict__ xv, int T, int H, int K,
                          const int32_t *__restrict__ inv, int P, uint8_t *__restrict__ xq,
                          uint8_t *__restrict__ xs) {
  const int G = H / kGroup;
  const long long n = (long long)T * G;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(i / G), g = (int)(i % G);
    float r[32];
    if (XF32) {
      const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(xv) +
                                                           (size_t)t * H + g * kGroup);
#pragma unroll
      for (int c = 0; c < 8; c++) {
        const float4 v = __ldg(src + c);
        r[4 * c] = v.x;
        r[4 * c + 1] = v.y;
        r[4 * c + 2] = v.z;
        r[4 * c + 3] = v.w;
      }
    } else {
      const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(xv) +
                                                         (size_t)t * H + g * kGroup);
#pragma unroll
      for (int c = 0; c < 4; c++) {
        const uint4 v = __ldg(src + c);
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; k++) {
          r[8 * c + 2 * k] = bf16_lo(w4[k]);
          r[8 * c + 2 * k + 1] = bf16_hi(w4[k]);
        }
      }
    }
    uint4 q[kTcTermsX];
    uint8_t sb[kTcTermsX];
    encode_terms<kTcTermsX>(r, q, sb);
    for (int j = 0; j < K; j++) {
      const int s = inv[(size_t)t * K + j];
      if (s < 0) continue;
#pragma unroll
      for (int tt = 0; tt < kTcTermsX; tt++) {
        reinterpret_cast<uint4 *>(xq + ((size_t)tt * P + s) * (H / 2))[g] = q[tt];
        xs[(((size_t)tt * ((G + 7) / 8) + g / 8) * P + s) * 8 + (g % 8)] = sb[tt];
      }
    }
  }
}

cudaError_t launch_quant_x(bool x_f32, int grid, cudaStream_t st, const void *x, int T, int H,
                           int K, const int32_t *inv, int P, uint8_t *xq, uint8_t *xs) {
  if (x_f32)
    k_quant_x<true><<<grid, 256, 0, st>>>(x, T, H, K, inv, P, xq, xs);
  else
    k_quant_x<false><<<grid, 256, 0, st>>>(x, T, H, K, inv, P, xq, xs);
  return cudaGetLastError();
}

// act [P][I] float -> kTcTermsAct-term encoding: aq [term][P][I/2], scale bytes as
// [term][K chunk][P][8].
__global__ void k_quant_act(const float *__restrict__ act, int P, int I,
                            uint8_t *__restrict__ aq, uint8_t *__restrict__ as) {
  const int G = I / kGroup;
  const long long n = (long long)P * G;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const int s = (int)(i / G), g = (int)(i % G);
    const float4 *src = reinterpret_cast<const float4 *>(act + (size_t)s * I + g * kGroup);
    float r[32];
#pragma unroll
    for (int c = 0; c < 8; c++) {
      const float4 v = __ldg(src + c);
      r[4 * c] = v.x;
      r[4 * c + 1] = v.y;
      r[4 * c + 2] = v.z;
      r[4 * c + 3] = v.w;
    }
    uint4 q[kTcTermsAct];
    uint8_t sb[kTcTermsAct];
    encode_terms<kTcTermsAct>(r, q, sb);
#pragma unroll
    for (int tt = 0; tt < kTcTermsAct; tt++) {
      reinterpret_cast<uint4 *>(aq + ((size_t)tt * P + s) * (I / 2))[g] = q[tt];
      as[(((size_t)tt * ((G + 7) / 8) + g / 8) * P + s) * 8 + (g % 8)] = sb[tt];
    }
  }
}

// float [n] -> two bf16 terms hi = bf16(v), lo = bf16(v - hi) (round to nearest even):
// out[0][n] = hi, out[1][n] = lo.  hi + lo carries 16 significant bits of v.
__global__ void k_split_bf16(const float *__restrict__ v, long long n, uint16_t *__restrict__ out) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const float f = v[i];
    const uint16_t hi = f32_to_bf16(f);
    const float r = __fsub_rn(f, __uint_as_float((uint32_t)hi << 16));
    out[i] = hi;
    out[n + i] = f32_to_bf16(r);
  }
}

// Group table of a single dense group of n rows: off = {0, n}, tile_off = {0, tiles}.
__global__ void k_group1(int n, int ntile, int32_t *off, int32_t *tile_off) {
  if (threadIdx.x == 0) {
    off[0] = 0;
    off[1] = n;
    tile_off[0] = 0;
    tile_off[1] = (n + ntile - 1) / ntile;
  }
}

// y[t] (=|+=) sum_j w[t,j] * dpair[inv[t*K+j]] (float, slot order j) + ds[t] (shared
// expert, unweighted, added last).  One block per token.
__global__ void k_combine(int T, int H, int K, const float *__restrict__ w,
                          const int32_t *__restrict__ inv, const float *__restrict__ dpair,
                          const float *__restrict__ ds, void *y, int ydt, int accumulate) {
  const int t = blockIdx.x;
  extern __shared__ int32_t s_slot[];  // [K] slots, then [K] weights (as float bits)
  float *s_w = reinterpret_cast<float *>(s_slot + K);
  for (int j = threadIdx.x; j < K; j += blockDim.x) {
    s_slot[j] = inv[(size_t)t * K + j];
    s_w[j] = w[(size_t)t * K + j];
  }
  __syncthreads();
  for (int h4 = blockIdx.y * blockDim.x + threadIdx.x; h4 < H / 4; h4 += gridDim.y * blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < K; j++) {
      const int s = s_slot[j];
      if (s < 0) continue;
      const float wj = s_w[j];
      const float4 d = __ldg(reinterpret_cast<const float4 *>(dpair + (size_t)s * H) + h4);
      acc.x = __fadd_rn(acc.x, __fmul_rn(wj, d.x));
      acc.y = __fadd_rn(acc.y, __fmul_rn(wj, d.y));
      acc.z = __fadd_rn(acc.z, __fmul_rn(wj, d.z));
      acc.w = __fadd_rn(acc.w, __fmul_rn(wj, d.w));
    }
    if (ds) {
      const float4 v = __ldg(reinterpret_cast<const float4 *>(ds + (size_t)t * H) + h4);
      acc.x = __fadd_rn(acc.x, v.x);
      acc.y = __fadd_rn(acc.y, v.y);
      acc.z = __fadd_rn(acc.z, v.z);
      acc.w = __fadd_rn(acc.w, v.w);
    }
    const float o[4] = {acc.x, acc.y, acc.z, acc.w};
    if (ydt == K3MOE_F32) {
      float *yp = static_cast<float *>(y) + (size_t)t * H + 4 * h4;
#pragma unroll
      for (int c = 0; c < 4; c++) yp[c] = accumulate ? __fadd_rn(yp[c], o[c]) : o[c];
    } else {
      uint16_t *yp = static_cast<uint16_t *>(y) + (size_t)t * H + 4 * h4;
#pragma unroll
      for (int c = 0; c < 4; c++) {
        const float prev = accumulate ? __uint_as_float((uint32_t)yp[c] << 16) : 0.f;
        yp[c] = f32_to_bf16(accumulate ? __fadd_rn(prev, o[c]) : o[c]);
      }
    }
  }
}

}  // namespace k3

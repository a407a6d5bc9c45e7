// k3moe_ffn.cu -- the routed expert FFN read straight from packed MXFP4, the
// router-order combine and the shared expert's down projection.
//
// Arithmetic (README of FareedKhan-dev/kimi-k3-in-c):
//   section 4 "Reduction one": y[r] = sum over groups of 32 of
//       (sum_k x[k] * E2M1[nibble]) * 2^(scale - 127), scale byte 255 contributing 0,
//       the low nibble of a byte being the even column; nothing is dequantised to memory.
//   section 9 (LatentMoE listing, step 3 and the activation listing): per selected
//       expert g = W1 x, u = W3 x, a = SiTU(g, u), d = W2 a; the routed sum
//       accL += w[j] * d accumulated in router order j; step 6: the shared expert's
//       output is added unweighted after the routed sum.
//   README of Maknee/Kimi-K3.cpp, "The consumer-memory idea" item 7: reduce in router
//       order, never in completion order (here: never in the order work items finish).
//
// GPU mapping.  Each 16-byte chunk of a packed row is exactly one scale group (32
// columns).  A thread owns one group column for the whole work item and keeps its 32
// activations in registers as f16 (scaled by a power of two so every bf16 input is an
// exact f16); the E2M1 pairs are converted to f16x2 in registers by the hardware
// conversion and multiplied with fp32 accumulation (each product exact).  The group sum
// is then scaled by 2^(s - 127 + ex) and the row sums are reduced across threads in a
// fixed order, so every result is bitwise reproducible.
#include "k3moe_kernels.cuh"

namespace k3 {

// ------------------------------------------------------------------------------------
// Dispatch: sort the T*K (token, slot) pairs by (expert, pair id) and list the distinct
// experts.  One CTA; bitonic sort in shared memory.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) k_dispatch(const int32_t *__restrict__ idx, int P, int E,
                                                   int32_t *__restrict__ disp, int32_t *status) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  int Pp = 1;
  while (Pp < P) Pp <<= 1;
  int *key = reinterpret_cast<int *>(smem_raw);  // [Pp]
  int *flag = key + Pp;                          // [Pp]
  __shared__ int wsum[32];
  const int nt = blockDim.x;
  for (int i = threadIdx.x; i < Pp; i += nt) {
    int k = 0x7fffffff;
    if (i < P) {
      const int e = idx[i];
      if (e >= 0 && e < E)
        k = (e << kPairKeyShift) | i;
      else
        set_status(status, K3MOE_ERR_BAD_EXPERT);
    }
    key[i] = k;
  }
  __syncthreads();
  for (int size = 2; size <= Pp; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < Pp; i += nt) {
        const int j = i ^ stride;
        if (j > i) {
          const bool up = (i & size) == 0;
          const int a = key[i], b = key[j];
          if ((a > b) == up) {
            key[i] = b;
            key[j] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  // flag = first pair of a distinct expert; exclusive scan gives its slot u
  for (int i = threadIdx.x; i < Pp; i += nt) {
    const int k = key[i];
    flag[i] = (k != 0x7fffffff) && (i == 0 || (key[i - 1] >> kPairKeyShift) != (k >> kPairKeyShift));
  }
  __syncthreads();
  // block-wide inclusive scan of flag (Pp <= 4096, each thread a contiguous run)
  const int per = (Pp + nt - 1) / nt;
  const int beg = threadIdx.x * per, end = min(Pp, beg + per);
  int run = 0;
  for (int i = beg; i < end; i++) run += flag[i];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int nw = (nt + 31) >> 5;
    int v = lane < nw ? wsum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    if (lane < nw) wsum[lane] = v;
  }
  __syncthreads();
  int base = inc - run + (warp > 0 ? wsum[warp - 1] : 0);  // exclusive prefix of this run
  int *uexp = disp + 4;
  int *uoff = uexp + P;
  int *plist = uoff + P + 1;
  for (int i = beg; i < end; i++) {
    const int k = key[i];
    if (k != 0x7fffffff) {
      plist[i] = k & ((1 << kPairKeyShift) - 1);
      if (flag[i]) {
        uexp[base] = k >> kPairKeyShift;
        uoff[base] = i;
      }
    }
    base += flag[i];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int nwarp = (nt + 31) >> 5;
    const int U = wsum[nwarp - 1];
    int nvalid = 0;
    for (int i = Pp; i > 0; i--)
      if (key[i - 1] != 0x7fffffff) {
        nvalid = i;
        break;
      }
    disp[0] = U;
    uoff[U] = nvalid;
  }
}

// ------------------------------------------------------------------------------------
// Expert gate/up + SiTU.  Work item = (distinct expert u, 32-row tile of the I rows).
// Path A (G = H/32 >= 32 or not a power of two): one thread per group column, the CTA
// covers one row at a time, 4-row blocks software-pipelined; the 8 partial sums of a
// block (4 rows x gate/up) per token are reduced across the CTA.
// Path B (G in {1,2,4,8,16}): G consecutive lanes form a row lane; the CTA covers 32
// rows at once.
// Output per (token, slot) pair i: act = SiTU(g, u) for the tile's 32 rows, stored as
// f16 hi + f16 lo of act * 2^-ex with one exponent ex per 32 rows (= one group of the
// down projection's input).
// ------------------------------------------------------------------------------------
// XF32: x is float [T][H] (the LatentMoE's latent input) instead of bf16; each group is
// prescaled the same way into two f16 terms (hi + residual, about 22 significant bits)
// and the products take both terms (group_dot2).
template <int MB, bool XF32>
__global__ void __launch_bounds__(256) k_expert_gateup(
    const void *__restrict__ xv, int H, int I, int K, ExpertArgs ex,
    const int32_t *__restrict__ disp, int P, float b1, float b2,
    uint16_t *__restrict__ act_hi, uint16_t *__restrict__ act_lo, int32_t *__restrict__ act_ex) {
  __shared__ float gu[MB][kTileRows][2];
  __shared__ float red[8][8 * MB];
  const int G = H / kGroup;
  const int tiles = I / kTileRows;
  const int U = disp[0];
  const int *uexp = disp + 4;
  const int *uoff = uexp + P;
  const int *plist = uoff + P + 1;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const bool pathB = (G <= 16) && ((G & (G - 1)) == 0);
  const int rowbytes = H / 2;

  for (int item = blockIdx.x; item < U * tiles; item += gridDim.x) {
    const int u = item / tiles, tile = item % tiles;
    const int e = uexp[u];
    const int pbeg = uoff[u], pend = uoff[u + 1];
    const uint8_t *rec = ex.base + (long long)e * ex.stride;
    const uint8_t *w1p = rec + ex.off[0], *w1s = rec + ex.off[1];
    const uint8_t *w3p = rec + ex.off[4], *w3s = rec + ex.off[5];
    const int r0 = tile * kTileRows;

    for (int pc = pbeg; pc < pend; pc += MB) {
      const int mcount = min(MB, pend - pc);
      // ---- this thread's group column of x for each token of the chunk, as f16
      const int g = pathB ? (tid % G) : tid;
      const bool gact = g < G;
      uint32_t xr[MB][16], xl[MB][16];
      int xe[MB];
#pragma unroll
      for (int m = 0; m < MB; m++) {
        xe[m] = 0;
#pragma unroll
        for (int p = 0; p < 16; p++) xr[m][p] = xl[m][p] = 0u;
        if (m < mcount && gact) {
          const int t = plist[pc + m] / K;
          float v[32];
          if (XF32) {
            const float4 *src = reinterpret_cast<const float4 *>(
                static_cast<const float *>(xv) + (size_t)t * H + g * kGroup);
#pragma unroll
            for (int q = 0; q < 8; q++) {
              const float4 c = __ldg(src + q);
              v[4 * q] = c.x;
              v[4 * q + 1] = c.y;
              v[4 * q + 2] = c.z;
              v[4 * q + 3] = c.w;
            }
          } else {
            const uint4 *src = reinterpret_cast<const uint4 *>(
                static_cast<const uint16_t *>(xv) + (size_t)t * H + g * kGroup);
#pragma unroll
            for (int q = 0; q < 4; q++) {
              const uint4 c = __ldg(src + q);
              const uint32_t a[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
              for (int k = 0; k < 4; k++) {
                v[8 * q + 2 * k] = bf16_lo(a[k]);
                v[8 * q + 2 * k + 1] = bf16_hi(a[k]);
              }
            }
          }
          xe[m] = XF32 ? prescale_group_f16_hilo(v, xr[m], xl[m]) : prescale_group_f16(v, xr[m]);
        }
      }

      if (!pathB) {
        // ---- path A: rows in blocks of 4, next block's weights loaded before compute
        uint4 wc[8], wn[8];
        uint32_t sc[8], sn[8];
        auto load_block = [&](int rb, uint4 (&w)[8], uint32_t (&s)[8]) {
#pragma unroll
          for (int q = 0; q < 4; q++) {
            const int r = r0 + 4 * rb + q;
            if (gact) {
              w[q] = __ldg(reinterpret_cast<const uint4 *>(w1p + (size_t)r * rowbytes) + g);
              w[4 + q] = __ldg(reinterpret_cast<const uint4 *>(w3p + (size_t)r * rowbytes) + g);
              s[q] = __ldg(w1s + (size_t)r * G + g);
              s[4 + q] = __ldg(w3s + (size_t)r * G + g);
            } else {
              w[q] = w[4 + q] = make_uint4(0u, 0u, 0u, 0u);
              s[q] = s[4 + q] = 255u;
            }
          }
        };
        load_block(0, wc, sc);
        for (int rb = 0; rb < kTileRows / 4; rb++) {
          if (rb + 1 < kTileRows / 4) load_block(rb + 1, wn, sn);
          float vals[8 * MB];
#pragma unroll
          for (int m = 0; m < MB; m++) {
#pragma unroll
            for (int c = 0; c < 8; c++) {
              const float part = XF32 ? group_dot2(xr[m], xl[m], wc[c]) : group_dot(xr[m], wc[c]);
              vals[m * 8 + c] = (sc[c] == 255u) ? 0.f : part * group_factor(sc[c], xe[m]);
            }
          }
          const float tot = warp_transpose_reduce<8 * MB>(vals);
          if (lane < 8 * MB) red[warp][lane] = tot;
          __syncthreads();
          if (tid < 8 * MB) {
            float s = 0.f;
            for (int w = 0; w < nwarps; w++) s += red[w][tid];
            const int m = tid / 8, c = tid % 8;
            gu[m][4 * rb + (c & 3)][c >> 2] = s;
          }
          __syncthreads();
          if (rb + 1 < kTileRows / 4) {
#pragma unroll
            for (int c = 0; c < 8; c++) {
              wc[c] = wn[c];
              sc[c] = sn[c];
            }
          }
        }
      } else {
        // ---- path B: row lanes of G threads, 32 rows per pass
        const int RL = min(32, (int)blockDim.x / G);
        const int p = tid / G;
        const int rows_per = kTileRows / RL;
        if (p < RL) {
          for (int q = 0; q < rows_per; q++) {
            const int rl = p * rows_per + q;
            const int r = r0 + rl;
            const uint4 wg = __ldg(reinterpret_cast<const uint4 *>(w1p + (size_t)r * rowbytes) + g);
            const uint4 wu = __ldg(reinterpret_cast<const uint4 *>(w3p + (size_t)r * rowbytes) + g);
            const uint32_t sg = __ldg(w1s + (size_t)r * G + g);
            const uint32_t su = __ldg(w3s + (size_t)r * G + g);
#pragma unroll
            for (int m = 0; m < MB; m++) {
              const float dg = XF32 ? group_dot2(xr[m], xl[m], wg) : group_dot(xr[m], wg);
              const float du = XF32 ? group_dot2(xr[m], xl[m], wu) : group_dot(xr[m], wu);
              float a = (sg == 255u) ? 0.f : dg * group_factor(sg, xe[m]);
              float b = (su == 255u) ? 0.f : du * group_factor(su, xe[m]);
              for (int o = G >> 1; o > 0; o >>= 1) {
                a += __shfl_xor_sync(0xffffffffu, a, o);
                b += __shfl_xor_sync(0xffffffffu, b, o);
              }
              if (g == 0) {
                gu[m][rl][0] = a;
                gu[m][rl][1] = b;
              }
            }
          }
        }
        __syncthreads();
      }

      // ---- SiTU, per-token exponent over the 32 rows, hi/lo f16 out; warp m = token m
      if (warp < mcount) {
        const int m = warp;
        const int i = plist[pc + m];
        const float a = situ(gu[m][lane][0], gu[m][lane][1], b1, b2);
        float mx = fabsf(a);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        int e2 = 0;
        if (mx > 0.f) {
          e2 = exponent_of(mx) - 14;
          e2 = e2 < -110 ? -110 : e2;
        }
        const float sa = a * pow2i(-e2);
        const __half hh = __float2half_rn(sa);
        const __half hl = __float2half_rn(sa - __half2float(hh));
        const size_t o = act_index(i, I, tile, lane);
        act_hi[o] = __half_as_ushort(hh);
        act_lo[o] = __half_as_ushort(hl);
        if (lane == 0) act_ex[(size_t)i * (I / kGroup) + tile] = e2;
      }
      __syncthreads();
    }
  }
}

// ------------------------------------------------------------------------------------
// Down projection + router-order combine + shared expert.  Work item = 16 output rows.
// Threads form "pair lanes" of LR threads; a pair lane computes d = W2_e act_i for one
// (token, slot) pair i over the 16 rows, each thread covering NG = G2 / LR consecutive
// groups of the I inputs.  The 16-row results land in dbuf[i][row]; then every token's
// output is the float sum over j in router order of w[t][j] * dbuf[t*K + j], plus the
// shared expert's row (bf16 weights, fp32 activations), added last and unweighted.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_down_combine(
    int T, int H, int I, int K, ExpertArgs ex, const int32_t *__restrict__ idx,
    const float *__restrict__ w, const int32_t *__restrict__ disp, int P,
    const uint16_t *__restrict__ act_hi, const uint16_t *__restrict__ act_lo,
    const int32_t *__restrict__ act_ex, const uint16_t *__restrict__ sh_down, int SI,
    const float *__restrict__ act_s, void *y, int ydt, int accumulate, int LR) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  float *dbuf = reinterpret_cast<float *>(smem_raw);       // [P][16]
  float *part = dbuf + (size_t)P * kDownRows;              // [blockDim][16]
  float *ds = part + (size_t)blockDim.x * kDownRows;       // [T][16]
  const int G2 = I / kGroup;
  const int NG = G2 / LR;
  const int tid = threadIdx.x;
  const int ul = tid / LR, l = tid % LR;
  const int ULANES = blockDim.x / LR;
  const int U = disp[0];
  const int *uoff = disp + 4 + P;
  const int *plist = uoff + P + 1;
  const int nvalid = uoff[U];
  const int rowbytes = I / 2;
  const int ntiles = H / kDownRows;

  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int r0 = tile * kDownRows;
    for (int i = tid; i < P * kDownRows; i += blockDim.x) dbuf[i] = 0.f;
    __syncthreads();

    for (int k0 = 0; k0 < nvalid; k0 += ULANES) {
      const int k = k0 + ul;
      const bool active = (ul < ULANES) && (k < nvalid);
      float acc[kDownRows];
#pragma unroll
      for (int r = 0; r < kDownRows; r++) acc[r] = 0.f;
      int i = 0;
      if (active) {
        i = plist[k];
        const int e = idx[i];
        const uint8_t *rec = ex.base + (long long)e * ex.stride;
        const uint8_t *w2p = rec + ex.off[2], *w2s = rec + ex.off[3];
        for (int q = 0; q < NG; q++) {
          const int gg = l * NG + q;
          uint32_t xh[16], xl[16];
          {
            const uint4 *ph = reinterpret_cast<const uint4 *>(act_hi + act_index(i, I, gg, 0));
            const uint4 *pl = reinterpret_cast<const uint4 *>(act_lo + act_index(i, I, gg, 0));
#pragma unroll
            for (int c = 0; c < 4; c++) {
              const uint4 a = ph[c * G2], b = pl[c * G2];
              xh[4 * c] = a.x; xh[4 * c + 1] = a.y; xh[4 * c + 2] = a.z; xh[4 * c + 3] = a.w;
              xl[4 * c] = b.x; xl[4 * c + 1] = b.y; xl[4 * c + 2] = b.z; xl[4 * c + 3] = b.w;
            }
          }
          const int e2 = act_ex[(size_t)i * G2 + gg];
#pragma unroll
          for (int h = 0; h < 2; h++) {
            uint4 wv[8];
            uint32_t sv[8];
#pragma unroll
            for (int r = 0; r < 8; r++) {
              const int row = r0 + 8 * h + r;
              wv[r] = __ldg(reinterpret_cast<const uint4 *>(w2p + (size_t)row * rowbytes) + gg);
              sv[r] = __ldg(w2s + (size_t)row * G2 + gg);
            }
#pragma unroll
            for (int r = 0; r < 8; r++) {
              if (sv[r] != 255u) acc[8 * h + r] += group_dot2(xh, xl, wv[r]) * group_factor(sv[r], e2);
            }
          }
        }
      }
      // reduce the LR lanes of each pair lane through shared memory, fixed order
#pragma unroll
      for (int r = 0; r < kDownRows; r++) part[(size_t)tid * kDownRows + r] = acc[r];
      __syncthreads();
      if (active) {
        for (int r = l; r < kDownRows; r += LR) {
          float s = 0.f;
          for (int l2 = 0; l2 < LR; l2++) s += part[(size_t)(ul * LR + l2) * kDownRows + r];
          dbuf[(size_t)i * kDownRows + r] = s;
        }
      }
      __syncthreads();
    }

    // shared expert rows r0..r0+15: 16 lanes per row, SI/8 chunks of 8 bf16
    if (sh_down != nullptr) {
      const int row = tid >> 4, ls = tid & 15;
      if (row < kDownRows) {
        const uint4 *w4 = reinterpret_cast<const uint4 *>(sh_down + (size_t)(r0 + row) * SI);
        const int nch = SI >> 3;
        for (int t = 0; t < T; t++) {
          const float4 *a4 = reinterpret_cast<const float4 *>(act_s + (size_t)t * SI);
          float s = 0.f;
          for (int c = ls; c < nch; c += 16) {
            const uint4 wv = __ldg(w4 + c);
            const float4 a0 = a4[2 * c], a1 = a4[2 * c + 1];
            s = fmaf(bf16_lo(wv.x), a0.x, s);
            s = fmaf(bf16_hi(wv.x), a0.y, s);
            s = fmaf(bf16_lo(wv.y), a0.z, s);
            s = fmaf(bf16_hi(wv.y), a0.w, s);
            s = fmaf(bf16_lo(wv.z), a1.x, s);
            s = fmaf(bf16_hi(wv.z), a1.y, s);
            s = fmaf(bf16_lo(wv.w), a1.z, s);
            s = fmaf(bf16_hi(wv.w), a1.w, s);
          }
#pragma unroll
          for (int o = 8; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
          if (ls == 0) ds[t * kDownRows + row] = s;
        }
      }
    }
    __syncthreads();

    // combine: routed sum in router order, then the shared expert, unweighted
    for (int q = tid; q < T * kDownRows; q += blockDim.x) {
      const int t = q / kDownRows, row = q % kDownRows;
      float s = 0.f;
      for (int j = 0; j < K; j++)
        s = __fadd_rn(s, __fmul_rn(w[t * K + j], dbuf[(size_t)(t * K + j) * kDownRows + row]));
      if (sh_down != nullptr) s = __fadd_rn(s, ds[t * kDownRows + row]);
      const size_t o = (size_t)t * H + r0 + row;
      if (ydt == K3MOE_F32) {
        float *yf = reinterpret_cast<float *>(y);
        yf[o] = accumulate ? __fadd_rn(yf[o], s) : s;
      } else {
        uint16_t *yb = reinterpret_cast<uint16_t *>(y);
        const float v = accumulate ? __fadd_rn(bf16_lo(yb[o]), s) : s;
        yb[o] = f32_to_bf16(v);
      }
    }
    __syncthreads();
  }
}

cudaError_t launch_expert_gateup(int mb, int grid, int block, cudaStream_t st, const void *x,
                                 bool x_f32, int H, int I, int K, const ExpertArgs &ex,
                                 const int32_t *disp, int P, float b1, float b2,
                                 uint16_t *act_hi, uint16_t *act_lo, int32_t *act_ex) {
  if (x_f32) {  // one token per register block: two f16 terms per input use the registers
    k_expert_gateup<1, true><<<grid, block, 0, st>>>(x, H, I, K, ex, disp, P, b1, b2, act_hi,
                                                     act_lo, act_ex);
  } else {
    if (mb == 1)
      k_expert_gateup<1, false><<<grid, block, 0, st>>>(x, H, I, K, ex, disp, P, b1, b2, act_hi,
                                                        act_lo, act_ex);
    else
      k_expert_gateup<2, false><<<grid, block, 0, st>>>(x, H, I, K, ex, disp, P, b1, b2, act_hi,
                                                        act_lo, act_ex);
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------------------------------
// Test hook: dequantise through the same conversion (E2M1 pair -> f16x2 -> float) and
// the same scale factor the FFN uses.  One thread per 32-column group.
// ------------------------------------------------------------------------------------
__global__ void k_dequant(const uint8_t *__restrict__ packed, const uint8_t *__restrict__ scales,
                          int rows, int cols, float *__restrict__ out) {
  const int G = cols / kGroup;
  const long long n = (long long)rows * G;
  for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < n;
       q += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(q / G), g = (int)(q % G);
    const uint4 wv = *(reinterpret_cast<const uint4 *>(packed + (size_t)r * (cols / 2)) + g);
    const uint32_t s = scales[(size_t)r * G + g];
    const float f = group_factor(s, 0);
    const uint32_t wa[4] = {wv.x, wv.y, wv.z, wv.w};
    float *o = out + (size_t)r * cols + (size_t)g * kGroup;
#pragma unroll
    for (int k = 0; k < 4; k++) {
      uint32_t h[4];
      e2m1x8_to_f16x2x4(wa[k], h[0], h[1], h[2], h[3]);
#pragma unroll
      for (int b = 0; b < 4; b++) {
        const __half2 v = *reinterpret_cast<__half2 *>(&h[b]);
        o[8 * k + 2 * b] = __low2float(v) * f;
        o[8 * k + 2 * b + 1] = __high2float(v) * f;
      }
    }
  }
}

// ------------------------------------------------------------------------------------
// RMSNorm to bf16 (kimi-k3-in-c, section 5): one CTA per row; sum of squares in double.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kRmsThreads) k_rmsnorm_bf16(const float *__restrict__ h, int T,
                                                              int n, float eps,
                                                              uint16_t *__restrict__ out) {
  // Each thread loads its (up to kRmsVec) float4 of the row at once and keeps them for the
  // output pass; the sum of squares is exact per product in double, reduced in a fixed
  // tree.  Rows whose width is not a multiple of 4 or above kRmsThreads * 4 * kRmsVec take
  // the strided loop.
  __shared__ double wsum[kRmsThreads / 32];
  __shared__ float s_inv;
  const int t = blockIdx.x;
  pdl_wait();  // h is written by the previous kernel when launched as a dependent
  pdl_launch_dependents();
  if (t >= T) return;
  const float *row = h + (size_t)t * n;
  const bool vec = (n % 4 == 0) && (n <= kRmsThreads * 4 * kRmsVec);
  float4 v[kRmsVec];
  double ss = 0.0;
  if (vec) {
    const float4 *r4 = reinterpret_cast<const float4 *>(row);
#pragma unroll
    for (int k = 0; k < kRmsVec; k++) {
      const int i = threadIdx.x + k * kRmsThreads;
      v[k] = (4 * i < n) ? __ldg(r4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < kRmsVec; k++)
      ss += (double)v[k].x * v[k].x + (double)v[k].y * v[k].y + (double)v[k].z * v[k].z +
            (double)v[k].w * v[k].w;
  } else {
    for (int i = threadIdx.x; i < n; i += blockDim.x) ss += (double)row[i] * (double)row[i];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    double tot = 0.0;
    for (int w = 0; w < (int)(blockDim.x >> 5); w++) tot += wsum[w];
    s_inv = (float)(1.0 / sqrt(tot / (double)n + (double)eps));
  }
  __syncthreads();
  const float inv = s_inv;
  uint16_t *orow = out + (size_t)t * n;
  if (vec) {
#pragma unroll
    for (int k = 0; k < kRmsVec; k++) {
      const int i = threadIdx.x + k * kRmsThreads;
      if (4 * i < n) {
        const uint32_t lo = (uint32_t)f32_to_bf16(__fmul_rn(v[k].x, inv)) |
                            ((uint32_t)f32_to_bf16(__fmul_rn(v[k].y, inv)) << 16);
        const uint32_t hi = (uint32_t)f32_to_bf16(__fmul_rn(v[k].z, inv)) |
                            ((uint32_t)f32_to_bf16(__fmul_rn(v[k].w, inv)) << 16);
        reinterpret_cast<uint2 *>(orow)[i] = make_uint2(lo, hi);
      }
    }
  } else {
    for (int i = threadIdx.x; i < n; i += blockDim.x) orow[i] = f32_to_bf16(__fmul_rn(row[i], inv));
  }
}

}  // namespace k3

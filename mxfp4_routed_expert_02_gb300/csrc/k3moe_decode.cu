// k3moe_decode.cu -- decode-path kernels that stream expert tiles through shared memory
// with bulk asynchronous copies (TMA, cp.async.bulk) into a ring of mbarrier-guarded
// slots: one producer thread keeps up to ~200 KB per SM in flight while the consumer
// warps decode MXFP4 in registers.
//
// Arithmetic is the same as k3moe_ffn.cu (README of FareedKhan-dev/kimi-k3-in-c,
// section 4 for the MXFP4 product, section 9 for the expert FFN, SiTU and the router-order
// sum; README of Maknee/Kimi-K3.cpp, "The consumer-memory idea" item 7).
#include "k3moe_kernels.cuh"

namespace k3 {

// ------------------------------------------------------------------------------------
// Gate/up + SiTU for ONE token, TMA ring.  Block = HP x C consumer threads (C =
// ceil(G/32)*32, one per 32-column group of the H inputs in each of HP row phases) + a
// producer warp + an epilogue warp.  Work items = (selected expert j, 32-row tile),
// statically strided over the grid.  A stage holds RB rows of gate and up (packed) and
// their scale bytes; a consumer keeps the partial sums of its group column in registers.
// Each CTA recomputes the top-k from the router's scores (a few microseconds, no extra
// launch); CTA 0 publishes the route (idx, w) and the dispatch lists.
// ------------------------------------------------------------------------------------
// shared-memory map of k_gateup_t1 (bytes)
constexpr int kGuBars = 0;       // full[16], empty[16]
constexpr int kGuRedBars = 256;  // redbar[2], redfree[2] (inside the 256..288 gap)
constexpr int kGuLst = 320;      // int [8][32]
constexpr int kGuSel = 1344;     // int [32]
constexpr int kGuWsel = 1472;    // float [32]
constexpr int kGuAbort = 1600;   // int
constexpr int kGuRed = 1664;     // float [2 parities][16 warps][32 rows][2]
constexpr int kGuScores = kGuRed + 2 * 16 * 64 * 4;  // top-k scratch (uint64)
__host__ __device__ inline int gu_ring_offset(int E, int K) {
  return (kGuScores + 8 * topk_scratch_keys(E, K) + 127) & ~127;
}

// HP consumer threads per group column (HP = 2, or 4 when the row is at most 128 groups
// long, so that narrow inputs still keep 16 consumer warps streaming): thread (h, g),
// h < HP, takes the rows q of a stage with q % HP == h.  Every two stages a thread's
// 4*RB/HP partial sums (RB/HP rows x gate/up x 2 stages) are transpose-reduced inside its
// warp and parked in shared memory (one of two buffers, by tile parity).  An epilogue warp adds the warps' parts of a 32-row tile in a
// fixed order, applies SiTU and writes the activations; consumers hand tiles to it
// through mbarriers and never wait for one another.
// XF32: the input is a.xf (float, the LatentMoE's latent), prescaled into two f16 terms
// per group (hi + residual) and multiplied with both (group_dot2).
template <int RB, bool XF32, int HP>
__global__ void __launch_bounds__(HP == 4 ? 576 : 512, 1) k_gateup_t1(GateUpT1Args a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int H = a.H, I = a.I, K = a.K;
  const int G = H / kGroup;
  const int C = ((G + 31) / 32) * 32;   // threads per row phase
  const int nwc = C / 32;               // warps per row phase
  const int NS = a.NS;
  const int rowb = H / 2;
  const uint32_t stage_bytes = (uint32_t)(2 * RB * (rowb + G));
  const int tiles = I / kTileRows;
  constexpr int nblk = kTileRows / RB;  // stages per tile (even)
  constexpr int RP = RB / HP;           // rows of a stage per consumer thread
  constexpr int V = 4 * RP;             // values per two stages: RP rows x 2 mats x 2

  uint64_t *full = reinterpret_cast<uint64_t *>(smem + kGuBars);
  uint64_t *empty = full + 16;
  uint64_t *redbar = reinterpret_cast<uint64_t *>(smem + kGuRedBars);  // [2]
  uint64_t *redfree = redbar + 2;                                       // [2]
  int *sel = reinterpret_cast<int *>(smem + kGuSel);
  float *wsel = reinterpret_cast<float *>(smem + kGuWsel);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kGuAbort);
  float *red = reinterpret_cast<float *>(smem + kGuRed);
  float *s_scores = reinterpret_cast<float *>(smem + kGuScores);  // top-k key scratch
  uint8_t *ring = smem + gu_ring_offset(a.E, a.K);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int s = 0; s < NS; s++) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], HP * nwc);
    }
    for (int p = 0; p < 2; p++) {
      mbar_init(&redbar[p], HP * nwc);
      mbar_init(&redfree[p], 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();

  cta_topk(a.sc, a.ch, a.E, K, a.renorm, a.routed_scale,
           reinterpret_cast<unsigned long long *>(s_scores), sel, wsel);
  if (blockIdx.x == 0) {
    if (tid < K) {
      a.idx_out[tid] = sel[tid];
      a.w_out[tid] = wsel[tid];
      int *uexp = a.disp + 4;
      int *uoff = uexp + K;
      int *plist = uoff + K + 1;
      uexp[tid] = sel[tid];
      uoff[tid] = tid;
      plist[tid] = tid;
    }
    if (tid == 0) {
      a.disp[0] = K;
      a.disp[4 + K + K] = K;  // uoff[U] = number of pairs
    }
  }
  pdl_launch_dependents();

  const int nitems = K * tiles;
  if (warp == HP * nwc) {
    // ---------------- producer: lane p < NS owns ring slot p ----------------
    // A single thread issues only a few bulk copies per microsecond, so the stages are
    // spread over NS lanes; each slot's fills are issued by one lane, in phase order.
    if (lane < NS) {
      const int p = lane;
      const int nmine = (nitems - blockIdx.x + gridDim.x - 1) / gridDim.x;  // items of this CTA
      const int nst = nmine > 0 ? nmine * nblk : 0;                            // stages
      int it = p;
      bool ok = true;
      for (; it < nst; it += NS) {
        const int item = blockIdx.x + (it / nblk) * gridDim.x;
        const int b = it % nblk;
        const int j = item / tiles, tile = item % tiles;
        const uint8_t *rec = a.ex.base + (long long)sel[j] * a.ex.stride;
        if (!mbar_wait(&empty[p], ((it / NS) & 1) ^ 1)) {
          set_status(a.status, K3MOE_ERR_TIMEOUT);
          ok = false;
          break;
        }
        const int r = tile * kTileRows + b * RB;
        uint8_t *dst = ring + (size_t)p * stage_bytes;
        mbar_arrive_expect_tx(&full[p], stage_bytes);
        // weights are read once: first out of L2
        const uint64_t pol = l2_evict_first();
        bulk_g2s_pol(dst, rec + a.ex.off[0] + (size_t)r * rowb, RB * rowb, &full[p], pol);
        bulk_g2s_pol(dst + RB * rowb, rec + a.ex.off[4] + (size_t)r * rowb, RB * rowb, &full[p],
                     pol);
        bulk_g2s_pol(dst + 2 * RB * rowb, rec + a.ex.off[1] + (size_t)r * G, RB * G, &full[p],
                     pol);
        bulk_g2s_pol(dst + 2 * RB * rowb + RB * G, rec + a.ex.off[5] + (size_t)r * G, RB * G,
                     &full[p], pol);
      }
      if (!ok && it - NS >= 0)  // bounded wait for this slot's last issued fill
        mbar_wait(&full[p], ((it - NS) / NS) & 1, 400000000LL);
    }
    return;
  }

  if (warp == HP * nwc + 1) {
    // ---------------- epilogue: SiTU and activation output per tile ----------------
    int n = 0;
    for (int item = blockIdx.x; item < nitems; item += gridDim.x, n++) {
      const int j = item / tiles, tile = item % tiles;
      const int par = n & 1;
      const float *rt = red + par * (16 * 64);
      if (!mbar_wait(&redbar[par], (n >> 1) & 1)) {
        set_status(a.status, K3MOE_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      // row `lane` of the tile was computed by the warps of row phase lane % HP
      const int hp = lane % HP;
      float gs = 0.f, us = 0.f;
      for (int w = hp * nwc; w < (hp + 1) * nwc; w++) {
        gs += rt[(w * 32 + lane) * 2];
        us += rt[(w * 32 + lane) * 2 + 1];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&redfree[par]);
      float act = situ(gs, us, a.b1, a.b2);
      if (*abort_flag) act = 0.f;
      float mx = fabsf(act);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      int e2 = 0;
      if (mx > 0.f) {
        e2 = exponent_of(mx) - 14;
        e2 = e2 < -110 ? -110 : e2;
      }
      const float sa = act * pow2i(-e2);
      const __half hh = __float2half_rn(sa);
      const __half hl = __float2half_rn(sa - __half2float(hh));
      const size_t o = act_index(j, I, tile, lane);
      a.act_hi[o] = __half_as_ushort(hh);
      a.act_lo[o] = __half_as_ushort(hl);
      if (lane == 0) a.act_ex[(size_t)j * (I / kGroup) + tile] = e2;
    }
    return;
  }

  // ---------------- consumers: thread (h, g) ----------------
  const int h = tid / C, g = tid % C;
  const bool gact = g < G;
  uint32_t xr[16], xl[16];
  int xe = 0;
#pragma unroll
  for (int p = 0; p < 16; p++) xr[p] = xl[p] = 0u;
  if (gact) {
    float v[32];
    if (XF32) {
      const float4 *src = reinterpret_cast<const float4 *>(a.xf + g * kGroup);
#pragma unroll
      for (int q = 0; q < 8; q++) {
        const float4 c = __ldg(src + q);
        v[4 * q] = c.x;
        v[4 * q + 1] = c.y;
        v[4 * q + 2] = c.z;
        v[4 * q + 3] = c.w;
      }
      xe = prescale_group_f16_hilo(v, xr, xl);
    } else {
      const uint4 *src = reinterpret_cast<const uint4 *>(a.x + g * kGroup);
#pragma unroll
      for (int q = 0; q < 4; q++) {
        const uint4 c = __ldg(src + q);
        const uint32_t w4[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int k = 0; k < 4; k++) {
          v[8 * q + 2 * k] = bf16_lo(w4[k]);
          v[8 * q + 2 * k + 1] = bf16_hi(w4[k]);
        }
      }
      xe = prescale_group_f16(v, xr);
    }
  }

  int it = 0, n = 0;
  bool aborted = false;
  for (int item = blockIdx.x; item < nitems; item += gridDim.x, n++) {
    const int par = n & 1;
    float *rt = red + par * (16 * 64);  // [warp][row 0..31][mat]
    // the epilogue must be done with this buffer's previous tile (two tiles back)
    if (!aborted && !mbar_wait(&redfree[par], ((n >> 1) & 1) ^ 1)) {
      set_status(a.status, K3MOE_ERR_TIMEOUT);
      aborted = true;
      *abort_flag = 1;
    }
#pragma unroll 1
    for (int b = 0; b < nblk; b += 2) {
      float vals[V];
#pragma unroll
      for (int v = 0; v < V; v++) vals[v] = 0.f;
#pragma unroll
      for (int b2 = 0; b2 < 2; b2++, it++) {
        const int s = it % NS;
        if (!aborted && !mbar_wait(&full[s], (it / NS) & 1)) {
          set_status(a.status, K3MOE_ERR_TIMEOUT);
          aborted = true;
          *abort_flag = 1;
        }
        if (!aborted && gact) {
          const uint8_t *st = ring + (size_t)s * stage_bytes;
          const uint8_t *sgs = st + 2 * RB * rowb;
          const uint8_t *sus = sgs + RB * G;
#pragma unroll
          for (int k = 0; k < RP; k++) {
            const int q = h + HP * k;  // row within the stage
            const uint4 wg = reinterpret_cast<const uint4 *>(st + q * rowb)[g];
            const uint4 wu = reinterpret_cast<const uint4 *>(st + (RB + q) * rowb)[g];
            const uint32_t sg = sgs[q * G + g], su = sus[q * G + g];
            if (sg != 255u)
              vals[b2 * 2 * RP + 2 * k] =
                  (XF32 ? group_dot2(xr, xl, wg) : group_dot(xr, wg)) * group_factor(sg, xe);
            if (su != 255u)
              vals[b2 * 2 * RP + 2 * k + 1] =
                  (XF32 ? group_dot2(xr, xl, wu) : group_dot(xr, wu)) * group_factor(su, xe);
          }
        }
        __syncwarp();
        if (lane == 0 && !aborted) mbar_arrive(&empty[s]);
      }
      // value v = b2*2*RP + 2k + m  ->  tile row (b + b2)*RB + h + HP*k, matrix m
      const float tot = warp_transpose_reduce<V>(vals);
      if (lane < V) {
        const int b2 = lane / (2 * RP), k = (lane % (2 * RP)) / 2, m = lane & 1;
        rt[(warp * 32 + ((b + b2) * RB + h + HP * k)) * 2 + m] = tot;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&redbar[par]);  // also when aborted: the epilogue never hangs
  }
}

size_t gateup_t1_smem(int H, int E, int K, int RB, int NS) {
  const int G = H / kGroup;
  return gu_ring_offset(E, K) + (size_t)NS * 2 * RB * (H / 2 + G);
}

int gateup_t1_phases(int H) { return H / kGroup <= 128 ? 4 : 2; }

cudaError_t launch_gateup_t1(const GateUpT1Args &a, int grid, cudaStream_t st, bool pdl) {
  const int G = a.H / kGroup;
  const int C = ((G + 31) / 32) * 32;
  const int HP = gateup_t1_phases(a.H);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(HP * C + 64);
  cfg.dynamicSmemBytes = gateup_t1_smem(a.H, a.E, a.K, a.RB, a.NS);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.RB != 8 && a.RB != 16) return cudaErrorInvalidValue;
  const bool r8 = a.RB == 8;
  if (HP == 4) {
    if (a.xf)
      return r8 ? cudaLaunchKernelEx(&cfg, k_gateup_t1<8, true, 4>, a)
                : cudaLaunchKernelEx(&cfg, k_gateup_t1<16, true, 4>, a);
    return r8 ? cudaLaunchKernelEx(&cfg, k_gateup_t1<8, false, 4>, a)
              : cudaLaunchKernelEx(&cfg, k_gateup_t1<16, false, 4>, a);
  }
  if (a.xf)
    return r8 ? cudaLaunchKernelEx(&cfg, k_gateup_t1<8, true, 2>, a)
              : cudaLaunchKernelEx(&cfg, k_gateup_t1<16, true, 2>, a);
  return r8 ? cudaLaunchKernelEx(&cfg, k_gateup_t1<8, false, 2>, a)
            : cudaLaunchKernelEx(&cfg, k_gateup_t1<16, false, 2>, a);
}

// ------------------------------------------------------------------------------------
// Down projection + router-order combine + shared expert, TMA ring.  Work item = 16
// output rows.  A stage holds one distinct expert's 16 rows of W2 (packed + scales);
// stages of an item go round-robin to NS "expert lanes" of LR threads (one slot per
// lane); an expert lane computes d = W2_e act for every (token, slot) pair routed to e,
// each thread covering NG = (I/32)/LR groups, and writes dbuf[pair][row].  After all
// stages of the item: y[t] = sum_j w[t][j] dbuf[t*K+j] in router order (float), plus the
// shared expert's rows (bf16 weights, fp32 activations), added last and unweighted.
// ------------------------------------------------------------------------------------
// A stage is one distinct expert's 8-row half of the 16-row tile (packed + scales).  Ring
// slot p belongs to consumer warp p: a warp consumes the phases of its own slot in order,
// so no two waiters ever wait on different phases of one barrier.  In a warp, lane =
// (row quarter rq, group lane l): a thread covers 4 rows x NG = (I/32)/16 groups.
// ACT_SMEM: the activations of all pairs are bulk-copied into shared memory once per CTA
// (they are the same for every row tile); otherwise they are read from global memory (L2)
// per pair and group.
constexpr int kDnLanes = 16;   // group lanes per row quarter (a half warp)
constexpr int kDnWarps = 16;   // consumer warps = ring slots
constexpr int kDnStageRows = 8;

template <bool ACT_SMEM>
__global__ void __launch_bounds__(544, 1) k_down_tma(DownArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int H = a.H, I = a.I, K = a.K, P = a.P, T = a.T;
  const int G2 = I / kGroup;
  const int NG = G2 / kDnLanes, NS = a.NS;
  const int rowb = I / 2;
  const uint32_t stage_bytes = (uint32_t)(kDnStageRows * (rowb + G2));
  const int ntiles = H / kDownRows;
  const int NC = kDnWarps * 32;  // consumer threads

  uint64_t *full = reinterpret_cast<uint64_t *>(smem);
  uint64_t *empty = full + 32;
  uint64_t *actbar = empty + 32;
  const int ntl = (ntiles + gridDim.x - 1) / gridDim.x;  // row tiles per CTA (at most)
  float *dbuf = reinterpret_cast<float *>(smem + 1024);   // [P][16]
  float *ds = dbuf + (size_t)P * kDownRows;               // [ntl][T][16] shared-expert rows
  float *wsm = ds + (size_t)ntl * T * kDownRows;          // [P] route weights
  // byte offsets inside the dynamic shared array (kept as smem + offset so the compiler
  // sees shared-space accesses)
  const size_t o_act = (1024 + ((size_t)P * kDownRows + (size_t)ntl * T * kDownRows + P) * 4 +
                        127) & ~size_t(127);
  const size_t n_act = ACT_SMEM ? (size_t)P * I * 2 : 0;
  uint16_t *s_hi = reinterpret_cast<uint16_t *>(smem + o_act);      // [P][I] (ACT_SMEM)
  uint16_t *s_lo = reinterpret_cast<uint16_t *>(smem + o_act + n_act);
  int32_t *s_ex = reinterpret_cast<int32_t *>(smem + o_act + 2 * n_act);
  const size_t o_ring = (o_act + 2 * n_act + (ACT_SMEM ? (size_t)P * G2 * 4 : 0) + 127) & ~size_t(127);
  uint8_t *ring = smem + o_ring;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int s = 0; s < NS; s++) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(actbar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();
  // the next kernel (a following layer's first kernel) may launch now; it waits for this
  // grid to complete before it reads anything
  pdl_launch_dependents();

  const int U = a.disp[0];
  const int *uexp = a.disp + 4;
  const int *uoff = uexp + P;
  const int *plist = uoff + P + 1;

  if (warp == kDnWarps) {
    // producer: lane p < NS owns ring slot p (stages it with it % NS == p), lane 31 stages
    // the activations and prefetches the shared-expert rows
    if (lane == 31) {
      if (ACT_SMEM) {
        const uint32_t nb = (uint32_t)((size_t)P * I * 2);
        const uint32_t ne = (uint32_t)((size_t)P * G2 * 4);
        mbar_arrive_expect_tx(actbar, 2 * nb + ne);
        bulk_g2s(s_hi, a.act_hi, nb, actbar);
        bulk_g2s(s_lo, a.act_lo, nb, actbar);
        bulk_g2s(s_ex, a.act_ex, ne, actbar);
      }
      if (a.sh_down != nullptr)
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x)
          bulk_prefetch_l2(a.sh_down + (size_t)tile * kDownRows * a.SI, kDownRows * a.SI * 2);
      if (ACT_SMEM) mbar_wait(actbar, 0, 400000000LL);
    } else if (lane < NS) {
      const int p = lane;
      const int per_tile = 2 * U;
      const int nmine = (ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x;
      const int nst = nmine > 0 ? nmine * per_tile : 0;
      int it = p;
      bool ok = true;
      for (; it < nst && per_tile > 0; it += NS) {
        const int tile = blockIdx.x + (it / per_tile) * gridDim.x;
        const int k = it % per_tile;
        const int r0 = tile * kDownRows;
        if (!mbar_wait(&empty[p], ((it / NS) & 1) ^ 1)) {
          set_status(a.status, K3MOE_ERR_TIMEOUT);
          ok = false;
          break;
        }
        const int u = k >> 1, rh = k & 1;
        const int rs = r0 + rh * kDnStageRows;
        const uint8_t *rec = a.ex.base + (long long)uexp[u] * a.ex.stride;
        uint8_t *dst = ring + (size_t)p * stage_bytes;
        mbar_arrive_expect_tx(&full[p], stage_bytes);
        const uint64_t pol = l2_evict_first();  // weights are read once: first out of L2
        bulk_g2s_pol(dst, rec + a.ex.off[2] + (size_t)rs * rowb, kDnStageRows * rowb, &full[p],
                     pol);
        bulk_g2s_pol(dst + kDnStageRows * rowb, rec + a.ex.off[3] + (size_t)rs * G2,
                     kDnStageRows * G2, &full[p], pol);
      }
      if (!ok && it - NS >= 0) mbar_wait(&full[p], ((it - NS) / NS) & 1, 400000000LL);
    }
    return;
  }

  const int rq = lane >> 4, l = lane & 15;  // row quarter (4 rows), group lane
  bool aborted = false;
  if (ACT_SMEM && !mbar_wait(actbar, 0)) {
    set_status(a.status, K3MOE_ERR_TIMEOUT);
    aborted = true;
  }
  const uint16_t *act_hi = ACT_SMEM ? s_hi : a.act_hi;
  const uint16_t *act_lo = ACT_SMEM ? s_lo : a.act_lo;
  const int32_t *act_ex = ACT_SMEM ? s_ex : a.act_ex;

  // Before the first tile, while the ring fills: the route weights into shared memory and
  // the shared expert's rows of every tile of this CTA (bf16 weights, prefetched into L2
  // by the producer, x fp32 activations; one warp per row).
  for (int i = tid; i < P; i += NC) wsm[i] = a.w[i];
  if (a.sh_down != nullptr) {
    const int nch = a.SI >> 3;
    for (int n = 0; n < ntl; n++) {
      const int tile = blockIdx.x + n * gridDim.x;
      if (tile >= ntiles) break;
      const int row = tile * kDownRows + warp;  // warp < 16 = kDownRows
      const uint4 *w4 = reinterpret_cast<const uint4 *>(a.sh_down + (size_t)row * a.SI);
      for (int t = 0; t < T; t++) {
        const float4 *a4 = reinterpret_cast<const float4 *>(a.act_s + (size_t)t * a.SI);
        float sacc = 0.f;
        for (int c = lane; c < nch; c += 32) {
          const uint4 wv = __ldg(w4 + c);
          const float4 a0 = a4[2 * c], a1 = a4[2 * c + 1];
          sacc = fmaf(bf16_lo(wv.x), a0.x, sacc);
          sacc = fmaf(bf16_hi(wv.x), a0.y, sacc);
          sacc = fmaf(bf16_lo(wv.y), a0.z, sacc);
          sacc = fmaf(bf16_hi(wv.y), a0.w, sacc);
          sacc = fmaf(bf16_lo(wv.z), a1.x, sacc);
          sacc = fmaf(bf16_hi(wv.z), a1.y, sacc);
          sacc = fmaf(bf16_lo(wv.w), a1.z, sacc);
          sacc = fmaf(bf16_hi(wv.w), a1.w, sacc);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sacc += __shfl_xor_sync(0xffffffffu, sacc, o);
        if (lane == 0) ds[((size_t)n * T + t) * kDownRows + warp] = sacc;
      }
    }
  }

  int it0 = 0, ntl_i = 0;
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ntl_i++) {
    const int r0 = tile * kDownRows;
    for (int i = tid; i < P * kDownRows; i += NC) dbuf[i] = 0.f;
    asm volatile("bar.sync 1, %0;" ::"r"(NC) : "memory");
    // this warp's stages of the tile: those in its own slot (it % NS == warp)
    for (int k = (warp < NS) ? (((warp - it0) % NS) + NS) % NS : 2 * U; k < 2 * U; k += NS) {
      const int it = it0 + k;
      const int s = warp;
      if (!aborted && !mbar_wait(&full[s], (it / NS) & 1)) {
        set_status(a.status, K3MOE_ERR_TIMEOUT);
        aborted = true;
      }
      const int u = k >> 1, rh = k & 1;
      const uint8_t *st = ring + (size_t)s * stage_bytes;
      const uint8_t *ss = st + kDnStageRows * rowb;
      for (int pk = uoff[u]; pk < uoff[u + 1] && !aborted; pk++) {
        const int i = plist[pk];
        float acc[4];
#pragma unroll
        for (int r = 0; r < 4; r++) acc[r] = 0.f;
        for (int q = 0; q < NG; q++) {
          // group lanes interleave (gg = q*16 + l): the 16 lanes read 16 consecutive
          // 16-byte weight chunks, and activation chunks 64 B apart
          const int gg = q * kDnLanes + l;
          uint32_t xh[16], xl[16];
          const uint4 *ph = reinterpret_cast<const uint4 *>(act_hi + act_index(i, I, gg, 0));
          const uint4 *pl = reinterpret_cast<const uint4 *>(act_lo + act_index(i, I, gg, 0));
#pragma unroll
          for (int c = 0; c < 4; c++) {
            const uint4 x0 = ph[c * G2], x1 = pl[c * G2];
            xh[4 * c] = x0.x; xh[4 * c + 1] = x0.y; xh[4 * c + 2] = x0.z; xh[4 * c + 3] = x0.w;
            xl[4 * c] = x1.x; xl[4 * c + 1] = x1.y; xl[4 * c + 2] = x1.z; xl[4 * c + 3] = x1.w;
          }
          const int e2 = act_ex[(size_t)i * G2 + gg];
#pragma unroll
          for (int r = 0; r < 4; r++) {
            const int row = rq * 4 + r;
            const uint4 wv = reinterpret_cast<const uint4 *>(st + row * rowb)[gg];
            const uint32_t sv = ss[row * G2 + gg];
            if (sv != 255u) acc[r] += group_dot2(xh, xl, wv) * group_factor(sv, e2);
          }
        }
        // reduce the 4 row partials over the 16 group lanes of this half warp
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) {
#pragma unroll
          for (int r = 0; r < 4; r++) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], o);
        }
        if (l == 0) {
#pragma unroll
          for (int r = 0; r < 4; r++)
            dbuf[(size_t)i * kDownRows + rh * kDnStageRows + rq * 4 + r] = acc[r];
        }
      }
      __syncwarp();
      if (lane == 0 && !aborted) mbar_arrive(&empty[s]);
    }
    it0 += 2 * U;

    asm volatile("bar.sync 1, %0;" ::"r"(NC) : "memory");

    for (int q = tid; q < T * kDownRows; q += NC) {
      const int t = q / kDownRows, row = q % kDownRows;
      float sum = 0.f;
      for (int j = 0; j < K; j++)
        sum = __fadd_rn(sum, __fmul_rn(wsm[t * K + j], dbuf[(size_t)(t * K + j) * kDownRows + row]));
      if (a.sh_down != nullptr) sum = __fadd_rn(sum, ds[((size_t)ntl_i * T + t) * kDownRows + row]);
      const size_t o = (size_t)t * H + r0 + row;
      if (aborted) sum = 0.f;
      if (a.ydt == K3MOE_F32) {
        float *yf = reinterpret_cast<float *>(a.y);
        yf[o] = a.accumulate ? __fadd_rn(yf[o], sum) : sum;
      } else {
        uint16_t *yb = reinterpret_cast<uint16_t *>(a.y);
        const float v = a.accumulate ? __fadd_rn(bf16_lo(yb[o]), sum) : sum;
        yb[o] = f32_to_bf16(v);
      }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(NC) : "memory");
  }
}

// Shared memory of k_down_tma for ntl row tiles per CTA: barriers, dbuf, shared-expert
// rows, route weights, [activations], NS ring slots.
size_t down_tma_smem(int I, int T, int P, int NS, bool act_smem, int ntl) {
  const int G2 = I / kGroup;
  const size_t stage = (size_t)kDnStageRows * (I / 2 + G2);
  size_t b = (1024 + ((size_t)P * kDownRows + (size_t)ntl * T * kDownRows + P) * 4 + 127) &
             ~size_t(127);
  if (act_smem) b += (size_t)P * I * 4 + (size_t)P * G2 * 4;
  b = (b + 127) & ~size_t(127);
  return b + NS * stage;
}

// ------------------------------------------------------------------------------------
// Down projection + router-order sum for ONE token without a shared expert (the
// LatentMoE's experts), bulk-copy ring of whole-expert stages.  CTA b owns output rows
// [b R, b R + R) (R a multiple of 8 chosen so that the rows spread evenly over the SMs: no
// SM has a second tile to do while others are idle).  A stage holds one distinct expert's
// R rows of W2 (packed + scales) AND that expert's activations (the f16 term scaled by
// its group's exponent, and the exponents), so no activation is read from global memory
// in the dot products.  The f16 term alone carries 11 significant bits of every
// activation (relative rounding at most 2^-12, as the single-token fused kernel hands its
// activations over); the residual term the gate/up kernels also write is not read here.
// Stage u goes to worker group u % 2 (eight warps); warp wg takes rows wg, wg + 8, .. of
// the stage, its 32 lanes the input groups l, l + 32, .. (each group's activations loaded
// once for all the warp's rows).  Then y[row] = sum_j w[j] d_j[row] in router order
// (float), as in the other down kernels.
// ------------------------------------------------------------------------------------
constexpr int kD1Workers = 16;  // worker warps (two groups of eight)
constexpr int kD1MaxSlots = 8;
constexpr int kD1MaxRows = 48;  // rows per CTA at most

__host__ __device__ inline uint32_t down_t1_stage_bytes(int I, int R) {
  const uint32_t w = (uint32_t)R * (I / 2 + I / kGroup);  // rows: packed + scales
  const uint32_t act = (uint32_t)I * 2 + (uint32_t)(I / kGroup) * 4;
  return (w + act + 127u) & ~127u;
}
__host__ __device__ inline uint32_t down_t1_head_bytes(int K, int R) {  // bars, dbuf, w
  return (uint32_t)((1024 + (K * R + K) * 4 + 127) & ~127);
}

__global__ void __launch_bounds__(kD1Workers * 32 + 32, 1) k_down_t1(DownArgs a, int R) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int H = a.H, I = a.I, K = a.K;
  const int G2 = I / kGroup, NGL = G2 / 32, NS = a.NS;
  const int rowb = I / 2;
  const int r0 = (int)blockIdx.x * R;
  const int nr = H - r0 < R ? H - r0 : R;  // rows of this CTA (the last may have fewer)
  const uint32_t wbytes = (uint32_t)nr * rowb, sbytes = (uint32_t)nr * G2;
  const uint32_t wcap = (uint32_t)R * rowb, scap = (uint32_t)R * G2;  // stage layout
  const uint32_t abytes = (uint32_t)I * 2, ebytes = (uint32_t)G2 * 4;
  const uint32_t stage_bytes = down_t1_stage_bytes(I, R);
  const uint32_t tx = wbytes + sbytes + abytes + ebytes;
  constexpr int NW = kD1Workers * 32;

  uint64_t *full = reinterpret_cast<uint64_t *>(smem);  // [NS]
  uint64_t *empty = full + kD1MaxSlots;                  // [NS]
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + 512);
  float *dbuf = reinterpret_cast<float *>(smem + 1024);  // [K][R]
  float *wsm = dbuf + K * R;                             // [K]
  uint8_t *ring = smem + down_t1_head_bytes(K, R);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int q = 0; q < NS; q++) {
      mbar_init(&full[q], 1);
      mbar_init(&empty[q], 8);  // the eight warps of the group that consumes the stage
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();

  const int U = r0 < H ? a.disp[0] : 0;  // distinct experts (one pair each: one token)
  const int *uexp = a.disp + 4;
  const int *uoff = uexp + a.P;
  const int *plist = uoff + a.P + 1;

  if (warp == kD1Workers) {
    // producer: lane p < NS fills ring slot p with the stages u = p, p + NS, ...
    if (lane < NS) {
      int u = lane;
      bool ok = true;
      for (; u < U; u += NS) {
        const int pi = plist[uoff[u]];  // the pair of expert u
        if (!mbar_wait(&empty[lane], ((u / NS) & 1) ^ 1)) {
          set_status(a.status, K3MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          ok = false;
          break;
        }
        const uint8_t *rec = a.ex.base + (long long)uexp[u] * a.ex.stride;
        uint8_t *dst = ring + (size_t)lane * stage_bytes;
        mbar_arrive_expect_tx(&full[lane], tx);
        const uint64_t pol = l2_evict_first();  // weights are read once: first out of L2
        bulk_g2s_pol(dst, rec + a.ex.off[2] + (size_t)r0 * rowb, wbytes, &full[lane], pol);
        bulk_g2s_pol(dst + wcap, rec + a.ex.off[3] + (size_t)r0 * G2, sbytes, &full[lane], pol);
        bulk_g2s(dst + wcap + scap, a.act_hi + (size_t)pi * I, abytes, &full[lane]);
        bulk_g2s(dst + wcap + scap + abytes, a.act_ex + (size_t)pi * G2, ebytes, &full[lane]);
      }
      if (!ok && u - NS >= 0)  // bounded wait for this slot's last issued fill
        mbar_wait(&full[lane], ((u - NS) / NS) & 1, 400000000LL);
    }
    return;
  }

  const int gd = warp >> 3, wg = warp & 7;
  bool aborted = false;
  for (int i = tid; i < K; i += NW) wsm[i] = a.w[i];
  for (int i = tid; i < K * R; i += NW) dbuf[i] = 0.f;
  asm volatile("bar.sync 1, %0;" ::"r"(NW) : "memory");
  for (int u = gd; u < U; u += 2) {
    const int q = u % NS;
    if (!aborted && !mbar_wait(&full[q], (u / NS) & 1)) {
      set_status(a.status, K3MOE_ERR_TIMEOUT);
      aborted = true;
      *abort_flag = 1;
    }
    if (!aborted) {
      const uint8_t *st = ring + (size_t)q * stage_bytes;
      const uint8_t *ss = st + wcap;
      const uint16_t *s_hi = reinterpret_cast<const uint16_t *>(st + wcap + scap);
      const int32_t *s_ex = reinterpret_cast<const int32_t *>(st + wcap + scap + abytes);
      const int pi = plist[uoff[u]];
      float acc[kD1MaxRows / 8];
#pragma unroll
      for (int k = 0; k < kD1MaxRows / 8; k++) acc[k] = 0.f;
      for (int g = 0; g < NGL; g++) {
        const int gg = g * 32 + lane;
        uint32_t xh[16];
        const uint4 *ph = reinterpret_cast<const uint4 *>(s_hi + act_index(0, I, gg, 0));
#pragma unroll
        for (int c = 0; c < 4; c++) {
          const uint4 x0 = ph[c * G2];
          xh[4 * c] = x0.x; xh[4 * c + 1] = x0.y; xh[4 * c + 2] = x0.z; xh[4 * c + 3] = x0.w;
        }
        const int ex = s_ex[gg];
#pragma unroll
        for (int k = 0; k < kD1MaxRows / 8; k++) {
          const int row = wg + 8 * k;
          if (row < nr) {
            const uint4 wv = reinterpret_cast<const uint4 *>(st + row * rowb)[gg];
            const uint32_t sv = ss[row * G2 + gg];
            if (sv != 255u) acc[k] += group_dot(xh, wv) * group_factor(sv, ex);
          }
        }
      }
#pragma unroll
      for (int k = 0; k < kD1MaxRows / 8; k++) {
        if (wg + 8 * k < nr) {
          float v = acc[k];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == 0) dbuf[pi * R + wg + 8 * k] = v;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[q]);  // also when aborted: the producer never hangs
  }
  asm volatile("bar.sync 1, %0;" ::"r"(NW) : "memory");
  if (tid < nr) {
    float sum = 0.f;
    for (int j = 0; j < K; j++) sum = __fadd_rn(sum, __fmul_rn(wsm[j], dbuf[j * R + tid]));
    if (*abort_flag) sum = 0.f;
    const size_t o = (size_t)r0 + tid;
    if (a.ydt == K3MOE_F32) {
      float *yf = reinterpret_cast<float *>(a.y);
      yf[o] = a.accumulate ? __fadd_rn(yf[o], sum) : sum;
    } else {
      uint16_t *yb = reinterpret_cast<uint16_t *>(a.y);
      yb[o] = f32_to_bf16(a.accumulate ? __fadd_rn(bf16_lo(yb[o]), sum) : sum);
    }
  }
}

// Rows per CTA of k_down_t1 for H outputs on `sms` SMs (a multiple of 8, even spread).
int down_t1_rows(int H, int sms) {
  int R = (H + sms - 1) / sms;
  R = (R + 7) / 8 * 8;
  return R < 8 ? 8 : R;
}

// Ring slots of k_down_t1 for (H, I, K) on `sms` SMs (0: the kernel does not apply).
int down_t1_slots(int H, int I, int K, int sms) {
  if (I % 1024 != 0 || K > 32 || H % 8 != 0) return 0;  // 32 group lanes x NGL groups
  const int R = down_t1_rows(H, sms);
  if (R > kD1MaxRows) return 0;
  const size_t avail = 227 * 1024 - down_t1_head_bytes(K, R);
  int ns = (int)(avail / down_t1_stage_bytes(I, R));
  if (ns > kD1MaxSlots) ns = kD1MaxSlots;
  return ns >= 3 ? ns : 0;
}

cudaError_t launch_down_t1(const DownArgs &a, int sms, cudaStream_t st, bool pdl) {
  const int R = down_t1_rows(a.H, sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.H + R - 1) / R);
  cfg.blockDim = dim3(kD1Workers * 32 + 32);
  cfg.dynamicSmemBytes = down_t1_head_bytes(a.K, R) + (size_t)a.NS * down_t1_stage_bytes(a.I, R);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_down_t1, a, R);
}

cudaError_t launch_down_tma(const DownArgs &a, int grid, cudaStream_t st, bool pdl,
                            bool act_smem) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDnWarps * 32 + 32);
  cfg.dynamicSmemBytes =
      down_tma_smem(a.I, a.T, a.P, a.NS, act_smem, (a.H / kDownRows + grid - 1) / grid);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (act_smem) return cudaLaunchKernelEx(&cfg, k_down_tma<true>, a);
  return cudaLaunchKernelEx(&cfg, k_down_tma<false>, a);
}

cudaError_t set_decode_smem_limits() {
  const int big = 227 * 1024;
  const void *fns[] = {reinterpret_cast<const void *>(k_gateup_t1<8, false, 2>),
                       reinterpret_cast<const void *>(k_gateup_t1<16, false, 2>),
                       reinterpret_cast<const void *>(k_gateup_t1<8, true, 2>),
                       reinterpret_cast<const void *>(k_gateup_t1<16, true, 2>),
                       reinterpret_cast<const void *>(k_gateup_t1<8, false, 4>),
                       reinterpret_cast<const void *>(k_gateup_t1<16, false, 4>),
                       reinterpret_cast<const void *>(k_gateup_t1<8, true, 4>),
                       reinterpret_cast<const void *>(k_gateup_t1<16, true, 4>),
                       reinterpret_cast<const void *>(k_down_tma<true>),
                       reinterpret_cast<const void *>(k_down_tma<false>),
                       reinterpret_cast<const void *>(k_down_t1)};
  for (const void *f : fns) {
    const cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, big);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace k3

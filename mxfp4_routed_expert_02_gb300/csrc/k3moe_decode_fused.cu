// k3moe_decode_fused.cu -- the whole MoE layer step for one decode token in one persistent
// kernel: one CTA per SM, launched cooperatively so that every CTA is resident, with two
// grid-wide dependencies (bounded waits on counters in the workspace header, which the
// last CTA to finish leaves zero for the next call).
//
// What it computes is the single-token layer step of the other decode kernels (README of
// FareedKhan-dev/kimi-k3-in-c: section 9 "Picking 16 experts of 896" for the router and
// the top-k, the LatentMoE listing steps 3 and 6 for the expert FFN, the routed sum and
// the shared expert, the activation listing for SiTU; section 4 for the MXFP4 format;
// README of Maknee/Kimi-K3.cpp, "The consumer-memory idea" item 7, for the router order of
// the sum).  The schedule is what changes: every weight byte -- router rows, the shared
// expert, the selected experts -- goes through one ring of bulk-copy stages per SM, in
// the order
//
//   X  the token's input (once per CTA: every consumer thread takes its inputs from it)
//   R  router rows (two per stage)           -> logits, scores, selection scores
//   S  shared-expert gate/up row pairs       -> SiTU activations of the shared expert
//   G  the selected experts' gate/up rows    -> SiTU activations of the 16 experts
//   D  down rows of 16-row output tiles: the selected experts (two per stage) and the
//      shared expert, then the router-order combine of the tile
//
// so the stream never drains: the top-k needs every CTA's R rows (dependency 1: a counter
// the epilogue warp bumps once its router rows are written) and is computed by one warp
// of every CTA while the consumers take the S stages; each selection is published as soon
// as it is known, and the G stages of an expert slot go out once its selection is; D
// needs every activation (dependency 2: all worker warps of every CTA), while the ring
// already holds the first D stages.
//
// Warp roles: workers 0..2n-1 (n = H/1024) consume X, R, S and G stages (thread (h, g):
// input group g, row parity h); warp 14 reduces their partial sums (logits and scores,
// SiTU); warp 15 selects the top-k; warp 16 issues the bulk copies (lane s owns ring slot
// s).  In D all 16 worker warps (0..15) consume.
// Every wait is bounded: on expiry the kernel reports K3MOE_ERR_TIMEOUT, keeps arriving on
// the barriers it owes, and writes zeros.
#include "k3moe_kernels.cuh"

namespace k3 {

namespace {

constexpr int kFuWorkers = 16;   // worker warps
constexpr int kFuEpi = 14;       // warp index of the reduction epilogue
constexpr int kFuTopk = 15;      // warp index of the top-k (a worker only in D)
constexpr int kFuProducer = 16;  // warp index of the bulk-copy producer
constexpr int kFuThreads = 32 * (kFuWorkers + 1);
constexpr int kFuItemRows = 8;   // gate/up rows per reduction item (two G stages: the gate
                                 // rows, then the up rows)
constexpr int kFuNSD = 6;        // D ring slots: three per group of eight worker warps
constexpr int kFuMaxNS = 8;      // R/S/G ring slots at most
constexpr int kFuDownRows = 16;  // output rows per down tile
constexpr int kFuRedBytes = 2 * 16 * 64 * 4;  // partial sums [parity][warp][row][2]
constexpr int kBarDown = 1;      // named barrier of the 16 worker warps (0 is __syncthreads)
constexpr int kBarCons = 2;      // named barrier of the R/S/G consumer warps
constexpr long long kExpireBudget = 200000000LL;  // ~0.1 s: the expiry test's wait limit

// shared-memory map: barriers and small arrays; the ring (X/R/S/G slots, then D slots);
// the partial sums
constexpr int kFuBars = 0;       // fullG[8] emptyG[8] fullD[6] emptyD[6] redbar[2] redfree[2]
                                 // selbar topbar
constexpr int kFuSel = 384;      // int[32]
constexpr int kFuWsel = 512;     // float[32]
constexpr int kFuMisc = 640;     // int[8]: abort flag [4], RMSNorm factor [5], selections
                                 // published [7]
constexpr int kFuGDone = 704;    // int[8]: X/R/S/G slot s fully consumed (set by its owner)
constexpr int kFuSmall = 1024;   // X (RMSNorm): per-warp sums; top-k: the selection scores;
                                 // D: dbuf [K][16] + ds [16]
constexpr int kFuSmallBytes = 4096;
static_assert((16 + 2 * kFuNSD + 6) * 8 <= kFuSel, "the barriers overlap the small arrays");
static_assert(kFuNSD % 2 == 0, "every D slot serves one worker group");
constexpr int kFuRing = kFuSmall + kFuSmallBytes;

__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Order this thread's generic-proxy accesses before later async-proxy (bulk copy) ones.
__device__ __forceinline__ void fence_proxy_async_all() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
// Bounded wait until a counter (zeroed by the host before the launch) reaches n.
__device__ bool wait_count(const unsigned *cnt, unsigned n, long long budget = kWaitBudget) {
  const long long t0 = clock64();
  while (ld_acquire_u32(cnt) < n) {
    if (clock64() - t0 > budget) return false;
    __nanosleep(64);  // let the other lanes of the warp issue
  }
  return true;
}
// D slot of D stage i: stages alternate between the two worker groups (i % 2, which is
// also the slot's parity), and each group cycles through its three slots, so a group
// computes on one slot while the other two fill.
__host__ __device__ __forceinline__ int d_slot_of(int i) { return i % kFuNSD; }
// The factor 2^(s-127) * pe of an MXFP4 group with scale byte s, without a branch: the
// byte's bits become the float exponent (exact powers of two, subnormal products
// included).  Byte 255 contributes nothing (the group's NaN code); byte 0 gives 0 where
// the exact factor is 2^-127 * pe, a contribution some 30 orders of magnitude below the
// output's tolerance.
__device__ __forceinline__ float group_scale(uint32_t s, float pe) {
  const float f = __uint_as_float(s << 23) * pe;
  return s == 255u ? 0.f : f;
}

// Top-k of one token by one warp, once every CTA's scores are in the workspace.  Keys as
// in cta_topk: the selection score's order-preserving bits, then the complemented expert
// index, so the unsigned order is (score desc, index asc) and keys are distinct.  Lane l
// scans experts l, l + 32, ... and keeps its kTopQ largest keys in order; K rounds of a
// warp-wide maximum over the lanes' first keys then pick the selection in order, the
// winning lane dropping its first key.  A lane whose kept keys run out rescans its
// experts for the kTopQ largest below the last one it gave up, so the result is exact
// whatever the distribution.  The selection scores are read from ch_s (a shared-memory
// copy) when given, else from ch.  Selection j goes to sel[j] as soon as it is known, and
// *ready = j + 1 publishes it.  Lane j < K returns selection j: its expert index and its
// weight (the unbiased score, divided by the sum of the K scores in selection order when
// renorm is set, times routed_scale).
constexpr int kTopQ = 4;
__device__ void topk_warp(const float *sc, const float *ch, const float *ch_s, int E, int K,
                          int renorm, float routed_scale, int *sel, volatile int *ready,
                          int &e_out, float &w_out) {
  const int lane = threadIdx.x & 31;
  unsigned long long top[kTopQ];
  // the kTopQ largest keys of this lane's experts that are below `below`
  auto scan = [&](unsigned long long below) {
#pragma unroll
    for (int q = 0; q < kTopQ; q++) top[q] = 0ull;
#pragma unroll 4
    for (int e = lane; e < E; e += 32) {
      float c = __fadd_rn(ch_s ? ch_s[e] : __ldcg(ch + e), 0.f);  // -0 -> +0
      if (c != c) c = -__int_as_float(0x7f800000);  // a NaN never wins (it is reported)
      const unsigned long long k = ((unsigned long long)float_order_key(c) << 32) |
                                   (unsigned long long)(0xffffffffu - (uint32_t)e);
      if (k < below && k > top[kTopQ - 1]) {
        top[kTopQ - 1] = k;
#pragma unroll
        for (int q = kTopQ - 1; q > 0; q--) {
          if (top[q] > top[q - 1]) {
            const unsigned long long tk = top[q];
            top[q] = top[q - 1];
            top[q - 1] = tk;
          }
        }
      }
    }
  };
  scan(~0ull);
  unsigned long long mine = 0ull;
#pragma unroll 1
  for (int j = 0; j < K; j++) {
    const unsigned long long head = top[0];
    const unsigned hi = (unsigned)(head >> 32), lo = (unsigned)head;
    const unsigned mhi = __reduce_max_sync(0xffffffffu, hi);
    const unsigned mlo = __reduce_max_sync(0xffffffffu, hi == mhi ? lo : 0u);
    const unsigned long long best = ((unsigned long long)mhi << 32) | mlo;
    if (lane == j) mine = best;
    if (lane == 0) {  // publish selection j at once: the producer waits for it
      sel[j] = best ? (int)(0xffffffffu - (uint32_t)(best & 0xffffffffull)) : 0;
      __threadfence_block();
      *ready = j + 1;
    }
    if (head == best && head != 0ull) {  // distinct keys: one lane at most
#pragma unroll
      for (int q = 0; q < kTopQ - 1; q++) top[q] = top[q + 1];
      top[kTopQ - 1] = 0ull;
      if (top[0] == 0ull) scan(best);  // kept keys used up: the next ones below `best`
    }
  }
  e_out = (lane < K && mine != 0ull) ? (int)(0xffffffffu - (uint32_t)(mine & 0xffffffffull)) : 0;
  const float s = lane < K ? __ldcg(sc + e_out) : 0.f;
  float wsum = 0.f;  // float sum of the chosen scores in selection order
  for (int j = 0; j < K; j++) wsum = __fadd_rn(wsum, __shfl_sync(0xffffffffu, s, j));
  float w = s;
  if (renorm && wsum > 0.f) w = __fdiv_rn(w, wsum);
  w_out = __fmul_rn(w, routed_scale);
}

}  // namespace

// ---- layout of the fused kernel, shared by the host and the device ----------------------
// [small arrays | ring | partial sums].  The ring holds NSG X/R/S/G slots (the largest of
// a G stage -- the 8 rows of one item of the gate or the up matrix, packed + scales -- and
// an R/S stage of two bf16 rows of H); in phase D the same bytes hold kFuNSD D slots: the larger of a routed
// stage (16 rows of two experts, packed + scales, and those experts' activations) and a
// shared stage (8 bf16 rows of the shared down matrix and its activations).
__host__ __device__ inline uint32_t fused_gslot_bytes(int H) {
  const uint32_t g = (uint32_t)(kFuItemRows * (H / 2 + H / kGroup));
  const uint32_t r = (uint32_t)(2 * H * 2);
  return ((g > r ? g : r) + 127u) & ~127u;
}
__host__ __device__ inline uint32_t fused_dexp_bytes(int I) {  // one expert's 16 down rows
  return (uint32_t)(kFuDownRows * (I / 2 + I / kGroup));
}
__host__ __device__ inline uint32_t fused_dslot_bytes(int I, int SI) {
  const uint32_t r = 2 * fused_dexp_bytes(I) + 2u * (uint32_t)I * 2u;
  const uint32_t sh = SI > 0 ? 8u * (uint32_t)SI * 2u + (uint32_t)SI * 4u : 0u;
  return ((r > sh ? r : sh) + 127u) & ~127u;
}
constexpr size_t kFuSmemMax = 227 * 1024;
__host__ __device__ inline int fused_nsg(int H) {
  const int ns = (int)((kFuSmemMax - kFuRing - kFuRedBytes) / fused_gslot_bytes(H));
  return ns > kFuMaxNS ? kFuMaxNS : ns;
}
__host__ __device__ inline uint32_t fused_ring_bytes(int H, int I, int SI) {
  const uint32_t g = (uint32_t)fused_nsg(H) * fused_gslot_bytes(H);
  const uint32_t d = (uint32_t)kFuNSD * fused_dslot_bytes(I, SI);
  return g > d ? g : d;
}

// One layer of the step (layer `layer` of a stack): everything below runs once per layer, the
// CTA's roles meeting at a __syncthreads between layers.  kMulti: several layers share the
// launch, so no copy may outlive a layer (after an expiry the consumers stop waiting for
// their stages): the producer then also waits for a slot's previous fill to land before it
// refills the slot.
template <bool kMulti>
__device__ __forceinline__ void fused_layer(const FusedT1Args &a, const int layer, uint8_t *smem) {
  const FusedLayer &lw = a.lay[layer];
  unsigned *const bar = a.bar + 4 * layer;  // this layer's grid counters
  const int H = a.H, I = a.I, K = a.K, E = a.E, SI = a.SI;
  const int G = H / kGroup, nwc = G / 32;  // consumer warps per row parity
  const int rowb = H / 2;                  // packed bytes of a gate/up row
  const int rowh = H * 2;                  // bytes of a bf16 row of H
  const uint32_t gstage = (uint32_t)(kFuItemRows * (rowb + G));
  const int G2 = I / kGroup, rowb2 = I / 2;
  const uint32_t dexp = fused_dexp_bytes(I);    // one expert's 16 down rows
  const uint32_t gslot = fused_gslot_bytes(H);
  const uint32_t dslot = fused_dslot_bytes(I, SI);
  const int NSG = fused_nsg(H);
  constexpr int RS = 8;                          // shared down rows per D stage
  const int nSD = SI > 0 ? kFuDownRows / RS : 0;  // shared-down stages per tile
  const int bx = blockIdx.x, nb = gridDim.x;
  // this CTA's work
  const int cntR = bx < E ? (E - bx + nb - 1) / nb : 0;  // router rows bx + nb k
  const int nR = (cntR + 1) / 2;                          // R stages
  const int nS = bx < SI ? (SI - bx + nb - 1) / nb : 0;   // shared pairs bx + nb k
  const int blocks = I / kFuItemRows;                     // 8-row blocks per expert
  const int nitems = K * blocks;
  const int nI = bx < nitems ? (nitems - bx + nb - 1) / nb : 0;  // items bx + nb k
  const int tR = 1, tS = 1 + nR, tG = 1 + nR + nS;          // first X, R, S, G stages
  const int nRSG = tG + 2 * nI;
  const int ntiles = H / kFuDownRows;
  const int nT = bx < ntiles ? (ntiles - bx + nb - 1) / nb : 0;  // tiles bx + nb k
  const int hk = K / 2;
  const int dpt = hk + nSD;  // D stages per tile
  const int nD = nT * dpt;

  uint8_t *ring = smem + kFuRing;
  auto slot_ptr = [&](int s) -> uint8_t * { return ring + (size_t)s * gslot; };
  auto dslot_ptr = [&](int d) -> uint8_t * { return ring + (size_t)d * dslot; };
  uint64_t *fullG = reinterpret_cast<uint64_t *>(smem + kFuBars);
  uint64_t *emptyG = fullG + 8;
  uint64_t *fullD = fullG + 16;
  uint64_t *emptyD = fullD + kFuNSD;
  uint64_t *redbar = emptyD + kFuNSD;
  uint64_t *redfree = redbar + 2;
  uint64_t *selbar = redfree + 2;
  uint64_t *topbar = selbar + 1;
  int *sel = reinterpret_cast<int *>(smem + kFuSel);
  float *wsel = reinterpret_cast<float *>(smem + kFuWsel);
  int *misc = reinterpret_cast<int *>(smem + kFuMisc);
  volatile int *abort_flag = misc + 4;
  volatile int *selready = misc + 7;  // selections 0 .. *selready-1 are in sel
  volatile int *gdone = reinterpret_cast<volatile int *>(smem + kFuGDone);
  float *wss = reinterpret_cast<float *>(smem + kFuSmall);  // [warp][2] (X)
  float *dbuf = reinterpret_cast<float *>(smem + kFuSmall);  // [K][16] (D)
  float *ds = dbuf + K * kFuDownRows;                        // [16] (D)
  float *red = reinterpret_cast<float *>(ring + fused_ring_bytes(H, I, SI));

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    if (layer > 0) {  // the previous layer's barriers are idle: invalidate, then set up again
      for (int b = 0; b < 16 + 2 * kFuNSD + 6; b++) mbar_inval(fullG + b);
    }
    for (int s = 0; s < NSG; s++) {
      mbar_init(&fullG[s], 1);
      mbar_init(&emptyG[s], 2 * nwc);
    }
    for (int d = 0; d < kFuNSD; d++) {
      mbar_init(&fullD[d], 1);
      mbar_init(&emptyD[d], 8);
    }
    for (int p = 0; p < 2; p++) {
      mbar_init(&redbar[p], 2 * nwc);
      mbar_init(&redfree[p], 1);
    }
    mbar_init(selbar, 1);
    mbar_init(topbar, 1);
    misc[4] = 0;
    misc[7] = 0;
    for (int s = 0; s < kFuMaxNS; s++) gdone[s] = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kFuProducer) {
    // ---------------- producer: lane p < NSG owns ring slot p ----------------
    bool ab = false;
    int last_g = -1;  // this lane's last R/S/G stage
    // every weight byte is read once per step: its lines are the first L2 evicts (the
    // lines the step finds in L2 stay, so dirty ones are not written back during it)
    const uint64_t pol_first = l2_evict_first();
    if (lane < NSG) {
      int ready = 0;  // selections this lane has seen published
      for (int t = lane; t < nRSG; t += NSG) {
        if (t >= tG) {  // a routed stage needs its expert slot's selection
          const int j = (bx + nb * ((t - tG) >> 1)) / blocks;
          if (j >= ready) {
            const long long t0 = clock64();
            while ((ready = *selready) <= j) {
              if (clock64() - t0 > kWaitBudget) {
                set_status(a.status, K3MOE_ERR_TIMEOUT);
                ab = true;
                break;
              }
              __nanosleep(32);
            }
            if (ab) break;
            __threadfence_block();  // the published selections before their use
          }
        }
        // the slot's previous stage consumed and landed (after an expiry its consumers
        // stop waiting for it): one fill per slot at a time, so no copy outlives the layer
        if (!mbar_wait(&emptyG[lane], ((t / NSG) & 1) ^ 1) ||
            (kMulti && t >= NSG && !mbar_wait(&fullG[lane], ((t / NSG) & 1) ^ 1))) {
          set_status(a.status, K3MOE_ERR_TIMEOUT);
          ab = true;
          break;
        }
        uint8_t *dst = slot_ptr(lane);
        if (t == 0) {
          // the token's input: bf16 x, or the float residual stream to normalise -- in a
          // stack, once every CTA has added its tiles of the previous layer to it (the
          // other lanes meanwhile issue this layer's router and shared-expert stages)
          if (layer > 0) {
            if (!wait_count(a.bar + 4 * (layer - 1) + 2, (unsigned)nb)) {
              set_status(a.status, K3MOE_ERR_TIMEOUT);
              ab = true;
              break;
            }
            fence_proxy_async_all();  // the other CTAs' stores before the async-proxy read
          }
          const uint32_t xbytes = a.h ? (uint32_t)(H * 4) : (uint32_t)rowh;
          mbar_arrive_expect_tx(&fullG[lane], xbytes);
          bulk_g2s(dst, a.h ? static_cast<const void *>(a.h) : static_cast<const void *>(a.x),
                   xbytes, &fullG[lane]);
        } else if (t < tS) {
          const int k0 = 2 * (t - tR);
          const int nrow = cntR - k0 < 2 ? cntR - k0 : 2;
          mbar_arrive_expect_tx(&fullG[lane], (uint32_t)(nrow * rowh));
          for (int rr = 0; rr < nrow; rr++)
            bulk_g2s_pol(dst + rr * rowh, lw.wr + (size_t)(bx + nb * (k0 + rr)) * H, rowh,
                         &fullG[lane], pol_first);
        } else if (t < tG) {
          const int p = bx + nb * (t - tS);
          mbar_arrive_expect_tx(&fullG[lane], (uint32_t)(2 * rowh));
          bulk_g2s_pol(dst, lw.sh_gate + (size_t)p * H, rowh, &fullG[lane], pol_first);
          bulk_g2s_pol(dst + rowh, lw.sh_up + (size_t)p * H, rowh, &fullG[lane], pol_first);
        } else {
          // the item's 8 rows of one matrix per stage (gate, then up): two copies, each
          // one contiguous run of the record
          const int tg = t - tG;
          const int item = bx + nb * (tg >> 1);
          const int j = item / blocks, blk = item % blocks;
          const int r = blk * kFuItemRows;
          const bool up = tg & 1;
          const uint8_t *rec = lw.experts + (long long)sel[j] * lw.stride;
          mbar_arrive_expect_tx(&fullG[lane], gstage);
          bulk_g2s_pol(dst, rec + a.ex.off[up ? 4 : 0] + (size_t)r * rowb, kFuItemRows * rowb,
                       &fullG[lane], pol_first);
          bulk_g2s_pol(dst + kFuItemRows * rowb, rec + a.ex.off[up ? 5 : 1] + (size_t)r * G,
                       kFuItemRows * G, &fullG[lane], pol_first);
        }
        last_g = t;
      }
    }
    // D stages: stage i = (tile n = i / dpt, m = i % dpt): m < hk the routed experts
    // 2m, 2m+1 with their activations, else rows (m - hk) RS .. of the shared expert with
    // its activations.  Stage i goes to worker group i % 2 and to that group's slots in
    // turn (d_slot_of); lane d issues the stages of slot d once the X/R/S/G slots that
    // share its bytes are consumed.  Weights go in flight at once; the activations only
    // once every CTA has written them (dependency 2, polled here).
    // every lane waits for the consumption of its own slot's last stage (a parity wait is
    // only safe on a barrier at most one phase behind: the owner's) and publishes it
    if (lane < NSG) {
      if (!ab && last_g >= 0 && !mbar_wait(&emptyG[lane], (last_g / NSG) & 1)) {
        set_status(a.status, K3MOE_ERR_TIMEOUT);
        ab = true;
      }
      // and landed, before D copies may overwrite the slot's bytes (bounded)
      if (last_g >= 0 && (kMulti || ab)) mbar_wait(&fullG[lane], (last_g / NSG) & 1, 400000000LL);
      __threadfence_block();
      gdone[lane] = 1;
    }
    int iD = lane;  // the first stage of slot `lane`
    if (lane < kFuNSD && !ab && nD > 0) {
      const int g0 = (int)((uint32_t)lane * dslot / gslot);
      int g1 = (int)((((uint32_t)lane + 1u) * dslot - 1u) / gslot);
      g1 = g1 < NSG - 1 ? g1 : NSG - 1;
      for (int gs = g0; gs <= g1 && !ab; gs++) {
        const long long t0 = clock64();
        while (!gdone[gs]) {
          if (clock64() - t0 > kWaitBudget) {
            set_status(a.status, K3MOE_ERR_TIMEOUT);
            ab = true;
            break;
          }
          __nanosleep(32);
        }
      }
      __threadfence_block();
      if (!ab && !mbar_wait(selbar, 0)) {
        set_status(a.status, K3MOE_ERR_TIMEOUT);
        ab = true;
      }
      bool dep2 = false;
      for (; !ab && iD < nD; iD += kFuNSD) {
        const int q = lane, u = iD / kFuNSD;
        if (!mbar_wait(&emptyD[q], (u & 1) ^ 1) ||
            (kMulti && u > 0 && !mbar_wait(&fullD[q], (u & 1) ^ 1))) {
          set_status(a.status, K3MOE_ERR_TIMEOUT);
          ab = true;
          break;
        }
        const int n = iD / dpt, m = iD % dpt;
        const int r0 = (bx + nb * n) * kFuDownRows;
        uint8_t *dst = dslot_ptr(q);
        const bool routed = m < hk;
        const uint32_t wbytes = routed ? 2 * dexp : (uint32_t)(RS * SI * 2);
        const uint32_t abytes = routed ? (uint32_t)(2 * I * 2) : (uint32_t)(SI * 4);
        mbar_arrive_expect_tx(&fullD[q], wbytes + abytes);
        if (routed) {
          for (int e2 = 0; e2 < 2; e2++) {
            const uint8_t *rec = lw.experts + (long long)sel[2 * m + e2] * lw.stride;
            bulk_g2s_pol(dst + e2 * dexp, rec + a.ex.off[2] + (size_t)r0 * rowb2,
                         kFuDownRows * rowb2, &fullD[q], pol_first);
            bulk_g2s_pol(dst + e2 * dexp + kFuDownRows * rowb2,
                         rec + a.ex.off[3] + (size_t)r0 * G2, kFuDownRows * G2, &fullD[q],
                         pol_first);
          }
        } else {
          const int rs0 = r0 + (m - hk) * RS;
          bulk_g2s_pol(dst, lw.sh_down + (size_t)rs0 * SI, wbytes, &fullD[q], pol_first);
        }
        if (!dep2) {
          // (the expiry test waits for one arrival more than there are CTAs, briefly)
          const unsigned need = (unsigned)nb + (a.expire_dep2 ? 1u : 0u);
          if (!wait_count(bar + 1, need, a.expire_dep2 ? kExpireBudget : kWaitBudget)) {
            set_status(a.status, K3MOE_ERR_TIMEOUT);
            *abort_flag = 1;
            __threadfence_block();  // before the copies whose landing the workers wait for
          }
          fence_proxy_async_all();
          dep2 = true;
        }
        if (routed) {
          // experts 2m, 2m+1: I f16 activations each, after the weights
          bulk_g2s(dst + 2 * dexp, a.act + (size_t)(2 * m) * I, (uint32_t)(2 * I * 2),
                   &fullD[q]);
        } else {
          bulk_g2s(dst + wbytes, a.act_s, abytes, &fullD[q]);
        }
      }
    }
    // bounded wait for this lane's last D copy (a worker whose wait expired no longer
    // waits for it, and neither the CTA's exit nor the next layer's barrier set-up may
    // come before it lands); its R/S/G fills have all landed above
    if (lane < kFuNSD && iD - kFuNSD >= 0 && iD - kFuNSD < nD)
      mbar_wait(&fullD[lane], ((iD - kFuNSD) / kFuNSD) & 1, 400000000LL);
    return;
  }

  if (warp == kFuEpi) {
    // ---------------- epilogue: the partial sums of each reduction item ----------------
    int n = 0;
    auto take = [&](int nn) -> const float * {
      const int par = nn & 1;
      if (!mbar_wait(&redbar[par], (nn >> 1) & 1)) {
        set_status(a.status, K3MOE_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      return red + par * (16 * 64);
    };
    auto release = [&](int nn) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&redfree[nn & 1]);
    };
    // R: router rows 2s, 2s+1 of this CTA -> logit (float-float sum of the warps' pairs),
    // collected in lane 2s + r; then every lane's unbiased score (logistic in double,
    // rounded once; the slow double pipe runs once for all rows) and selection score
    float mylogit = 0.f;
    // this lane's router-row bias, fetched now: by the time it is added the stream of
    // weight stages keeps every memory queue long
    const float mybias = (lw.bias && lane < cntR) ? __ldg(lw.bias + bx + nb * lane) : 0.f;
    for (int s = 0; s < nR; s++, n++) {
      const float *rt = take(n);
      float hi = 0.f, lo = 0.f;
      if (lane < 2) {
        for (int w = lane * nwc; w < (lane + 1) * nwc; w++) ff_add(hi, lo, rt[w * 64], rt[w * 64 + 1]);
      }
      release(n);
      const float h0 = __shfl_sync(0xffffffffu, hi, 0), h1 = __shfl_sync(0xffffffffu, hi, 1);
      if (lane == 2 * s) mylogit = h0;
      if (lane == 2 * s + 1) mylogit = h1;
    }
    if (lane < cntR) {
      const int row = bx + nb * lane;
      const float sv = (float)(1.0 / (1.0 + exp(-(double)mylogit)));
      const float cv = __fadd_rn(sv, mybias);
      a.sc[row] = sv;
      a.ch[row] = cv;
      if (!(fabsf(cv) <= 3.402823466e38f)) set_status(a.status, K3MOE_ERR_NONFINITE);
    }
    __syncwarp();  // the lanes' score writes before lane 0's fence, which covers them all
    if (lane == 0) {  // dependency 1: this CTA's router rows are written
      __threadfence();
      atomicAdd(bar, 1u);
    }
    // S: shared pair p -> SiTU(gate, up)
    for (int s = 0; s < nS; s++, n++) {
      const float *rt = take(n);
      float gs = 0.f, us = 0.f;
      if (lane == 0) {
        for (int w = 0; w < nwc; w++) gs += rt[w * 64];
        for (int w = nwc; w < 2 * nwc; w++) us += rt[w * 64];
      }
      release(n);
      if (lane == 0) a.act_s[bx + nb * s] = situ(gs, us, a.b1, a.b2);
    }
    // G: rows of an 8-row block of expert slot j -> SiTU -> f16 at the fixed scale
    // 2^-act_exp (|SiTU| <= b1 b2, so the scaled value stays below 2^15)
    const float inv = pow2i(-a.act_exp);
    for (int s = 0; s < nI; s++, n++) {
      const float *rt = take(n);
      const int item = bx + nb * s;
      const int j = item / blocks, blk = item % blocks;
      const int r = lane & (kFuItemRows - 1), hp = r & 1;
      float gs = 0.f, us = 0.f;
      for (int w = hp * nwc; w < (hp + 1) * nwc; w++) {
        gs += rt[(w * 32 + r) * 2];
        us += rt[(w * 32 + r) * 2 + 1];
      }
      release(n);
      if (lane < kFuItemRows) {
        float act = situ(gs, us, a.b1, a.b2);
        if (*abort_flag) act = 0.f;
        const float sa = act * inv;
        const int row = blk * kFuItemRows + r;
        const size_t o = act_index(j, I, row / kTileRows, row % kTileRows);
        a.act[o] = __half_as_ushort(__float2half_rn(sa));
      }
    }
  } else if (warp < 2 * nwc) {
    // ---------------- consumers: thread (h, g) ----------------
    const int h = tid / G, g = tid % G;
    const int nt = 2 * nwc * 32;  // consumer threads
    int t = 0, n = 0;
    bool aborted = false;
    auto begin_item = [&](int nn) -> float * {
      const int par = nn & 1;
      if (!aborted && !mbar_wait(&redfree[par], ((nn >> 1) & 1) ^ 1)) {
        set_status(a.status, K3MOE_ERR_TIMEOUT);
        aborted = true;
        *abort_flag = 1;
      }
      return red + par * (16 * 64);
    };
    auto stage_in = [&](int tt) -> const uint8_t * {
      const int s = tt % NSG;
      if (!aborted && !mbar_wait(&fullG[s], (tt / NSG) & 1)) {
        set_status(a.status, K3MOE_ERR_TIMEOUT);
        aborted = true;
        *abort_flag = 1;
      }
      return slot_ptr(s);
    };
    auto stage_out = [&](int tt) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&emptyG[tt % NSG]);
    };
    auto end_item = [&](int nn) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&redbar[nn & 1]);  // also when aborted: no one hangs
    };
    // X: MXFP4 rows use input group g (32 inputs prescaled to f16); bf16 rows use the
    // 16-byte chunks g + G c (c < 4) of the row, so a warp reads consecutive chunks
    uint32_t xr[16];
    int xe;
    uint4 xb[4];
    if (a.h == nullptr) {
      const uint4 *xs = reinterpret_cast<const uint4 *>(stage_in(t));
      float v[32];
#pragma unroll
      for (int q = 0; q < 4; q++) {
        const uint4 c = xs[g * 4 + q];
        const uint32_t w4[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int k = 0; k < 4; k++) {
          v[8 * q + 2 * k] = bf16_lo(w4[k]);
          v[8 * q + 2 * k + 1] = bf16_hi(w4[k]);
        }
      }
      xe = prescale_group_f16(v, xr);
#pragma unroll
      for (int c = 0; c < 4; c++) xb[c] = xs[g + G * c];
      stage_out(t);
      t++;
    } else {
      // x = bf16(h * inv), inv = 1 / sqrt(mean(h^2) + eps) (kimi-k3-in-c, section 5): the
      // sum of squares as a float-float sum of exact squares (parity-0 threads cover each
      // input group once; fixed warp and cross-warp order), one double-precision root
      const float *hs = reinterpret_cast<const float *>(stage_in(t));
      float sh = 0.f, sl = 0.f;
      if (h == 0) {
        const float4 *h4 = reinterpret_cast<const float4 *>(hs + g * kGroup);
#pragma unroll
        for (int q = 0; q < 8; q++) {
          const float4 c = h4[q];
          const float e4[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
          for (int k = 0; k < 4; k++) {
            const float p = __fmul_rn(e4[k], e4[k]);
            const float pe = fmaf(e4[k], e4[k], -p);  // exact square = p + pe
            float sx, ex;
            two_sum(sh, p, sx, ex);
            sh = sx;
            sl = __fadd_rn(sl, __fadd_rn(ex, pe));
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float oh = __shfl_xor_sync(0xffffffffu, sh, o);
        const float ol = __shfl_xor_sync(0xffffffffu, sl, o);
        ff_add(sh, sl, oh, ol);
      }
      if (lane == 0) {
        wss[2 * warp] = sh;
        wss[2 * warp + 1] = sl;
      }
      named_bar_sync(kBarCons, nt);
      if (tid == 0) {
        float th = 0.f, tl = 0.f;
        for (int w = 0; w < nwc; w++) ff_add(th, tl, wss[2 * w], wss[2 * w + 1]);
        const double tot = (double)th + (double)tl;
        misc[5] = __float_as_int((float)(1.0 / sqrt(tot / (double)H + (double)a.eps)));
      }
      named_bar_sync(kBarCons, nt);
      const float inv = __int_as_float(misc[5]);
      float v[32];
#pragma unroll
      for (int k = 0; k < 32; k++)
        v[k] = bf16_lo(f32_to_bf16(__fmul_rn(hs[g * kGroup + k], inv)));
      xe = prescale_group_f16(v, xr);
      auto pair = [&](const float *p2) -> uint32_t {
        return (uint32_t)f32_to_bf16(__fmul_rn(p2[0], inv)) |
               ((uint32_t)f32_to_bf16(__fmul_rn(p2[1], inv)) << 16);
      };
#pragma unroll
      for (int c = 0; c < 4; c++) {
        const float *p8 = hs + 8 * (g + G * c);
        xb[c] = make_uint4(pair(p8), pair(p8 + 2), pair(p8 + 4), pair(p8 + 6));
      }
      stage_out(t);
      t++;
    }
    // R: row h of the stage, exact bf16 products summed as a float-float pair
    for (int s = 0; s < nR; s++, t++, n++) {
      float *rt = begin_item(n);
      const uint8_t *st = stage_in(t);
      float hi = 0.f, lo = 0.f;
      if (!aborted && 2 * s + h < cntR) {
        const uint4 *w4 = reinterpret_cast<const uint4 *>(st + h * rowh);
#pragma unroll
        for (int c = 0; c < 4; c++) {
          const uint4 wv = w4[g + G * c];
          const uint32_t wa[4] = {wv.x, wv.y, wv.z, wv.w};
          const uint32_t xa[4] = {xb[c].x, xb[c].y, xb[c].z, xb[c].w};
#pragma unroll
          for (int q = 0; q < 4; q++) {
            float p0, p1, sx, ex;
            mul2_bf16_f32(xa[q], wa[q], p0, p1);  // exact products
            two_sum(hi, p0, sx, ex);
            hi = sx;
            lo = __fadd_rn(lo, ex);
            two_sum(hi, p1, sx, ex);
            hi = sx;
            lo = __fadd_rn(lo, ex);
          }
        }
      }
      stage_out(t);
      {
        const float sx = __fadd_rn(hi, lo);
        lo = __fsub_rn(lo, __fsub_rn(sx, hi));
        hi = sx;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float oh = __shfl_xor_sync(0xffffffffu, hi, o);
        const float ol = __shfl_xor_sync(0xffffffffu, lo, o);
        ff_add(hi, lo, oh, ol);
      }
      if (lane == 0) {
        rt[warp * 64] = hi;
        rt[warp * 64 + 1] = lo;
      }
      end_item(n);
    }
    // S: gate row (h = 0) or up row (h = 1) of shared pair s, fp32 sums of exact products
    for (int s = 0; s < nS; s++, t++, n++) {
      float *rt = begin_item(n);
      const uint8_t *st = stage_in(t);
      float acc = 0.f;
      if (!aborted) {
        const uint4 *w4 = reinterpret_cast<const uint4 *>(st + h * rowh);
#pragma unroll
        for (int c = 0; c < 4; c++) {
          const uint4 wv = w4[g + G * c];
          const uint32_t wa[4] = {wv.x, wv.y, wv.z, wv.w};
          const uint32_t xa[4] = {xb[c].x, xb[c].y, xb[c].z, xb[c].w};
#pragma unroll
          for (int q = 0; q < 4; q++) acc = fma2_bf16_f32(xa[q], wa[q], acc);
        }
      }
      stage_out(t);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) rt[warp * 64] = acc;
      end_item(n);
    }
    // G: an 8-row block = two stages, its gate rows and then its up rows; thread (h, g)
    // takes the rows of parity h in input group g
    constexpr int RH = kFuItemRows / 2;  // rows of one parity in an item
    constexpr int V = 2 * RH;            // (4 rows) x (2 matrices)
    const float pxe = pow2i(xe);  // this thread's inputs are stored times 2^-xe
    for (int s = 0; s < nI; s++, n++) {
      float *rt = begin_item(n);
      float vals[V];
#pragma unroll
      for (int v = 0; v < V; v++) vals[v] = 0.f;
      // both stages of the item first: eight independent dot products per thread
      const uint8_t *stA = stage_in(t);
      const uint8_t *stB = stage_in(t + 1);
#pragma unroll
      for (int m = 0; m < 2; m++) {  // m: the stage's matrix, 0 gate, 1 up
        const uint8_t *st = m ? stB : stA;
        if (!aborted) {
          const uint8_t *ss = st + kFuItemRows * rowb;  // the rows' scale bytes
#pragma unroll
          for (int k = 0; k < RH; k++) {
            const int q = h + 2 * k;  // row within the block
            const uint4 w = reinterpret_cast<const uint4 *>(st + q * rowb)[g];
            vals[m * RH + k] = group_dot(xr, w) * group_scale(ss[q * G + g], pxe);
          }
        }
      }
      stage_out(t);
      stage_out(t + 1);
      t += 2;
      // value v = m * RH + k  ->  block row h + 2k, matrix m
      const float tot = warp_transpose_reduce<V>(vals);
      if (lane < V) {
        const int m = lane / RH, k = lane % RH;
        rt[(warp * 32 + h + 2 * k) * 2 + m] = tot;
      }
      end_item(n);
    }
  } else if (warp == kFuTopk) {
    // ---------------- top-k, once every CTA's router rows are in the workspace ----------
    // (meanwhile the consumers take the S stages; the producer issues G stages once the
    // selection is published)
    // the selection scores come into shared memory in one bulk copy when they fit
    const uint32_t chb = ((uint32_t)E * 4u + 15u) & ~15u;  // the workspace pads them to 16
    const bool bulk = chb <= (uint32_t)kFuSmallBytes;
    bool ok = true;
    if (lane == 0) {
      if (!wait_count(bar, (unsigned)nb)) {
        set_status(a.status, K3MOE_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      if (bulk) {
        fence_proxy_async_all();  // the other CTAs' score writes before the async-proxy read
        mbar_arrive_expect_tx(topbar, chb);
        bulk_g2s(smem + kFuSmall, a.ch, chb, topbar);
      }
    }
    __syncwarp();
    if (bulk && !mbar_wait(topbar, 0)) {
      set_status(a.status, K3MOE_ERR_TIMEOUT);
      *abort_flag = 1;
      ok = false;
      mbar_wait(topbar, 0, 400000000LL);  // bounded wait for the copy still in flight
    }
    int e_sel = 0;
    float w_sel = 0.f;
    if (__all_sync(0xffffffffu, ok)) {
      topk_warp(a.sc, a.ch, bulk ? reinterpret_cast<const float *>(smem + kFuSmall) : nullptr, E,
                K, a.renorm, a.routed_scale, sel, selready, e_sel, w_sel);
    } else {  // after an expiry: expert 0 everywhere, output zero (the abort flag is set)
      if (lane < K) sel[lane] = 0;
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        *selready = K;
      }
    }
    if (lane < K) {
      wsel[lane] = w_sel;
      if (bx == 0 && lw.idx_out) {
        lw.idx_out[lane] = e_sel;
        lw.w_out[lane] = w_sel;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(selbar);
  }

  // ---------------- dependency 2: this CTA's activations are written ----------------
  // (the producer waits for every CTA's before it copies activations into D stages)
  constexpr int NDT = kFuWorkers * 32;  // worker threads
  fence_proxy_async_all();              // generic writes before the bulk copies that read them
  named_bar_sync(kBarDown, NDT);
  if (tid == 0) {
    __threadfence();
    atomicAdd(bar + 1, 1u);
  }

  // ---------------- D: down rows, shared down rows, router-order combine ----------------
  // worker group gD (eight warps) takes the D stages i with i % 2 == gD; warp wg of the
  // group takes expert wg / 4 of a routed stage, rows 4 (wg % 4) .. + 4
  const int gD = warp >> 3, wg = warp & 7;
  bool aborted = *abort_flag != 0;
  const int NG = G2 / 16;                   // groups per lane
  const int rp = lane >> 4, l = lane & 15;  // row pair, group lane
  const float pe2 = pow2i(a.act_exp);  // activations are stored times 2^-act_exp
  for (int n = 0; n < nT; n++) {
    const int r0 = (bx + nb * n) * kFuDownRows;
    for (int i = tid; i < (K + 1) * kFuDownRows; i += NDT) dbuf[i] = 0.f;  // dbuf and ds
    named_bar_sync(kBarDown, NDT);
    for (int m = 0; m < dpt; m++) {
      const int i = n * dpt + m;
      if ((i & 1) != gD) continue;
      const int q = d_slot_of(i);
      if (!aborted && !mbar_wait(&fullD[q], (i / kFuNSD) & 1)) {
        set_status(a.status, K3MOE_ERR_TIMEOUT);
        aborted = true;
      }
      const uint8_t *st = dslot_ptr(q);
      if (!aborted && m < hk) {
        // expert slot j = 2m + wg/4; each lane: rows rb + 2 rp, +1 over NG input groups
        const int ex = wg >> 2, j = 2 * m + ex, rb = (wg & 3) * 4 + rp * 2;
        const uint8_t *sp = st + ex * dexp;
        const uint8_t *ss = sp + kFuDownRows * rowb2;
        const uint16_t *s_act = reinterpret_cast<const uint16_t *>(st + 2 * dexp + ex * (I * 2));
        float acc[2] = {0.f, 0.f};
        for (int qq = 0; qq < NG; qq++) {
          // the 16 group lanes read 16 consecutive 16-byte weight chunks of a row
          const int gg = qq * 16 + l;
          uint32_t xa[16];
          const uint4 *pa = reinterpret_cast<const uint4 *>(s_act + act_index(0, I, gg, 0));
#pragma unroll
          for (int c = 0; c < 4; c++) {
            const uint4 x0 = pa[c * G2];
            xa[4 * c] = x0.x; xa[4 * c + 1] = x0.y; xa[4 * c + 2] = x0.z; xa[4 * c + 3] = x0.w;
          }
#pragma unroll
          for (int r = 0; r < 2; r++) {
            const int row = rb + r;
            const uint4 wv = reinterpret_cast<const uint4 *>(sp + row * rowb2)[gg];
            const uint32_t sv = ss[row * G2 + gg];
            acc[r] += group_dot(xa, wv) * group_scale(sv, pe2);
          }
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) {
          acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], o);
          acc[1] += __shfl_xor_sync(0xffffffffu, acc[1], o);
        }
        if (l == 0) {
          dbuf[j * kFuDownRows + rb] = acc[0];
          dbuf[j * kFuDownRows + rb + 1] = acc[1];
        }
      } else if (!aborted) {
        // shared expert: row wg of this stage; bf16 weights, fp32 inputs
        const int nch = SI >> 3;
        for (int rr = wg; rr < RS; rr += 8) {
          const uint4 *w4 = reinterpret_cast<const uint4 *>(st + (size_t)rr * SI * 2);
          const float4 *a4 = reinterpret_cast<const float4 *>(st + RS * SI * 2);
          float sacc = 0.f;
          for (int c = lane; c < nch; c += 32) {
            const uint4 wv = w4[c];
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
          if (lane == 0) ds[(m - hk) * RS + rr] = sacc;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&emptyD[q]);
    }
    if (aborted) *abort_flag = 1;
    named_bar_sync(kBarDown, NDT);
    if (tid < kFuDownRows) {
      const int row = tid;
      float sum = 0.f;
      for (int j = 0; j < K; j++)
        sum = __fadd_rn(sum, __fmul_rn(wsel[j], dbuf[j * kFuDownRows + row]));
      if (SI > 0) sum = __fadd_rn(sum, ds[row]);  // the shared expert, unweighted, last
      if (*abort_flag) sum = 0.f;
      const size_t o = (size_t)r0 + row;
      if (a.ydt == K3MOE_F32) {
        float *yf = reinterpret_cast<float *>(a.y);
        yf[o] = a.accumulate ? __fadd_rn(yf[o], sum) : sum;
      } else {
        uint16_t *yb = reinterpret_cast<uint16_t *>(a.y);
        const float vv = a.accumulate ? __fadd_rn(bf16_lo(yb[o]), sum) : sum;
        yb[o] = f32_to_bf16(vv);
      }
    }
    named_bar_sync(kBarDown, NDT);
  }
  // exit of the layer: its tiles of y (or of the residual stream) are written; the next
  // layer's input stage waits for every CTA's exit.  After the last layer every use of the
  // counters is over (a CTA reads them only before its own exit), so the last CTA to get
  // here leaves all of them zero for the next call.
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(bar + 2, 1u) == (unsigned)nb - 1 && layer == a.L - 1) {
      for (int k = 0; k < 4 * a.L; k++) a.bar[k] = 0u;
      __threadfence();
    }
  }
}

template <bool kMulti>
__global__ void __launch_bounds__(kFuThreads, 1) k_decode_fused(FusedT1Args a) {
  extern __shared__ __align__(128) uint8_t smem[];
  if (!kMulti) {
    fused_layer<false>(a, 0, smem);
    return;
  }
  for (int l = 0; l < a.L; l++) {
    if (l > 0) __syncthreads();  // every role of the CTA is done with layer l - 1
    fused_layer<true>(a, l, smem);
  }
}

size_t fused_t1_smem(int H, int I, int E, int K, int SI, int grid) {
  const int G = H / kGroup, G2 = I / kGroup;
  if (H % 1024 != 0 || G / 32 < 1 || G / 32 > 7) return 0;  // 2 G/32 consumer warps <= 14
  if (I % 512 != 0 || G2 / 16 > 8) return 0;               // 16 group lanes, <= 8 groups each
  if (K < 2 || K > 16 || K % 2 != 0) return 0;             // two experts per down stage
  if (SI < 0 || SI % 256 != 0) return 0;                   // shared rows in 32 lanes x 8
  if (grid < 1) return 0;
  if ((E + grid - 1) / grid > 32) return 0;  // R rows of a CTA: one epilogue lane each
  if (fused_nsg(H) < 2) return 0;
  const size_t total = (size_t)kFuRing + fused_ring_bytes(H, I, SI) + kFuRedBytes;
  return total <= kFuSmemMax ? total : 0;
}

cudaError_t set_fused_smem_limit() {
  cudaError_t e = cudaFuncSetAttribute(k_decode_fused<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k_decode_fused<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              227 * 1024);
}

// Cooperative launch: the runtime refuses it unless every CTA can be resident at once,
// which the grid-wide dependencies need.
cudaError_t launch_fused_t1(const FusedT1Args &a, int grid, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kFuThreads);
  cfg.dynamicSmemBytes = fused_t1_smem(a.H, a.I, a.E, a.K, a.SI, grid);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return a.L > 1 ? cudaLaunchKernelEx(&cfg, k_decode_fused<true>, a)
                 : cudaLaunchKernelEx(&cfg, k_decode_fused<false>, a);
}

}  // namespace k3

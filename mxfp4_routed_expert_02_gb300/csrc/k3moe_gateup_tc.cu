// k3moe_gateup_tc.cu -- gate/up + SiTU for ONE token on the 5th-generation tensor cores
// (tcgen05, block-scaled MXFP4).  The experts' gate and up operands stream in 128-row x
// 128-byte boxes straight from the records into the MMAs, with no E2M1 conversion on the
// CUDA cores; the token's input sits in shared memory as kTcTermsX MXFP4 terms (the B
// operand); the accumulators and the scale vectors live in tensor memory.
//
// What it computes is k_gateup_t1's (README of FareedKhan-dev/kimi-k3-in-c, section 9
// "Picking 16 experts of 896" for the top-k and the LatentMoE listing step 3 for the expert
// FFN, section 4 for MXFP4, the activation listing for SiTU), with the same outputs: the
// route and the dispatch lists (CTA 0), and the activations of the K (token, slot) pairs
// as f16 hi + lo terms with one exponent per 32 rows (k_down_tma reads both terms,
// k_down_t1 the hi term alone).  The
// input enters as four MXFP4 terms per 32 values (the multi-token path's encoding), so
// the products differ from k_gateup_t1's f16 ones by a relative ~4e-5.
//
// Work: the K x (I / 128) row tiles, each over H / 256 chunks of 128 bytes of K.  The
// (tile, chunk) steps in tile order are cut into one contiguous run per CTA, so a tile is
// done by one CTA or split between two; the CTA whose run ends inside a tile finishes it
// once the next CTA's part of it is in (a counter per tile in the workspace header), adding
// the parts in CTA order.
// Warps: 0-3 place each stage's scale vectors in tensor memory (warp q owns TMEM lanes
// 32q .. 32q + 31), 4-7 drain the accumulators (SiTU, activations), 8 issues the MMAs (and
// holds the TMEM allocation), 9 issues the TMA copies; warps 0-7 first encode the input.
// Every wait is bounded: on expiry the kernel reports K3MOE_ERR_TIMEOUT, keeps arriving
// on what it owes, writes zero activations and leaves the counters zero.
#include "k3moe_tcgen05.cuh"

namespace k3 {

namespace {

constexpr int kT1Warps = 10;
constexpr int kT1Threads = 32 * kT1Warps;
constexpr int kT1WarpEpi = 4;                 // warps 4..7
constexpr int kT1WarpMma = 8;
constexpr int kT1WarpTma = 9;
constexpr int kT1N = 16;                      // MMA columns: the term rows, then unused rows
constexpr uint32_t kT1A = 2 * kTcBox;         // gate + up boxes of a stage
constexpr uint32_t kT1Sf = 2 * kTcTile * 16;  // their scale words: chunks (c & ~1, c | 1)
constexpr uint32_t kT1Stage = kT1A + kT1Sf;   // 36 KB (a 1 KB multiple)
constexpr int kT1AccCols = 2 * 2 * kT1N;      // two buffers of (gate, up) accumulators
constexpr int kT1SfSlot = 3 * kSfW;           // scale columns per ring slot: B, gate, up
constexpr int kT1TmemCols = 512;
constexpr int kT1MaxNS = 8;
constexpr int kBarT1Epi = 1;                  // named barrier of the four epilogue warps
// the first 1 KB of shared memory: barriers, then small arrays
constexpr int kT1Bars = 0;     // full[8] empty[8] sfull[8] dfull[2] dempty[2] bready
constexpr int kT1Tmem = 256;   // u32: TMEM base address
constexpr int kT1Abort = 260;  // int
constexpr int kT1Sel = 384;    // int[32]
constexpr int kT1Wsel = 512;   // float[32]
constexpr int kT1Small = 1024;

__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// Bounded wait until a counter in global memory reaches n (acquire).
__device__ bool t1_wait_count(const unsigned *cnt, unsigned n) {
  const long long t0 = clock64();
  while (true) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
    if (v >= n) return true;
    if (clock64() - t0 > kWaitBudget) return false;
    __nanosleep(64);
  }
}

}  // namespace

// Shared-memory map (from a 1 KB-aligned base): [small | top-k scratch | B image | B scale
// bytes | ring].  The B image holds one 8-row x 128-byte swizzle atom per 128 bytes of K
// (rows 0..3 the input's terms, 4..7 zero) and a spare zero atom, which the unused MMA
// rows 8..15 of the last chunk read.
__host__ __device__ inline uint32_t t1_scratch_bytes(int E, int K) {
  return ((uint32_t)topk_scratch_keys(E, K) * 8u + 1023u) & ~1023u;
}
__host__ __device__ inline uint32_t t1_bimg_bytes(int H) { return (uint32_t)(H / 256 + 1) * 1024u; }
__host__ __device__ inline uint32_t t1_bsf_bytes(int H) {
  return ((uint32_t)(kTcTermsX * (H / kGroup)) + 1023u) & ~1023u;
}
__host__ __device__ inline uint32_t t1_fixed_bytes(int H, int E, int K) {
  return kT1Small + t1_scratch_bytes(E, K) + t1_bimg_bytes(H) + t1_bsf_bytes(H);
}
// The CTA whose run [S b / nb, S (b + 1) / nb) holds step `step`.
__host__ __device__ inline int t1_cta_of(int S, int nb, int step) {
  int b = (int)((long long)step * nb / S);
  if (b > nb - 1) b = nb - 1;
  while (b < nb - 1 && (int)((long long)S * (b + 1) / nb) <= step) b++;
  while (b > 0 && (int)((long long)S * b / nb) > step) b--;
  return b;
}

// Input group g (32 values of x, bf16 or float) as kTcTermsX MXFP4 terms: term t is row t
// of the swizzle atom of its 128-byte K chunk (16-byte unit u of row r at unit u ^ r, the
// 128-byte swizzle), rows 4..7 zero; the terms' scale bytes go to bsf[t][g].
template <bool XF32>
__device__ __forceinline__ void t1_encode_group(const GateUpT1Args &g, int gi, int G,
                                                uint8_t *bimg, uint8_t *bsf) {
  float r[32];
  if (XF32) {
    const float4 *src = reinterpret_cast<const float4 *>(g.xf + (size_t)gi * kGroup);
#pragma unroll
    for (int q = 0; q < 8; q++) {
      const float4 c = __ldg(src + q);
      r[4 * q] = c.x;
      r[4 * q + 1] = c.y;
      r[4 * q + 2] = c.z;
      r[4 * q + 3] = c.w;
    }
  } else {
    const uint4 *src = reinterpret_cast<const uint4 *>(g.x + (size_t)gi * kGroup);
#pragma unroll
    for (int q = 0; q < 4; q++) {
      const uint4 c = __ldg(src + q);
      const uint32_t w4[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
      for (int k = 0; k < 4; k++) {
        r[8 * q + 2 * k] = bf16_lo(w4[k]);
        r[8 * q + 2 * k + 1] = bf16_hi(w4[k]);
      }
    }
  }
  uint4 q4[kTcTermsX];
  uint8_t sb[kTcTermsX];
  encode_terms<kTcTermsX>(r, q4, sb);
  const int u = gi & 7;
  uint8_t *atom = bimg + (size_t)(gi >> 3) * 1024;
#pragma unroll
  for (int t = 0; t < 8; t++)
    *reinterpret_cast<uint4 *>(atom + 128 * t + 16 * (u ^ t)) =
        t < kTcTermsX ? q4[t < kTcTermsX ? t : 0] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
  for (int t = 0; t < kTcTermsX; t++) bsf[t * G + gi] = sb[t];
}

template <bool XF32>
__global__ void __launch_bounds__(kT1Threads, 1)
    k_gateup_tc1(const GateUpTc1Args a, const __grid_constant__ CUtensorMap tmw,
                 const __grid_constant__ CUtensorMap tms) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const GateUpT1Args &g = a.g;
  const int H = g.H, I = g.I, K = g.K, E = g.E;
  const int G = H / kGroup, CH = H / 256, MT = I / kTcTile;
  const int NS = a.NS;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + kT1Bars);  // [8] a stage landed
  uint64_t *empty = full + 8;    // [8] a stage's MMAs done (ring slot and scale columns free)
  uint64_t *sfull = full + 16;   // [8] a stage's scale vectors in tensor memory
  uint64_t *dfull = full + 24;   // [2] accumulator buffer complete
  uint64_t *dempty = full + 26;  // [2] accumulator buffer drained
  uint64_t *bready = full + 28;  // the B image and its scale bytes written
  uint32_t *tmem_base = reinterpret_cast<uint32_t *>(smem + kT1Tmem);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kT1Abort);
  int *sel = reinterpret_cast<int *>(smem + kT1Sel);
  float *wsel = reinterpret_cast<float *>(smem + kT1Wsel);
  unsigned long long *cand = reinterpret_cast<unsigned long long *>(smem + kT1Small);
  uint8_t *bimg = smem + kT1Small + t1_scratch_bytes(E, K);
  uint8_t *bsf = bimg + t1_bimg_bytes(H);
  uint8_t *ring = bsf + t1_bsf_bytes(H);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bx = blockIdx.x, nb = gridDim.x;

  if (tid == 0) {
    for (int s = 0; s < NS; s++) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&sfull[s], 4);
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(&dfull[b], 1);
      mbar_init(&dempty[b], 4);
    }
    mbar_init(bready, 8);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kT1WarpMma) tmem_alloc(tmem_base, kT1TmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tmem_base;
  pdl_wait();

  // the route, recomputed by every CTA from the router's scores (a few microseconds)
  cta_topk(g.sc, g.ch, E, K, g.renorm, g.routed_scale, cand, sel, wsel);
  if (bx == 0) {
    if (tid < K) {
      g.idx_out[tid] = sel[tid];
      g.w_out[tid] = wsel[tid];
      int *uexp = g.disp + 4;
      int *uoff = uexp + K;
      int *plist = uoff + K + 1;
      uexp[tid] = sel[tid];
      uoff[tid] = tid;
      plist[tid] = tid;
    }
    if (tid == 0) {
      g.disp[0] = K;
      g.disp[4 + K + K] = K;  // uoff[U] = number of pairs
    }
  }
  pdl_launch_dependents();

  // this CTA's run of (tile, chunk) steps; step k -> tile, chunk
  const int S = K * MT * CH;
  const int r0 = (int)((long long)S * bx / nb);
  const int nG = (int)((long long)S * (bx + 1) / nb) - r0;
  auto same_tile = [&](int k0, int k1) -> bool { return (r0 + k0) / CH == (r0 + k1) / CH; };

  if (warp == kT1WarpTma) {
    // ---------------- TMA: lane p < NS owns ring slot p (stages p, p + NS, ...) ----------
    if (lane < NS) {
      uint64_t pol;  // the weights are read once: first out of L2
      asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
      bool ok = true;
      int k = lane;
      for (; k < nG; k += NS) {
        const int u = k / NS;
        if (u > 0 && !mbar_wait(&empty[lane], (u - 1) & 1)) {
          set_status(g.status, K3MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          ok = false;
          break;
        }
        const int st = r0 + k, tile = st / CH, c = st % CH;
        const int e = sel[tile / MT], mt = tile % MT;
        uint8_t *dst = ring + (size_t)lane * kT1Stage;
        mbar_arrive_expect_tx(&full[lane], kT1Stage);
        tma_load4d_pol(dst, &tmw, c * kTcChunkBytes, mt * kTcTile, 0, e, &full[lane], pol);
        tma_load4d(dst + kT1A, &tms, c & ~1, mt * kTcTile, 0, e, &full[lane]);
      }
      // a fill no MMA will consume (after an expiry) lands before the CTA exits (bounded)
      if (!ok && k - NS >= 0) mbar_wait(&full[lane], ((k - NS) / NS) & 1, 400000000LL);
    }
  } else {
    if (warp < 8) {
      // ---------------- the input's terms (warps 0..7, one group per thread) -------------
      for (int gi = tid; gi < G; gi += 256) t1_encode_group<XF32>(g, gi, G, bimg, bsf);
      if (tid < 64) *reinterpret_cast<uint4 *>(bimg + (size_t)CH * 1024 + 16 * tid) =
          make_uint4(0u, 0u, 0u, 0u);  // the spare atom
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // before the MMAs read
      __syncwarp();
      if (lane == 0) mbar_arrive(bready);
    }
    bool aborted = false;
    if (warp < 4) {
      // ---------------- scale writers ----------------
      // A: K step i of matrix m reads column slot + kSfW (1 + m) + 4i + (row / 32); scale
      // byte 255 (no contribution) becomes 0.  B: K step i of row n reads column slot + 4i
      // + n / 32 at lane n % 32 of every lane quarter; rows n < 4 are the terms.
      const int q = warp;
      const uint32_t lane_sel = (uint32_t)(32 * q) << 16;
      if (nG > 0 && !mbar_wait(bready, 0)) {
        set_status(g.status, K3MOE_ERR_TIMEOUT);
        aborted = true;
        *abort_flag = 1;
      }
      for (int k = 0; k < nG; k++) {
        const int s = k % NS, u = k / NS;
        if (!aborted && (!mbar_wait(&full[s], u & 1) || !mbar_wait(&empty[s], (u & 1) ^ 1))) {
          set_status(g.status, K3MOE_ERR_TIMEOUT);
          aborted = true;
          *abort_flag = 1;
        }
        tc_fence_after();
        if (!aborted) {
          const int c = (r0 + k) % CH;
          const uint8_t *sfs = ring + (size_t)s * kT1Stage + kT1A;
          const uint32_t col = tm + (uint32_t)(kT1AccCols + s * kT1SfSlot);
          const int r = 32 * q + lane;
#pragma unroll
          for (int m = 0; m < 2; m++) {
            uint2 v = *reinterpret_cast<const uint2 *>(sfs + m * (kTcTile * 16) + r * 16 +
                                                       (c & 1) * 8);
            v.x &= ~__vcmpeq4(v.x, 0xffffffffu);
            v.y &= ~__vcmpeq4(v.y, 0xffffffffu);
#pragma unroll
            for (int i = 0; i < kTcSteps; i++)
              tmem_st_x1(col + lane_sel + kSfW * (1 + m) + 4 * i + q, step_scales(v, i));
          }
          uint32_t vb[kSfW];
#pragma unroll
          for (int i = 0; i < kSfW; i++) vb[i] = 0u;
          if (lane < kTcTermsX) {
            const uint2 v = *reinterpret_cast<const uint2 *>(bsf + lane * G + 8 * c);
#pragma unroll
            for (int i = 0; i < kTcSteps; i++) vb[4 * i] = step_scales(v, i);
          }
          tmem_st_sf(col + lane_sel, vb);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfull[s]);
      }
    } else if (warp < 8) {
      // ---------------- epilogue ----------------
      // warp q drains rows 32q .. 32q + 31 of each tile segment (the sum of the four term
      // columns of gate and of up), then SiTU and the activations of that 32-row group
      const int q = warp & 3;
      const uint32_t lane_sel = (uint32_t)(32 * q) << 16;
      const int rt = 32 * q + lane;
      int sg = 0;
      for (int k = 0; k < nG; sg++) {
        int ke = k + 1;
        while (ke < nG && same_tile(ke - 1, ke)) ke++;
        const int tile = (r0 + k) / CH, j = tile / MT, mt = tile % MT;
        const int db = sg & 1;
        bool got = false;
        if (!aborted) {
          got = mbar_wait(&dfull[db], (sg >> 1) & 1);
          if (!got) {
            set_status(g.status, K3MOE_ERR_TIMEOUT);
            aborted = true;
            *abort_flag = 1;
          }
        }
        tc_fence_after();
        float gsum = 0.f, usum = 0.f;
        if (got) {
          uint32_t dg[4], du[4];
          const uint32_t d0 = tm + lane_sel + (uint32_t)(db * 2 * kT1N);
          tmem_ld4_nowait(d0, dg);
          tmem_ld4_nowait(d0 + kT1N, du);
          tmem_wait_ld4(dg, du);
          gsum = (__uint_as_float(dg[0]) + __uint_as_float(dg[1])) +
                 (__uint_as_float(dg[2]) + __uint_as_float(dg[3]));
          usum = (__uint_as_float(du[0]) + __uint_as_float(du[1])) +
                 (__uint_as_float(du[2]) + __uint_as_float(du[3]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&dempty[db]);
        const int first = t1_cta_of(S, nb, tile * CH);
        const int np = t1_cta_of(S, nb, tile * CH + CH - 1) - first + 1;
        const int piece = bx - first;
        bool mine = true;
        if (np > 1 && piece > 0) {
          // the start of this CTA's run: published for the CTA that ends its run here
          float *pp = a.gpart + ((size_t)tile * kTc1Pieces + piece) * 256;
          pp[rt] = gsum;
          pp[128 + rt] = usum;
          __threadfence();
          named_bar_sync(kBarT1Epi, 128);
          if (warp == kT1WarpEpi && lane == 0) atomicAdd(a.cnt + 1 + tile, 1u);
          mine = false;
        } else if (np > 1) {
          // the finisher: once the other parts are in (bounded wait), they are added after
          // its own, in piece order
          if (warp == kT1WarpEpi && lane == 0) {
            if (!t1_wait_count(a.cnt + 1 + tile, (unsigned)(np - 1))) {
              set_status(g.status, K3MOE_ERR_TIMEOUT);
              *abort_flag = 1;
            }
            a.cnt[1 + tile] = 0u;  // no other arrival this call: zero for the next one
          }
          named_bar_sync(kBarT1Epi, 128);
          for (int pc = 1; pc < np; pc++) {
            const float *qq = a.gpart + ((size_t)tile * kTc1Pieces + pc) * 256;
            gsum += __ldcg(qq + rt);
            usum += __ldcg(qq + 128 + rt);
          }
        }
        if (mine) {
          // SiTU, then f16 hi + lo at one power-of-two scale per 32-row group
          float act = situ(gsum, usum, g.b1, g.b2);
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
          const int t32 = mt * (kTcTile / kTileRows) + q;  // this warp's 32-row group
          const size_t o = act_index(j, I, t32, lane);
          g.act_hi[o] = __half_as_ushort(hh);
          g.act_lo[o] = __half_as_ushort(hl);
          if (lane == 0) g.act_ex[(size_t)j * (I / kGroup) + t32] = e2;
        }
        k = ke;
      }
    } else if (warp == kT1WarpMma) {
      // ---------------- MMA issue ----------------
      // per tile segment, every stage's 4 K steps x (gate, up) block-scaled MMAs of N = 16
      // into the segment's accumulator buffer; the stage's commit frees its slot and scale
      // columns, the segment's commit hands the buffer to the epilogue
      const uint32_t idesc = (1u << 7) | (1u << 10) | ((uint32_t)(kT1N >> 3) << 17) |
                             (1u << 23) | ((uint32_t)(kTcTile >> 4) << 24);
      bool ok = __all_sync(0xffffffffu, nG == 0 || mbar_wait(bready, 0));
      uint64_t *lastbar = nullptr;
      uint32_t lastpar = 0;
      int sg = 0;
      for (int k = 0; k < nG && ok; sg++) {
        int ke = k + 1;
        while (ke < nG && same_tile(ke - 1, ke)) ke++;
        const int db = sg & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&dempty[db], ((sg >> 1) & 1) ^ 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dg = tm + (uint32_t)(db * 2 * kT1N), du = dg + kT1N;
        for (int kk = k; kk < ke; kk++) {
          const int s = kk % NS, u = kk / NS;
          const bool got = mbar_wait(&full[s], u & 1) && mbar_wait(&sfull[s], u & 1);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int c = (r0 + kk) % CH;
          const uint32_t alo = sw_desc_lo(smem_u32(ring + (size_t)s * kT1Stage));
          const uint32_t blo = sw_desc_lo(smem_u32(bimg + (size_t)c * 1024));
          const uint32_t col = tm + (uint32_t)(kT1AccCols + s * kT1SfSlot);
#pragma unroll
          for (int i = 0; i < kTcSteps; i++) {
            const uint32_t acc = (kk == k && i == 0) ? 0u : 1u;
            mma_mxf4_el_lo(dg, alo + (uint32_t)((32 * i) >> 4), blo + (uint32_t)(2 * i),
                           kDescHi, idesc, col + kSfW + 4 * i, col + 4 * i, acc);
            mma_mxf4_el_lo(du, alo + (uint32_t)((kTcBox + 32 * i) >> 4), blo + (uint32_t)(2 * i),
                           kDescHi, idesc, col + 2 * kSfW + 4 * i, col + 4 * i, acc);
          }
          tc_commit_el(&empty[s]);
          lastbar = &empty[s];
          lastpar = (uint32_t)(u & 1);
        }
        if (!ok) break;
        tc_commit_el(&dfull[db]);
        lastbar = &dfull[db];
        lastpar = (uint32_t)((sg >> 1) & 1);
        k = ke;
      }
      if (!ok && lane == 0) {
        set_status(g.status, K3MOE_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      // every MMA issued is done before the tensor memory is freed (bounded)
      if (lastbar) mbar_wait(lastbar, lastpar, 400000000LL);
      __syncwarp();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kT1WarpMma) tmem_dealloc(tm, kT1TmemCols);
  // exit: the last CTA leaves every tile counter zero (they are zero already unless a wait
  // expired), and the exit counter
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(a.cnt, 1u) == (unsigned)nb - 1) {
      for (int t = 0; t < K * MT; t++) a.cnt[1 + t] = 0u;
      a.cnt[0] = 0u;
      __threadfence();
    }
  }
}

size_t gateup_tc1_smem(int H, int I, int E, int K, int grid, int *ns_out) {
  if (H % 512 != 0 || H / kGroup > 256 || I % kTcTile != 0 || K < 1 || K > 32 || grid < 1)
    return 0;
  const int CH = H / 256, MT = I / kTcTile;
  if (K * MT > kTc1MaxTiles) return 0;
  const int S = K * MT * CH;
  for (int t = 0; t < K * MT; t++) {  // the parts of every tile
    const int np = t1_cta_of(S, grid, t * CH + CH - 1) - t1_cta_of(S, grid, t * CH) + 1;
    if (np > kTc1Pieces) return 0;
  }
  const size_t budget = 227 * 1024 - 1024 - t1_fixed_bytes(H, E, K);
  int ns = (int)(budget / kT1Stage);
  if (ns > kT1MaxNS) ns = kT1MaxNS;
  if (ns < 3 || kT1AccCols + ns * kT1SfSlot > kT1TmemCols) return 0;
  if (ns_out) *ns_out = ns;
  return 1024 + t1_fixed_bytes(H, E, K) + (size_t)ns * kT1Stage;
}

cudaError_t set_gateup_tc1_smem_limit() {
  cudaError_t e = cudaFuncSetAttribute(k_gateup_tc1<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k_gateup_tc1<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              227 * 1024);
}

cudaError_t launch_gateup_tc1(const GateUpTc1Args &a, const CUtensorMap &tmw,
                              const CUtensorMap &tms, int grid, cudaStream_t st, bool pdl) {
  int ns = 0;
  const size_t smem = gateup_tc1_smem(a.g.H, a.g.I, a.g.E, a.g.K, grid, &ns);
  if (smem == 0 || ns != a.NS) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kT1Threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return a.g.xf ? cudaLaunchKernelEx(&cfg, k_gateup_tc1<true>, a, tmw, tms)
                : cudaLaunchKernelEx(&cfg, k_gateup_tc1<false>, a, tmw, tms);
}

}  // namespace k3

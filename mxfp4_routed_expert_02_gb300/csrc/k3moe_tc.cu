// k3moe_tc.cu -- grouped GEMM on the 5th-generation tensor cores (tcgen05) for the
// multi-token expert path (prefill and batched decode).
//
// What it computes (README of FareedKhan-dev/kimi-k3-in-c, section 4 for MXFP4 and
// section 9, LatentMoE listing, for the expert FFN): for every group g (a routed expert,
// or the shared expert) and every B row n routed to it,
//     D[m][n] = sum_k A_g[m][k] * B[n][k]        (m: output feature, k: input feature)
// with A_g the expert's weight matrix (rows = outputs, K-major) and B the activations of
// the group's tokens.  Two kinds:
//   MXF4: A is the expert's packed MXFP4 operand as stored in the record (E2M1 nibbles,
//         one E8M0 scale per 32 along K) and B is the activation written as a sum of
//         NT MXFP4 terms (each E2M1 with its own E8M0 scale per 32; 4 for x and for the
//         activations, relative error ~4e-5 and ~3e-4 of a row's product); every term is one
//         block-scaled MMA (kind::mxf4, scale vectors of 2 per 64-wide K step), all
//         accumulated in one fp32 accumulator.  Scale byte 255 of A (the page's "no
//         contribution") is written to tensor memory as 0, i.e. 2^-127.
//   F16:  A and B bf16 (kind::f16, fp32 accumulate); B may be NT bf16 terms (hi + lo).
// Epilogues: SITU (two A matrices, gate and up: act = SiTU(D_gate, D_up)) or STORE
// (D as is; with two A matrices they are two consecutive 128-row tiles of one matrix,
// which then share every B stage); both write fp32 [B row][feature].
//
// Design: one CTA per SM (persistent), work item = (group, 128- or 256-row tile of A, tile
// of up to 128 B rows).  Warp roles: 0-3 write the scale vectors of each stage into tensor
// memory (warp q owns TMEM lanes 32q..32q+31; A row m's scales sit in lane m, B's are
// replicated in every lane quarter, column n / 32, lane n % 32), 4 issues TMA loads
// (swizzled tiles of 128 rows x kTcChunk bytes of K; 128-byte chunks: 64-byte ones would fit
// twice as many stages but measured 1.6-1.7x slower, each row segment then being half a
// 128-byte line), 5 issues the MMAs (one thread), 6-13 drain the
// accumulator (two warps per lane quarter).  Shared-memory stages and the scale slots in
// tensor memory are released together by tcgen05.commit on the stage's "empty" barrier.
#include <cuda.h>

#include "k3moe_tcgen05.cuh"

namespace k3 {

namespace {

constexpr int kTcThreads = 448;           // 14 warps
constexpr int kTcWarpSf = 0;              // warps 0..3
constexpr int kTcWarpTma = 4;
constexpr int kTcWarpMma = 5;
constexpr int kTcWarpEpi = 6;             // warps 6..13
constexpr int kTcTmemCols = 512;
constexpr int kTcItemTable = 512;         // per-CTA work items kept in shared memory
constexpr uint32_t kTcItemTableBytes = kTcItemTable * 16;

}  // namespace

struct TcItem {
  int g, mt, brow0, nvalid;
};

// Maps a flat item index to (group, A-row tile, first B row, valid B rows).
__device__ __forceinline__ TcItem tc_item(const TcGemmArgs &a, int item) {
  TcItem it;
  const int tile = item / a.mtiles;
  it.mt = item - tile * a.mtiles;
  int lo = 0, hi = a.ngroups - 1;  // last group with tile_off[g] <= tile
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.tile_off[mid] <= tile)
      lo = mid;
    else
      hi = mid - 1;
  }
  it.g = lo;
  const int nt = tile - a.tile_off[lo];
  it.brow0 = a.off[lo] + nt * a.ntile;
  const int rem = a.off[lo + 1] - it.brow0;
  it.nvalid = rem < a.ntile ? rem : a.ntile;
  return it;
}

// Non-blocking test of an mbarrier phase (unlike try_wait, never suspends the thread).
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, "
      "p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Copies kSfB bytes (both addresses kSfB-aligned).
__device__ __forceinline__ void cp_async_sf(void *dst, const void *src) {
  if (kSfB == 8)
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}
// Arrives on `bar` once every cp.async this thread issued so far has landed.
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Shared memory after the 1 KB header: NS data stages [A_0 .. A_{NA-1}: 128 rows x kTcChunk]
// [B_0 .. B_{NT-1}: ntile rows x kTcChunk] (1 KB aligned), then NSF scale slots [A scales:
// NA x 128 rows x kSfB][B scales: NT x ntile rows x kSfB].
__host__ __device__ inline uint32_t tc_stage_bytes(int na, int nt, int ntile) {
  const uint32_t b = (uint32_t)na * kTcBox + (uint32_t)nt * ntile * kTcChunkBytes;
  return (b + 1023u) & ~1023u;
}
__host__ __device__ inline uint32_t tc_sf_bytes(int na, int nt, int ntile) {
  return ((uint32_t)na * kTcTile * kSfB + (uint32_t)nt * ntile * kSfB + 15u) & ~15u;
}

// SiTU-GLU in the tensor-core epilogue: b1 tanh(g/b1) sigmoid(g) * b2 tanh(u/b2) with the
// fast exponential; within ~1e-6 of the value (absolute near zero), far inside the layer
// tolerance.
__device__ __forceinline__ float tanh_fast(float y) {
  const float e = __expf(-2.f * fabsf(y));
  return copysignf(__fdividef(1.f - e, 1.f + e), y);
}
__device__ __forceinline__ float situ_fast(float g, float u, float b1, float ib1, float b2,
                                           float ib2) {
  const float sg = __fdividef(1.f, 1.f + __expf(-g));
  return (b1 * tanh_fast(g * ib1)) * sg * (b2 * tanh_fast(u * ib2));
}

// The MMAs of one stage, issued by a converged warp: NQ groups of B terms side by side, NA A
// matrices, K steps 0 .. nk-1 of the stage's chunk.  Everything but the stage's
// descriptor low word, its scale-slot column, the accumulator columns and the first-chunk
// flag is a compile-time offset, so the issuing warp spends few instructions per MMA (the
// issue loop runs on the pipeline's critical path: commit, refill, landing, issue).
template <int KIND, int NA, int NQ>
__device__ __forceinline__ void tc_issue_stage(uint32_t alo, uint32_t blo, uint32_t bstep, int nk,
                                               uint32_t slot, uint32_t dcol0, uint32_t dcol1,
                                               uint32_t idesc, bool first) {
#pragma unroll
  for (int i = 0; i < kTcSteps; i++) {
    if (i < nk) {
#pragma unroll
      for (int m = 0; m < NA; m++) {
        const uint32_t a_lo = alo + (uint32_t)((m * kTcBox + 32 * i) >> 4);
        const uint32_t dcol = m == 0 ? dcol0 : dcol1;
#pragma unroll
        for (int u = 0; u < NQ; u++) {
          const uint32_t b_lo = blo + (uint32_t)u * bstep + (uint32_t)(2 * i);
          const uint32_t acc = (i == 0 && u == 0 && first) ? 0u : 1u;
          if (KIND == 0)
            mma_mxf4_el_lo(dcol, a_lo, b_lo, kDescHi, idesc, slot + kSfW * (NQ + m) + 4 * i,
                           slot + kSfW * u + 4 * i, acc);
          else
            mma_f16_el_lo(dcol, a_lo, b_lo, kDescHi, idesc, acc);
        }
      }
    }
  }
}

template <int KIND, int NA, int NT, int EPI>
__global__ void __launch_bounds__(kTcThreads, 1)
    k_tc_gemm(const TcGemmArgs a, const __grid_constant__ CUtensorMap tmA0,
              const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // barriers and the TMEM base address in the first 1 KB; stages 1024-aligned after it
  uint8_t *smem = smem_raw;
  const uint32_t base_u32 = smem_u32(smem);
  const uint32_t pad = ((base_u32 + 1023u) & ~1023u) - base_u32;
  smem += pad;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);  // [NS] TMA landed
  uint64_t *sfull = full + 8;                           // [NS] scale vectors in TMEM
  uint64_t *empty = full + 16;                          // [NS] MMAs of the stage done
  uint64_t *sfload = full + 24;                         // [NSF] scale bytes landed
  uint64_t *sffree = full + 32;                         // [NSF] scale slot read by all
  uint64_t *dfull = full + 40;   // [2] accumulator buffer complete
  uint64_t *dempty = full + 42;  // [2] accumulator buffer drained
  uint32_t *tmem_base = reinterpret_cast<uint32_t *>(smem + 512);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + 520);
  uint8_t *stages = smem + 1024;
  uint8_t *sfring = stages + (size_t)a.nstages * tc_stage_bytes(NA, NT, a.ntile);
  constexpr bool kScales = (KIND == 0);
  // B terms side by side: one MMA of N = TG * ntile columns covers TG terms (their tiles
  // are adjacent in the stage), NQ = NT / TG such groups per K step accumulate into the
  // same TG column blocks, which the epilogue adds up
  const int TG = a.tgroup, NQ = NT / TG;
  // TMEM columns per stage of scale vectors: B term groups first (16 columns each), then
  // the A matrices (16 each); multi-column accesses stay aligned to their width
  const int kSfSlot = kScales ? kSfW * (NQ + NA) : 0;
  const int NS = a.nstages, NSF = a.nsf, ntile = a.ntile;
  const int aw = TG * ntile;  // accumulator columns of one A matrix
  const uint32_t stage_bytes = tc_stage_bytes(NA, NT, ntile);
  const uint32_t tma_bytes = (uint32_t)NA * kTcBox + (uint32_t)NT * ntile * kTcChunkBytes;
  const uint32_t sf_bytes = tc_sf_bytes(NA, NT, ntile);
  const uint32_t off_sfa = 0, off_sfb = (uint32_t)NA * kTcTile * kSfB;
  // output rows of an item: A matrices side by side (gate, up) share the item's 128 rows;
  // in the row-pair mode matrix m holds rows 128 m .. of the item's 256
  const int mrows = a.a_pair == 2 ? 2 * kTcTile : kTcTile;
  const int moff = a.a_pair == 2 ? kTcTile : 0;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < NS; s++) {
      mbar_init(&full[s], 1);
      mbar_init(&sfull[s], 4);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < NSF; s++) {
      mbar_init(&sfload[s], 128);
      mbar_init(&sffree[s], 4);
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(&dfull[b], 1);
      mbar_init(&dempty[b], 8);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kTcWarpMma) tmem_alloc(tmem_base, kTcTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base;
  // accumulators: buffer b, matrix m at columns (b * NA + m) * aw; scale slots after them
  const int ND = a.nacc;
  const uint32_t sf_col0 = (uint32_t)((ND * NA * aw + 15) & ~15);

  pdl_wait();
  // split K: an item is (tile, M tile, K range ks of KS), its kc chunks from ks * kc on; its
  // output goes to the ks-th partial buffer
  const int KS = a.ksplit > 1 ? a.ksplit : 1;
  const int kc = a.kchunks / KS;
  const int nitems = a.tile_off[a.ngroups] * a.mtiles * KS;
  const int my_items = nitems > (int)blockIdx.x ? (nitems - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
  const int total = my_items * kc;  // stages this CTA runs
  const int G = a.sf_rowb;                 // scale bytes per A row
  // this CTA's work items (the k-th is item blockIdx.x + k * gridDim.x), looked up once
  int4 *itab = reinterpret_cast<int4 *>(sfring + (size_t)NSF * sf_bytes);
  for (int k = tid; k < my_items && k < kTcItemTable; k += blockDim.x) {
    const TcItem ti = tc_item(a, ((int)blockIdx.x + k * (int)gridDim.x) / KS);
    itab[k] = make_int4(ti.g, ti.mt, ti.brow0, ti.nvalid);
  }
  __syncthreads();
  auto item_at = [&](int k) -> TcItem {
    if (k < kTcItemTable) {
      const int4 v = itab[k];
      return TcItem{v.x, v.y, v.z, v.w};
    }
    return tc_item(a, ((int)blockIdx.x + k * (int)gridDim.x) / KS);
  };
  // the K range of the CTA's k-th item
  auto ks_at = [&](int k) -> int { return ((int)blockIdx.x + k * (int)gridDim.x) % KS; };

  if (warp == kTcWarpTma) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      uint64_t apol;
      if (a.a_once)
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(apol));
      else
        asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(apol));
      for (int it = 0; it < total && !*abort_flag; it++) {
        const int c = ks_at(it / kc) * kc + it % kc;
        const TcItem ti = item_at(it / kc);
        const int ga = a.gid ? a.gid[ti.g] : ti.g;
        const int s = it % NS;
        if (!mbar_wait(&empty[s], ((it / NS) & 1) ^ 1)) {
          set_status(a.status, K3MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        uint8_t *st = stages + (size_t)s * stage_bytes;
        mbar_arrive_expect_tx(&full[s], tma_bytes);
        // few large copies: a stage costs the TMA unit about the same whether it moves 4 KB
        // or 32 KB, so both A matrices come in one 4-D box where their layout allows, and
        // all NT terms of B in one box of depth NT
        // A tiles read by this item only go first out of L2 (evict first; else normal)
        if (NA > 1 && a.a_pair == 2) {
          tma_load4d_pol(st, &tmA0, c * kTcChunkBytes, 0, 2 * ti.mt, ga, &full[s], apol);
        } else if (NA > 1 && a.a_pair) {
          tma_load4d_pol(st, &tmA0, c * kTcChunkBytes, ti.mt * kTcTile, 0, ga, &full[s], apol);
        } else {
          tma_load3d_pol(st, &tmA0, c * kTcChunkBytes, ti.mt * kTcTile, ga, &full[s], apol);
          if (NA > 1)
            tma_load3d_pol(st + kTcBox, &tmA1, c * kTcChunkBytes, ti.mt * kTcTile, ga, &full[s],
                           apol);
        }
        tma_load3d(st + NA * kTcBox, &tmB, c * kTcChunkBytes, ti.brow0, 0, &full[s]);
      }
    }
  } else if (warp < 4) {
    // ---------------------------------------------------------------- scale writers
    // Two streams: load stage ld's scale bytes into scale slot ld % NSF (cp.async, arriving
    // on sfload) as soon as every writer has finished with that slot's previous stage (up
    // to NSF stages ahead), and place stage stn's bytes in TMEM once they have landed and
    // the stage's TMEM slot is free.
    if (kScales) {
      const int q = warp;
      const bool gal = (G % kSfB) == 0;  // a row's chunk bytes are kSfB-aligned
      const uint32_t lane_sel = (uint32_t)(32 * q) << 16;
      int ld = 0, stn = 0;
      while (stn < total && !*abort_flag) {
        while (ld < total && ld < stn + NSF &&
               (ld == stn ? mbar_wait(&sffree[ld % NSF], ((ld / NSF) & 1) ^ 1)
                          : mbar_test(&sffree[ld % NSF], ((ld / NSF) & 1) ^ 1))) {
          const int c = ks_at(ld / kc) * kc + ld % kc;
          const TcItem ti = item_at(ld / kc);
          const int ga = a.gid ? a.gid[ti.g] : ti.g;
          const int k = ld % NSF;
          uint8_t *sfs = sfring + (size_t)k * sf_bytes;
          const int r = 32 * q + lane;  // this thread's A row and B row in the tile
#pragma unroll
          for (int m = 0; m < NA; m++) {
            const int row = ti.mt * mrows + m * moff + r;
            uint8_t *dst = sfs + off_sfa + (m * kTcTile + r) * kSfB;
            const uint8_t *src = a.sfa[m] + (long long)ga * a.sfa_gstride + (long long)row * G;
            if (row < a.M_rows && gal && kSfB * c + kSfB <= G) {
              cp_async_sf(dst, src + kSfB * c);
            } else {
              const uint2 v = row < a.M_rows ? load_scales(src, G, c) : make_uint2(0u, 0u);
              st_staged_scales(dst, v);
            }
          }
          if (r < ntile) {
            // B scales are stored 8 per row per 256-column K group: this chunk's kSfB of them
            const long long boff = (long long)(c / (8 / kSfB)) * a.sfb_cstride +
                                   (long long)(ti.brow0 + r) * 8 + (c % (8 / kSfB)) * kSfB;
#pragma unroll
            for (int t = 0; t < NT; t++) {
              uint8_t *dst = sfs + off_sfb + (t * ntile + r) * kSfB;
              if (r < ti.nvalid)
                cp_async_sf(dst, a.sfb + (long long)t * a.sfb_tstride + boff);
              else
                st_staged_scales(dst, make_uint2(0u, 0u));
            }
          }
          cp_async_arrive(&sfload[k]);
          ld++;
        }
        if (stn >= ld) {  // the slot wait above timed out
          set_status(a.status, K3MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        const int k = stn % NSF, sj = stn % NS;
        if (!mbar_wait(&sfload[k], (stn / NSF) & 1) ||
            !mbar_wait(&empty[sj], ((stn / NS) & 1) ^ 1)) {
          set_status(a.status, K3MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint8_t *sfs = sfring + (size_t)k * sf_bytes;
        const uint32_t slot = tmem + sf_col0 + (uint32_t)(sj * kSfSlot);
        // A: K step i of matrix m reads column slot + kSfW(NQ + m) + 4i + (row / 32);
        // scale byte 255 (no contribution) becomes 0
#pragma unroll
        for (int m = 0; m < NA; m++) {
          uint2 v = ld_staged_scales(sfs + off_sfa + (m * kTcTile + 32 * q + lane) * kSfB);
          v.x &= ~__vcmpeq4(v.x, 0xffffffffu);
          v.y &= ~__vcmpeq4(v.y, 0xffffffffu);
#pragma unroll
          for (int i = 0; i < kTcSteps; i++)
            tmem_st_x1(slot + lane_sel + kSfW * (NQ + m) + 4 * i + q, step_scales(v, i));
        }
        // B: K step i of term group u reads column slot + kSfW u + 4i + n/32 at lane n % 32
        // of every lane quarter (each 32-row quarter of the MMA reads its own copy), for
        // the group's rows n = 0 .. aw-1 (term u*TG + n / ntile, row n % ntile; those are
        // consecutive in the staged scale bytes)
#pragma unroll
        for (int u = 0; u < NT; u++) {
          if (u < NQ) {
            uint32_t vb[kSfW];
#pragma unroll
            for (int jj = 0; jj < 4; jj++) {
              const int n = 32 * jj + lane;
              const uint2 v = (n < aw) ? ld_staged_scales(sfs + off_sfb + (u * aw + n) * kSfB)
                                       : make_uint2(0u, 0u);
#pragma unroll
              for (int i = 0; i < kTcSteps; i++) vb[4 * i + jj] = step_scales(v, i);
            }
            tmem_st_sf(slot + lane_sel + kSfW * u, vb);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sfull[sj]);
          mbar_arrive(&sffree[k]);
        }
        stn++;
      }
      // every cp.async of this thread must land before the CTA can exit
      asm volatile("cp.async.wait_all;" ::: "memory");
    }
  } else if (warp == kTcWarpMma) {
    // ---------------------------------------------------------------- MMA issuer
    // The whole warp runs the loop (waits and operands warp-uniform); one elected lane
    // issues each tcgen05 instruction.
    {
      int it = 0, n = 0;
      bool ok = true;
      // B: group u of TG terms starts TG * ntile rows of 128 bytes after group u - 1
      const uint32_t bstep = (uint32_t)(TG * ntile * kTcChunkBytes) >> 4;
      for (; n < my_items && ok; n++) {
        const TcItem ti = item_at(n);
        // the last term block of a group needs only the tile's valid rows
        const int nmma = (TG - 1) * ntile + ((ti.nvalid + 15) / 16) * 16;
        uint32_t idesc;
        if (KIND == 0)
          idesc = (1u << 7) | (1u << 10) | ((uint32_t)(nmma >> 3) << 17) | (1u << 23) |
                  ((uint32_t)(kTcTile >> 4) << 24);
        else
          idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(nmma >> 3) << 17) |
                  ((uint32_t)(kTcTile >> 4) << 24);
        // the epilogue must have drained this accumulator buffer's previous item
        const int db = n % ND;
        const uint32_t dcol0 = tmem + (uint32_t)((db * NA) * aw);
        const uint32_t dcol1 = dcol0 + (uint32_t)aw;
        if (!__all_sync(0xffffffffu, mbar_wait(&dempty[db], ((n / ND) & 1) ^ 1))) {
          if (lane == 0) {
            set_status(a.status, K3MOE_ERR_TIMEOUT);
            *abort_flag = 1;
          }
          ok = false;
          break;
        }
        tc_fence_after();
        const int c0k = ks_at(n) * kc;
        for (int c = 0; c < kc; c++, it++) {
          const int s = it % NS;
          const uint32_t par = (it / NS) & 1;
          const bool got = mbar_wait(&full[s], par) && (!kScales || mbar_wait(&sfull[s], par));
          if (!__all_sync(0xffffffffu, got)) {
            if (lane == 0) {
              set_status(a.status, K3MOE_ERR_TIMEOUT);
              *abort_flag = 1;
            }
            ok = false;
            break;
          }
          tc_fence_after();
          {
            const uint32_t alo = sw_desc_lo(smem_u32(stages + (size_t)s * stage_bytes));
            const uint32_t blo = alo + ((uint32_t)(NA * kTcBox) >> 4);
            const uint32_t slot = tmem + sf_col0 + (uint32_t)(s * kSfSlot);
            const int nk = (c0k + c == a.kchunks - 1) ? a.ksteps_last : kTcSteps;
            if (NQ == 1)
              tc_issue_stage<KIND, NA, 1>(alo, blo, bstep, nk, slot, dcol0, dcol1, idesc, c == 0);
            else if (NQ == 2)
              tc_issue_stage<KIND, NA, (NT >= 2 ? 2 : 1)>(alo, blo, bstep, nk, slot, dcol0, dcol1,
                                                          idesc, c == 0);
            else
              tc_issue_stage<KIND, NA, (NT >= 4 ? 4 : 1)>(alo, blo, bstep, nk, slot, dcol0, dcol1,
                                                          idesc, c == 0);
          }
          tc_commit_el(&empty[s]);
        }
        tc_commit_el(&dfull[db]);
      }
      // before the accumulator is freed: wait (bounded) for every MMA issued
      if (!ok && it > 0) {
        const int s = (it - 1) % NS;
        mbar_wait(&empty[s], ((it - 1) / NS) & 1, 400000000LL);
      }
      __syncwarp();
    }
  } else if (warp >= kTcWarpEpi) {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;              // TMEM lane quarter this warp may access
    const int half = (warp - kTcWarpEpi) >> 2;
    const int hcols = ((ntile / 2) + 15) & ~15;  // columns per half (multiple of 16)
    const float ib1 = 1.f / a.b1, ib2 = 1.f / a.b2;
    for (int n = 0; n < my_items; n++) {
      const TcItem ti = item_at(n);
      const int db = n % ND;
      const bool got = mbar_wait(&dfull[db], (n / ND) & 1);
      if (!got) {
        set_status(a.status, K3MOE_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      tc_fence_after();
      const int row = ti.mt * mrows + 32 * q + lane;
      const uint32_t lane_sel = (uint32_t)(32 * q) << 16;
      if (got && !*abort_flag) {
        const uint32_t dbase = tmem + lane_sel + (uint32_t)(db * NA * aw);
        for (int c0 = half * hcols; c0 < (half + 1) * hcols && c0 < ti.nvalid; c0 += 16) {
          // the sum of the TG term blocks of each matrix
          uint32_t d0[16], d1[16];
          tmem_ld16_nowait(dbase + (uint32_t)c0, d0);
          if (NA > 1) tmem_ld16_nowait(dbase + (uint32_t)(aw + c0), d1);
          tmem_wait_ld2(d0, d1);
          for (int tb = 1; tb < TG; tb++) {
            uint32_t e0[16], e1[16];
            tmem_ld16_nowait(dbase + (uint32_t)(tb * ntile + c0), e0);
            if (NA > 1) tmem_ld16_nowait(dbase + (uint32_t)(aw + tb * ntile + c0), e1);
            tmem_wait_ld2(e0, e1);
#pragma unroll
            for (int j = 0; j < 16; j++) {
              d0[j] = __float_as_uint(__uint_as_float(d0[j]) + __uint_as_float(e0[j]));
              if (NA > 1) d1[j] = __float_as_uint(__uint_as_float(d1[j]) + __uint_as_float(e1[j]));
            }
          }
          float *obase = a.out + (long long)ks_at(n) * a.out_kstride;
          if (row < a.M_rows) {
            float *orow = obase + (long long)(ti.brow0 + c0) * a.out_ld + row;
#pragma unroll
            for (int j = 0; j < 16; j++) {
              if (c0 + j < ti.nvalid) {
                float v = __uint_as_float(d0[j]);
                if (EPI == 0)
                  v = situ_fast(v, __uint_as_float(d1[j]), a.b1, ib1, a.b2, ib2);
                orow[(long long)j * a.out_ld] = v;
              }
            }
          }
          if (EPI == 1 && NA > 1 && row + moff < a.M_rows) {  // row-pair mode: second half
            float *orow = obase + (long long)(ti.brow0 + c0) * a.out_ld + row + moff;
#pragma unroll
            for (int j = 0; j < 16; j++)
              if (c0 + j < ti.nvalid) orow[(long long)j * a.out_ld] = __uint_as_float(d1[j]);
          }
          if (EPI == 2 && row < a.M_rows) {  // both matrices stored: the second at + mstride
            float *orow = obase + a.out_mstride + (long long)(ti.brow0 + c0) * a.out_ld + row;
#pragma unroll
            for (int j = 0; j < 16; j++)
              if (c0 + j < ti.nvalid) orow[(long long)j * a.out_ld] = __uint_as_float(d1[j]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&dempty[db]);
      if (!got) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kTcWarpMma) tmem_dealloc(tmem, kTcTmemCols);
}

// ---------------------------------------------------------------------------------------
// Host side: tensor maps (through the driver entry point, no link against libcuda) and
// launches.
namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  }
  return fn;
}
}  // namespace

bool tc_map(CUtensorMap *m, const void *base, int rank, const unsigned long long *dims,
            const unsigned long long *strides, const unsigned *box) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rank < 3 || rank > 5) return false;
  if (reinterpret_cast<uintptr_t>(base) & 15) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; i++) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) {
      if (strides[i] & 15) return false;
      st[i] = strides[i];
    }
  }
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, (cuuint32_t)rank, const_cast<void *>(base), d, st,
            bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            kTcChunkBytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map of 8-byte words (scale bytes read in 16-byte boxes), no swizzle: rank 3..5,
// dims[0] in words, strides in bytes of dims 1..rank-1.
bool tc_map_words(CUtensorMap *m, const void *base, int rank, const unsigned long long *dims,
                  const unsigned long long *strides, const unsigned *box) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rank < 3 || rank > 5) return false;
  if (reinterpret_cast<uintptr_t>(base) & 15) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; i++) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) {
      if (strides[i] & 15) return false;
      st[i] = strides[i];
    }
  }
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT64, (cuuint32_t)rank, const_cast<void *>(base), d, st,
            bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_map3d(CUtensorMap *m, const void *base, unsigned long long inner_bytes,
              unsigned long long rows, unsigned long long depth, unsigned long long row_stride,
              unsigned long long depth_stride, int box_rows, int box_depth) {
  if (depth_stride == 0) depth_stride = row_stride * rows;
  const unsigned long long dims[3] = {inner_bytes, rows, depth};
  const unsigned long long strides[2] = {row_stride, depth_stride};
  const unsigned box[3] = {(unsigned)kTcChunkBytes, (unsigned)box_rows, (unsigned)box_depth};
  return tc_map(m, base, 3, dims, strides, box);
}

// Ring depths: NSF scale slots (8 when they fit), then as many data stages as fit in
// shared memory (and, with scale slots, in TMEM next to the accumulators), at most 8.
// tg: B terms per MMA (accumulator columns tg * ntile per A matrix).
static void tc_depths(int na, int nt, int ntile, int tg, bool scales, int *ns, int *nsf) {
  const size_t budget = 227 * 1024 - 2048 - kTcItemTableBytes;
  const size_t stage = tc_stage_bytes(na, nt, ntile), sfb = scales ? tc_sf_bytes(na, nt, ntile) : 0;
  int by_tmem = 8;
  if (scales) {
    const int free_cols = kTcTmemCols - ((na * tg * ntile + 15) & ~15);
    by_tmem = free_cols / (kSfW * (na + nt / tg));
  }
  // the most data stages (at most 8, and what TMEM holds), then the most scale slots
  int best_s = -1, best_f = 0;
  for (int f = scales ? 8 : 0; f >= (scales ? 2 : 0); f -= 2) {
    if ((size_t)f * sfb >= budget) continue;
    int s = (int)((budget - f * sfb) / stage);
    if (s > 8) s = 8;
    if (s > by_tmem) s = by_tmem;
    if (s > best_s) {
      best_s = s;
      best_f = f;
    }
    if (!scales) break;
  }
  *ns = best_s < 0 ? 0 : best_s;
  *nsf = best_f;
}

// Accumulator buffers: two (the epilogue of one item overlaps the next item's MMAs) when
// they fit in TMEM next to the scale slots, else one.
static int tc_nacc(int na, int nt, int ntile, int tg, bool scales, int ns) {
  const int sf = scales ? ns * kSfW * (na + nt / tg) : 0;
  return (((2 * na * tg * ntile + 15) & ~15) + sf <= kTcTmemCols) ? 2 : 1;
}

// B terms per MMA: the largest divisor of nt with tg * ntile <= 128 (the scale layout of
// up to four 32-row column groups) that still leaves room for two accumulator buffers and
// two data stages; else the largest that leaves two stages.
static int tc_tgroup(int na, int nt, int ntile, bool scales) {
  int best = 1, best2 = 0;
  for (int tg = 1; tg <= nt; tg *= 2) {
    if (nt % tg || tg * ntile > 128) continue;
    int ns = 0, nsf = 0;
    tc_depths(na, nt, ntile, tg, scales, &ns, &nsf);
    if (ns < 2) continue;
    best = tg;
    if (tc_nacc(na, nt, ntile, tg, scales, ns) == 2) best2 = tg;
  }
  return best2 ? best2 : best;
}

template <int KIND, int NA, int NT, int EPI>
static cudaError_t launch_tc(const TcGemmArgs &a, const CUtensorMap &A0, const CUtensorMap &A1,
                             const CUtensorMap &B, int grid, cudaStream_t st) {
  auto fn = k_tc_gemm<KIND, NA, NT, EPI>;
  if (a.ntile < 16 || a.ntile > kTcTile || a.ntile % 16) return cudaErrorInvalidValue;
  const int tg = tc_tgroup(NA, NT, a.ntile, KIND == 0);
  int ns = 0, nsf = 0;
  tc_depths(NA, NT, a.ntile, tg, KIND == 0, &ns, &nsf);
  if (ns < 2 || (KIND == 0 && nsf < 2)) return cudaErrorInvalidValue;
  const size_t smem = 2048 + (size_t)ns * tc_stage_bytes(NA, NT, a.ntile) +
                      (size_t)nsf * (KIND == 0 ? tc_sf_bytes(NA, NT, a.ntile) : 0) +
                      kTcItemTableBytes;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  TcGemmArgs aa = a;
  aa.nstages = ns;
  aa.nsf = nsf;
  aa.nacc = tc_nacc(NA, NT, a.ntile, tg, KIND == 0, ns);
  aa.tgroup = tg;
  fn<<<grid, kTcThreads, smem, st>>>(aa, A0, A1, B);
  return cudaGetLastError();
}

cudaError_t launch_tc_gemm(TcKind kind, const TcGemmArgs &a, const CUtensorMap &A0,
                           const CUtensorMap &A1, const CUtensorMap &B, int grid,
                           cudaStream_t st) {
  switch (kind) {
    case TcKind::kMxf4GateUp: return launch_tc<0, 2, kTcTermsX, 0>(a, A0, A1, B, grid, st);
    case TcKind::kMxf4Down: return launch_tc<0, 1, kTcTermsAct, 1>(a, A0, A1, B, grid, st);
    case TcKind::kMxf4DownPair: return launch_tc<0, 2, kTcTermsAct, 1>(a, A0, A1, B, grid, st);
    case TcKind::kBf16GateUp: return launch_tc<1, 2, 1, 0>(a, A0, A1, B, grid, st);
    case TcKind::kBf16Pair: return launch_tc<1, 2, 1, 2>(a, A0, A1, B, grid, st);
    case TcKind::kBf16Down: return launch_tc<1, 1, 2, 1>(a, A0, A1, B, grid, st);
    case TcKind::kBf16Store: return launch_tc<1, 1, 1, 1>(a, A0, A1, B, grid, st);
  }
  return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------------------
// Split-K partial sums, added in partial order k = 0 .. KS-1 (the same on every run).
// out[i] = sum_k part[k * kstride + i]
__global__ void k_sum_parts(const float *__restrict__ part, int KS, long long kstride,
                            long long n, float *__restrict__ out) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    float v = part[i];
    for (int k = 1; k < KS; k++) v = __fadd_rn(v, part[k * kstride + i]);
    out[i] = v;
  }
}
// act[i] = SiTU(sum_k part[k * kstride + i], sum_k part[k * kstride + mstride + i]), the
// gate/up epilogue's SiTU.
__global__ void k_situ_parts(const float *__restrict__ part, int KS, long long kstride,
                             long long mstride, long long n, float b1, float b2,
                             float *__restrict__ act) {
  const float ib1 = 1.f / b1, ib2 = 1.f / b2;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    float g = part[i], u = part[mstride + i];
    for (int k = 1; k < KS; k++) {
      g = __fadd_rn(g, part[k * kstride + i]);
      u = __fadd_rn(u, part[k * kstride + mstride + i]);
    }
    act[i] = situ_fast(g, u, b1, ib1, b2, ib2);
  }
}

cudaError_t launch_sum_parts(cudaStream_t st, int sms, const float *part, int KS,
                             long long kstride, long long n, float *out) {
  long long g = (n + 255) / 256;
  if (g > 8LL * sms) g = 8LL * sms;
  k_sum_parts<<<(int)g, 256, 0, st>>>(part, KS, kstride, n, out);
  return cudaGetLastError();
}

cudaError_t launch_situ_parts(cudaStream_t st, int sms, const float *part, int KS,
                              long long kstride, long long mstride, long long n, float b1,
                              float b2, float *act) {
  long long g = (n + 255) / 256;
  if (g > 8LL * sms) g = 8LL * sms;
  k_situ_parts<<<(int)g, 256, 0, st>>>(part, KS, kstride, mstride, n, b1, b2, act);
  return cudaGetLastError();
}

}  // namespace k3

// k3moe_tc.cuh -- declarations of the multi-token path: the tensor-core grouped GEMM
// (k3moe_tc.cu), its routing and quantisation helpers (k3moe_prefill.cu) and the screening
// router (k3moe_router_tc.cu).
#pragma once
#include <cuda.h>
#include "k3moe_kernels.cuh"

namespace k3 {

constexpr int kTcRows = 128;     // A rows / B rows per tensor-core tile
constexpr int kTcChunk = 128;    // K bytes per pipeline stage (one swizzle atom: 128 or 64)
constexpr int kTcSteps = kTcChunk / 32;  // MMA K steps (32 bytes of K each) per stage
constexpr int kTcTermsX = 4;     // MXFP4 terms of the layer input x (bf16)
constexpr int kTcTermsAct = 4;   // MXFP4 terms of the SiTU activations (float)
constexpr int kTcTokens = 4096;  // tokens per pass of the multi-token path

// Arguments of k_tc_gemm.  Groups g = 0..ngroups-1 own B rows [off[g], off[g+1]) and
// tile_off[g] = sum over earlier groups of ceil(rows / 128); gid[g] is the A index of
// group g in the A tensor map's third dimension (NULL: g itself).
struct TcGemmArgs {
  const int32_t *off, *tile_off, *gid;
  int ngroups;
  int mtiles;        // ceil(M_rows / 128)
  int M_rows;        // rows of each A matrix (outputs)
  int kchunks;       // kTcChunk-byte chunks of K
  int ksteps_last;   // 32-byte MMA steps in the last chunk (1..kTcSteps)
  int ntile;         // B rows per tile (multiple of 16, at most 128)
  int nstages;       // data stages, set by the launcher
  int nsf;           // scale-byte slots, set by the launcher
  int nacc;          // accumulator buffers (1 or 2), set by the launcher
  int tgroup;        // B terms side by side in one MMA (divides the term count), set by
                     // the launcher
  int a_pair;        // 1: A matrices 0 and 1 are one 4-D map (third dimension = matrix),
                     // fetched by one copy per stage; 2: they are two consecutive 128-row
                     // tiles of ONE matrix (4-D map: K bytes, 128 rows, tile, group), so an
                     // item's M tile covers 256 output rows and both halves share the B
                     // stage
  const uint8_t *sfa[2];   // MXF4: scale bytes of A matrix m for group 0, rows of sf_rowb
  long long sfa_gstride;   // bytes between consecutive groups' A scales
  int sf_rowb;             // scale bytes per row (K / 32)
  const uint8_t *sfb;      // MXF4: B scale bytes [term][256-column K group][B row][8]
  long long sfb_tstride;   // bytes between terms
  long long sfb_cstride;   // bytes between 256-column K groups (B rows x 8)
  float *out;              // [B row][out_ld]
  long long out_ld;
  int ksplit;              // K ranges per item (0 or 1: none); kchunks must divide by it.
                           // The partial sum of range ks goes to out + ks * out_kstride
  long long out_kstride;
  long long out_mstride;   // kBf16Pair: the second matrix's output at out + out_mstride
  float b1, b2;            // SiTU caps (gate/up epilogue)
  int32_t *status;
  int a_once;              // every A tile is read by one item only (each group's B rows fit
                           // one tile): its loads are marked first out of L2
};

// kBf16Pair: two bf16 matrices on one B, both products stored (the gate/up pair's partial
// sums under split K; k_situ_parts then adds them up and applies SiTU).
enum class TcKind { kMxf4GateUp, kMxf4Down, kMxf4DownPair, kBf16GateUp, kBf16Pair, kBf16Down,
                    kBf16Store };

// Tensor map of bytes of rank 3..5 (dims[0] = K bytes, innermost; strides in bytes of
// dims 1..rank-1) with the kTcChunk-byte swizzle and boxes of box[0] = kTcChunk bytes x
// box[1..]; false if the driver entry point is missing or the layout is refused.
bool tc_map(CUtensorMap *m, const void *base, int rank, const unsigned long long *dims,
            const unsigned long long *strides, const unsigned *box);
// The same for 8-byte words without swizzle (dims[0] in words).
bool tc_map_words(CUtensorMap *m, const void *base, int rank, const unsigned long long *dims,
                  const unsigned long long *strides, const unsigned *box);
// The 3-D case (inner = K bytes, rows, depth) with boxes of kTcChunk bytes x box_rows x
// box_depth.
bool tc_map3d(CUtensorMap *m, const void *base, unsigned long long inner_bytes,
              unsigned long long rows, unsigned long long depth, unsigned long long row_stride,
              unsigned long long depth_stride, int box_rows, int box_depth = 1);
// Split-K partials added in range order: out = sum_k part_k; act = SiTU(gate, up) sums.
cudaError_t launch_sum_parts(cudaStream_t st, int sms, const float *part, int KS,
                             long long kstride, long long n, float *out);
cudaError_t launch_situ_parts(cudaStream_t st, int sms, const float *part, int KS,
                              long long kstride, long long mstride, long long n, float b1,
                              float b2, float *act);
cudaError_t launch_tc_gemm(TcKind kind, const TcGemmArgs &a, const CUtensorMap &A0,
                           const CUtensorMap &A1, const CUtensorMap &B, int grid,
                           cudaStream_t st);

// Gate/up + SiTU of one token on the tensor cores (k3moe_gateup_tc.cu): the arguments of
// k_gateup_t1, the split tiles' partial sums [tile][kTc1Pieces][2][128], and the counters
// (cnt[0] exit, cnt[1 + tile]; zero on entry, left zero).  tmw: the experts' gate and up
// operands (K bytes, rows, {gate, up}, expert; 128-row x 128-byte boxes of both); tms:
// their scale bytes as 8-byte words (words, rows, {gate, up}, expert; boxes of 2 x 128 x 2).
struct GateUpTc1Args {
  GateUpT1Args g;
  float *gpart;
  unsigned *cnt;
  int NS;  // ring slots, set from gateup_tc1_smem
};
// Shared memory of the kernel for this shape and grid (0: it does not apply), ring slots
// in *ns_out.
size_t gateup_tc1_smem(int H, int I, int E, int K, int grid, int *ns_out);
cudaError_t set_gateup_tc1_smem_limit();
cudaError_t launch_gateup_tc1(const GateUpTc1Args &a, const CUtensorMap &tmw,
                              const CUtensorMap &tms, int grid, cudaStream_t st, bool pdl);

// Pairs per block of the dispatch's counting sort: small chunks spread a small batch over
// several blocks, larger ones keep the per-chunk tables of a large batch short.
inline int route_chunk(int P) { return P <= 16384 ? 256 : 1024; }
__global__ void k_route_count(const int32_t *__restrict__ idx, int P, int E, int chunk,
                              int32_t *__restrict__ counts, int32_t *inv, int32_t *status);
__global__ void k_route_hist(int32_t *__restrict__ counts, int nch, int E, int ntile,
                             int32_t *off, int32_t *tile_off);
__global__ void k_route_scatter(const int32_t *__restrict__ idx, int P, int E, int chunk,
                                const int32_t *__restrict__ first, int32_t *perm,
                                int32_t *inv);
// k_quant_x on 256-thread blocks: x bf16, or float when x_f32.
cudaError_t launch_quant_x(bool x_f32, int grid, cudaStream_t st, const void *x, int T, int H,
                           int K, const int32_t *inv, int P, uint8_t *xq, uint8_t *xs);
__global__ void k_quant_act(const float *__restrict__ act, int P, int I,
                            uint8_t *__restrict__ aq, uint8_t *__restrict__ as);
__global__ void k_split_bf16(const float *__restrict__ v, long long n, uint16_t *__restrict__ out);
__global__ void k_group1(int n, int ntile, int32_t *off, int32_t *tile_off);
__global__ void k_row_norms(const uint16_t *__restrict__ v0, int R0, float *__restrict__ out0,
                            const uint16_t *__restrict__ v1, int R1, float *__restrict__ out1,
                            int H);
__global__ void k_route_candidates(const float *__restrict__ Lt, const float *__restrict__ xn,
                                   const float *__restrict__ wn,
                                   const uint16_t *__restrict__ x, const uint16_t *__restrict__ wr,
                                   const float *__restrict__ bias, int H, int E, int K,
                                   int nadd, float *__restrict__ sc, float *__restrict__ ch,
                                   int32_t *__restrict__ ncand, int32_t *status);
size_t route_candidates_smem(int H, int E, int K);
__global__ void k_combine(int T, int H, int K, const float *__restrict__ w,
                          const int32_t *__restrict__ inv, const float *__restrict__ dpair,
                          const float *__restrict__ ds, void *y, int ydt, int accumulate);

}  // namespace k3

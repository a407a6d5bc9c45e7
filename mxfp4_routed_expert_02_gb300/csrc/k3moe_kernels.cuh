// k3moe_kernels.cuh -- kernel declarations and launch-shape constants of libk3moe.
#pragma once
#include "k3moe_device.cuh"
#include "k3moe_topk.cuh"

namespace k3 {

constexpr int kTokChunk = 8;      // tokens of x staged in shared memory by k_router_shared
constexpr int kDecodeTokens = 64; // tokens per pass of the decode expert path
constexpr int kTileRows = 32;     // gate/up output rows per work item (one down-input group)
constexpr int kDownRows = 16;     // down output rows per work item
constexpr int kPairKeyShift = 12; // dispatch sort key = expert << 12 | pair id (pairs < 4096)

// Dispatch buffer (int32), for P = T*K (token, slot) pairs:
//   [0]            U, the number of distinct experts used
//   [4 .. 4+P)     uexp[u], the distinct experts, ascending
//   [4+P .. 5+2P)  uoff[u], start of expert u's pairs in plist (uoff[U] = valid pairs)
//   [5+2P .. 5+3P) plist, pair ids t*K + j sorted by (expert, pair id)
__host__ __device__ inline int disp_words(int P) { return 5 + 3 * P; }

// Launches k_router_shared with tc tokens per chunk (1: a decode step; else up to
// kTokChunk).
cudaError_t launch_router_shared(int tc, int grid, size_t smem, cudaStream_t st, const uint16_t *x,
                                 int T, int H, const uint16_t *wr, int E, const float *bias,
                                 const uint16_t *sh_gate, const uint16_t *sh_up, int SI, float b1,
                                 float b2, float *sc, float *ch, float *act_s, int32_t *status);
cudaError_t set_router_smem_limits(int bytes);
// One decode token: router rows and shared gate/up rows, one warp each.
cudaError_t launch_router_t1(cudaStream_t st, const uint16_t *x, int H, const uint16_t *wr,
                             int E, const float *bias, const uint16_t *sh_gate,
                             const uint16_t *sh_up, int SI, float b1, float b2, float *sc,
                             float *ch, float *act_s, int32_t *status, bool pdl);

__global__ void k_topk(const float *__restrict__ scores, const float *__restrict__ choice, int T,
                       int E, int K, int renorm, float routed_scale, int32_t *__restrict__ idx,
                       float *__restrict__ w, int32_t *status);

__global__ void k_dispatch(const int32_t *__restrict__ idx, int P, int E,
                           int32_t *__restrict__ disp, int32_t *status);

struct ExpertArgs {
  const uint8_t *base;
  long long stride;
  long long off[6];  // w1p, w1s, w2p, w2s, w3p, w3s
};

// Launches k_expert_gateup<mb> (mb = tokens per register block: 1 or 2); x is bf16
// [T][H], or float [T][H] when x_f32.
cudaError_t launch_expert_gateup(int mb, int grid, int block, cudaStream_t st, const void *x,
                                 bool x_f32, int H, int I, int K, const ExpertArgs &ex,
                                 const int32_t *disp, int P, float b1, float b2,
                                 uint16_t *act_hi, uint16_t *act_lo, int32_t *act_ex);

__global__ void k_down_combine(int T, int H, int I, int K, ExpertArgs ex,
                               const int32_t *__restrict__ idx, const float *__restrict__ w,
                               const int32_t *__restrict__ disp, int P,
                               const uint16_t *__restrict__ act_hi,
                               const uint16_t *__restrict__ act_lo,
                               const int32_t *__restrict__ act_ex,
                               const uint16_t *__restrict__ sh_down, int SI,
                               const float *__restrict__ act_s, void *y, int ydt,
                               int accumulate, int LR);

// ---- decode kernels with bulk-copy rings (k3moe_decode.cu)
struct GateUpT1Args {
  const uint16_t *x;
  const float *xf;  // when set, the input is this float row instead of x (two f16 terms)
  int H, I, E, K;
  ExpertArgs ex;
  const float *sc, *ch;  // [E] router scores / selection scores
  int renorm;
  float routed_scale;
  int32_t *idx_out;
  float *w_out;
  int32_t *disp;
  float b1, b2;
  uint16_t *act_hi, *act_lo;
  int32_t *act_ex;
  int32_t *status;
  int RB, NS;
};

struct DownArgs {
  int T, H, I, K, P;
  ExpertArgs ex;
  const int32_t *idx;
  const float *w;
  const int32_t *disp;
  const uint16_t *act_hi, *act_lo;
  const int32_t *act_ex;
  const uint16_t *sh_down;
  int SI;
  const float *act_s;
  void *y;
  int ydt, accumulate, LR, NS;
  int32_t *status;
};

// ---- the single-token layer step as one persistent kernel (k3moe_decode_fused.cu)
// Weights and route outputs of one layer of the step (a stack of layers runs several in
// one launch).
struct FusedLayer {
  const uint16_t *wr;                         // [E][H]
  const float *bias;                          // [E] or null
  const uint16_t *sh_gate, *sh_up, *sh_down;  // null when SI == 0
  const uint8_t *experts;                     // expert e at experts + e * stride
  long long stride;
  int32_t *idx_out;                           // [K] or null
  float *w_out;                               // [K] or null
};
// Layers per launch: each uses four grid counters of the 256-byte workspace header.
constexpr int kFuMaxLayers = 16;
// The tensor-core single-token gate/up (k_gateup_tc1): row tiles (expert slots x 128 rows)
// at most, and the parts one tile may be split into between CTAs.
constexpr int kTc1MaxTiles = 768;
constexpr int kTc1Pieces = 2;
struct FusedT1Args {
  const uint16_t *x;  // [H] bf16 (unused when h is set)
  const float *h;     // [H] residual stream: when set, x = bf16(RMSNorm(h)) in the kernel
  float eps;          // RMSNorm epsilon (with h)
  int H, I, E, K, SI;
  int L;                        // layers, 1 .. kFuMaxLayers (more than one needs h)
  FusedLayer lay[kFuMaxLayers];
  ExpertArgs ex;                // record offsets (base and stride are per layer)
  int renorm;
  float routed_scale, b1, b2;
  float *sc, *ch;       // [E] workspace
  float *act_s;         // [SI] workspace
  uint16_t *act;              // [K][I] workspace
  unsigned *bar;              // per layer l, bar[4l ..]: dependency 1, dependency 2, exit;
                              // zero on entry and on exit
  int act_exp;                // activations are stored as f16 of act * 2^-act_exp
  void *y;
  int ydt, accumulate;
  int32_t *status;
  int expire_dep2;  // test of the expiry path: dependency 2 cannot complete, its wait is short
};
// Shared memory the fused kernel needs for this shape (0: the shape does not fit it).
size_t fused_t1_smem(int H, int I, int E, int K, int SI, int grid);
cudaError_t launch_fused_t1(const FusedT1Args &a, int grid, cudaStream_t st);
cudaError_t set_fused_smem_limit();

size_t gateup_t1_smem(int H, int E, int K, int RB, int NS);
cudaError_t launch_gateup_t1(const GateUpT1Args &a, int grid, cudaStream_t st, bool pdl);
size_t down_tma_smem(int I, int T, int P, int NS, bool act_smem, int ntl);
cudaError_t launch_down_tma(const DownArgs &a, int grid, cudaStream_t st, bool pdl,
                            bool act_smem);
// The single-token down without a shared expert, whole-expert stages with their
// activations (k_down_t1): ring slots for (I, K), 0 when it does not apply.
int down_t1_slots(int H, int I, int K, int sms);
cudaError_t launch_down_t1(const DownArgs &a, int sms, cudaStream_t st, bool pdl);
cudaError_t set_decode_smem_limits();

__global__ void k_dequant(const uint8_t *__restrict__ packed, const uint8_t *__restrict__ scales,
                          int rows, int cols, float *__restrict__ out);

__global__ void k_rmsnorm_bf16(const float *__restrict__ h, int T, int n, float eps,
                               uint16_t *__restrict__ out);

// ---- LatentMoE pieces (k3moe_latent.cu)
// out = W in (bf16 W [R][C], T input rows of C, bf16 or float); with W2 the shared gate/up
// pair, SiTU applied; with y the layer output y (=|+=) addend + value (ydt), else float out.
// norm (float input, no W2, T <= kProjRows): the input rows RMS-normalised with weight nw
// on the fly, as launch_rmsnorm_f32w would write them.
constexpr int kProjRows = 4;
cudaError_t launch_proj(cudaStream_t st, int sms, const uint16_t *W, const uint16_t *W2, int R,
                        int C, const void *in, bool in_f32, int T, float *out,
                        const float *addend, void *y, int ydt, int accumulate, float b1,
                        float b2, bool pdl, bool norm = false, const float *nw = nullptr,
                        float eps = 0.f);
// y (=|+=) up + ds elementwise over n values (ds may be nullptr), float or bf16 y.
cudaError_t launch_add_out(cudaStream_t st, int sms, const float *up, const float *ds, void *y,
                           int ydt, int accumulate, long long n);
// RMSNorm of T float rows of n with weight w (nullptr: 1), sum of squares as a float-float
// pair.
cudaError_t launch_rmsnorm_f32w(cudaStream_t st, const float *in, int T, int n, const float *w,
                                float eps, float *out, bool pdl);
constexpr int kRmsThreads = 256;  // threads per row of k_rmsnorm_bf16
constexpr int kRmsVec = 8;        // float4 per thread held in registers (rows up to 8192)

}  // namespace k3

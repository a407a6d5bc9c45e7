// k3moe_api.cu -- the C ABI of libk3moe: argument checks, workspace layout, launches.
//
// Operation definitions and the error contract are in include/k3moe.h.  Every step of
// the path runs in this library's kernels; nothing here computes on the host.
#include <cstdio>
#include <cstring>
#include <cmath>
#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "k3moe_cache.h"
#include "k3moe_tc.cuh"

using namespace k3;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  int sms = 0;
  bool attrs_set = false;
  cudaStream_t side = nullptr;  // a second stream for work that overlaps the caller's
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t up16(size_t n) { return (n + 15) & ~size_t(15); }

// Per-device one-time set-up: SM count and the dynamic shared-memory limits.
const DeviceInfo *device_info() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo &d = g_dev[dev];
  if (!d.attrs_set) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return nullptr;
    const int big = 200 * 1024;
    if (set_router_smem_limits(big) != cudaSuccess ||
        cudaFuncSetAttribute(k_down_combine, cudaFuncAttributeMaxDynamicSharedMemorySize, big) !=
            cudaSuccess ||
        cudaFuncSetAttribute(k_topk, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024) !=
            cudaSuccess ||
        cudaFuncSetAttribute(k_dispatch, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024) !=
            cudaSuccess ||
        cudaFuncSetAttribute(k_route_candidates, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             128 * 1024) != cudaSuccess ||
        set_decode_smem_limits() != cudaSuccess || set_fused_smem_limit() != cudaSuccess ||
        set_gateup_tc1_smem_limit() != cudaSuccess)
      return nullptr;
    d.attrs_set = true;
  }
  return &d;
}

// This device's side stream (non-blocking, created once): independent parts of a call run
// on it, forked from and joined back into the caller's stream by events.
cudaStream_t side_stream() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo &d = g_dev[dev];
  if (!d.side && cudaStreamCreateWithFlags(&d.side, cudaStreamNonBlocking) != cudaSuccess)
    d.side = nullptr;
  return d.side;
}

// Lanes per pair in the down kernel: the largest power of two <= 32 dividing I/32 with
// at most 8 groups per lane; 0 if none.
int down_lanes(int I) {
  const int G2 = I / kGroup;
  for (int lr = 32; lr >= 1; lr >>= 1)
    if (G2 % lr == 0 && G2 / lr <= 8) return lr;
  return 0;
}

k3moe_status check_dims(const k3moe_dims *d) {
  if (!d) return K3MOE_ERR_ARG;
  if (d->group != kGroup) return K3MOE_ERR_SHAPE;
  if (d->hidden < 32 || d->hidden > 8192 || d->hidden % 32) return K3MOE_ERR_SHAPE;
  if (d->inter < 32 || d->inter > 16384 || d->inter % 32) return K3MOE_ERR_SHAPE;
  if (d->n_experts < 1 || d->n_experts > 4096) return K3MOE_ERR_SHAPE;
  if (d->topk < 1 || d->topk > 32 || d->topk > d->n_experts) return K3MOE_ERR_SHAPE;
  if (d->shared_inter < 0 || d->shared_inter > 65536 || d->shared_inter % 32) return K3MOE_ERR_SHAPE;
  if (!(d->situ_b1 > 0.f) || !(d->situ_b2 > 0.f)) return K3MOE_ERR_ARG;
  if (!(d->routed_scale == d->routed_scale)) return K3MOE_ERR_ARG;
  if (down_lanes(d->inter) == 0) return K3MOE_ERR_SHAPE;
  return K3MOE_OK;
}

void record_offsets(const k3moe_dims *d, int64_t off[7]) {
  const int64_t H = d->hidden, I = d->inter;
  const int64_t gp = I * (H / 2), gs = I * (H / 32), dp = H * (I / 2), ds = H * (I / 32);
  off[0] = 0;
  off[1] = gp;
  off[2] = off[1] + gs;
  off[3] = off[2] + dp;
  off[4] = off[3] + ds;
  off[5] = off[4] + gp;
  off[6] = off[5] + gs;
}

// Workspace carve-up for one pass of up to kDecodeTokens tokens.
struct Ws {
  float *sc, *ch;
  int32_t *idx;
  float *w;
  int32_t *disp;
  uint16_t *act_hi, *act_lo;
  int32_t *act_ex;
  float *act_s;
  unsigned *bar;  // grid-barrier counters of the single-token kernels (the header)
  float *gpart;   // one token: partial gate/up sums of row tiles split between CTAs
  size_t total;
};

// The first kWsHeader bytes of every workspace hold the single-token kernels' grid-wide
// counters, which must be zero before a call and are zero again after it; no layout
// places anything else there: words [0, 4 kFuMaxLayers) the fused kernel's (4 per layer),
// then those of the tensor-core gate/up (an exit counter and one per row tile).
constexpr size_t kWsHeader = 4096;
static_assert(4 * kFuMaxLayers + 1 + kTc1MaxTiles <= kWsHeader / 4, "counters overflow");

Ws ws_layout(const k3moe_dims *d, int T, void *base) {
  const int Tc = T < kDecodeTokens ? T : kDecodeTokens;
  const size_t P = (size_t)Tc * d->topk;
  size_t o = kWsHeader;
  Ws w{};
  const uintptr_t b = reinterpret_cast<uintptr_t>(base);
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += up16(bytes);
    return reinterpret_cast<uint8_t *>(b + at);
  };
  w.sc = reinterpret_cast<float *>(take((size_t)Tc * d->n_experts * 4));
  w.ch = reinterpret_cast<float *>(take((size_t)Tc * d->n_experts * 4));
  w.idx = reinterpret_cast<int32_t *>(take(P * 4));
  w.w = reinterpret_cast<float *>(take(P * 4));
  w.disp = reinterpret_cast<int32_t *>(take((size_t)disp_words((int)P) * 4));
  w.act_hi = reinterpret_cast<uint16_t *>(take(P * d->inter * 2));
  w.act_lo = reinterpret_cast<uint16_t *>(take(P * d->inter * 2));
  w.act_ex = reinterpret_cast<int32_t *>(take(P * (d->inter / kGroup) * 4));
  w.act_s = reinterpret_cast<float *>(take((size_t)Tc * (d->shared_inter > 0 ? d->shared_inter : 1) * 4));
  if (Tc == 1) {  // the tensor-core gate/up's split tiles: kTc1Pieces x 256 floats each
    const int tiles = d->topk * ((d->inter + 127) / 128);
    if (tiles <= kTc1MaxTiles)
      w.gpart = reinterpret_cast<float *>(take((size_t)tiles * kTc1Pieces * 256 * 4));
  }
  w.bar = reinterpret_cast<unsigned *>(b);  // the header
  w.total = o;
  return w;
}

k3moe_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ERR_CUDA;
}

// ---- tracing: CUDA events around every launch, durations summed per kernel ---------
enum KernelId { KID_ROUTER = 0, KID_TOPK, KID_DISPATCH, KID_GATEUP, KID_DOWN, KID_RMSNORM,
                KID_DEQUANT, KID_GATEUP_T1, KID_DOWN_TMA, KID_ROUTE_HIST, KID_ROUTE_SCATTER,
                KID_QUANT_X, KID_TC_GATEUP, KID_QUANT_ACT, KID_TC_DOWN, KID_TC_SH_GATEUP,
                KID_SPLIT, KID_TC_SH_DOWN, KID_COMBINE, KID_NORMS, KID_TC_ROUTER,
                KID_ROUTE_CAND, KID_DECODE_FUSED, KID_PROJ, KID_SHARED_GATEUP, KID_RMSNORM_F32,
                KID_PROJ_UP, KID_PROJ_SHARED_DOWN, KID_GATEUP_TC1, KID_ROUTER_T1, KID_DOWN_T1,
                KID_COUNT };
const char *const kKernelNames[KID_COUNT] = {
    "k_router_shared", "k_topk", "k_dispatch", "k_expert_gateup", "k_down_combine",
    "k_rmsnorm_bf16", "k_dequant", "k_gateup_t1", "k_down_tma", "k_route_hist",
    "k_route_scatter", "k_quant_x", "k_tc_gemm_gateup", "k_quant_act", "k_tc_gemm_down",
    "k_tc_gemm_shared_gateup", "k_split_bf16", "k_tc_gemm_shared_down", "k_combine",
    "k_row_norms", "k_tc_gemm_router", "k_route_candidates", "k_decode_fused", "k_proj_down",
    "k_proj_shared_gateup", "k_rmsnorm_f32w", "k_proj_up", "k_proj_shared_down",
    "k_gateup_tc1", "k_router_t1", "k_down_t1"};
struct TraceRec {
  int kid;
  cudaEvent_t a, b;
};
struct Trace {
  bool on = false;
  std::vector<TraceRec> pending;
  std::vector<cudaEvent_t> pool;
  double total_ms[KID_COUNT] = {};
  long long launches[KID_COUNT] = {};
} g_trace;

cudaEvent_t trace_event() {
  if (!g_trace.pool.empty()) {
    cudaEvent_t e = g_trace.pool.back();
    g_trace.pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Brackets one launch: call with the kernel id before (returns a token) and after.
struct TraceScope {
  int kid;
  cudaStream_t st;
  cudaEvent_t a = nullptr;
  TraceScope(int k, cudaStream_t s) : kid(k), st(s) {
    if (g_trace.on) {
      std::lock_guard<std::mutex> lk(g_mu);
      a = trace_event();
      cudaEventRecord(a, st);
    }
  }
  ~TraceScope() {
    if (a) {
      std::lock_guard<std::mutex> lk(g_mu);
      cudaEvent_t b = trace_event();
      cudaEventRecord(b, st);
      g_trace.pending.push_back({kid, a, b});
    }
  }
};

void trace_drain() {
  for (auto &r : g_trace.pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) == cudaSuccess && cudaEventElapsedTime(&ms, r.a, r.b) == cudaSuccess) {
      g_trace.total_ms[r.kid] += ms;
      g_trace.launches[r.kid] += 1;
    }
    g_trace.pool.push_back(r.a);
    g_trace.pool.push_back(r.b);
  }
  g_trace.pending.clear();
}

int tok_chunk_router(int H) {
  int tc = (160 * 1024) / (2 * H);
  if (tc > kTokChunk) tc = kTokChunk;
  return tc < 1 ? 1 : tc;
}

// Router scores (+ shared gate/up when sh_gate != NULL) for Tc tokens; then the top-k
// kernel unless the caller fuses it into the next kernel (topk = false).
k3moe_status run_route(const DeviceInfo *di, const k3moe_dims *d, const uint16_t *x, int Tc,
                       const uint16_t *wr, const float *bias, const uint16_t *sh_gate,
                       const uint16_t *sh_up, Ws &ws, int32_t *idx, float *w, int32_t *status,
                       cudaStream_t st, bool topk) {
  const int H = d->hidden, E = d->n_experts, SI = sh_gate ? d->shared_inter : 0;
  int tc = tok_chunk_router(H);
  if (tc > Tc) tc = Tc;
  const int rows = E + SI;
  int grid = (rows + 7) / 8;
  if (grid > 8 * di->sms) grid = 8 * di->sms;
  {
    TraceScope ts(Tc == 1 ? KID_ROUTER_T1 : KID_ROUTER, st);
    const cudaError_t e =
        (Tc == 1) ? launch_router_t1(st, x, H, wr, E, bias, sh_gate, sh_up, SI, d->situ_b1,
                                     d->situ_b2, ws.sc, ws.ch, ws.act_s, status, !g_trace.on)
                  : launch_router_shared(tc, grid, (size_t)tc * H * 2, st, x, Tc, H, wr, E, bias,
                                         sh_gate, sh_up, SI, d->situ_b1, d->situ_b2, ws.sc,
                                         ws.ch, ws.act_s, status);
    if (e != cudaSuccess) return K3MOE_ERR_CUDA;
  }
  if (topk) {
    TraceScope ts(KID_TOPK, st);
    k_topk<<<Tc, 512, (size_t)topk_scratch_keys(E, d->topk) * 8, st>>>(
        ws.sc, ws.ch, Tc, E, d->topk, d->renorm, d->routed_scale, idx, w, status);
  }
  return launch_status();
}

// Row-block size of the single-token gate/up kernel: 8 rows (fewer, larger stages: less
// per-stage work in the consumers and larger bulk copies) when 8 rows of scale bytes are
// a 16-byte multiple, else 16; 0 if the kernel does not apply (fewer than 32 or more
// than 224 groups per row, or a stage above 64 KB).
int t1_row_block(int H) {
  const int G = H / kGroup;
  if (G < 32 || G > 224) return 0;
  const int rb = (G % 2 == 0) ? 8 : 16;
  if ((size_t)2 * rb * (H / 2 + G) > 64 * 1024) return 0;
  return rb;
}

// Ring slots of the bulk-copy down kernel for this shape (0: use the register kernel) and
// whether the activations of all pairs are staged in its shared memory.
int down_slots(int I, int Tc, int K, int ntl, bool *act_smem) {
  const int G2 = I / kGroup;
  *act_smem = false;
  if (G2 % 16 != 0 || G2 / 16 > 8) return 0;
  const int P = Tc * K;
  const size_t stage = (size_t)8 * (I / 2 + G2);  // 8-row half tiles
  const size_t avail = 227 * 1024;
  // one slot per consumer warp (16): all of them when they fit
  const size_t fa = down_tma_smem(I, Tc, P, 0, true, ntl);
  if (fa + 16 * stage <= avail) {
    *act_smem = true;
    return 16;
  }
  const size_t fg = down_tma_smem(I, Tc, P, 0, false, ntl);
  if (fg + stage > avail) return 0;
  const int ns = (int)((avail - fg) / stage);
  return ns > 16 ? 16 : ns;
}

ExpertArgs expert_args(const k3moe_dims *d, const k3moe_experts *ex) {
  ExpertArgs ea;
  ea.base = ex->experts;
  ea.stride = ex->expert_stride;
  int64_t off[7];
  record_offsets(d, off);
  for (int i = 0; i < 6; i++) ea.off[i] = off[i];
  return ea;
}

// Down projection + combine (+ shared expert) for Tc tokens: the bulk-copy ring kernel
// when its slots fit in shared memory, else the register kernel.
k3moe_status run_down(const DeviceInfo *di, const k3moe_dims *d, int Tc, const ExpertArgs &ea,
                      const int32_t *idx, const float *w, const uint16_t *sh_down, Ws &ws,
                      void *y, k3moe_dtype ydt, int accumulate, int32_t *status, cudaStream_t st,
                      bool pdl) {
  const int H = d->hidden, I = d->inter, K = d->topk;
  const int P = Tc * K;
  const int LR = down_lanes(I);
  bool act_smem = false;
  int dgrid = H / kDownRows;
  if (dgrid > di->sms) dgrid = di->sms;
  const int ns1 = (Tc == 1 && sh_down == nullptr) ? down_t1_slots(H, I, K, di->sms) : 0;
  if (ns1 >= 3) {
    // one token, no shared expert: whole-expert stages carrying their activations
    TraceScope ts(KID_DOWN_T1, st);
    DownArgs a{};
    a.T = 1; a.H = H; a.I = I; a.K = K; a.P = P;
    a.ex = ea;
    a.idx = idx; a.w = w; a.disp = ws.disp;
    a.act_hi = ws.act_hi; a.act_lo = ws.act_lo; a.act_ex = ws.act_ex;
    a.y = y; a.ydt = (int)ydt; a.accumulate = accumulate; a.NS = ns1;
    a.status = status;
    return launch_down_t1(a, di->sms, st, pdl) == cudaSuccess ? K3MOE_OK : K3MOE_ERR_CUDA;
  }
  const int ns = down_slots(I, Tc, K, (H / kDownRows + dgrid - 1) / dgrid, &act_smem);
  TraceScope ts(ns >= 1 ? KID_DOWN_TMA : KID_DOWN, st);
  if (ns >= 1) {
    DownArgs a;
    a.T = Tc; a.H = H; a.I = I; a.K = K; a.P = P;
    a.ex = ea;
    a.idx = idx; a.w = w; a.disp = ws.disp;
    a.act_hi = ws.act_hi; a.act_lo = ws.act_lo; a.act_ex = ws.act_ex;
    a.sh_down = sh_down; a.SI = sh_down ? d->shared_inter : 0; a.act_s = ws.act_s;
    a.y = y; a.ydt = (int)ydt; a.accumulate = accumulate; a.LR = LR; a.NS = ns;
    a.status = status;
    return launch_down_tma(a, dgrid, st, pdl, act_smem) == cudaSuccess ? K3MOE_OK : K3MOE_ERR_CUDA;
  }
  const size_t dsmem = ((size_t)P * kDownRows + 256 * kDownRows + (size_t)Tc * kDownRows) * 4;
  k_down_combine<<<H / kDownRows, 256, dsmem, st>>>(Tc, H, I, K, ea, idx, w, ws.disp, P,
                                                    ws.act_hi, ws.act_lo, ws.act_ex, sh_down,
                                                    sh_down ? d->shared_inter : 0, ws.act_s, y,
                                                    (int)ydt, accumulate, LR);
  return launch_status();
}

// Dispatch + gate/up + down/combine for Tc tokens with a given route; x is bf16 [Tc][H],
// or float [Tc][H] when x_f32 (the LatentMoE's latent).
k3moe_status run_ffn(const DeviceInfo *di, const k3moe_dims *d, const void *x, int Tc,
                     const k3moe_experts *ex, const int32_t *idx, const float *w,
                     const uint16_t *sh_down, Ws &ws, void *y, k3moe_dtype ydt, int accumulate,
                     int32_t *status, cudaStream_t st, bool x_f32 = false) {
  const int H = d->hidden, I = d->inter, K = d->topk, E = d->n_experts;
  const int P = Tc * K;
  int Pp = 1;
  while (Pp < P) Pp <<= 1;
  int nt = Pp < 32 ? 32 : (Pp > 1024 ? 1024 : Pp);
  {
    TraceScope ts(KID_DISPATCH, st);
    k_dispatch<<<1, nt, (size_t)2 * Pp * 4, st>>>(idx, P, E, ws.disp, status);
  }
  const ExpertArgs ea = expert_args(d, ex);
  const int G = H / kGroup;
  const bool pathB = (G <= 16) && ((G & (G - 1)) == 0);
  const int maxU = P < E ? P : E;
  const int tiles = I / kTileRows;
  int grid = maxU * tiles;
  if (grid > 16 * di->sms) grid = 16 * di->sms;
  const int mb = (Tc == 1 || x_f32) ? 1 : 2;
  int bd = pathB ? 256 : ((G + 31) / 32) * 32;
  if (bd < 32 * mb) bd = 32 * mb;
  {
    TraceScope ts(KID_GATEUP, st);
    if (launch_expert_gateup(mb, grid, bd, st, x, x_f32, H, I, K, ea, ws.disp, P, d->situ_b1,
                             d->situ_b2, ws.act_hi, ws.act_lo, ws.act_ex) != cudaSuccess)
      return K3MOE_ERR_CUDA;
  }
  return run_down(di, d, Tc, ea, idx, w, sh_down, ws, y, ydt, accumulate, status, st, false);
}

// Exponent e with |b1 b2| 2^-e < 2^15 (at least one binade of headroom below the f16
// maximum), clamped to a range where every scale is a normal float.
int act_scale_exp(float b1, float b2) {
  const double m = std::fabs((double)b1 * (double)b2);
  int e = -100;
  if (m > 0.0) e = std::ilogb(m) + 1 - 15;
  return e < -100 ? -100 : (e > 100 ? 100 : e);
}

// Whether the single-token fused kernel takes this shape.
bool fused_takes(const DeviceInfo *di, const k3moe_dims *d) {
  return fused_t1_smem(d->hidden, d->inter, d->n_experts, d->topk, d->shared_inter, di->sms) > 0;
}

// While set, single-token fused launches wait for an arrival that never comes (test of the
// bounded-wait path).
std::atomic<int> g_expire_wait{0};

// One token through the fused kernel, for L layers (1 .. kFuMaxLayers) in one launch:
// input x (bf16; one layer), or h (float, the residual stream) normalised in the kernel
// before every layer (x = bf16(RMSNorm(h)) with eps).  Its grid-wide counters (workspace
// header) are zero on entry and left zero by the kernel's last CTA.
k3moe_status run_fused(const DeviceInfo *di, const k3moe_dims *d, const uint16_t *x,
                       const float *h, float eps, const FusedLayer *layers, int L, Ws &ws,
                       void *y, k3moe_dtype ydt, int accumulate, int32_t *status,
                       cudaStream_t st) {
  if (L < 1 || L > kFuMaxLayers || (L > 1 && !h)) return K3MOE_ERR_ARG;
  FusedT1Args a{};
  a.x = x; a.h = h; a.eps = eps;
  a.H = d->hidden; a.I = d->inter; a.E = d->n_experts; a.K = d->topk;
  a.SI = d->shared_inter;
  a.L = L;
  for (int l = 0; l < L; l++) a.lay[l] = layers[l];
  int64_t off[7];
  record_offsets(d, off);
  for (int i = 0; i < 6; i++) a.ex.off[i] = off[i];
  a.renorm = d->renorm; a.routed_scale = d->routed_scale;
  a.b1 = d->situ_b1; a.b2 = d->situ_b2;
  a.sc = ws.sc; a.ch = ws.ch; a.act_s = ws.act_s;
  a.act = ws.act_hi;
  a.bar = ws.bar;
  // |SiTU| <= b1 b2: scale the activations so that the largest stays below 2^15
  a.act_exp = act_scale_exp(d->situ_b1, d->situ_b2);
  a.y = y; a.ydt = (int)ydt; a.accumulate = accumulate;
  a.status = status;
  a.expire_dep2 = g_expire_wait.load(std::memory_order_relaxed);
  TraceScope ts(KID_DECODE_FUSED, st);
  return launch_fused_t1(a, di->sms, st) == cudaSuccess ? K3MOE_OK : K3MOE_ERR_CUDA;
}

FusedLayer fused_layer_of(const uint16_t *wr, const float *bias, const k3moe_experts *ex,
                          const uint16_t *sh_gate, const uint16_t *sh_up,
                          const uint16_t *sh_down, int32_t *idx, float *w) {
  FusedLayer f{};
  f.wr = wr; f.bias = bias;
  f.sh_gate = sh_gate; f.sh_up = sh_up; f.sh_down = sh_down;
  f.experts = ex->experts; f.stride = ex->expert_stride;
  f.idx_out = idx; f.w_out = w;
  return f;
}

// The single-token gate/up + SiTU (with the top-k and the dispatch lists): on the tensor
// cores (k_gateup_tc1, one CTA per SM) where the shape, the grid and the workspace allow
// it and the tensor maps of the expert pool encode, else k_gateup_t1 on grid_t1 CTAs.
k3moe_status run_gateup1(const DeviceInfo *di, const k3moe_dims *d, const k3moe_experts *ex,
                         const GateUpT1Args &a, Ws &ws, int grid_t1, cudaStream_t st, bool pdl) {
  int ns = 0;
  if (ws.gpart &&
      gateup_tc1_smem(d->hidden, d->inter, d->n_experts, d->topk, di->sms, &ns) > 0) {
    int64_t off[7];
    record_offsets(d, off);
    const unsigned long long H = (unsigned long long)d->hidden, I = (unsigned long long)d->inter;
    const unsigned long long E = (unsigned long long)d->n_experts;
    const unsigned long long es = (unsigned long long)ex->expert_stride;
    // gate and up as one 4-D map: K bytes, rows, {gate, up}, expert; boxes of 128 rows x
    // 128 bytes of both.  Their scales: 8-byte words (8 groups), rows, {gate, up}, expert.
    const unsigned long long dw[4] = {H / 2, I, 2, E};
    const unsigned long long sw[3] = {H / 2, (unsigned long long)(off[4] - off[0]), es};
    const unsigned bw[4] = {(unsigned)kTcChunk, (unsigned)kTcRows, 2, 1};
    const unsigned long long ds[4] = {H / 256, I, 2, E};
    const unsigned long long ss[3] = {H / kGroup, (unsigned long long)(off[5] - off[1]), es};
    const unsigned bs[4] = {2, (unsigned)kTcRows, 2, 1};
    CUtensorMap mw, ms;
    if (off[4] > off[0] && off[5] > off[1] && tc_map(&mw, ex->experts + off[0], 4, dw, sw, bw) &&
        tc_map_words(&ms, ex->experts + off[1], 4, ds, ss, bs)) {
      GateUpTc1Args t{};
      t.g = a;
      t.gpart = ws.gpart;
      t.cnt = ws.bar + 4 * kFuMaxLayers;
      t.NS = ns;
      TraceScope ts(KID_GATEUP_TC1, st);
      return launch_gateup_tc1(t, mw, ms, di->sms, st, pdl) == cudaSuccess ? K3MOE_OK
                                                                            : K3MOE_ERR_CUDA;
    }
  }
  TraceScope ts(KID_GATEUP_T1, st);
  return launch_gateup_t1(a, grid_t1, st, pdl) == cudaSuccess ? K3MOE_OK : K3MOE_ERR_CUDA;
}

// The whole layer for Tc tokens.  One token with a supported width: router kernel, then
// the single-token gate/up kernel (top-k and dispatch fused), then the down kernel, the
// last two launched as programmatic dependents so their prologues overlap the previous
// kernel's tail.  Otherwise router, top-k, dispatch, gate/up and down kernels.
k3moe_status run_layer(const DeviceInfo *di, const k3moe_dims *d, const uint16_t *x, int Tc,
                       const uint16_t *wr, const float *bias, const k3moe_experts *ex,
                       const uint16_t *sh_gate, const uint16_t *sh_up, const uint16_t *sh_down,
                       Ws &ws, int32_t *idx, float *w, void *y, k3moe_dtype ydt, int accumulate,
                       int32_t *status, cudaStream_t st) {
  if (Tc == 1 && fused_takes(di, d)) {
    const FusedLayer f = fused_layer_of(wr, bias, ex, sh_gate, sh_up, sh_down, idx, w);
    return run_fused(di, d, x, nullptr, 0.f, &f, 1, ws, y, ydt, accumulate, status, st);
  }
  const int rb = t1_row_block(d->hidden);
  if (Tc == 1 && rb > 0) {
    k3moe_status s = run_route(di, d, x, Tc, wr, bias, sh_gate, sh_up, ws, idx, w, status, st,
                               false);
    if (s != K3MOE_OK) return s;
    const ExpertArgs ea = expert_args(d, ex);
    const int H = d->hidden, G = H / kGroup;
    const size_t stage = (size_t)2 * rb * (H / 2 + G);
    int ns = (int)((227 * 1024 - gateup_t1_smem(H, d->n_experts, d->topk, rb, 0)) / stage);
    if (ns > 16) ns = 16;
    GateUpT1Args a{};
    a.x = x; a.xf = nullptr; a.H = H; a.I = d->inter; a.E = d->n_experts; a.K = d->topk;
    a.ex = ea; a.sc = ws.sc; a.ch = ws.ch; a.renorm = d->renorm;
    a.routed_scale = d->routed_scale; a.idx_out = idx; a.w_out = w; a.disp = ws.disp;
    a.b1 = d->situ_b1; a.b2 = d->situ_b2;
    a.act_hi = ws.act_hi; a.act_lo = ws.act_lo; a.act_ex = ws.act_ex;
    a.status = status; a.RB = rb; a.NS = ns;
    const bool pdl = !g_trace.on;
    {
      int grid = d->topk * (d->inter / kTileRows);
      if (grid > di->sms) grid = di->sms;
      s = run_gateup1(di, d, ex, a, ws, grid, st, pdl);
      if (s != K3MOE_OK) return s;
    }
    return run_down(di, d, Tc, ea, idx, w, sh_down, ws, y, ydt, accumulate, status, st, pdl);
  }
  k3moe_status s = run_route(di, d, x, Tc, wr, bias, sh_gate, sh_up, ws, idx, w, status, st,
                             true);
  if (s != K3MOE_OK) return s;
  return run_ffn(di, d, x, Tc, ex, idx, w, sh_down, ws, y, ydt, accumulate, status, st);
}

size_t dtype_size(k3moe_dtype t) { return t == K3MOE_F32 ? 4 : 2; }

// ---- multi-token path on the tensor cores -------------------------------------------
// Shapes it takes: H, I (and SI) multiples of 64 with rows of at least 128 bytes of
// packed MXFP4 (H, I >= 256) and of bf16 (SI >= 64).
bool tc_shape_ok(const k3moe_dims *d) {
  const int H = d->hidden, I = d->inter, SI = d->shared_inter;
  if (H % 64 || I % 64 || H < 256 || I < 256) return false;
  if (SI > 0 && (SI % 64 || SI < 64)) return false;
  return true;
}

// Workspace of one pass of up to kTcTokens tokens (P = Tc * K pairs).
struct WsTc {
  float *sc, *ch;                 // router scores [Tc][E]
  float *Lt;                      // screening logits [Tc][E]
  float *xn, *wn;                 // row norms of x [Tc] and Wr [E]
  int32_t *ncand;                 // candidates per token [Tc]
  int32_t *idx;
  float *w;
  int32_t *off, *tile_off, *inv, *perm, *off1, *tile_off1;
  int32_t *rcount;                // [ceil(P / kRouteChunk)][E] pairs per chunk and expert,
                                  // then each chunk's first position per expert
  uint8_t *xq, *xs;               // [kTcTermsX][P][H/2], [kTcTermsX][P][H/32]
  float *act;                     // [P][I]
  uint8_t *aq, *as;               // [kTcTermsAct][P][I/2], [kTcTermsAct][P][I/32]
  float *dpair;                   // [P][H]
  float *act_s;                   // [Tc][SI]
  uint16_t *hs;                   // [2][Tc][SI]
  float *ds;                      // [Tc][H]
  size_t total;
};

WsTc ws_tc_layout(const k3moe_dims *d, int T, void *base) {
  const int Tc = T < kTcTokens ? T : kTcTokens;
  const size_t H = d->hidden, I = d->inter, E = d->n_experts, SI = d->shared_inter;
  const size_t P = (size_t)Tc * d->topk;
  size_t o = kWsHeader;
  const uintptr_t b = reinterpret_cast<uintptr_t>(base);
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += (bytes + 255) & ~size_t(255);
    return reinterpret_cast<uint8_t *>(b + at);
  };
  WsTc w{};
  w.sc = reinterpret_cast<float *>(take((size_t)Tc * E * 4));
  w.ch = reinterpret_cast<float *>(take((size_t)Tc * E * 4));
  w.Lt = reinterpret_cast<float *>(take((size_t)Tc * E * 4));
  w.xn = reinterpret_cast<float *>(take((size_t)Tc * 4));
  w.wn = reinterpret_cast<float *>(take(E * 4));
  w.ncand = reinterpret_cast<int32_t *>(take((size_t)Tc * 4));
  w.idx = reinterpret_cast<int32_t *>(take(P * 4));
  w.w = reinterpret_cast<float *>(take(P * 4));
  w.off = reinterpret_cast<int32_t *>(take((E + 1) * 4));
  w.tile_off = reinterpret_cast<int32_t *>(take((E + 1) * 4));
  w.inv = reinterpret_cast<int32_t *>(take(P * 4));
  w.perm = reinterpret_cast<int32_t *>(take(P * 4));
  w.rcount = reinterpret_cast<int32_t *>(
      take((P + route_chunk((int)P) - 1) / route_chunk((int)P) * E * 4));
  w.off1 = reinterpret_cast<int32_t *>(take(8));
  w.tile_off1 = reinterpret_cast<int32_t *>(take(8));
  w.xq = take((size_t)kTcTermsX * P * (H / 2));
  w.xs = take((size_t)kTcTermsX * ((H / kGroup + 7) / 8) * P * 8);
  w.act = reinterpret_cast<float *>(take(P * I * 4));
  w.aq = take((size_t)kTcTermsAct * P * (I / 2));
  w.as = take((size_t)kTcTermsAct * ((I / kGroup + 7) / 8) * P * 8);
  w.dpair = reinterpret_cast<float *>(take(P * H * 4));
  if (SI > 0) {
    w.act_s = reinterpret_cast<float *>(take((size_t)Tc * SI * 4));
    w.hs = reinterpret_cast<uint16_t *>(take((size_t)2 * Tc * SI * 2));
    w.ds = reinterpret_cast<float *>(take((size_t)Tc * H * 4));
  }
  w.total = o;
  return w;
}

// K ranges per item for a GEMM of `items` work items over `kchunks` K chunks whose items
// alone would leave most SMs idle (few output tiles, one B tile): the largest divisor of
// kchunks up to `cap` with items x ranges <= sms.  The partial sums go to a buffer and are
// added in range order by a small kernel.
int tc_ksplit(int items, int kchunks, int sms, int cap) {
  if (2 * items > sms) return 1;
  int best = 1;
  for (int k = 2; k <= cap && k <= kchunks; k++)
    if (kchunks % k == 0 && items * k <= sms) best = k;
  return best;
}

// Token/pair tables of a tensor-core GEMM over K_bytes of K per row.
void tc_k_split(long long k_bytes, TcGemmArgs &a) {
  a.kchunks = (int)((k_bytes + kTcChunk - 1) / kTcChunk);
  a.ksteps_last = (int)((k_bytes - (long long)kTcChunk * (a.kchunks - 1) + 31) / 32);
}
// Bytes between terms of the quantised scales ([term][256-column group][row][8]).
long long tc_sf_tstride(long long k_bytes, long long cstride) {
  return (k_bytes + 127) / 128 * cstride;
}

// The shared expert of Tc tokens on the tensor cores: ds [Tc][H] = Wsd SiTU(Wsg x, Wsu x)
// (bf16 weights; the activations as bf16 hi + lo for the down GEMM).  Under split K its
// partial sums use ws.act, which the routed gate/up writes: callers run this either after
// the routed down GEMM or before the routed gate/up.  group1_done: ws.off1 / tile_off1
// already hold the one-group table of Tc rows.
k3moe_status run_shared_tc(const DeviceInfo *di, const k3moe_dims *d, const uint16_t *x, int Tc,
                           const uint16_t *sh_gate, const uint16_t *sh_up,
                           const uint16_t *sh_down, WsTc &ws, int32_t *status, cudaStream_t st,
                           bool group1_done) {
  const int H = d->hidden, I = d->inter, K = d->topk, SI = d->shared_inter;
  {
    CUtensorMap msg, msu, msd, mxs, mhs;
    const int nt1 = kTcRows;
    if (!tc_map3d(&msg, sh_gate, 2ull * H, SI, 1, 2ull * H, 2ull * H * SI, kTcRows) ||
        !tc_map3d(&msu, sh_up, 2ull * H, SI, 1, 2ull * H, 2ull * H * SI, kTcRows) ||
        !tc_map3d(&msd, sh_down, 2ull * SI, H, 1, 2ull * SI, 2ull * SI * H, kTcRows) ||
        !tc_map3d(&mxs, x, 2ull * H, Tc, 1, 2ull * H, 2ull * H * Tc, nt1) ||
        !tc_map3d(&mhs, ws.hs, 2ull * SI, Tc, 2, 2ull * SI, 2ull * SI * Tc, nt1, 2))
      return K3MOE_ERR_CUDA;
    if (!group1_done) k_group1<<<1, 32, 0, st>>>(Tc, nt1, ws.off1, ws.tile_off1);
    TcGemmArgs s1{};
    s1.b1 = d->situ_b1;
    s1.b2 = d->situ_b2;
    s1.status = status;
    s1.off = ws.off1;
    s1.tile_off = ws.tile_off1;
    s1.ngroups = 1;
    s1.ntile = nt1;
    s1.a_once = Tc <= nt1;
    {
      TcGemmArgs a = s1;
      a.mtiles = (SI + kTcRows - 1) / kTcRows;
      a.M_rows = SI;
      tc_k_split(2LL * H, a);
      a.out_ld = SI;
      TraceScope ts(KID_TC_SH_GATEUP, st);
      // few output tiles at a small batch: split K, the gate and up partials in the routed
      // activations' buffer (free once they are encoded), P x I >= KS x 2 x Tc x SI floats
      const int cap = std::min(16, (K * I) / (2 * SI));
      const int KS = Tc <= nt1 ? tc_ksplit(a.mtiles, a.kchunks, di->sms, cap) : 1;
      if (KS > 1) {
        a.ksplit = KS;
        a.out = ws.act;
        a.out_mstride = (long long)Tc * SI;
        a.out_kstride = 2LL * Tc * SI;
        if (launch_tc_gemm(TcKind::kBf16Pair, a, msg, msu, mxs, di->sms, st) != cudaSuccess ||
            launch_situ_parts(st, di->sms, ws.act, KS, 2LL * Tc * SI, (long long)Tc * SI,
                              (long long)Tc * SI, d->situ_b1, d->situ_b2, ws.act_s) !=
                cudaSuccess)
          return K3MOE_ERR_CUDA;
      } else {
        a.out = ws.act_s;
        if (launch_tc_gemm(TcKind::kBf16GateUp, a, msg, msu, mxs, di->sms, st) != cudaSuccess)
          return K3MOE_ERR_CUDA;
      }
    }
    {
      TraceScope ts(KID_SPLIT, st);
      const long long n = (long long)Tc * SI;
      int grid = (int)((n + 255) / 256);
      if (grid > 16 * di->sms) grid = 16 * di->sms;
      k_split_bf16<<<grid, 256, 0, st>>>(ws.act_s, n, ws.hs);
    }
    {
      TcGemmArgs a = s1;
      a.mtiles = (H + kTcRows - 1) / kTcRows;
      a.M_rows = H;
      tc_k_split(2LL * SI, a);
      a.out = ws.ds;
      a.out_ld = H;
      TraceScope ts(KID_TC_SH_DOWN, st);
      if (launch_tc_gemm(TcKind::kBf16Down, a, msd, msd, mhs, di->sms, st) != cudaSuccess)
        return K3MOE_ERR_CUDA;
    }
  }
  return launch_status();
}

// Expert FFN of Tc tokens on the tensor cores, given the route (idx, w [Tc][K]):
// dispatch, x encoding, gate/up + SiTU, activation encoding, down, then (with the shared
// expert when sh_gate != NULL) the router-order combine into y.  shared_done: ws.ds
// already holds the shared expert's output (run_shared_tc, run before).
k3moe_status run_ffn_tc(const DeviceInfo *di, const k3moe_dims *d, const void *x, int Tc,
                        const k3moe_experts *ex, const int32_t *idx, const float *w,
                        const uint16_t *sh_gate, const uint16_t *sh_up, const uint16_t *sh_down,
                        WsTc &ws, void *y, k3moe_dtype ydt, int accumulate, int32_t *status,
                        cudaStream_t st, bool x_f32 = false, bool shared_done = false) {
  if (x_f32 && sh_gate) return K3MOE_ERR_ARG;  // the shared GEMMs take bf16 x
  const int H = d->hidden, I = d->inter, E = d->n_experts, K = d->topk;
  const int SI = sh_gate ? d->shared_inter : 0;
  const int P = Tc * K;
  int64_t off[7];
  record_offsets(d, off);
  const uint8_t *rec = ex->experts;
  const unsigned long long es = (unsigned long long)ex->expert_stride;
  // B rows per tile: 1.25 x the mean number of pairs per expert, rounded up to a power of
  // two from 16 to 128 (few experts then need a second tile; measured, heights of 48 and
  // 96 rows run slower than the powers of two beside them: 4096 tokens 7.40 ms at 96 rows,
  // 6.85 ms at 128)
  const int used = P < E ? P : E;
  const int want = (5 * P + 4 * used - 1) / (4 * used);
  int ntile = 16;
  while (ntile < want && ntile < kTcRows) ntile *= 2;
  const int chunk = route_chunk(P), nch = (P + chunk - 1) / chunk;
  {
    TraceScope ts(KID_ROUTE_HIST, st);
    k_route_count<<<nch, 256, (size_t)E * 4, st>>>(idx, P, E, chunk, ws.rcount, ws.inv, status);
    k_route_hist<<<1, 1024, (size_t)E * 4, st>>>(ws.rcount, nch, E, ntile, ws.off, ws.tile_off);
  }
  {
    TraceScope ts(KID_ROUTE_SCATTER, st);
    k_route_scatter<<<nch, 256, (size_t)(E + chunk) * 4, st>>>(idx, P, E, chunk, ws.rcount,
                                                               ws.perm, ws.inv);
  }
  {
    TraceScope ts(KID_QUANT_X, st);
    const long long n = (long long)Tc * (H / kGroup);
    int grid = (int)((n + 255) / 256);
    if (grid > 16 * di->sms) grid = 16 * di->sms;
    if (launch_quant_x(x_f32, grid, st, x, Tc, H, K, ws.inv, P, ws.xq, ws.xs) != cudaSuccess)
      return K3MOE_ERR_CUDA;
  }
  if (launch_status() != K3MOE_OK) return K3MOE_ERR_CUDA;
  // gate and up packed matrices of every expert as one 4-D map (K bytes, rows, matrix,
  // expert): the up matrix sits at a fixed offset after the gate matrix in each record
  CUtensorMap mgu, md, mx, ma;
  const unsigned long long gu_dims[4] = {(unsigned long long)H / 2, (unsigned long long)I, 2,
                                         (unsigned long long)E};
  const unsigned long long gu_strides[3] = {(unsigned long long)H / 2,
                                            (unsigned long long)(off[4] - off[0]),
                                            (unsigned long long)es};
  const unsigned gu_box[4] = {(unsigned)kTcChunk, (unsigned)kTcRows, 2, 1};  // K chunk x 128 rows x both
  if (!tc_map(&mgu, rec + off[0], 4, gu_dims, gu_strides, gu_box) ||
      !tc_map3d(&md, rec + off[2], I / 2, H, E, I / 2, es, kTcRows) ||
      !tc_map3d(&mx, ws.xq, H / 2, P, kTcTermsX, H / 2, (unsigned long long)P * (H / 2), ntile,
                kTcTermsX) ||
      !tc_map3d(&ma, ws.aq, I / 2, P, kTcTermsAct, I / 2, (unsigned long long)P * (I / 2), ntile,
                kTcTermsAct))
    return K3MOE_ERR_CUDA;
  TcGemmArgs g{};
  g.off = ws.off;
  g.tile_off = ws.tile_off;
  g.gid = nullptr;
  g.ngroups = E;
  g.ntile = ntile;
  g.a_once = Tc <= ntile;  // a token picks an expert once: at most Tc rows per group
  g.b1 = d->situ_b1;
  g.b2 = d->situ_b2;
  g.status = status;
  {
    TcGemmArgs a = g;
    a.mtiles = (I + kTcRows - 1) / kTcRows;
    a.M_rows = I;
    tc_k_split(H / 2, a);
    a.sfa[0] = rec + off[1];
    a.sfa[1] = rec + off[5];
    a.sfa_gstride = ex->expert_stride;
    a.sf_rowb = H / kGroup;
    a.sfb = ws.xs;
    a.sfb_cstride = (long long)P * 8;
    a.sfb_tstride = tc_sf_tstride(H / 2, a.sfb_cstride);
    a.out = ws.act;
    a.out_ld = I;
    a.a_pair = 1;
    TraceScope ts(KID_TC_GATEUP, st);
    if (launch_tc_gemm(TcKind::kMxf4GateUp, a, mgu, mgu, mx, di->sms, st) != cudaSuccess)
      return K3MOE_ERR_CUDA;
  }
  {
    TraceScope ts(KID_QUANT_ACT, st);
    const long long n = (long long)P * (I / kGroup);
    int grid = (int)((n + 255) / 256);
    if (grid > 16 * di->sms) grid = 16 * di->sms;
    k_quant_act<<<grid, 256, 0, st>>>(ws.act, P, I, ws.aq, ws.as);
  }
  {
    // down: two consecutive 128-row tiles of W2 per item when H is a multiple of 256, so
    // that they share one B stage (half the activation traffic per output row)
    const bool pair = H % (2 * kTcRows) == 0;
    TcGemmArgs a = g;
    a.mtiles = pair ? H / (2 * kTcRows) : (H + kTcRows - 1) / kTcRows;
    a.M_rows = H;
    tc_k_split(I / 2, a);
    a.sfa[0] = rec + off[3];
    a.sfa[1] = pair ? rec + off[3] : nullptr;
    a.sfa_gstride = ex->expert_stride;
    a.sf_rowb = I / kGroup;
    a.sfb = ws.as;
    a.sfb_cstride = (long long)P * 8;
    a.sfb_tstride = tc_sf_tstride(I / 2, a.sfb_cstride);
    a.out = ws.dpair;
    a.out_ld = H;
    a.a_pair = pair ? 2 : 0;
    CUtensorMap md2;
    if (pair) {
      const unsigned long long d_dims[4] = {(unsigned long long)I / 2, (unsigned long long)kTcRows,
                                            (unsigned long long)H / kTcRows,
                                            (unsigned long long)E};
      const unsigned long long d_strides[3] = {(unsigned long long)I / 2,
                                               (unsigned long long)kTcRows * (I / 2), es};
      const unsigned d_box[4] = {(unsigned)kTcChunk, (unsigned)kTcRows, 2, 1};
      if (!tc_map(&md2, rec + off[2], 4, d_dims, d_strides, d_box)) return K3MOE_ERR_CUDA;
    }
    TraceScope ts(KID_TC_DOWN, st);
    if (launch_tc_gemm(pair ? TcKind::kMxf4DownPair : TcKind::kMxf4Down, a, pair ? md2 : md,
                       pair ? md2 : md, ma, di->sms, st) != cudaSuccess)
      return K3MOE_ERR_CUDA;
  }
  if (SI > 0 && !shared_done) {
    const k3moe_status r = run_shared_tc(di, d, static_cast<const uint16_t *>(x), Tc, sh_gate,
                                         sh_up, sh_down, ws, status, st, false);
    if (r != K3MOE_OK) return r;
  }
  {
    TraceScope ts(KID_COMBINE, st);
    k_combine<<<dim3(Tc, (H / 4 + 255) / 256), 256, (size_t)2 * K * 4, st>>>(Tc, H, K, w, ws.inv, ws.dpair,
                                                 SI > 0 ? ws.ds : nullptr, y, (int)ydt,
                                                 accumulate);
  }
  return launch_status();
}

// Route Tc tokens into idx/w [Tc][K] for the tensor-core path: screening logits and
// their error bounds on the tensor cores, exact scores for the candidates, then top-k.
k3moe_status run_route_tc(const DeviceInfo *di, const k3moe_dims *d, const uint16_t *x, int Tc,
                          const uint16_t *wr, const float *bias, WsTc &wt, int32_t *idx,
                          float *w, int32_t *status, cudaStream_t st,
                          bool group1_done = false) {
  const int H = d->hidden, E = d->n_experts, K = d->topk;
  {
    TraceScope ts(KID_NORMS, st);
    k_row_norms<<<Tc + E, 128, 0, st>>>(x, Tc, wt.xn, wr, E, wt.wn, H);
  }
  if (!group1_done) k_group1<<<1, 32, 0, st>>>(Tc, kTcRows, wt.off1, wt.tile_off1);
  CUtensorMap mw, mx;
  if (!tc_map3d(&mw, wr, 2ull * H, E, 1, 2ull * H, 2ull * H * E, kTcRows) ||
      !tc_map3d(&mx, x, 2ull * H, Tc, 1, 2ull * H, 2ull * H * Tc, kTcRows))
    return K3MOE_ERR_CUDA;
  TcGemmArgs a{};
  int nadd = H;
  a.off = wt.off1;
  a.tile_off = wt.tile_off1;
  a.ngroups = 1;
  a.ntile = kTcRows;
  a.a_once = Tc <= kTcRows;
  a.mtiles = (E + kTcRows - 1) / kTcRows;
  a.M_rows = E;
  tc_k_split(2LL * H, a);
  a.out_ld = E;
  a.status = status;
  {
    TraceScope ts(KID_TC_ROUTER, st);
    // split K, partials in the (still unused) per-pair down-output buffer, which holds
    // P x H >= KS x Tc x E floats for KS <= K H / E: at a small batch because its few
    // output tiles alone would leave most SMs idle; at a large one for the screening
    // bound (H / KS + KS additions instead of H, so fewer candidates need exact logits)
    const int cap = std::min(16, (int)((long long)K * H / E));
    int KS = Tc <= kTcRows ? tc_ksplit(a.mtiles, a.kchunks, di->sms, cap) : 1;
    if (Tc > kTcRows && cap >= 8 && a.kchunks % 8 == 0) KS = 8;
    nadd = KS > 1 ? H / KS + KS : H;  // the longest chain of additions behind a logit
    a.ksplit = KS;
    a.out_kstride = (long long)Tc * E;
    a.out = KS > 1 ? wt.dpair : wt.Lt;
    if (launch_tc_gemm(TcKind::kBf16Store, a, mw, mw, mx, di->sms, st) != cudaSuccess)
      return K3MOE_ERR_CUDA;
    if (KS > 1 && launch_sum_parts(st, di->sms, wt.dpair, KS, (long long)Tc * E,
                                   (long long)Tc * E, wt.Lt) != cudaSuccess)
      return K3MOE_ERR_CUDA;
  }
  {
    TraceScope ts(KID_ROUTE_CAND, st);
    // enough blocks per token to cover the SMs twice, at most 8
    const int split = std::max(1, std::min(8, (2 * di->sms + Tc - 1) / Tc));
    k_route_candidates<<<dim3(Tc, split), 256, route_candidates_smem(H, E, K), st>>>(
        wt.Lt, wt.xn, wt.wn, x, wr, bias, H, E, K, nadd, wt.sc, wt.ch, wt.ncand, status);
  }
  {
    TraceScope ts(KID_TOPK, st);
    k_topk<<<Tc, 512, (size_t)topk_scratch_keys(E, K) * 8, st>>>(
        wt.sc, wt.ch, Tc, E, K, d->renorm, d->routed_scale, idx, w, status);
  }
  return launch_status();
}

// The tensor-core path applies from two tokens on, for the shapes it takes.
bool use_tc(const k3moe_dims *d, int T) { return T >= 2 && tc_shape_ok(d); }

// ---- the LatentMoE layer ---------------------------------------------------------------
// The router's dims (full width) and the experts' dims (in the latent, no shared expert)
// of a LatentMoE layer.
k3moe_status latent_dims(const k3moe_latent_dims *d, k3moe_dims *full, k3moe_dims *lat) {
  if (!d) return K3MOE_ERR_ARG;
  if (d->latent < 32 || d->latent > 8192 || d->latent % 32) return K3MOE_ERR_SHAPE;
  if (d->latent_norm && !(d->rms_eps >= 0.f)) return K3MOE_ERR_ARG;
  *full = k3moe_dims{d->hidden, d->inter, d->n_experts, d->topk, d->group, d->shared_inter,
                     d->situ_b1, d->situ_b2, d->routed_scale, d->renorm};
  *lat = k3moe_dims{d->latent, d->inter, d->n_experts, d->topk, d->group, 0,
                    d->situ_b1, d->situ_b2, d->routed_scale, d->renorm};
  k3moe_status s = check_dims(full);
  return s != K3MOE_OK ? s : check_dims(lat);
}

// Workspace of one pass of up to kDecodeTokens tokens: the router's part, the experts'
// part, then z [Tc][L], the latent sum [Tc][L], the up-projection [Tc][H] and the shared
// activations [Tc][SI] (float); for passes of two tokens or more at a latent shape the
// grouped GEMMs take, the tensor-core experts' part after them.
struct WsLatent {
  Ws route, ffn;
  float *z, *accl, *up, *act_s;
  bool has_tc;
  WsTc tc;
  uint16_t *hs;    // [2][Tc][L] bf16 hi / lo terms of the latent sum (tensor-core passes)
  uint16_t *hs_s;  // [2][Tc][SI] the same of the shared activations
  float *ds;       // [Tc][H] shared experts' output
  size_t total;
};

WsLatent ws_latent_layout(const k3moe_dims *full, const k3moe_dims *lat, int T, void *base) {
  const int Tc = T < kDecodeTokens ? T : kDecodeTokens;
  WsLatent w{};
  const uintptr_t b = reinterpret_cast<uintptr_t>(base);
  w.route = ws_layout(full, Tc, base);
  size_t o = w.route.total;
  w.ffn = ws_layout(lat, Tc, reinterpret_cast<void *>(b + o));
  o += w.ffn.total;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += up16(bytes);
    return reinterpret_cast<float *>(b + at);
  };
  const size_t L = lat->hidden, H = full->hidden, SI = full->shared_inter;
  w.z = take((size_t)Tc * L * 4);
  w.accl = take((size_t)Tc * L * 4);
  w.up = take((size_t)Tc * H * 4);
  w.act_s = take((size_t)Tc * (SI > 0 ? SI : 1) * 4);
  w.ds = take((size_t)Tc * H * 4);
  w.has_tc = use_tc(lat, Tc) && use_tc(full, Tc);
  if (w.has_tc) {
    w.tc = ws_tc_layout(lat, Tc, reinterpret_cast<void *>(b + o));
    o += up16(w.tc.total);
    w.hs = reinterpret_cast<uint16_t *>(take((size_t)2 * Tc * L * 2));
    w.hs_s = reinterpret_cast<uint16_t *>(take((size_t)2 * Tc * (SI > 0 ? SI : 1) * 2));
  }
  w.total = o;
  return w;
}

// out[t][r] (float, row length R) = sum_c A0[r][c] B[t][c] on the tensor cores for a bf16
// matrix A0 [R][C] and B given as nb bf16 terms [nb][Tc][C] (their products summed); with A1
// (the same shape) the output is SiTU(A0 B, A1 B).  g carries the one-group table of the Tc
// rows (k_group1), the SiTU caps and the status word.
k3moe_status tc_bf16_gemm(const DeviceInfo *di, TcKind kind, const uint16_t *A0,
                          const uint16_t *A1, int R, int C, const uint16_t *B, int nb, int Tc,
                          float *out, const TcGemmArgs &g, cudaStream_t st) {
  CUtensorMap ma0, ma1, mb;
  const unsigned long long rb = 2ull * C;
  if (!tc_map3d(&ma0, A0, rb, R, 1, rb, rb * R, kTcRows) ||
      (A1 && !tc_map3d(&ma1, A1, rb, R, 1, rb, rb * R, kTcRows)) ||
      !tc_map3d(&mb, B, rb, Tc, nb, rb, rb * Tc, g.ntile, nb))
    return K3MOE_ERR_CUDA;
  TcGemmArgs a = g;
  a.mtiles = (R + kTcRows - 1) / kTcRows;
  a.M_rows = R;
  tc_k_split((long long)rb, a);
  a.out = out;
  a.out_ld = R;
  return launch_tc_gemm(kind, a, ma0, A1 ? ma1 : ma0, mb, di->sms, st) == cudaSuccess
             ? K3MOE_OK
             : K3MOE_ERR_CUDA;
}

k3moe_status launch_split(const DeviceInfo *di, const float *v, long long n, uint16_t *out,
                          cudaStream_t st) {
  TraceScope ts(KID_SPLIT, st);
  int grid = (int)((n + 255) / 256);
  if (grid > 16 * di->sms) grid = 16 * di->sms;
  k_split_bf16<<<grid, 256, 0, st>>>(v, n, out);
  return launch_status();
}

// The LatentMoE's shared experts of one pass, ds = Wsd SiTU(Wsg x, Wsu x) [Tc][H] float,
// enqueued on the side stream after an event recorded on st (they read only x and write
// only act_s / hs_s / ds); *join is recorded after them for st to wait on.
k3moe_status run_latent_shared(const DeviceInfo *di, const k3moe_latent_weights *lw,
                               const uint16_t *xc, int Tc, int H, int SI, bool proj_tc,
                               const TcGemmArgs &g1, const WsLatent &ws, float b1, float b2,
                               cudaStream_t st, cudaEvent_t *join) {
  cudaStream_t ss = side_stream();
  cudaEvent_t fork = nullptr;
  if (!ss || cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) != cudaSuccess)
    return K3MOE_ERR_CUDA;
  if (cudaEventCreateWithFlags(join, cudaEventDisableTiming) != cudaSuccess) {
    cudaEventDestroy(fork);
    return K3MOE_ERR_CUDA;
  }
  const bool forked = cudaEventRecord(fork, st) == cudaSuccess &&
                      cudaStreamWaitEvent(ss, fork, 0) == cudaSuccess;
  cudaEventDestroy(fork);
  if (!forked) return K3MOE_ERR_CUDA;
  k3moe_status s = K3MOE_OK;
  if (proj_tc) {
    {
      TraceScope ts(KID_SHARED_GATEUP, ss);
      s = tc_bf16_gemm(di, TcKind::kBf16GateUp, lw->sh_gate, lw->sh_up, SI, H, xc, 1, Tc,
                       ws.act_s, g1, ss);
    }
    if (s == K3MOE_OK) s = launch_split(di, ws.act_s, (long long)Tc * SI, ws.hs_s, ss);
    if (s == K3MOE_OK) {
      TraceScope ts(KID_PROJ_SHARED_DOWN, ss);
      s = tc_bf16_gemm(di, TcKind::kBf16Down, lw->sh_down, nullptr, H, SI, ws.hs_s, 2, Tc,
                       ws.ds, g1, ss);
    }
  } else {
    {
      TraceScope ts(KID_SHARED_GATEUP, ss);
      if (launch_proj(ss, di->sms, lw->sh_gate, lw->sh_up, SI, H, xc, false, Tc, ws.act_s,
                      nullptr, nullptr, 0, 0, b1, b2, false) != cudaSuccess)
        s = K3MOE_ERR_CUDA;
    }
    if (s == K3MOE_OK) {
      TraceScope ts(KID_PROJ_SHARED_DOWN, ss);
      if (launch_proj(ss, di->sms, lw->sh_down, nullptr, H, SI, ws.act_s, true, Tc, ws.ds,
                      nullptr, nullptr, 0, 0, b1, b2, false) != cudaSuccess)
        s = K3MOE_ERR_CUDA;
    }
  }
  // recorded whatever happened, so that st never waits on an event with nothing behind it
  if (cudaEventRecord(*join, ss) != cudaSuccess) s = K3MOE_ERR_CUDA;
  return s;
}

}  // namespace

// ---- scratch of k3moe_layer_static_scratch -------------------------------------------
// A static device array: every device that loads this library's device code gets its own
// copy, reserved when the code is loaded, so the call that uses it allocates nothing.
static __device__ __align__(256) uint8_t g_static_scratch[K3MOE_STATIC_SCRATCH_BYTES];

namespace {

void *g_static_scratch_addr[kMaxDevices];

// Device address of the current device's copy of g_static_scratch, looked up on the
// first call made with that device current; nullptr if the lookup fails.
void *static_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_static_scratch_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // leave no stale error for the next launch check
      return nullptr;
    }
    g_static_scratch_addr[dev] = p;
  }
  return g_static_scratch_addr[dev];
}

}  // namespace

extern "C" {

const char *k3moe_status_str(k3moe_status s) {
  switch (s) {
    case K3MOE_OK: return "ok";
    case K3MOE_ERR_ARG: return "invalid argument";
    case K3MOE_ERR_SHAPE: return "unsupported shape";
    case K3MOE_ERR_ALIGN: return "pointer or stride not 16-byte aligned";
    case K3MOE_ERR_WORKSPACE: return "workspace too small";
    case K3MOE_ERR_CUDA: return "CUDA launch failed";
    case K3MOE_ERR_TIMEOUT: return "device wait timed out";
    case K3MOE_ERR_BAD_EXPERT: return "expert index out of range";
    case K3MOE_ERR_NONFINITE: return "non-finite router score";
    case K3MOE_ERR_SCRATCH_LIMIT:
      return "call needs more scratch than the static array holds (K3MOE_STATIC_SCRATCH_BYTES)";
    case K3MOE_ERR_CACHE_FULL: return "the call's distinct experts exceed the cache's slots";
  }
  return "unknown status";
}

k3moe_status k3moe_record_layout(const k3moe_dims *dims, int64_t offsets[7]) {
  const k3moe_status s = check_dims(dims);
  if (s != K3MOE_OK) return s;
  if (!offsets) return K3MOE_ERR_ARG;
  record_offsets(dims, offsets);
  return K3MOE_OK;
}

size_t k3moe_workspace_size(const k3moe_dims *dims, int32_t T) {
  if (check_dims(dims) != K3MOE_OK || T < 0) return 0;
  if (T == 0) return 16;
  const size_t base = ws_layout(dims, T, nullptr).total;
  if (use_tc(dims, T)) {
    const size_t tc = ws_tc_layout(dims, T, nullptr).total;
    return tc > base ? tc : base;
  }
  return base;
}

k3moe_status k3moe_route(const k3moe_dims *dims, const uint16_t *x_bf16, const uint16_t *wr_bf16,
                         const float *bias, int32_t T, int32_t *idx, float *w, void *workspace,
                         size_t ws_bytes, int32_t *status_dev, k3moe_stream_t stream) {
  k3moe_status s = check_dims(dims);
  if (s != K3MOE_OK) return s;
  if (T < 0) return K3MOE_ERR_ARG;
  if (T == 0) return K3MOE_OK;
  if (!x_bf16 || !wr_bf16 || !idx || !w || !workspace || !status_dev) return K3MOE_ERR_ARG;
  if (!aligned16(x_bf16) || !aligned16(wr_bf16) || !aligned16(workspace) ||
      (bias && !aligned16(bias)) || !aligned16(idx) || !aligned16(w))
    return K3MOE_ERR_ALIGN;
  if (ws_bytes < k3moe_workspace_size(dims, T)) return K3MOE_ERR_WORKSPACE;
  const DeviceInfo *di = device_info();
  if (!di) return K3MOE_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  Ws ws = ws_layout(dims, T, workspace);
  const int H = dims->hidden, K = dims->topk;
  for (int t0 = 0; t0 < T; t0 += kDecodeTokens) {
    const int Tc = (T - t0) < kDecodeTokens ? (T - t0) : kDecodeTokens;
    s = run_route(di, dims, x_bf16 + (size_t)t0 * H, Tc, wr_bf16, bias, nullptr, nullptr, ws,
                  idx + (size_t)t0 * K, w + (size_t)t0 * K, status_dev, st, true);
    if (s != K3MOE_OK) return s;
  }
  return K3MOE_OK;
}

k3moe_status k3moe_expert_ffn_mxfp4(const k3moe_dims *dims, const uint16_t *x_bf16, int32_t T,
                                    const k3moe_experts *experts, const int32_t *idx,
                                    const float *w, void *y, k3moe_dtype ydt, int32_t accumulate,
                                    void *workspace, size_t ws_bytes, int32_t *status_dev,
                                    k3moe_stream_t stream) {
  k3moe_status s = check_dims(dims);
  if (s != K3MOE_OK) return s;
  if (T < 0 || (ydt != K3MOE_F32 && ydt != K3MOE_BF16)) return K3MOE_ERR_ARG;
  if (T == 0) return K3MOE_OK;
  if (!x_bf16 || !experts || !experts->experts || !idx || !w || !y || !workspace || !status_dev)
    return K3MOE_ERR_ARG;
  int64_t off[7];
  record_offsets(dims, off);
  if (experts->expert_stride < off[6] || experts->expert_stride % 16) return K3MOE_ERR_ALIGN;
  if (!aligned16(x_bf16) || !aligned16(experts->experts) || !aligned16(idx) || !aligned16(w) ||
      !aligned16(y) || !aligned16(workspace))
    return K3MOE_ERR_ALIGN;
  if (ws_bytes < k3moe_workspace_size(dims, T)) return K3MOE_ERR_WORKSPACE;
  const DeviceInfo *di = device_info();
  if (!di) return K3MOE_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int H = dims->hidden, K = dims->topk;
  if (use_tc(dims, T)) {
    WsTc wt = ws_tc_layout(dims, T, workspace);
    for (int t0 = 0; t0 < T; t0 += kTcTokens) {
      const int Tc = (T - t0) < kTcTokens ? (T - t0) : kTcTokens;
      s = run_ffn_tc(di, dims, x_bf16 + (size_t)t0 * H, Tc, experts, idx + (size_t)t0 * K,
                     w + (size_t)t0 * K, nullptr, nullptr, nullptr, wt,
                     static_cast<uint8_t *>(y) + (size_t)t0 * H * dtype_size(ydt), ydt,
                     accumulate, status_dev, st);
      if (s != K3MOE_OK) return s;
    }
    return K3MOE_OK;
  }
  Ws ws = ws_layout(dims, T, workspace);
  for (int t0 = 0; t0 < T; t0 += kDecodeTokens) {
    const int Tc = (T - t0) < kDecodeTokens ? (T - t0) : kDecodeTokens;
    s = run_ffn(di, dims, x_bf16 + (size_t)t0 * H, Tc, experts, idx + (size_t)t0 * K,
                w + (size_t)t0 * K, nullptr, ws,
                static_cast<uint8_t *>(y) + (size_t)t0 * H * dtype_size(ydt), ydt, accumulate,
                status_dev, st);
    if (s != K3MOE_OK) return s;
  }
  return K3MOE_OK;
}

// Host-side argument checks of k3moe_layer (x is the layer input, or the residual
// stream of a stacked step; only its pointer and alignment are checked).
static k3moe_status check_layer_args(const k3moe_dims *dims, const void *x, int32_t T,
                                     const uint16_t *wr_bf16, const float *bias,
                                     const k3moe_experts *experts, const uint16_t *sh_gate,
                                     const uint16_t *sh_up, const uint16_t *sh_down,
                                     const int32_t *idx_out, const float *w_out, const void *y,
                                     k3moe_dtype ydt, const void *workspace, size_t ws_bytes,
                                     const int32_t *status_dev) {
  k3moe_status s = check_dims(dims);
  if (s != K3MOE_OK) return s;
  if (T < 0 || (ydt != K3MOE_F32 && ydt != K3MOE_BF16)) return K3MOE_ERR_ARG;
  if (T == 0) return K3MOE_OK;
  if (!x || !wr_bf16 || !experts || !experts->experts || !y || !workspace || !status_dev)
    return K3MOE_ERR_ARG;
  const bool shared = dims->shared_inter > 0;
  if (shared && (!sh_gate || !sh_up || !sh_down)) return K3MOE_ERR_ARG;
  if ((idx_out == nullptr) != (w_out == nullptr)) return K3MOE_ERR_ARG;
  int64_t off[7];
  record_offsets(dims, off);
  if (experts->expert_stride < off[6] || experts->expert_stride % 16) return K3MOE_ERR_ALIGN;
  if (!aligned16(x) || !aligned16(wr_bf16) || !aligned16(experts->experts) ||
      !aligned16(y) || !aligned16(workspace) || (bias && !aligned16(bias)) ||
      (idx_out && (!aligned16(idx_out) || !aligned16(w_out))) ||
      (shared && (!aligned16(sh_gate) || !aligned16(sh_up) || !aligned16(sh_down))))
    return K3MOE_ERR_ALIGN;
  if (ws_bytes < k3moe_workspace_size(dims, T)) return K3MOE_ERR_WORKSPACE;
  return K3MOE_OK;
}

namespace {

// The layer step.  overlap: on the tensor-core path the shared expert (it reads only x)
// runs on the side stream while the tokens are routed, joined before the routed GEMMs
// (off for the static-scratch entry, which creates nothing).
k3moe_status layer_impl(const k3moe_dims *dims, const uint16_t *x_bf16, int32_t T,
                        const uint16_t *wr_bf16, const float *bias, const k3moe_experts *experts,
                        const uint16_t *sh_gate, const uint16_t *sh_up, const uint16_t *sh_down,
                        int32_t *idx_out, float *w_out, void *y, k3moe_dtype ydt,
                        int32_t accumulate, void *workspace, size_t ws_bytes,
                        int32_t *status_dev, k3moe_stream_t stream, bool overlap) {
  k3moe_status s = check_layer_args(dims, x_bf16, T, wr_bf16, bias, experts, sh_gate, sh_up,
                                    sh_down, idx_out, w_out, y, ydt, workspace, ws_bytes,
                                    status_dev);
  if (s != K3MOE_OK || T == 0) return s;
  const bool shared = dims->shared_inter > 0;
  const DeviceInfo *di = device_info();
  if (!di) return K3MOE_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int H = dims->hidden, K = dims->topk;
  if (use_tc(dims, T)) {
    WsTc wt = ws_tc_layout(dims, T, workspace);
    for (int t0 = 0; t0 < T; t0 += kTcTokens) {
      const int Tc = (T - t0) < kTcTokens ? (T - t0) : kTcTokens;
      int32_t *idx_c = idx_out ? idx_out + (size_t)t0 * K : wt.idx;
      float *w_c = w_out ? w_out + (size_t)t0 * K : wt.w;
      const uint16_t *xc = x_bf16 + (size_t)t0 * H;
      struct EventGuard {
        cudaEvent_t e = nullptr;
        ~EventGuard() {
          if (e) cudaEventDestroy(e);
        }
      } fork, join;
      cudaStream_t ss = overlap && shared ? side_stream() : nullptr;
      if (ss) {
        k_group1<<<1, 32, 0, st>>>(Tc, kTcRows, wt.off1, wt.tile_off1);
        if (cudaEventCreateWithFlags(&fork.e, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&join.e, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventRecord(fork.e, st) != cudaSuccess ||
            cudaStreamWaitEvent(ss, fork.e, 0) != cudaSuccess)
          return K3MOE_ERR_CUDA;
        s = run_shared_tc(di, dims, xc, Tc, sh_gate, sh_up, sh_down, wt, status_dev, ss, true);
        if (cudaEventRecord(join.e, ss) != cudaSuccess && s == K3MOE_OK) s = K3MOE_ERR_CUDA;
        if (s != K3MOE_OK) return s;
      }
      s = run_route_tc(di, dims, xc, Tc, wr_bf16, bias, wt, idx_c, w_c, status_dev, st, ss);
      if (s != K3MOE_OK) return s;
      if (ss && cudaStreamWaitEvent(st, join.e, 0) != cudaSuccess) return K3MOE_ERR_CUDA;
      s = run_ffn_tc(di, dims, xc, Tc, experts, idx_c, w_c, shared ? sh_gate : nullptr,
                     shared ? sh_up : nullptr, shared ? sh_down : nullptr, wt,
                     static_cast<uint8_t *>(y) + (size_t)t0 * H * dtype_size(ydt), ydt,
                     accumulate, status_dev, st, false, ss != nullptr);
      if (s != K3MOE_OK) return s;
    }
    return K3MOE_OK;
  }
  Ws ws = ws_layout(dims, T, workspace);
  for (int t0 = 0; t0 < T; t0 += kDecodeTokens) {
    const int Tc = (T - t0) < kDecodeTokens ? (T - t0) : kDecodeTokens;
    int32_t *idx_c = idx_out ? idx_out + (size_t)t0 * K : ws.idx;
    float *w_c = w_out ? w_out + (size_t)t0 * K : ws.w;
    const uint16_t *xc = x_bf16 + (size_t)t0 * H;
    s = run_layer(di, dims, xc, Tc, wr_bf16, bias, experts, shared ? sh_gate : nullptr,
                  shared ? sh_up : nullptr, shared ? sh_down : nullptr, ws, idx_c, w_c,
                  static_cast<uint8_t *>(y) + (size_t)t0 * H * dtype_size(ydt), ydt, accumulate,
                  status_dev, st);
    if (s != K3MOE_OK) return s;
  }
  return K3MOE_OK;
}

}  // namespace

k3moe_status k3moe_layer(const k3moe_dims *dims, const uint16_t *x_bf16, int32_t T,
                         const uint16_t *wr_bf16, const float *bias, const k3moe_experts *experts,
                         const uint16_t *sh_gate, const uint16_t *sh_up, const uint16_t *sh_down,
                         int32_t *idx_out, float *w_out, void *y, k3moe_dtype ydt,
                         int32_t accumulate, void *workspace, size_t ws_bytes,
                         int32_t *status_dev, k3moe_stream_t stream) {
  return layer_impl(dims, x_bf16, T, wr_bf16, bias, experts, sh_gate, sh_up, sh_down, idx_out,
                    w_out, y, ydt, accumulate, workspace, ws_bytes, status_dev, stream, true);
}

// k3moe_layer with the static array as its workspace: size check first (nothing is
// launched when the request does not fit), then the per-device address lookup and the
// argument checks, then the counter words cleared on the caller's stream.
k3moe_status k3moe_layer_static_scratch(const k3moe_dims *dims, const uint16_t *x_bf16,
                                        int32_t T, const uint16_t *wr_bf16, const float *bias,
                                        const k3moe_experts *experts, const uint16_t *sh_gate,
                                        const uint16_t *sh_up, const uint16_t *sh_down,
                                        int32_t *idx_out, float *w_out, void *y,
                                        k3moe_dtype ydt, int32_t accumulate,
                                        int32_t *status_dev, k3moe_stream_t stream) {
  const k3moe_status s = check_dims(dims);
  if (s != K3MOE_OK) return s;
  if (T < 0) return K3MOE_ERR_ARG;
  if (T == 0) return K3MOE_OK;
  if (k3moe_workspace_size(dims, T) > (size_t)K3MOE_STATIC_SCRATCH_BYTES)
    return K3MOE_ERR_SCRATCH_LIMIT;
  void *scratch = static_scratch();
  if (!scratch) return K3MOE_ERR_CUDA;
  const k3moe_status a = check_layer_args(dims, x_bf16, T, wr_bf16, bias, experts, sh_gate,
                                          sh_up, sh_down, idx_out, w_out, y, ydt, scratch,
                                          K3MOE_STATIC_SCRATCH_BYTES, status_dev);
  if (a != K3MOE_OK) return a;
  // the counter words at the array's start must be zero when the kernels start; clearing
  // them on the call's stream also undoes what calls that raced on the array left there
  if (cudaMemsetAsync(scratch, 0, kWsHeader, reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return K3MOE_ERR_CUDA;
  return layer_impl(dims, x_bf16, T, wr_bf16, bias, experts, sh_gate, sh_up, sh_down, idx_out,
                    w_out, y, ydt, accumulate, scratch, K3MOE_STATIC_SCRATCH_BYTES, status_dev,
                    stream, false);
}

size_t k3moe_latent_workspace_size(const k3moe_latent_dims *dims, int32_t T) {
  k3moe_dims full, lat;
  if (latent_dims(dims, &full, &lat) != K3MOE_OK || T < 0) return 0;
  if (T == 0) return 16;
  return ws_latent_layout(&full, &lat, T, nullptr).total;
}

// The LatentMoE layer in passes of up to kDecodeTokens tokens: route on the full-width x,
// project into the latent, the experts in the latent (float input) with their router-order
// sum, RMSNorm of that sum, project back up, then the shared experts on x, whose down
// projection adds the up-projection and writes y.
k3moe_status k3moe_latent_layer(const k3moe_latent_dims *dims, const k3moe_latent_weights *lw,
                                const uint16_t *x_bf16, int32_t T, int32_t *idx_out,
                                float *w_out, void *y, k3moe_dtype ydt, int32_t accumulate,
                                void *workspace, size_t ws_bytes, int32_t *status_dev,
                                k3moe_stream_t stream) {
  k3moe_dims full, lat;
  k3moe_status s = latent_dims(dims, &full, &lat);
  if (s != K3MOE_OK) return s;
  if (T < 0 || (ydt != K3MOE_F32 && ydt != K3MOE_BF16)) return K3MOE_ERR_ARG;
  if (T == 0) return K3MOE_OK;
  if (!lw || !x_bf16 || !lw->wr_bf16 || !lw->w_down || !lw->w_up || !lw->experts.experts ||
      !y || !workspace || !status_dev)
    return K3MOE_ERR_ARG;
  if (dims->latent_norm && !lw->latent_norm_w) return K3MOE_ERR_ARG;
  const bool shared = dims->shared_inter > 0;
  if (shared && (!lw->sh_gate || !lw->sh_up || !lw->sh_down)) return K3MOE_ERR_ARG;
  if ((idx_out == nullptr) != (w_out == nullptr)) return K3MOE_ERR_ARG;
  int64_t off[7];
  record_offsets(&lat, off);
  if (lw->experts.expert_stride < off[6] || lw->experts.expert_stride % 16) return K3MOE_ERR_ALIGN;
  if (!aligned16(x_bf16) || !aligned16(lw->wr_bf16) || !aligned16(lw->w_down) ||
      !aligned16(lw->w_up) || !aligned16(lw->experts.experts) || !aligned16(y) ||
      !aligned16(workspace) || (lw->bias && !aligned16(lw->bias)) ||
      (lw->latent_norm_w && !aligned16(lw->latent_norm_w)) ||
      (idx_out && (!aligned16(idx_out) || !aligned16(w_out))) ||
      (shared && (!aligned16(lw->sh_gate) || !aligned16(lw->sh_up) || !aligned16(lw->sh_down))))
    return K3MOE_ERR_ALIGN;
  if (ws_bytes < k3moe_latent_workspace_size(dims, T)) return K3MOE_ERR_WORKSPACE;
  const DeviceInfo *di = device_info();
  if (!di) return K3MOE_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  WsLatent ws = ws_latent_layout(&full, &lat, T, workspace);
  const int H = dims->hidden, L = dims->latent, K = dims->topk, SI = dims->shared_inter;
  const float b1 = dims->situ_b1, b2 = dims->situ_b2;
  for (int t0 = 0; t0 < T; t0 += kDecodeTokens) {
    const int Tc = (T - t0) < kDecodeTokens ? (T - t0) : kDecodeTokens;
    const uint16_t *xc = x_bf16 + (size_t)t0 * H;
    int32_t *idx_c = idx_out ? idx_out + (size_t)t0 * K : ws.route.idx;
    float *w_c = w_out ? w_out + (size_t)t0 * K : ws.route.w;
    void *yc = static_cast<uint8_t *>(y) + (size_t)t0 * H * dtype_size(ydt);
    // one token at a latent width the single-token gate/up kernel takes: it selects the
    // top-k itself from the router's scores and streams the experts through its ring
    const int rb = Tc == 1 ? t1_row_block(L) : 0;
    // more tokens than one pass of the GEMV kernels takes: the four bf16 projections as
    // GEMMs on the tensor cores (one group of Tc rows)
    const bool proj_tc = ws.has_tc && Tc > kProjRows;
    TcGemmArgs g1{};
    if (proj_tc) {
      k_group1<<<1, 32, 0, st>>>(Tc, kTcRows, ws.tc.off1, ws.tc.tile_off1);
      g1.off = ws.tc.off1;
      g1.tile_off = ws.tc.tile_off1;
      g1.gid = nullptr;
      g1.ngroups = 1;
      g1.ntile = kTcRows;
      g1.a_once = Tc <= kTcRows;
      g1.b1 = b1;
      g1.b2 = b2;
      g1.status = status_dev;
    }
    // 6 (first, on the side stream). The shared experts read only x: their SiTU(Wg x, Wu x)
    // and down projection into ds run alongside the routed chain and join before the
    // final add y (=|+=) up + ds.
    struct EventGuard {  // destroys the join event on every way out of the pass
      cudaEvent_t e = nullptr;
      ~EventGuard() {
        if (e) cudaEventDestroy(e);
      }
    } ev_join;
    if (shared) {
      s = run_latent_shared(di, lw, xc, Tc, H, SI, proj_tc, g1, ws, b1, b2, st, &ev_join.e);
      if (s != K3MOE_OK) return s;
    }
    // 1. route on the full-width x
    s = run_route(di, &full, xc, Tc, lw->wr_bf16, lw->bias, nullptr, nullptr, ws.route, idx_c,
                  w_c, status_dev, st, rb == 0);
    if (s != K3MOE_OK) return s;
    // 2. z = Wdn x
    if (proj_tc) {
      TraceScope ts(KID_PROJ, st);
      s = tc_bf16_gemm(di, TcKind::kBf16Store, lw->w_down, nullptr, L, H, xc, 1, Tc, ws.z, g1,
                       st);
      if (s != K3MOE_OK) return s;
    } else {
      TraceScope ts(KID_PROJ, st);
      if (launch_proj(st, di->sms, lw->w_down, nullptr, L, H, xc, false, Tc, ws.z, nullptr,
                      nullptr, 0, 0, b1, b2, !g_trace.on) != cudaSuccess)
        return K3MOE_ERR_CUDA;
    }
    // 3. the experts in the latent, summed in router order into accL
    if (rb > 0) {
      const ExpertArgs ea = expert_args(&lat, &lw->experts);
      const int G = L / kGroup;
      const size_t stage = (size_t)2 * rb * (L / 2 + G);
      int ns = (int)((227 * 1024 - gateup_t1_smem(L, dims->n_experts, K, rb, 0)) / stage);
      if (ns > 16) ns = 16;
      GateUpT1Args g{};
      g.x = nullptr; g.xf = ws.z; g.H = L; g.I = dims->inter; g.E = dims->n_experts; g.K = K;
      g.ex = ea; g.sc = ws.route.sc; g.ch = ws.route.ch; g.renorm = dims->renorm;
      g.routed_scale = dims->routed_scale; g.idx_out = idx_c; g.w_out = w_c;
      g.disp = ws.ffn.disp; g.b1 = b1; g.b2 = b2;
      g.act_hi = ws.ffn.act_hi; g.act_lo = ws.ffn.act_lo; g.act_ex = ws.ffn.act_ex;
      g.status = status_dev; g.RB = rb; g.NS = ns;
      {
        int grid = K * (dims->inter / kTileRows);
        if (grid > di->sms) grid = di->sms;
        s = run_gateup1(di, &lat, &lw->experts, g, ws.ffn, grid, st, !g_trace.on);
        if (s != K3MOE_OK) return s;
      }
      s = run_down(di, &lat, 1, ea, idx_c, w_c, nullptr, ws.ffn, ws.accl, K3MOE_F32, 0,
                   status_dev, st, !g_trace.on);
    } else if (ws.has_tc && Tc >= 2) {
      // two tokens or more: the grouped GEMMs on the tensor cores, z encoded as four
      // MXFP4 terms like the direct layer's x
      s = run_ffn_tc(di, &lat, ws.z, Tc, &lw->experts, idx_c, w_c, nullptr, nullptr, nullptr,
                     ws.tc, ws.accl, K3MOE_F32, 0, status_dev, st, true);
    } else {
      s = run_ffn(di, &lat, ws.z, Tc, &lw->experts, idx_c, w_c, nullptr, ws.ffn, ws.accl,
                  K3MOE_F32, 0, status_dev, st, true);
    }
    if (s != K3MOE_OK) return s;
    // 4. RMSNorm of the aggregate: its own kernel for a large pass, else done by every block
    //    of the up-projection on the rows it reads
    const bool fold_norm = dims->latent_norm && Tc <= kProjRows;
    if (dims->latent_norm && !fold_norm) {
      TraceScope ts(KID_RMSNORM_F32, st);
      if (launch_rmsnorm_f32w(st, ws.accl, Tc, L, lw->latent_norm_w, dims->rms_eps, ws.accl,
                              !g_trace.on) != cudaSuccess)
        return K3MOE_ERR_CUDA;
    }
    if (proj_tc) {
      // 5 on the tensor cores: up = Wup accL (accL as bf16 hi + lo)
      s = launch_split(di, ws.accl, (long long)Tc * L, ws.hs, st);
      if (s != K3MOE_OK) return s;
      {
        TraceScope ts(KID_PROJ_UP, st);
        s = tc_bf16_gemm(di, TcKind::kBf16Down, lw->w_up, nullptr, H, L, ws.hs, 2, Tc, ws.up,
                         g1, st);
        if (s != K3MOE_OK) return s;
      }
    } else {
      // 5. up = Wup accL (straight into y when there is no shared expert)
      TraceScope ts(KID_PROJ_UP, st);
      if (launch_proj(st, di->sms, lw->w_up, nullptr, H, L, ws.accl, true, Tc, ws.up, nullptr,
                      shared ? nullptr : yc, (int)ydt, accumulate, b1, b2, !g_trace.on,
                      fold_norm, lw->latent_norm_w, dims->rms_eps) != cudaSuccess)
        return K3MOE_ERR_CUDA;
    }
    if (shared || proj_tc) {
      if (ev_join.e && cudaStreamWaitEvent(st, ev_join.e, 0) != cudaSuccess)
        return K3MOE_ERR_CUDA;
      TraceScope ts(KID_COMBINE, st);
      if (launch_add_out(st, di->sms, ws.up, shared ? ws.ds : nullptr, yc, (int)ydt, accumulate,
                         (long long)Tc * H) != cudaSuccess)
        return K3MOE_ERR_CUDA;
    }
  }
  return K3MOE_OK;
}

// ---- host-tier expert streaming ---------------------------------------------------------
// Workspace: the decode path's (one pass of up to kDecodeTokens tokens) plus the pass's slot
// indices [Tc][K].
size_t k3moe_streamed_workspace_size(const k3moe_dims *dims, int32_t T) {
  if (check_dims(dims) != K3MOE_OK || T < 0) return 0;
  if (T == 0) return 16;
  const int Tc = T < kDecodeTokens ? T : kDecodeTokens;
  return ws_layout(dims, T, nullptr).total + up16((size_t)Tc * dims->topk * 4);
}

k3moe_status k3moe_layer_streamed(const k3moe_dims *dims, k3moe_expert_cache *cache,
                                  int32_t layer, const uint16_t *x_bf16, int32_t T,
                                  const uint16_t *wr_bf16, const float *bias,
                                  const uint16_t *sh_gate, const uint16_t *sh_up,
                                  const uint16_t *sh_down, int32_t *idx_out, float *w_out,
                                  void *y, k3moe_dtype ydt, int32_t accumulate,
                                  void *workspace, size_t ws_bytes, int32_t *status_dev,
                                  k3moe_stream_t stream) {
  k3moe_status s = check_dims(dims);
  if (s != K3MOE_OK) return s;
  if (!cache || layer < 0 || layer >= cache->n_layers) return K3MOE_ERR_ARG;
  int64_t off[7];
  record_offsets(dims, off);
  if (cache->n_experts != dims->n_experts || cache->record_bytes != off[6]) return K3MOE_ERR_ARG;
  if (dims->topk > cache->n_slots) return K3MOE_ERR_CACHE_FULL;
  // the slots stand in for the expert pool in the argument checks; the workspace is this
  // path's own (decode passes only), checked below
  const k3moe_experts slots{cache->slots, cache->slot_stride};
  s = check_layer_args(dims, x_bf16, T, wr_bf16, bias, &slots, sh_gate, sh_up, sh_down, idx_out,
                       w_out, y, ydt, workspace, ~size_t(0), status_dev);
  if (s != K3MOE_OK || T == 0) return s;
  if (ws_bytes < k3moe_streamed_workspace_size(dims, T)) return K3MOE_ERR_WORKSPACE;
  const DeviceInfo *di = device_info();
  if (!di) return K3MOE_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  Ws ws = ws_layout(dims, T, workspace);
  int32_t *slot_dev = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(workspace) + ws.total);
  const bool shared = dims->shared_inter > 0;
  const int H = dims->hidden, K = dims->topk;
  // the FFN addresses the slots as its expert pool
  k3moe_dims ds = *dims;
  ds.n_experts = cache->n_slots;
  for (int t0 = 0; t0 < T; t0 += kDecodeTokens) {
    const int Tc = (T - t0) < kDecodeTokens ? (T - t0) : kDecodeTokens;
    const int n = Tc * K;
    int32_t *idx_c = idx_out ? idx_out + (size_t)t0 * K : ws.idx;
    float *w_c = w_out ? w_out + (size_t)t0 * K : ws.w;
    const uint16_t *xc = x_bf16 + (size_t)t0 * H;
    // route, with the shared expert's gate/up (its activations stay in the workspace)
    s = run_route(di, dims, xc, Tc, wr_bf16, bias, shared ? sh_gate : nullptr,
                  shared ? sh_up : nullptr, ws, idx_c, w_c, status_dev, st, true);
    if (s != K3MOE_OK) return s;
    std::lock_guard<std::mutex> lk(cache->mu);
    cache->route_host.resize(n);
    cache->slot_host.resize(n);
    cache->load_host.resize(n);
    if (cudaMemcpyAsync(cache->route_host.data(), idx_c, (size_t)n * 4, cudaMemcpyDeviceToHost,
                        st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return K3MOE_ERR_CUDA;
    s = k3::cache_reserve(cache, layer, cache->route_host.data(), n, cache->slot_host.data(),
                          cache->load_host.data());
    if (s != K3MOE_OK) return s;
    // the misses as one batch of copies, in host address order
    std::vector<int> order;
    for (int j = 0; j < n; j++)
      if (cache->load_host[j]) order.push_back(j);
    std::sort(order.begin(), order.end(), [&](int a, int b) {
      return cache->route_host[a] < cache->route_host[b];
    });
    std::vector<int32_t> ok(n, 0);
    bool copied = true;
    for (int j : order) {
      const uint8_t *src = cache->host[layer] + (int64_t)cache->route_host[j] * cache->host_stride;
      uint8_t *dst = cache->slots + (int64_t)cache->slot_host[j] * cache->slot_stride;
      if (cudaMemcpyAsync(dst, src, (size_t)cache->record_bytes, cudaMemcpyHostToDevice, st) !=
          cudaSuccess) {
        copied = false;
        break;
      }
      ok[j] = 1;
    }
    k3::cache_publish(cache, layer, cache->route_host.data(), n, cache->slot_host.data(),
                      cache->load_host.data(), ok.data());
    if (!copied) {
      cudaGetLastError();
      return K3MOE_ERR_CUDA;
    }
    // slot indices to the device (a route outside the pool keeps slot -1: that pair is
    // dropped and reported by the FFN, after whatever the router reported), from pinned
    // memory and without waiting: the FFN follows the copies on the same stream
    if ((size_t)n > cache->slot_pin_n) {
      if (cache->slot_pin) cudaFreeHost(cache->slot_pin);
      cache->slot_pin = nullptr;
      cache->slot_pin_n = 0;
      if (cudaHostAlloc(&cache->slot_pin, (size_t)n * 4, cudaHostAllocDefault) != cudaSuccess) {
        cache->slot_pin = nullptr;
        return K3MOE_ERR_CUDA;
      }
      cache->slot_pin_n = (size_t)n;
    }
    std::copy(cache->slot_host.begin(), cache->slot_host.begin() + n, cache->slot_pin);
    if (cudaMemcpyAsync(slot_dev, cache->slot_pin, (size_t)n * 4, cudaMemcpyHostToDevice, st) !=
        cudaSuccess)
      return K3MOE_ERR_CUDA;
    s = run_ffn(di, &ds, xc, Tc, &slots, slot_dev, w_c, shared ? sh_down : nullptr, ws,
                static_cast<uint8_t *>(y) + (size_t)t0 * H * dtype_size(ydt), ydt, accumulate,
                status_dev, st);
    if (s != K3MOE_OK) return s;
  }
  return K3MOE_OK;
}

// The stacked decode loop: per layer, RMSNorm of the residual stream into bf16, then the
// layer step added to the stream (k3moe_layer with accumulate).
k3moe_status k3moe_decode_stack(const k3moe_dims *dims, int32_t L,
                                const k3moe_layer_weights *layers, int32_t T, float *h,
                                float eps, uint16_t *x_scratch, int32_t *idx_out, float *w_out,
                                void *workspace, size_t ws_bytes, int32_t *status_dev,
                                k3moe_stream_t stream) {
  k3moe_status s = check_dims(dims);
  if (s != K3MOE_OK) return s;
  if (L < 1 || T < 0 || !layers) return K3MOE_ERR_ARG;
  if (T == 0) return K3MOE_OK;
  if (!h || !x_scratch || !workspace || !status_dev) return K3MOE_ERR_ARG;
  if ((idx_out == nullptr) != (w_out == nullptr)) return K3MOE_ERR_ARG;
  const int H = dims->hidden, K = dims->topk;
  const DeviceInfo *di = device_info();
  if (!di) return K3MOE_ERR_CUDA;
  if (T == 1 && fused_takes(di, dims) && eps >= 0.f) {
    // up to kFuMaxLayers layers per launch: the fused kernel normalises h itself before
    // every layer (RMSNorm in every CTA), adds the layer's output to it, and streams the
    // next layer's router and shared-expert weights while it waits for every CTA to finish
    // the layer; x_scratch is not used
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    Ws ws = ws_layout(dims, T, workspace);
    const bool shared = dims->shared_inter > 0;
    FusedLayer f[kFuMaxLayers];
    for (int l0 = 0; l0 < L; l0 += kFuMaxLayers) {
      const int n = (L - l0) < kFuMaxLayers ? (L - l0) : kFuMaxLayers;
      for (int i = 0; i < n; i++) {
        const int l = l0 + i;
        const k3moe_layer_weights &lw = layers[l];
        s = check_layer_args(dims, h, T, lw.wr_bf16, lw.bias, &lw.experts, lw.sh_gate, lw.sh_up,
                             lw.sh_down, idx_out, w_out, h, K3MOE_F32, workspace, ws_bytes,
                             status_dev);
        if (s != K3MOE_OK) return s;
        const size_t ro = (size_t)l * K;
        f[i] = fused_layer_of(lw.wr_bf16, lw.bias, &lw.experts, shared ? lw.sh_gate : nullptr,
                              shared ? lw.sh_up : nullptr, shared ? lw.sh_down : nullptr,
                              idx_out ? idx_out + ro : nullptr, w_out ? w_out + ro : nullptr);
      }
      s = run_fused(di, dims, nullptr, h, eps, f, n, ws, h, K3MOE_F32, 1, status_dev, st);
      if (s != K3MOE_OK) return s;
    }
    return K3MOE_OK;
  }
  for (int l = 0; l < L; l++) {
    s = k3moe_rmsnorm_bf16(h, T, H, eps, x_scratch, stream);
    if (s != K3MOE_OK) return s;
    const k3moe_layer_weights &lw = layers[l];
    const size_t ro = (size_t)l * T * K;
    s = k3moe_layer(dims, x_scratch, T, lw.wr_bf16, lw.bias, &lw.experts, lw.sh_gate, lw.sh_up,
                    lw.sh_down, idx_out ? idx_out + ro : nullptr, w_out ? w_out + ro : nullptr, h,
                    K3MOE_F32, 1, workspace, ws_bytes, status_dev, stream);
    if (s != K3MOE_OK) return s;
  }
  return K3MOE_OK;
}

k3moe_status k3moe_rmsnorm_bf16(const float *h, int32_t T, int32_t n, float eps, uint16_t *out,
                                k3moe_stream_t stream) {
  if (T < 0 || n < 1 || !(eps >= 0.f)) return K3MOE_ERR_ARG;
  if (T == 0) return K3MOE_OK;
  if (!h || !out) return K3MOE_ERR_ARG;
  if (!aligned16(h) || !aligned16(out)) return K3MOE_ERR_ALIGN;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  TraceScope ts(KID_RMSNORM, st);
  // launched as a programmatic dependent (outside tracing): its launch overlaps the tail
  // of the kernel that wrote h, and the kernel waits for that kernel before reading
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(T);
  cfg.blockDim = dim3(kRmsThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = g_trace.on ? 0 : 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_rmsnorm_bf16, h, T, n, eps, out) == cudaSuccess ? K3MOE_OK
                                                                                  : K3MOE_ERR_CUDA;
}

k3moe_status k3moe_dequant_mxfp4(const uint8_t *packed, const uint8_t *scales, int32_t rows,
                                 int32_t cols, float *out, k3moe_stream_t stream) {
  if (rows < 0 || cols < 0 || cols % kGroup) return cols % kGroup ? K3MOE_ERR_SHAPE : K3MOE_ERR_ARG;
  if (rows == 0 || cols == 0) return K3MOE_OK;
  if (!packed || !scales || !out) return K3MOE_ERR_ARG;
  if (!aligned16(packed) || !aligned16(out)) return K3MOE_ERR_ALIGN;
  const long long n = (long long)rows * (cols / kGroup);
  int grid = (int)((n + 255) / 256);
  if (grid > 4096) grid = 4096;
  TraceScope ts(KID_DEQUANT, reinterpret_cast<cudaStream_t>(stream));
  k_dequant<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(packed, scales, rows, cols,
                                                                    out);
  return launch_status();
}

k3moe_status k3moe_test_expire_wait(int32_t on) {
  g_expire_wait.store(on != 0 ? 1 : 0, std::memory_order_relaxed);
  return K3MOE_OK;
}

k3moe_status k3moe_trace_enable(int32_t on) {
  std::lock_guard<std::mutex> lk(g_mu);
  trace_drain();
  for (int k = 0; k < KID_COUNT; k++) {
    g_trace.total_ms[k] = 0.0;
    g_trace.launches[k] = 0;
  }
  g_trace.on = on != 0;
  return K3MOE_OK;
}

int32_t k3moe_trace_read(int32_t kernel, const char **name, double *total_ms, int64_t *launches) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (kernel < 0) return KID_COUNT;
  if (kernel >= KID_COUNT) return -1;
  trace_drain();
  if (name) *name = kKernelNames[kernel];
  if (total_ms) *total_ms = g_trace.total_ms[kernel];
  if (launches) *launches = g_trace.launches[kernel];
  return KID_COUNT;
}

}  // extern "C"

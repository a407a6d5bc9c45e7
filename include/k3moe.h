/*
 * k3moe.h -- C ABI of the GB300 (sm_103a) MoE layer step of Kimi K3.
 *
 * The operation (what each call computes) is defined by the README of
 * FareedKhan-dev/kimi-k3-in-c ("kimi-k3-in-c" below):
 *   - the router: section 9 "Picking 16 experts of 896" (router listing) and
 *     "Three invariants", item 3 (the bias steers selection only);
 *   - the MXFP4 format and the nibble-direct product: section 4 "Reduction one: the
 *     experts already ship at half a byte";
 *   - the expert FFN with the SiTU-GLU activation, the routed sum and the shared
 *     expert: section 9 (LatentMoE listing, steps 3 and 6; activation listing);
 *   - RMSNorm: section 5 "Kernels with a floating point contract";
 * and the README of Maknee/Kimi-K3.cpp ("The consumer-memory idea", item 7: results are
 * reduced in router order).
 *
 * Conventions shared by every call
 *   - Every pointer argument is a DEVICE pointer owned by the caller, unless stated
 *     otherwise.  The library allocates no device memory on these paths and frees
 *     nothing; scratch space is the caller's `workspace`.
 *   - Calls are asynchronous on `stream` (0 = the legacy default stream).  Argument
 *     errors found on the host are returned at once and nothing is launched.
 *   - Errors found on the device are written to `*status_dev` (an int32 the caller
 *     allocates and zeroes; the first error wins, later ones do not overwrite it) and
 *     are read by the caller after synchronising.  A failing work item still writes
 *     defined output (zeros for its part), so results are never undefined memory.
 *   - bf16 tensors are passed as uint16_t bit patterns.  Row-major throughout.
 *   - Pointers must be 16-byte aligned (K3MOE_ERR_ALIGN otherwise).
 *   - Thread safety: calls are independent; two calls may run concurrently only if
 *     they use different workspaces.
 *   - Workspace: zero-fill it once before its first use (e.g. one cudaMemsetAsync).  Its
 *     first 4096 bytes hold counters of the single-token kernels that must be zero when a
 *     call starts; every call leaves them zero, so a workspace can be reused across calls,
 *     entry points, shapes and token counts without clearing it again.  Do not write to
 *     a workspace between calls.  The rest is scratch.
 */
#ifndef K3MOE_H
#define K3MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *k3moe_stream_t; /* a cudaStream_t */

typedef enum {
    K3MOE_OK = 0,
    K3MOE_ERR_ARG = 1,        /* NULL pointer, negative count, bad enum */
    K3MOE_ERR_SHAPE = 2,      /* a dimension the kernels do not support */
    K3MOE_ERR_ALIGN = 3,      /* a pointer or stride not 16-byte aligned */
    K3MOE_ERR_WORKSPACE = 4,  /* ws_bytes below k3moe_workspace_size() */
    K3MOE_ERR_CUDA = 5,       /* a CUDA launch failed (see cudaGetLastError) */
    K3MOE_ERR_TIMEOUT = 6,    /* a bounded device-side wait gave up */
    K3MOE_ERR_BAD_EXPERT = 7, /* an expert index outside [0, n_experts) */
    K3MOE_ERR_NONFINITE = 8,  /* a router score that is NaN or infinite */
    K3MOE_ERR_SCRATCH_LIMIT = 9, /* the call needs more than K3MOE_STATIC_SCRATCH_BYTES */
    K3MOE_ERR_CACHE_FULL = 10    /* one call's distinct experts exceed the cache's slots */
} k3moe_status;

typedef enum { K3MOE_F32 = 0, K3MOE_BF16 = 1 } k3moe_dtype;

/* Shapes and constants of one MoE layer (the model config fields of kimi-k3-in-c,
 * section 2, K3Cfg: n_experts, topk, moe_inter, routed_scale, moe_renorm, situ_b1,
 * situ_b2).
 *   hidden        H, the layer width (x and y are [T][H]); multiple of 32
 *   inter         I, the routed expert's intermediate width; multiple of 32
 *   n_experts     E, 1..4096
 *   topk          K, 1..32 and <= E
 *   group         MXFP4 block size; must be 32
 *   shared_inter  SI, the shared expert's intermediate width (multiple of 32), or 0 for
 *                 no shared expert
 *   situ_b1/b2    SiTU caps (4 and 25 in the model)
 *   routed_scale  factor applied to every routed weight after renormalisation
 *   renorm        1: divide the K selected scores by their sum when it is > 0          */
typedef struct {
    int32_t hidden, inter, n_experts, topk, group, shared_inter;
    float situ_b1, situ_b2, routed_scale;
    int32_t renorm;
} k3moe_dims;

/* Routed expert weights.  Expert e is the record at experts + e * expert_stride bytes.
 * One record holds six operands, in this order (byte offsets from
 * k3moe_record_layout):
 *   w1 (gate) packed [I][H/2]   w1 scales [I][H/32]
 *   w2 (down) packed [H][I/2]   w2 scales [H][I/32]
 *   w3 (up)   packed [I][H/2]   w3 scales [I][H/32]
 * Packed byte = two E2M1 codes, the low nibble the EVEN column (kimi-k3-in-c,
 * section 4); scale byte = E8M0, value 2^(s-127), with 255 read as 0 (the group then
 * contributes nothing).  For H = 7168, I = 1536 a record is 17,547,264 bytes
 * (kimi-k3-in-c, "The problem: a model that does not fit", shard census).
 * expert_stride must be >= the record size and a multiple of 16.                   */
typedef struct {
    const uint8_t *experts;
    int64_t expert_stride;
} k3moe_experts;

/* Byte offsets of the six operands and the record size:
 * offsets[0..5] = w1p, w1s, w2p, w2s, w3p, w3s; offsets[6] = total.  Host only. */
k3moe_status k3moe_record_layout(const k3moe_dims *dims, int64_t offsets[7]);

/* Bytes of workspace k3moe_route / k3moe_expert_ffn_mxfp4 / k3moe_layer need for T
 * tokens.  Host only; 0 for invalid dims. */
size_t k3moe_workspace_size(const k3moe_dims *dims, int32_t T);

/* Router (kimi-k3-in-c, section 9).  For each token t:
 *   logit[e] = sum_i x[t,i] Wr[e,i]  rounded to float; every bf16 product is exact in
 *              float and the sum is carried as a float-float pair (about 48
 *              significant bits), so the rounded logit agrees with a double sum
 *              except for a vanishing fraction of inputs;
 *   sc[e]    = 1 / (1 + exp(-logit[e])) evaluated in double, rounded to float;
 *   ch[e]    = sc[e] + bias[e] (one float add; bias may be NULL = 0);
 *   idx[t,:] = the K experts of largest ch, in descending ch, an equal ch going to the
 *              lower expert index (the page's repeated strict maximum);
 *   w[t,j]   = sc[idx[t,j]]; if renorm and s = sum_j w[t,j] (float, j order) > 0 then
 *              w[t,j] /= s; then w[t,j] *= routed_scale.
 * x_bf16 [T][H], wr_bf16 [E][H], bias [E] float, idx [T][K] int32, w [T][K] float.
 * A non-finite ch sets K3MOE_ERR_NONFINITE (idx/w of that token are then undefined
 * but written).  Needs k3moe_workspace_size(dims, T) bytes of workspace.          */
k3moe_status k3moe_route(const k3moe_dims *dims, const uint16_t *x_bf16,
                         const uint16_t *wr_bf16, const float *bias, int32_t T, int32_t *idx,
                         float *w, void *workspace, size_t ws_bytes, int32_t *status_dev,
                         k3moe_stream_t stream);

/* Routed expert FFN straight from MXFP4 (kimi-k3-in-c, sections 4 and 9):
 *   for each token t and slot j, e = idx[t,j]:
 *     g = W1_e x_t, u = W3_e x_t                         (MXFP4, fp32 accumulate)
 *     a = b1 tanh(g/b1) sigmoid(g) * b2 tanh(u/b2)      (SiTU-GLU, uncapped sigmoid)
 *     d_j = W2_e a
 *   y_t (=|+=) sum_{j=0}^{K-1} w[t,j] d_j               (float, in router order j)
 * x_bf16 [T][H]; idx/w [T][K]; y [T][H] of dtype ydt.  accumulate = 1 adds to the
 * existing y (for bf16: y = bf16(float(y) + sum)).  An idx outside [0, E) sets
 * K3MOE_ERR_BAD_EXPERT and that slot contributes zero.                                */
k3moe_status k3moe_expert_ffn_mxfp4(const k3moe_dims *dims, const uint16_t *x_bf16, int32_t T,
                                    const k3moe_experts *experts, const int32_t *idx,
                                    const float *w, void *y, k3moe_dtype ydt,
                                    int32_t accumulate, void *workspace, size_t ws_bytes,
                                    int32_t *status_dev, k3moe_stream_t stream);

/* The whole layer step: route, routed expert FFN, router-order combine, then the shared
 * expert added unweighted (kimi-k3-in-c, section 9, LatentMoE listing step 6):
 *   y_t (=|+=) sum_j w[t,j] d_j  +  W2s SiTU(W1s x_t, W3s x_t)
 * sh_gate/sh_up bf16 [SI][H], sh_down bf16 [H][SI] (all NULL when SI = 0).
 * idx_out [T][K] / w_out [T][K] receive the route when not NULL.                     */
k3moe_status k3moe_layer(const k3moe_dims *dims, const uint16_t *x_bf16, int32_t T,
                         const uint16_t *wr_bf16, const float *bias,
                         const k3moe_experts *experts, const uint16_t *sh_gate,
                         const uint16_t *sh_up, const uint16_t *sh_down, int32_t *idx_out,
                         float *w_out, void *y, k3moe_dtype ydt, int32_t accumulate,
                         void *workspace, size_t ws_bytes, int32_t *status_dev,
                         k3moe_stream_t stream);

/* Size of the library's static scratch array (8 MiB), the most scratch that
 * k3moe_layer_static_scratch can use.  At the model's shape (H 7168, I 1536, 896
 * experts, top 16, shared 1536) it holds the workspace of up to 9 tokens: 115,296 bytes
 * for one token, 8,157,952 for nine.                                                  */
#define K3MOE_STATIC_SCRATCH_BYTES (8u * 1024u * 1024u)

/* k3moe_layer without a workspace argument: the same kernels, arguments, results and
 * error codes, with the scratch taken from an array of K3MOE_STATIC_SCRATCH_BYTES that
 * the library declares as a static device variable (one copy per device).  The pages
 * have no counterpart; it serves callers that must not allocate device memory while
 * they run the layer: cudaMalloc and cudaFree can synchronise the whole device and
 * stall a latency-bound decode loop, a host program may have handed all free memory to
 * a cache pool already, and a plug-in may receive only the tensors of the step with no
 * allocator to obtain a workspace from.  This call allocates and frees nothing.
 *   - K3MOE_ERR_SCRATCH_LIMIT, with nothing launched, when k3moe_workspace_size(dims, T)
 *     exceeds K3MOE_STATIC_SCRATCH_BYTES.
 *   - The first call on a device, with that device current, does one-time set-up: it
 *     looks up the device address of the array (which may load the library's device
 *     code) and sets kernel attributes.  Make that first call before any stream capture
 *     starts on the device.  K3MOE_ERR_CUDA if the lookup fails.
 *   - Each call first clears the counter words at the array's start (the 4096 bytes that
 *     Workspace above describes) with one cudaMemsetAsync on `stream`, which allocates
 *     nothing; so a call starts clean even after earlier calls raced on the array.  The
 *     rest of the array is written before it is read.
 *   - Every call on a device shares the one array.  Calls ordered on one stream are
 *     safe; two calls whose work can overlap on the device (different streams without
 *     an ordering between them, or concurrent host threads) race on the array and
 *     their results are undefined.  *status_dev stays the caller's.                  */
k3moe_status k3moe_layer_static_scratch(const k3moe_dims *dims, const uint16_t *x_bf16,
                                        int32_t T, const uint16_t *wr_bf16, const float *bias,
                                        const k3moe_experts *experts, const uint16_t *sh_gate,
                                        const uint16_t *sh_up, const uint16_t *sh_down,
                                        int32_t *idx_out, float *w_out, void *y,
                                        k3moe_dtype ydt, int32_t accumulate,
                                        int32_t *status_dev, k3moe_stream_t stream);

/* The pages' LatentMoE layer (kimi-k3-in-c, section 9, LatentMoE listing steps 1-6; its
 * config fields in section 2, K3Cfg: latent, moe_inter, n_shared, latent_norm, rms_eps).
 *   hidden        H, the layer width (x and y are [T][H])
 *   latent        L, the width the routed experts run in (3584 in the model); multiple of 32
 *   inter         I, the routed experts' intermediate width (3072 in the model)
 *   n_experts, topk, group, situ_b1, situ_b2, routed_scale, renorm: as in k3moe_dims
 *   shared_inter  SI = I x n_shared (6144 in the model: two shared experts of width I,
 *                 which together are one SiTU-GLU of width SI), or 0
 *   rms_eps       epsilon of the latent RMSNorm (1e-5)
 *   latent_norm   1: RMSNorm the aggregated latent sum (with latent_norm_w), 0: skip it  */
typedef struct {
    int32_t hidden, latent, inter, n_experts, topk, group, shared_inter;
    float situ_b1, situ_b2, routed_scale, rms_eps;
    int32_t renorm, latent_norm;
} k3moe_latent_dims;

/* Weights of one LatentMoE layer (device pointers).                                    */
typedef struct {
    const uint16_t *wr_bf16;        /* [E][H] router, applied to the FULL-width x          */
    const float *bias;              /* [E] correction bias, or NULL                       */
    const uint16_t *w_down;         /* [L][H] bf16, x -> latent                           */
    const uint16_t *w_up;           /* [H][L] bf16, latent -> full width                  */
    const float *latent_norm_w;     /* [L] float weight of the latent RMSNorm             */
    k3moe_experts experts;          /* records of the (L, I) layout: w1/w3 [I][L/2],
                                       w2 [L][I/2] (17,547,264 bytes at L 3584, I 3072)   */
    const uint16_t *sh_gate, *sh_up; /* [SI][H] bf16 (NULL when SI == 0)                  */
    const uint16_t *sh_down;        /* [H][SI] bf16                                        */
} k3moe_latent_weights;

/* Bytes of workspace k3moe_latent_layer needs for T tokens (0 for invalid dims).        */
size_t k3moe_latent_workspace_size(const k3moe_latent_dims *dims, int32_t T);

/* One LatentMoE layer step for T tokens x (bf16 [T][H]), per token:
 *   1. route on the full-width x: idx, w as k3moe_route (same rules, ties, renorm);
 *   2. z = Wdn x                                  (float; bf16 weights, fp32 sums)
 *   3. accL = sum_{j=0}^{K-1} w[j] expert_idx[j](z)  (float, in router order; the experts
 *                                                   take z in float)
 *   4. accL = RMSNorm(accL) * latent_norm_w        (when latent_norm: on the AGGREGATE,
 *                                                   sum of squares in double)
 *   5. y = Wup accL
 *   6. y = y + W2s SiTU(W1s x, W3s x)              (the shared experts on the ORIGINAL x,
 *                                                   unweighted, one float add)
 * y [T][H] of dtype ydt (=, or += when accumulate).  idx_out / w_out [T][K] receive the
 * route when not NULL.  Errors as k3moe_layer (a NaN router score sets
 * K3MOE_ERR_NONFINITE, a bad shape K3MOE_ERR_SHAPE, ...).  Needs
 * k3moe_latent_workspace_size(dims, T) bytes of zero-filled workspace.                  */
k3moe_status k3moe_latent_layer(const k3moe_latent_dims *dims, const k3moe_latent_weights *w,
                                const uint16_t *x_bf16, int32_t T, int32_t *idx_out,
                                float *w_out, void *y, k3moe_dtype ydt, int32_t accumulate,
                                void *workspace, size_t ws_bytes, int32_t *status_dev,
                                k3moe_stream_t stream);

/* ---- Host-tier expert streaming --------------------------------------------------------
 * For layers whose experts do not all fit in HBM: the records stay in host memory (on a
 * GB300's Grace host, reached over NVLink-C2C) and a fixed pool of record-sized slots in
 * device memory caches them, the GPU counterpart of the pages' expert cache
 * (kimi-k3-in-c, section 12 "An LRU cache for the experts"; Kimi-K3.cpp, "The
 * consumer-memory idea", items 3-7):
 *   - a slot is empty, in flight (reserved, being read) or holds one expert of one layer;
 *   - a call first pins every selected expert already resident (a hit) and marks it used,
 *     then reserves a slot for each miss, serially, in router order: an empty slot if any
 *     (the first one), else the least recently used slot that is neither pinned nor in
 *     flight;
 *   - every miss is then read as one batch, one host-to-device copy per record (in host
 *     address order), on the call's stream, and the slots are published;
 *   - the layer is computed on the slots, the routed sum still in router order.
 * The cache is a host object; it allocates no device memory (it keeps a few KB of pinned
 * host memory for each pass's slot indices, freed by k3moe_cache_destroy).  Host memory of
 * the records should be pinned (cudaHostAlloc / cudaHostRegister) for the copies to run at
 * the link's rate; pageable memory works, slower.  One cache may serve several layers (a key is
 * (layer, expert)).  Calls on one cache must not run concurrently from several threads
 * with overlapping streams (the slots they publish would race); the host state itself is
 * locked. */
typedef struct k3moe_expert_cache k3moe_expert_cache;

/* Create a cache for n_layers layers of n_experts records of record_bytes each: layer l's
 * expert e at host_experts[l] + e * host_stride (HOST pointers, owned by the caller, alive
 * while the cache is); n_slots slots at slots + s * slot_stride (a DEVICE pointer, 16-byte
 * aligned, slot_stride >= record_bytes and a multiple of 16).  Host only (no CUDA call). */
k3moe_status k3moe_cache_create(int32_t n_layers, const uint8_t *const *host_experts,
                                int32_t n_experts, int64_t record_bytes, int64_t host_stride,
                                uint8_t *slots, int32_t n_slots, int64_t slot_stride,
                                k3moe_expert_cache **cache);
k3moe_status k3moe_cache_destroy(k3moe_expert_cache *cache);

/* Host only: the cache's decision for one call of n experts (router order, duplicates
 * allowed) of a layer, as k3moe_layer_streamed takes it -- slots[j] the slot of expert j,
 * load[j] = 1 where it has to be read -- with the reads taken as done.  For callers that
 * move the records themselves, and for tests of the policy.  K3MOE_ERR_CACHE_FULL (the
 * cache unchanged) when the call's distinct experts do not fit. */
k3moe_status k3moe_cache_lookup(k3moe_expert_cache *cache, int32_t layer,
                                const int32_t *experts, int32_t n, int32_t *slots,
                                int32_t *load);

/* Hits and misses counted per distinct expert of a call, and bytes read into slots. */
k3moe_status k3moe_cache_stats(k3moe_expert_cache *cache, int64_t *hits, int64_t *misses,
                               int64_t *bytes_loaded);

/* Bytes of workspace k3moe_layer_streamed needs for T tokens (0 for invalid dims). */
size_t k3moe_streamed_workspace_size(const k3moe_dims *dims, int32_t T);

/* k3moe_layer with the routed experts of layer `layer` taken from the cache, in passes of
 * up to 64 tokens: route (on the device), copy the routes to the host and wait for them
 * (the call synchronises `stream` once per pass), look up / reserve the slots, read the
 * misses, then the expert FFN and the shared expert on the device, the routed sum in router
 * order.  Same arguments, results and error codes as k3moe_layer, except that the expert
 * records come from the cache; K3MOE_ERR_CACHE_FULL (nothing computed for that pass) when
 * a pass's distinct experts exceed the slots; K3MOE_ERR_CUDA if a copy cannot be issued.
 * Needs k3moe_streamed_workspace_size(dims, T) bytes of workspace.                      */
k3moe_status k3moe_layer_streamed(const k3moe_dims *dims, k3moe_expert_cache *cache,
                                  int32_t layer, const uint16_t *x_bf16, int32_t T,
                                  const uint16_t *wr_bf16, const float *bias,
                                  const uint16_t *sh_gate, const uint16_t *sh_up,
                                  const uint16_t *sh_down, int32_t *idx_out, float *w_out,
                                  void *y, k3moe_dtype ydt, int32_t accumulate,
                                  void *workspace, size_t ws_bytes, int32_t *status_dev,
                                  k3moe_stream_t stream);

/* Weights of one layer of a stack (the arguments k3moe_layer takes for it). */
typedef struct {
    const uint16_t *wr_bf16;  /* [E][H] */
    const float *bias;        /* [E] or NULL */
    k3moe_experts experts;
    const uint16_t *sh_gate, *sh_up, *sh_down;  /* NULL when shared_inter == 0 */
} k3moe_layer_weights;

/* Decode through L stacked MoE layers with the residual stream between them (the
 * decoder loop of kimi-k3-in-c, section 5 for RMSNorm and section 9 for the layer): for
 * l = 0 .. L-1,
 *     x = bf16(RMSNorm(h))        (k3moe_rmsnorm_bf16 with eps; weight 1)
 *     h = h + layer_l(x)          (k3moe_layer, float output added to h)
 * h float [T][H] is updated in place; x_scratch bf16 [T][H] is caller scratch (for one
 * token at the shapes of the single-token kernel the RMSNorm runs inside that kernel, one
 * launch per layer, and x_scratch is not written);
 * idx_out / w_out ([L][T][K] each) receive every layer's route when not NULL.
 * layers is a HOST array of L entries (device pointers inside).  Needs
 * k3moe_workspace_size(dims, T) bytes of workspace, shared by the layers in turn.     */
k3moe_status k3moe_decode_stack(const k3moe_dims *dims, int32_t L,
                                const k3moe_layer_weights *layers, int32_t T, float *h,
                                float eps, uint16_t *x_scratch, int32_t *idx_out, float *w_out,
                                void *workspace, size_t ws_bytes, int32_t *status_dev,
                                k3moe_stream_t stream);

/* RMSNorm then bf16 (kimi-k3-in-c, section 5): for each of T rows of width n,
 *   inv = 1 / sqrt(mean(h^2) + eps) (sum of squares in double), out = bf16(h * inv),
 * round to nearest even.  h float [T][n], out bf16 [T][n].  The step between stacked
 * MoE layers (the decoder's residual stream feeds the next layer's input).            */
k3moe_status k3moe_rmsnorm_bf16(const float *h, int32_t T, int32_t n, float eps,
                                uint16_t *out, k3moe_stream_t stream);

/* Test hook, not on the hot path: dequantise an MXFP4 matrix to float through the same
 * device decode the FFN kernels use (E2M1 pair -> f16x2 in registers, then the E8M0
 * scale).  packed [rows][cols/2], scales [rows][cols/32], out [rows][cols] float;
 * cols a multiple of 32.  Exact: every E2M1 * 2^(s-127) is a float.                  */
k3moe_status k3moe_dequant_mxfp4(const uint8_t *packed, const uint8_t *scales, int32_t rows,
                                 int32_t cols, float *out, k3moe_stream_t stream);

/* Test hook for failure detection, not on the hot path.  While on (on != 0), every
 * single-token step that runs as one fused kernel (k3moe_layer and k3moe_decode_stack
 * with T == 1 at shapes that kernel takes) makes its second grid-wide dependency, the
 * one on every CTA's activations, wait for one arrival more than there are CTAs, with a
 * limit of about 0.1 s instead of the usual ~2 s.  The wait runs out: the launch
 * completes with the layer's output taken as zero (y = 0, or y unchanged when
 * accumulating, as the residual stream of a stack is) and *status_dev set to
 * K3MOE_ERR_TIMEOUT; the workspace counters are left zero, so the context and the
 * workspace stay usable.  Other kernels ignore it.  Process-wide; returns K3MOE_OK.     */
k3moe_status k3moe_test_expire_wait(int32_t on);

/* Tracing (no counterpart in the pages, which time whole tokens on the host).  When on,
 * every kernel the library launches is bracketed by two CUDA events on its stream and
 * its device duration is summed per kernel.  k3moe_trace_enable(1) clears the sums and
 * starts; (0) stops.  k3moe_trace_read(k, ...) synchronises on the recorded events and
 * returns kernel k's name (static string), total milliseconds and launch count; it
 * returns the number of kernels (k < 0 only queries that), or -1 for an invalid k.
 * Host only; not for use inside CUDA graph capture.                                  */
k3moe_status k3moe_trace_enable(int32_t on);
int32_t k3moe_trace_read(int32_t kernel, const char **name, double *total_ms, int64_t *launches);

/* Static string for a status code. */
const char *k3moe_status_str(k3moe_status s);

#ifdef __cplusplus
}
#endif
#endif /* K3MOE_H */

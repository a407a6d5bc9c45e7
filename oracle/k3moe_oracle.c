/*
 * k3moe_oracle.c -- plain, slow, CPU reference for the Kimi-K3 MoE layer step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls this
 * file: it is built into its own shared object and used by the tests, by the package's
 * smoke check and by the benchmark's CPU-baseline leg.  It shares no code, header or
 * table with the CUDA library.
 *
 * What it computes, and where each step is defined ("kimi-k3-in-c" is the README of
 * FareedKhan-dev/kimi-k3-in-c; "Kimi-K3.cpp" is the README of Maknee/Kimi-K3.cpp):
 *
 *   E2M1 value table, E8M0 scale ............ kimi-k3-in-c, section 4 "Reduction one:
 *                                              the experts already ship at half a byte"
 *   MXFP4 matrix-vector product ............. same section (the nibble-direct product)
 *   bf16 widening, bf16 matrix-vector ....... kimi-k3-in-c, section 5 "Kernels with a
 *                                              floating point contract"
 *   RMSNorm ................................. same section
 *   router: sigmoid scores, biased choice,
 *   repeated-max top-k, renorm, scale ....... kimi-k3-in-c, section 9 "Picking 16
 *                                              experts of 896" (router listing) and
 *                                              "Three invariants", item 3
 *   SiTU-GLU ................................ section 9 (activation listing)
 *   routed sum in router order, shared
 *   expert added unweighted ................. section 9 (LatentMoE listing, steps 3, 6);
 *                                              Kimi-K3.cpp "The consumer-memory idea" 7
 *   the LatentMoE: down-projection, experts
 *   in the latent, RMSNorm of the aggregate,
 *   up-projection, shared experts on the
 *   full-width input ........................ section 9 (LatentMoE listing, steps 1-6);
 *                                              section 2 (K3Cfg: latent, n_shared,
 *                                              latent_norm)
 *
 * Precision: every sum the page accumulates in double is accumulated in double here,
 * every sum the page accumulates in float (the routed sum in router order, the shared
 * expert's add) is a float sum here, term by term in the page's order, and every value
 * the page stores as float is rounded to float here.  Where the page uses a float libm
 * call (expf, tanhf) the oracle evaluates the same function in double and rounds once to
 * float: the float libm result differs from one C library to another, the
 * double-then-round one does not, so CPU and GPU can agree on it.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fopenmp -fPIC -shared (see build.py).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define K3O_GROUP 32

/* ---------------------------------------------------------------------------------
 * Number formats (section 4).  The page prints the sixteen E2M1 values; the table
 * below is that printed table.  E8M0 is 2^(b-127) with b = 255 (NaN in the MX
 * specification) mapped to 0.
 * ------------------------------------------------------------------------------- */
static const double K3O_E2M1[16] = {
    0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
    -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0};

double k3o_e2m1(int code) { return K3O_E2M1[code & 15]; }

double k3o_e8m0(int b) {
    b &= 255;
    return (b == 255) ? 0.0 : ldexp(1.0, b - 127);
}

/* bf16 -> f32 is the top half of the f32 bit pattern (section 5): exact. */
float k3o_bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* f32 -> bf16, round to nearest, ties to even; NaN stays NaN. */
uint16_t k3o_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return (uint16_t)((u >> 16) | 0x40);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

static int k3o_threads(int nt) {
#ifdef _OPENMP
    return nt > 0 ? nt : omp_get_max_threads();
#else
    (void)nt;
    return 1;
#endif
}

/* Weight (r, c) of an MXFP4 matrix: low nibble of byte c/2 is the even column, high
 * nibble the odd one; scale byte (r, c/32).  Rows hold (in+1)/2 packed bytes and
 * ceil(in/32) scale bytes (section 4). */
static inline int k3o_nibble(const uint8_t *packed_row, int c) {
    uint8_t b = packed_row[c >> 1];
    return (c & 1) ? (b >> 4) : (b & 15);
}

/* Dequantised weights as float: E2M1 * 2^(s-127).  Every such product is a float (at
 * worst a subnormal) except |code| >= 2 with s = 254, which is beyond the float range
 * and becomes +-inf; so this is exact wherever a float can hold the value. */
void k3o_dequant_mxfp4(int rows, int in, const uint8_t *packed, const uint8_t *scales,
                       float *out) {
    const int rowbytes = (in + 1) / 2, ngroup = (in + K3O_GROUP - 1) / K3O_GROUP;
    for (int r = 0; r < rows; r++)
        for (int c = 0; c < in; c++) {
            double v = k3o_e2m1(k3o_nibble(packed + (size_t)r * rowbytes, c)) *
                       k3o_e8m0(scales[(size_t)r * ngroup + c / K3O_GROUP]);
            out[(size_t)r * in + c] = (float)v;
        }
}

/* y[r] = sum_c W[r,c] x[c], straight from the nibbles (section 4): per group of 32, a
 * double partial of x * E2M1, skipped when the scale decodes to 0, then acc += part *
 * scale in double; the row result is rounded to float once. */
void k3o_mxfp4_gemv(int rows, int in, const uint8_t *packed, const uint8_t *scales,
                    const float *x, float *y, int nthreads) {
    const int rowbytes = (in + 1) / 2, ngroup = (in + K3O_GROUP - 1) / K3O_GROUP;
#pragma omp parallel for schedule(static) num_threads(k3o_threads(nthreads))
    for (int r = 0; r < rows; r++) {
        const uint8_t *pb = packed + (size_t)r * rowbytes;
        const uint8_t *sb = scales + (size_t)r * ngroup;
        double acc = 0.0;
        for (int g = 0; g < ngroup; g++) {
            const double s = k3o_e8m0(sb[g]);
            if (s == 0.0) continue;
            const int c0 = g * K3O_GROUP;
            const int n = (c0 + K3O_GROUP <= in) ? K3O_GROUP : in - c0;
            double part = 0.0;
            for (int k = 0; k < n; k++) part += (double)x[c0 + k] * k3o_e2m1(k3o_nibble(pb, c0 + k));
            acc += part * s;
        }
        y[r] = (float)acc;
    }
}

/* y[r] = sum_c bf16(W[r,c]) * x[c], accumulated in double, rounded to float
 * (section 5; plain sequential order -- the page's i%4 partition only pins the CPU's
 * own SIMD/scalar agreement). */
void k3o_bf16_gemv(int rows, int in, const uint16_t *W, const float *x, float *y,
                   int nthreads) {
#pragma omp parallel for schedule(static) num_threads(k3o_threads(nthreads))
    for (int r = 0; r < rows; r++) {
        const uint16_t *w = W + (size_t)r * in;
        double acc = 0.0;
        for (int c = 0; c < in; c++) acc += (double)k3o_bf16_to_f32(w[c]) * (double)x[c];
        y[r] = (float)acc;
    }
}

/* RMSNorm (section 5): double sum of squares, epsilon inside the square root,
 * inv rounded to float, out = x * inv * w (w == NULL means weight 1). */
void k3o_rmsnorm(int n, const float *x, const float *w, float eps, float *out) {
    double ss = 0.0;
    for (int i = 0; i < n; i++) ss += (double)x[i] * (double)x[i];
    const float inv = (float)(1.0 / sqrt(ss / (double)n + (double)eps));
    for (int i = 0; i < n; i++) {
        float t = x[i] * inv;
        out[i] = w ? t * w[i] : t;
    }
}

/* Logistic function evaluated in double, rounded once to float. */
static float k3o_sigmoid_f(double z) { return (float)(1.0 / (1.0 + exp(-z))); }

/* Router for T tokens (section 9, "Picking 16 experts of 896"):
 *   logit[e] = (float) sum_i x[i] * Wr[e,i]          (double accumulation)
 *   sc[e]    = sigmoid(logit[e])                       (unbiased score, float)
 *   ch[e]    = sc[e] + bias[e]                         (selection score, one float add)
 *   top-K by repeated strict maximum of ch, so an equal ch goes to the lower index;
 *   w[j] = sc[idx[j]];  s = float sum in j order;  if renorm and s > 0: w[j] /= s;
 *   w[j] *= routed_scale.
 * Returns 0, or 8 when some score is not finite (the choice is then undefined).
 * logits / scores may be NULL. */
int k3o_router(int T, int H, int E, int K, int renorm, float routed_scale,
               const uint16_t *x, const uint16_t *Wr, const float *bias, int32_t *idx,
               float *w, float *logits, float *scores, int nthreads) {
    int status = 0;
    float *sc = (float *)malloc(sizeof(float) * (size_t)E);
    float *ch = (float *)malloc(sizeof(float) * (size_t)E);
    float *xf = (float *)malloc(sizeof(float) * (size_t)H);
    char *taken = (char *)malloc((size_t)E);
    for (int t = 0; t < T; t++) {
        for (int i = 0; i < H; i++) xf[i] = k3o_bf16_to_f32(x[(size_t)t * H + i]);
#pragma omp parallel for schedule(static) num_threads(k3o_threads(nthreads))
        for (int e = 0; e < E; e++) {
            const uint16_t *row = Wr + (size_t)e * H;
            double acc = 0.0;
            for (int i = 0; i < H; i++) acc += (double)xf[i] * (double)k3o_bf16_to_f32(row[i]);
            const float lg = (float)acc;
            if (logits) logits[(size_t)t * E + e] = lg;
            sc[e] = k3o_sigmoid_f((double)lg);
            ch[e] = sc[e] + (bias ? bias[e] : 0.0f);
        }
        for (int e = 0; e < E; e++) {
            if (scores) scores[(size_t)t * E + e] = sc[e];
            if (!isfinite(ch[e]) || !isfinite(sc[e])) status = 8;
        }
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < K; j++) {
            int best = -1;
            for (int e = 0; e < E; e++)
                if (!taken[e] && (best < 0 || ch[e] > ch[best])) best = e;
            taken[best] = 1;
            idx[(size_t)t * K + j] = best;
            w[(size_t)t * K + j] = sc[best];
        }
        float *wt = w + (size_t)t * K;
        if (renorm) {
            float s = 0.0f;
            for (int j = 0; j < K; j++) s += wt[j];
            if (s > 0.0f)
                for (int j = 0; j < K; j++) wt[j] /= s;
        }
        for (int j = 0; j < K; j++) wt[j] *= routed_scale;
    }
    free(sc);
    free(ch);
    free(xf);
    free(taken);
    return status;
}

/* SiTU-GLU (section 9, activation listing): the sigmoid takes the UNCAPPED gate.
 *   a = b1 tanh(g / b1) sigmoid(g),  u' = b2 tanh(u / b2),  act = a u'.
 * Evaluated in double from the float inputs, rounded once to float. */
void k3o_situ(int n, float b1, float b2, const float *g, const float *u, float *act) {
    for (int i = 0; i < n; i++) {
        const double gd = g[i], ud = u[i];
        const double a = (double)b1 * tanh(gd / (double)b1) * (1.0 / (1.0 + exp(-gd)));
        const double v = (double)b2 * tanh(ud / (double)b2);
        act[i] = (float)(a * v);
    }
}

/* Byte offsets of the six operands inside one expert record: w1 (gate) packed, w1
 * scales, w2 (down) packed, w2 scales, w3 (up) packed, w3 scales -- the w1, w2, w3
 * order in which the page's loader walks an expert (section 12, k3_expert_load).
 * gate/up are [inter][hidden], down is [hidden][inter], rows packed along the input. */
void k3o_record_offsets(int H, int I, int64_t off[7]) {
    const int64_t gp = (int64_t)I * ((H + 1) / 2), gs = (int64_t)I * ((H + 31) / 32);
    const int64_t dp = (int64_t)H * ((I + 1) / 2), ds = (int64_t)H * ((I + 31) / 32);
    off[0] = 0;             /* w1 packed */
    off[1] = off[0] + gp;   /* w1 scales */
    off[2] = off[1] + gs;   /* w2 packed */
    off[3] = off[2] + dp;   /* w2 scales */
    off[4] = off[3] + ds;   /* w3 packed */
    off[5] = off[4] + gp;   /* w3 scales */
    off[6] = off[5] + gs;   /* record size */
}

/* One routed expert on one token: g = W1 x, u = W3 x, act = SiTU(g, u), d = W2 act
 * (section 9, LatentMoE listing step 3).  x is float (bf16 widened), d is float. */
void k3o_expert(int H, int I, const uint8_t *rec, const float *x, float b1, float b2,
                float *d, int nthreads) {
    int64_t off[7];
    k3o_record_offsets(H, I, off);
    float *g = (float *)malloc(sizeof(float) * (size_t)I);
    float *u = (float *)malloc(sizeof(float) * (size_t)I);
    float *act = (float *)malloc(sizeof(float) * (size_t)I);
    k3o_mxfp4_gemv(I, H, rec + off[0], rec + off[1], x, g, nthreads);
    k3o_mxfp4_gemv(I, H, rec + off[4], rec + off[5], x, u, nthreads);
    k3o_situ(I, b1, b2, g, u, act);
    k3o_mxfp4_gemv(H, I, rec + off[2], rec + off[3], act, d, nthreads);
    free(g);
    free(u);
    free(act);
}

/* Shared expert on one token (section 9, LatentMoE listing step 6): bf16 gate/up
 * [SI][H] and down [H][SI], SiTU in between; its output is added unweighted. */
void k3o_shared_expert(int H, int SI, const uint16_t *gate, const uint16_t *up,
                       const uint16_t *down, const float *x, float b1, float b2, float *ds,
                       int nthreads) {
    float *g = (float *)malloc(sizeof(float) * (size_t)SI);
    float *u = (float *)malloc(sizeof(float) * (size_t)SI);
    float *act = (float *)malloc(sizeof(float) * (size_t)SI);
    k3o_bf16_gemv(SI, H, gate, x, g, nthreads);
    k3o_bf16_gemv(SI, H, up, x, u, nthreads);
    k3o_situ(SI, b1, b2, g, u, act);
    k3o_bf16_gemv(H, SI, down, act, ds, nthreads);
    free(g);
    free(u);
    free(act);
}

/* The routed sum and the shared expert (section 9, LatentMoE listing steps 3 and 6):
 *   acc[i] = 0.0f;  for j = 0 .. K-1 in router order:  acc[i] = acc[i] + w[j] * d[j][i]
 * with one float product and one float sum per term (the build turns off contraction,
 * so no fused multiply-add), then y[i] = acc[i] + ds[i], one float add (skipped when ds
 * is NULL).  Float addition is not associative: the order of the terms is part of the
 * result.  d is [K][H]. */
void k3o_combine(int H, int K, const float *w, const float *d, const float *ds, float *y) {
    for (int i = 0; i < H; i++) {
        float acc = 0.0f;
        for (int j = 0; j < K; j++) {
            const float p = w[j] * d[(size_t)j * H + i];
            acc = acc + p;
        }
        y[i] = ds ? acc + ds[i] : acc;
    }
}

/* The layer for ONE token whose route is already known.
 *   recs[j]  : the expert record of the j-th selected expert (router order)
 *   w[j]     : its weight
 *   y        = the float router-order sum of w[j] d_j plus the shared expert's output
 *              (unweighted; no shared expert when gate == NULL), as k3o_combine forms it.
 * x is the token's bf16 input. */
void k3o_moe_token(int H, int I, int K, int SI, const uint16_t *x,
                   const uint8_t *const *recs, const float *w, const uint16_t *sh_gate,
                   const uint16_t *sh_up, const uint16_t *sh_down, float b1, float b2,
                   float *y, int nthreads) {
    float *xf = (float *)malloc(sizeof(float) * (size_t)H);
    float *d = (float *)malloc(sizeof(float) * (size_t)H * (size_t)(K > 0 ? K : 1));
    float *ds = sh_gate ? (float *)malloc(sizeof(float) * (size_t)H) : NULL;
    for (int i = 0; i < H; i++) xf[i] = k3o_bf16_to_f32(x[i]);
    for (int j = 0; j < K; j++) k3o_expert(H, I, recs[j], xf, b1, b2, d + (size_t)j * H, nthreads);
    if (sh_gate) k3o_shared_expert(H, SI, sh_gate, sh_up, sh_down, xf, b1, b2, ds, nthreads);
    k3o_combine(H, K, w, d, ds, y);
    free(xf);
    free(d);
    free(ds);
}

/* One token through the page's LatentMoE (section 9, LatentMoE listing), its route
 * (step 1, the router on the FULL-width x) already known:
 *   2. z = Wdn x              Wdn bf16 [L][H]; double accumulation, rounded to float
 *   3. accL = the float router-order sum of w[j] * expert_j(z)   (k3o_combine); the
 *                             experts run in the latent: input z (float), records of
 *                             the (L, I) layout
 *   4. if norm: accL = RMSNorm(accL) with weight nw [L] and eps -- on the AGGREGATE,
 *                             after the sum, not on each expert's output
 *   5. y = Wup accL           Wup bf16 [H][L]
 *   6. y = y + shared(x)      the shared experts (bf16 gate/up [SI][H], down [H][SI]; the
 *                             page's two experts of width I are one of width SI = 2 I)
 *                             on the ORIGINAL x, added unweighted with one float add per
 *                             element; skipped when sh_gate == NULL.
 * z_out and accl_out ([L] each, optional) receive z and the latent sum after step 4. */
void k3o_latent_moe_token(int H, int L, int I, int K, int SI, const uint16_t *x,
                          const uint16_t *wdn, const uint16_t *wup, const float *nw, int norm,
                          float eps, const uint8_t *const *recs, const float *w,
                          const uint16_t *sh_gate, const uint16_t *sh_up,
                          const uint16_t *sh_down, float b1, float b2, float *y, float *z_out,
                          float *accl_out, int nthreads) {
    float *xf = (float *)malloc(sizeof(float) * (size_t)H);
    float *z = (float *)malloc(sizeof(float) * (size_t)L);
    float *d = (float *)malloc(sizeof(float) * (size_t)L * (size_t)(K > 0 ? K : 1));
    float *acc = (float *)malloc(sizeof(float) * (size_t)L);
    for (int i = 0; i < H; i++) xf[i] = k3o_bf16_to_f32(x[i]);
    k3o_bf16_gemv(L, H, wdn, xf, z, nthreads);
    for (int j = 0; j < K; j++) k3o_expert(L, I, recs[j], z, b1, b2, d + (size_t)j * L, nthreads);
    k3o_combine(L, K, w, d, NULL, acc);
    if (norm) k3o_rmsnorm(L, acc, nw, eps, acc);
    k3o_bf16_gemv(H, L, wup, acc, y, nthreads);
    if (sh_gate) {
        float *ds = (float *)malloc(sizeof(float) * (size_t)H);
        k3o_shared_expert(H, SI, sh_gate, sh_up, sh_down, xf, b1, b2, ds, nthreads);
        for (int i = 0; i < H; i++) y[i] = y[i] + ds[i];
        free(ds);
    }
    if (z_out) memcpy(z_out, z, sizeof(float) * (size_t)L);
    if (accl_out) memcpy(accl_out, acc, sizeof(float) * (size_t)L);
    free(xf);
    free(z);
    free(d);
    free(acc);
}

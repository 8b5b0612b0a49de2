/*
 * moe_oracle.c -- plain, slow fp64 CPU reference for the routed mixture-of-experts
 * FFN layer (router, softmax top-k, bucketing, block-quantised experts, SwiGLU,
 * down projection, weighted combine, shared expert, RMSNorm chain step).
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load this file. It shares no code, header,
 * table or constant with the CUDA library; it is written from the pages' text:
 *
 *   [K]  Krasis white paper ("Phase-Separated Inference for Large Mixture-of-Experts
 *        Models on Memory-Constrained NVIDIA GPUs"), sec. 5.3 "Per-token routed expert
 *        execution", sec. 7.3/7.5 (zero-weight slots), Finding 2 (fixed reduction order).
 *   [S]  "Strata in the source: one verify window, three workers and a cache that
 *        learns", sections "The byte budget, in code" (Q2_0 block: 64 weights =
 *        16 bytes of 2-bit codes + an fp16 scale; expert = gate, up, down) and
 *        "The CPU kernels" (codes {0,1,2,3} mean {-1,0,1,2} x scale; the 2-bit
 *        unpack order).
 *   [R]  kairos-engine README, "The MoE forward" (normalise, router GEMM, top-k,
 *        expert-major buckets, routed and shared branches summed).
 *
 * Every floating-point step is fp64. Every loop runs in plain index order; no
 * blocking, fusion or reordering. Readings of points the pages leave open:
 *   - canonical block = fp16 scale (2 bytes, little-endian) followed by the codes;
 *   - Q4 blocks hold 32 weights, weight n in nibble (byte[n/2] >> 4*(n%2)) & 15;
 *   - blocks run along the reduction dimension of each output row; an expert blob
 *     is gate [F][H], then up [F][H], then down [H][F], rows in row-major order;
 *   - selection is on the logits: larger first, ties to the lower expert index,
 *     NaN ranks below every number; weights are the softmax over all experts,
 *     renormalised over the K selected;
 *   - the shared expert has weight 1 and is added after the routed sum.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_Q4 0 /* 32 weights per block, 4-bit codes */
#define ORC_Q2 1 /* 64 weights per block, 2-bit codes ("Q2_0") */

#define ORC_ACT_SWIGLU 0
#define ORC_ACT_GEGLU_TANH 1

/* status bits returned by orc_layer_forward */
#define ORC_ABSENT 1
#define ORC_NONFINITE 2

/* ---------------------------------------------------------------- format */

/* IEEE 754 binary16 -> double, exact (normal, subnormal, inf, nan). */
double orc_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 31;
    int mant = h & 1023;
    double v;
    if (expo == 0) {
        v = ldexp((double)mant, -24); /* subnormal: mant * 2^-24 */
    } else if (expo == 31) {
        v = mant ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + mant), expo - 25); /* 1.mant * 2^(expo-15) */
    }
    return sign ? -v : v;
}

int orc_block_weights(int kind) { return kind == ORC_Q2 ? 64 : 32; }

/* 2-byte scale + 16 bytes of codes, for both formats. */
int orc_block_bytes(int kind) { (void)kind; return 18; }

/* Bytes of one expert blob: gate and up (F rows of H) and down (H rows of F). */
int64_t orc_expert_bytes(int kind, int H, int F)
{
    int64_t weights = 3 * (int64_t)H * (int64_t)F;
    return weights / orc_block_weights(kind) * orc_block_bytes(kind);
}

/* The code (unsigned integer) of weight n of one block's code bytes. */
static int orc_code(int kind, const uint8_t *codes, int n)
{
    if (kind == ORC_Q2)
        return (codes[n / 4] >> (2 * (n % 4))) & 3;
    return (codes[n / 2] >> (4 * (n % 2))) & 15;
}

/* Dequantise n_weights consecutive weights stored as canonical blocks:
 * w = d * (q - zero_point), d the block's fp16 scale. */
void orc_dequant(int kind, int zero_point, const uint8_t *blocks, int64_t n_weights, double *out)
{
    int bw = orc_block_weights(kind);
    int bb = orc_block_bytes(kind);
    int64_t n_blocks = n_weights / bw;
    for (int64_t b = 0; b < n_blocks; b++) {
        const uint8_t *blk = blocks + b * bb;
        uint16_t dbits = (uint16_t)(blk[0] | (blk[1] << 8));
        double d = orc_f16_to_f64(dbits);
        for (int n = 0; n < bw; n++) {
            int q = orc_code(kind, blk + 2, n);
            out[b * bw + n] = d * (double)(q - zero_point);
        }
    }
}

/* Dense fp64 copies of the three matrices of one expert blob. */
static void orc_expert_matrices(int kind, int zp, const uint8_t *blob, int H, int F,
                                double *Wg, double *Wu, double *Wd)
{
    int64_t mat_bytes = (int64_t)H * F / orc_block_weights(kind) * orc_block_bytes(kind);
    orc_dequant(kind, zp, blob, (int64_t)F * H, Wg);
    orc_dequant(kind, zp, blob + mat_bytes, (int64_t)F * H, Wu);
    orc_dequant(kind, zp, blob + 2 * mat_bytes, (int64_t)H * F, Wd);
}

/* ---------------------------------------------------------------- router */

/* logits[t][e] = sum_h Wr[e][h] * x[t][h] (+ bias[e]). */
void orc_router_logits(const double *x, int T, int H, const double *Wr, int E,
                       const double *bias, double *logits)
{
    for (int t = 0; t < T; t++)
        for (int e = 0; e < E; e++) {
            double s = 0.0;
            for (int h = 0; h < H; h++)
                s += Wr[(int64_t)e * H + h] * x[(int64_t)t * H + h];
            if (bias)
                s += bias[e];
            logits[(int64_t)t * E + e] = s;
        }
}

/* 1 if expert a ranks before expert b: larger logit first, equal logits to the
 * lower index, NaN below every number (two NaNs: lower index first). */
static int orc_ranks_before(const double *l, int a, int b)
{
    int na = isnan(l[a]), nb = isnan(l[b]);
    if (na || nb) {
        if (na && nb)
            return a < b;
        return nb;
    }
    if (l[a] > l[b])
        return 1;
    if (l[a] < l[b])
        return 0;
    return a < b;
}

/* Top-K ids per token (in rank order) and their weights: the softmax over all E
 * logits, renormalised to sum 1 over the K selected. Returns 1 if any logit of
 * any token is not finite (weights are then left NaN), else 0. */
int orc_topk(const double *logits, int T, int E, int K, int *ids, double *w)
{
    int nonfinite = 0;
    char *taken = (char *)malloc((size_t)E);
    for (int t = 0; t < T; t++) {
        const double *l = logits + (int64_t)t * E;
        int bad = 0;
        for (int e = 0; e < E; e++)
            if (!isfinite(l[e]))
                bad = 1;
        memset(taken, 0, (size_t)E);
        for (int k = 0; k < K; k++) {
            int best = -1;
            for (int e = 0; e < E; e++) {
                if (taken[e])
                    continue;
                if (best < 0 || orc_ranks_before(l, e, best))
                    best = e;
            }
            taken[best] = 1;
            ids[t * K + k] = best;
        }
        if (bad) {
            nonfinite = 1;
            for (int k = 0; k < K; k++)
                w[t * K + k] = NAN;
            continue;
        }
        /* full softmax over all E experts */
        double m = l[0];
        for (int e = 1; e < E; e++)
            if (l[e] > m)
                m = l[e];
        double z = 0.0;
        for (int e = 0; e < E; e++)
            z += exp(l[e] - m);
        double sel = 0.0;
        for (int k = 0; k < K; k++)
            sel += exp(l[ids[t * K + k]] - m) / z;
        for (int k = 0; k < K; k++)
            w[t * K + k] = (exp(l[ids[t * K + k]] - m) / z) / sel;
    }
    free(taken);
    return nonfinite;
}

/* ---------------------------------------------------------------- bucket */

/* Expert-major grouping of the T*K (token, rank) pairs, pair p = t*K + k.
 * counts[e] = pairs routed to e; offsets = exclusive prefix sum (E+1 entries);
 * perm lists the pairs of expert 0 first, then expert 1, ..., each group in
 * increasing pair order; active lists the experts with count > 0, ascending. */
void orc_bucket(const int *ids, int T, int K, int E, int *counts, int *offsets, int *perm,
                int *active, int *n_active)
{
    int P = T * K;
    int pos = 0, na = 0;
    for (int e = 0; e < E; e++) {
        offsets[e] = pos;
        int c = 0;
        for (int p = 0; p < P; p++)
            if (ids[p] == e) {
                perm[pos++] = p;
                c++;
            }
        counts[e] = c;
        if (c > 0)
            active[na++] = e;
    }
    offsets[E] = pos;
    *n_active = na;
}

/* ---------------------------------------------------------------- expert */

static double orc_silu(double g) { return g / (1.0 + exp(-g)); }

/* tanh-approximated GELU: 0.5 g (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3))) */
static double orc_gelu_tanh(double g)
{
    const double c = sqrt(2.0 / M_PI);
    return 0.5 * g * (1.0 + tanh(c * (g + 0.044715 * g * g * g)));
}

/* y[r] = W_down * (act(W_gate x[r]) * (W_up x[r])) for n input rows. */
void orc_expert_ffn(int kind, int zero_point, int act, const uint8_t *blob, int H, int F,
                    const double *x, int n, double *y)
{
    double *Wg = (double *)malloc(sizeof(double) * (size_t)F * H);
    double *Wu = (double *)malloc(sizeof(double) * (size_t)F * H);
    double *Wd = (double *)malloc(sizeof(double) * (size_t)H * F);
    double *hid = (double *)malloc(sizeof(double) * (size_t)F);
    orc_expert_matrices(kind, zero_point, blob, H, F, Wg, Wu, Wd);
    for (int r = 0; r < n; r++) {
        const double *xr = x + (int64_t)r * H;
        for (int f = 0; f < F; f++) {
            double g = 0.0, u = 0.0;
            for (int h = 0; h < H; h++) {
                g += Wg[(int64_t)f * H + h] * xr[h];
                u += Wu[(int64_t)f * H + h] * xr[h];
            }
            double a = act == ORC_ACT_GEGLU_TANH ? orc_gelu_tanh(g) : orc_silu(g);
            hid[f] = a * u;
        }
        for (int j = 0; j < H; j++) {
            double s = 0.0;
            for (int f = 0; f < F; f++)
                s += Wd[(int64_t)j * F + f] * hid[f];
            y[(int64_t)r * H + j] = s;
        }
    }
    free(Wg);
    free(Wu);
    free(Wd);
    free(hid);
}

/* ---------------------------------------------------------------- layer */

/* One MoE layer for T tokens:
 *   logits = router(x) unless logits_in is given (then those logits are used,
 *   e.g. the fp32 logits another implementation produced, widened to fp64);
 *   ids, w = top-K with renormalised softmax weights;
 *   y[t] = sum_{k=0}^{K-1} w[t][k] * expert_{ids[t][k]}(x[t])   (k order)
 *          + shared(x[t])                                      (if present).
 * experts[e] == NULL means expert e is absent: it contributes nothing and the
 * ORC_ABSENT bit is returned. A pair with weight exactly 0 contributes nothing.
 * Returns status bits (ORC_ABSENT, ORC_NONFINITE). */
int orc_layer_forward(int kind, int zero_point, int act, int H, int E, int K, int F,
                      const double *Wr, const double *bias, const uint8_t *const *experts,
                      const uint8_t *shared, int F_shared, const double *x, int T,
                      const double *logits_in, double *y, int *ids, double *w,
                      double *logits_out)
{
    int status = 0;
    double *logits = (double *)malloc(sizeof(double) * (size_t)T * E);
    double *ye = (double *)malloc(sizeof(double) * (size_t)H);
    if (logits_in)
        memcpy(logits, logits_in, sizeof(double) * (size_t)T * E);
    else
        orc_router_logits(x, T, H, Wr, E, bias, logits);
    if (logits_out)
        memcpy(logits_out, logits, sizeof(double) * (size_t)T * E);
    if (orc_topk(logits, T, E, K, ids, w))
        status |= ORC_NONFINITE;
    for (int t = 0; t < T; t++) {
        double *yt = y + (int64_t)t * H;
        const double *xt = x + (int64_t)t * H;
        for (int j = 0; j < H; j++)
            yt[j] = 0.0;
        for (int k = 0; k < K; k++) {
            int e = ids[t * K + k];
            double wk = w[t * K + k];
            if (!experts[e]) {
                status |= ORC_ABSENT;
                continue;
            }
            if (wk == 0.0)
                continue;
            orc_expert_ffn(kind, zero_point, act, experts[e], H, F, xt, 1, ye);
            for (int j = 0; j < H; j++)
                yt[j] += wk * ye[j];
        }
        if (shared) {
            orc_expert_ffn(kind, zero_point, act, shared, H, F_shared, xt, 1, ye);
            for (int j = 0; j < H; j++)
                yt[j] += ye[j];
        }
    }
    free(logits);
    free(ye);
    return status;
}

/* ---------------------------------------------------------------- chain */

/* Weightless RMSNorm: out[t][h] = x[t][h] / sqrt(mean_h x[t][h]^2 + eps). */
void orc_rmsnorm(const double *x, int T, int H, double eps, double *out)
{
    for (int t = 0; t < T; t++) {
        double ss = 0.0;
        for (int h = 0; h < H; h++)
            ss += x[(int64_t)t * H + h] * x[(int64_t)t * H + h];
        double r = 1.0 / sqrt(ss / H + eps);
        for (int h = 0; h < H; h++)
            out[(int64_t)t * H + h] = x[(int64_t)t * H + h] * r;
    }
}

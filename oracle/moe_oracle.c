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
 *
 * Further routing forms, from the same pages:
 *   [R] "The MoE forward": the router scale is per input dimension, the down
 *       scale per expert (logits = Wr (x * s_r); expert e's output is scaled by s_e);
 *   [K] sec. 5.3: sigmoid top-k routers (scores 1 / (1 + e^-l), optionally
 *       normalised over the K chosen); the selection of the K largest logits is
 *       the selection of the K largest sigmoid scores, as the sigmoid is monotone;
 *   [K] sec. 7.2-7.3: the P/M route-drop rule (below, orc_route_drop), no
 *       renormalisation of the surviving weights.
 * The route-drop rule decides integers (which routes go) from floating-point sums;
 * it is written in fp32, the precision the GPU decides in, and fed fp32 weights.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_Q4 0 /* 32 weights per block, 4-bit codes */
#define ORC_Q2 1 /* 64 weights per block, 2-bit codes ("Q2_0") */

#define ORC_ACT_SWIGLU 0
#define ORC_ACT_GEGLU_TANH 1

#define ORC_ROUTER_SOFTMAX 0
#define ORC_ROUTER_SIGMOID 1
#define ORC_ROUTER_SIGMOID_NORM 2

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

/* logits[t][e] = sum_h Wr[e][h] * (x[t][h] * s[h]) (+ bias[e]): the router input
 * scaled per input dimension ([R]). */
void orc_router_logits_scaled(const double *x, int T, int H, const double *Wr, int E,
                              const double *bias, const double *s, double *logits)
{
    for (int t = 0; t < T; t++)
        for (int e = 0; e < E; e++) {
            double acc = 0.0;
            for (int h = 0; h < H; h++)
                acc += Wr[(int64_t)e * H + h] * (x[(int64_t)t * H + h] * s[h]);
            if (bias)
                acc += bias[e];
            logits[(int64_t)t * E + e] = acc;
        }
}

/* Route weights of the K chosen logits l[0..K) (rank order) for a router kind:
 * softmax over the K (= the full softmax renormalised over them), the sigmoid
 * 1 / (1 + e^-l), or the sigmoid divided by its sum over the K. */
void orc_route_weights(int kind, const double *l, int K, double *w)
{
    if (kind == ORC_ROUTER_SOFTMAX) {
        double sum = 0.0;
        for (int k = 0; k < K; k++)
            sum += exp(l[k] - l[0]);
        for (int k = 0; k < K; k++)
            w[k] = exp(l[k] - l[0]) / sum;
        return;
    }
    double sum = 0.0;
    for (int k = 0; k < K; k++) {
        w[k] = 1.0 / (1.0 + exp(-l[k]));
        sum += w[k];
    }
    if (kind == ORC_ROUTER_SIGMOID_NORM)
        for (int k = 0; k < K; k++)
            w[k] /= sum;
}

/* The P/M route-drop rule ([K] sec. 7.2) on one token's K route weights w[0..K)
 * (rank order, fp32) with eligible[k] (the expert of rank k may be dropped):
 *   1. the first ceil(K P / 100) ranks are kept;
 *   2. candidates: later ranks that are eligible and have a positive weight;
 *   3. taken from the smallest weight up (equal weights: the later rank first);
 *   4. a candidate is dropped while the dropped total c (fp32, in that order)
 *      stays at or below M percent of S, the sum of the K weights in rank order
 *      (fp32): c * 100 <= M * S; the first that does not fit ends the scan.
 * Dropped routes get weight 0; the others keep theirs ([K] sec. 7.3). Returns the
 * number dropped; *share = c / S (0 if S is 0); *margin = the smallest
 * |c' * 100 - M * S| / (M * S) over the comparisons made (how far each decision
 * was from flipping; 1 if none or M * S is 0). */
int orc_route_drop(const float *w, const uint8_t *eligible, int K, int P, int M, float *w_out,
                   float *share, double *margin)
{
    int protect = (K * P + 99) / 100;
    float S = 0.0f;
    for (int k = 0; k < K; k++)
        S += w[k];
    int order[64], n = 0;
    for (int k = protect; k < K; k++)
        if (eligible[k] && w[k] > 0.0f)
            order[n++] = k;
    /* insertion sort: ascending weight, equal weights later rank first */
    for (int i = 1; i < n; i++) {
        int v = order[i], j = i - 1;
        while (j >= 0 && (w[order[j]] > w[v] || (w[order[j]] == w[v] && order[j] < v))) {
            order[j + 1] = order[j];
            j--;
        }
        order[j + 1] = v;
    }
    for (int k = 0; k < K; k++)
        w_out[k] = w[k];
    float c = 0.0f, lim = (float)M * S;
    double mg = 1.0;
    int nd = 0;
    for (int i = 0; i < n; i++) {
        float c2 = c + w[order[i]];
        float lhs = c2 * 100.0f;
        if (lim > 0.0f) {
            double r = fabs((double)lhs - (double)lim) / (double)lim;
            if (r < mg)
                mg = r;
        }
        if (lhs <= lim) {
            c = c2;
            w_out[order[i]] = 0.0f;
            nd++;
        } else {
            break;
        }
    }
    *share = S > 0.0f ? c / S : 0.0f;
    *margin = mg;
    return nd;
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
/* The layer with the routing forms above: logits from the scaled router input
 * (router_scale may be NULL) unless logits_in is given; top-K selection as
 * orc_topk; route weights of router_kind (fp64); if drop_eligible is not NULL,
 * the drop rule on the fp32 rounding of those weights (drop_w32 may give the fp32
 * weights to decide on instead), dropped routes then count 0; then each weight is
 * multiplied by down_scale[e] (may be NULL); the combine as orc_layer_forward.
 * omitted [T] (may be NULL) gets each token's dropped share, margin [T] the
 * decision margin of orc_route_drop. Returns the status bits. */
int orc_layer_forward_routed(int kind, int zero_point, int act, int H, int E, int K, int F,
                             const double *Wr, const double *bias, const double *router_scale,
                             int router_kind, const double *down_scale, const uint8_t *drop_eligible,
                             int P, int M, const float *drop_w32, const uint8_t *const *experts,
                             const uint8_t *shared, int F_shared, const double *x, int T,
                             const double *logits_in, double *y, int *ids, double *w, float *omitted,
                             double *margin)
{
    int status = 0;
    double *logits = (double *)malloc(sizeof(double) * (size_t)T * E);
    double *ye = (double *)malloc(sizeof(double) * (size_t)H);
    if (logits_in)
        memcpy(logits, logits_in, sizeof(double) * (size_t)T * E);
    else if (router_scale)
        orc_router_logits_scaled(x, T, H, Wr, E, bias, router_scale, logits);
    else
        orc_router_logits(x, T, H, Wr, E, bias, logits);
    if (orc_topk(logits, T, E, K, ids, w))
        status |= ORC_NONFINITE;
    for (int t = 0; t < T; t++) {
        double lsel[32];
        float w32[32], wd[32], share = 0.0f;
        uint8_t el[32];
        double mg = 1.0;
        int bad = 0;
        for (int k = 0; k < K; k++) {
            lsel[k] = logits[(int64_t)t * E + ids[t * K + k]];
            if (!isfinite(lsel[k]))
                bad = 1;
        }
        if (!bad)
            orc_route_weights(router_kind, lsel, K, w + t * K);
        if (!bad && drop_eligible) {
            for (int k = 0; k < K; k++) {
                w32[k] = drop_w32 ? drop_w32[t * K + k] : (float)w[t * K + k];
                el[k] = drop_eligible[ids[t * K + k]] != 0;
            }
            orc_route_drop(w32, el, K, P, M, wd, &share, &mg);
            for (int k = 0; k < K; k++)
                if (wd[k] == 0.0f && w32[k] != 0.0f)
                    w[t * K + k] = 0.0;
        }
        if (omitted)
            omitted[t] = share;
        if (margin)
            margin[t] = mg;
        if (!bad && down_scale)
            for (int k = 0; k < K; k++)
                w[t * K + k] *= down_scale[ids[t * K + k]];
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

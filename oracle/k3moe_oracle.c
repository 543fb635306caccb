/*
 * CPU oracle for the Kimi K3 LatentMoE layer with MXFP4 routed experts.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, plainly written reference
 * that the CUDA library is checked against. Only the tests, the package
 * smoke check and bench.py's CPU-baseline leg may load it; the library never
 * does, and it shares no code, header or table with the library.
 *
 * Everything is computed in double precision. Inputs arrive in the checkpoint
 * formats (bf16 bit patterns, packed e2m1 nibbles, ue8m0 scale bytes, fp32
 * bias) and are widened exactly; intermediate values are never rounded.
 *
 * Sources (pages about "kimi-k3-in-c" and "colibri"):
 *  - MXFP4 format and matmul: kimi-k3-in-c README, Part II section 4
 *    ("the experts already ship at half a byte"): E2M1 table, E8M0 rule,
 *    low nibble = even column, fp64 accumulation per 32-group then x scale.
 *    colibri docs/kimi_k3.md, "Weights": bit 3 = sign, w = v * 2^(scale-127).
 *  - RMSNorm and the bf16 widening: kimi-k3-in-c README, section 5
 *    ("Kernels with a floating point contract").
 *  - Router, top-k, SiTU-GLU, the layer: kimi-k3-in-c README, section 9
 *    ("Picking 16 experts of 896"); colibri "Stable LatentMoE" bullet.
 *  - The cut of the picks to cumulative weight p: the README's run-time
 *    option K3_TOPP. The dense feed-forward layer 0: the README's K3Cfg
 *    ("first_dense", "dense_inter"), in the model's SiTU-GLU form.
 *
 * Parity pins for every function live in the tests (hand-packed bytes, closed
 * forms, invariants, and a dense fp64 route through the whole layer).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_GROUP 32

/* ------------------------------------------------------------------------ */
/* Formats                                                                   */
/* ------------------------------------------------------------------------ */

/* bf16 -> double: the bf16 bits are the top half of an fp32 (README section 5:
 * widening is a 16-bit left shift, exact). */
double orc_bf16(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* E2M1 nibble -> value. Bit 3 is the sign, the low three bits index the
 * magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6} (README section 4, E2M1 table). */
double orc_e2m1(unsigned nibble)
{
    static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    const double m = mag[nibble & 7u];
    return (nibble & 8u) ? -m : m;
}

/* ue8m0 scale byte -> 2^(b-127); 255 (NaN by the MX spec) maps to 0, which
 * zeroes its group (README section 4, E8M0 rule). */
double orc_e8m0(unsigned byte)
{
    if ((byte & 0xFFu) == 255u) return 0.0;
    return ldexp(1.0, (int)(byte & 0xFFu) - 127);
}

/* Weight at logical column c of one MXFP4 row: byte c/2, low nibble for an
 * even c and high nibble for an odd c, times the scale of group c/32. */
double orc_mxfp4_weight(const uint8_t *packed_row, const uint8_t *scale_row, int c)
{
    const uint8_t b = packed_row[c / 2];
    const unsigned nib = (c % 2 == 0) ? (b & 0x0Fu) : (b >> 4);
    return orc_e2m1(nib) * orc_e8m0(scale_row[c / ORC_GROUP]);
}

/* y[o] = sum_c W[o][c] * x[c] for an MXFP4 matrix of `rows` rows and `in`
 * logical columns (row pitch (in+1)/2 bytes, ceil(in/32) scales per row).
 * As in the README's k3_matmul_mxfp4: per group, the raw table values are
 * dotted with x in fp64, the partial sum is multiplied by the scale and added;
 * a group whose scale decodes to 0 is skipped; the last group may be short. */
void orc_mxfp4_matvec(double *y, const double *x, const uint8_t *packed,
                      const uint8_t *scales, int in, int rows)
{
    const int rowbytes = (in + 1) / 2;
    const int ngroup = (in + ORC_GROUP - 1) / ORC_GROUP;
    for (int o = 0; o < rows; o++) {
        const uint8_t *pb = packed + (size_t)o * (size_t)rowbytes;
        const uint8_t *sb = scales + (size_t)o * (size_t)ngroup;
        double acc = 0.0;
        for (int g = 0; g < ngroup; g++) {
            const double s = orc_e8m0(sb[g]);
            if (s == 0.0) continue;
            const int c0 = g * ORC_GROUP;
            const int c1 = (c0 + ORC_GROUP <= in) ? c0 + ORC_GROUP : in;
            double part = 0.0;
            for (int c = c0; c < c1; c++) {
                const uint8_t b = pb[c / 2];
                const unsigned nib = (c % 2 == 0) ? (b & 0x0Fu) : (b >> 4);
                part += x[c] * orc_e2m1(nib);
            }
            acc += part * s;
        }
        y[o] = acc;
    }
}

/* y[o] = sum_i W[o][i] * x[i], W bf16 [out, in] row-major (row = output). */
void orc_bf16_matvec(double *y, const double *x, const uint16_t *W, int in, int out)
{
    for (int o = 0; o < out; o++) {
        const uint16_t *row = W + (size_t)o * (size_t)in;
        double acc = 0.0;
        for (int i = 0; i < in; i++) acc += orc_bf16(row[i]) * x[i];
        y[o] = acc;
    }
}

/* ------------------------------------------------------------------------ */
/* Elementwise pieces                                                        */
/* ------------------------------------------------------------------------ */

double orc_sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }

/* SiTU-GLU of one (gate, up) pair: b1*tanh(g/b1) * sigmoid(g) * b2*tanh(u/b2).
 * The sigmoid reads the uncapped gate (README section 9, k3_situ_glu; colibri
 * "Activation is SiTU-GLU"). Its magnitude is below b1*b2. */
double orc_situ(double g, double u, double b1, double b2)
{
    return (b1 * tanh(g / b1)) * orc_sigmoid(g) * (b2 * tanh(u / b2));
}

/* RMSNorm: out = x / sqrt(mean(x^2) + eps) * gain, sum of squares in fp64 and
 * eps inside the square root (README section 5, k3_rmsnorm). gain may be NULL
 * (unit gain). out may alias x. */
void orc_rmsnorm(double *out, const double *x, const double *gain, int n, double eps)
{
    double ss = 0.0;
    for (int i = 0; i < n; i++) ss += x[i] * x[i];
    const double inv = 1.0 / sqrt(ss / (double)n + eps);
    for (int i = 0; i < n; i++) out[i] = x[i] * inv * (gain ? gain[i] : 1.0);
}

/* ------------------------------------------------------------------------ */
/* Router (README section 9, k3_router; colibri "Stable LatentMoE")          */
/* ------------------------------------------------------------------------ */

typedef struct { double ch; int e; } orc_pick;

/* Order: larger selection score first; equal scores -> lower expert id first.
 * This is the order the README's repeated strict-'>' maximum produces. */
static int orc_pick_cmp(const void *a, const void *b)
{
    const orc_pick *p = (const orc_pick *)a, *q = (const orc_pick *)b;
    if (p->ch > q->ch) return -1;
    if (p->ch < q->ch) return 1;
    return (p->e < q->e) ? -1 : (p->e > q->e);
}

/* One token. logits[e] = x . Wr[e]; sc = sigmoid(logit) (the unbiased score);
 * ch = sc + bias[e] (the selection score). The top-k by ch are found by
 * sorting all E (ch, e) pairs; the weight of each winner is its UNBIASED sc,
 * divided by the winners' sum when renorm is set and the sum is positive, then
 * multiplied by routed_scale. ids/w are written in selection order.
 * sc_out / ch_out (length E) and margin (ch of the k-th pick minus ch of the
 * (k+1)-th; +inf when k == E) are optional diagnostics. */
void orc_router_token(int *ids, double *w, double *sc_out, double *ch_out, double *margin,
                      const double *x, const uint16_t *Wr, const float *bias,
                      int H, int E, int k, int renorm, double routed_scale)
{
    double *sc = (double *)malloc(sizeof(double) * (size_t)E);
    orc_pick *pk = (orc_pick *)malloc(sizeof(orc_pick) * (size_t)E);
    for (int e = 0; e < E; e++) {
        const uint16_t *row = Wr + (size_t)e * (size_t)H;
        double acc = 0.0;
        for (int i = 0; i < H; i++) acc += x[i] * orc_bf16(row[i]);
        sc[e] = orc_sigmoid(acc);
        pk[e].ch = sc[e] + (bias ? (double)bias[e] : 0.0);
        pk[e].e = e;
        if (sc_out) sc_out[e] = sc[e];
        if (ch_out) ch_out[e] = pk[e].ch;
    }
    qsort(pk, (size_t)E, sizeof(orc_pick), orc_pick_cmp);
    double sum = 0.0;
    for (int j = 0; j < k; j++) {
        ids[j] = pk[j].e;
        w[j] = sc[pk[j].e];
        sum += w[j];
    }
    if (renorm && sum > 0.0)
        for (int j = 0; j < k; j++) w[j] /= sum;
    for (int j = 0; j < k; j++) w[j] *= routed_scale;
    if (margin) *margin = (k < E) ? pk[k - 1].ch - pk[k].ch : INFINITY;
    free(pk);
    free(sc);
}

/* ------------------------------------------------------------------------ */
/* Token -> expert permutation                                               */
/* ------------------------------------------------------------------------ */

/* counts[e] = number of (t, j) with ids[t*k+j] == e; offsets = exclusive prefix
 * sum (E+1 entries); perm lists the flat pair index t*k+j grouped by expert in
 * ascending expert order, and inside one expert by ascending token (then slot).
 * Written as the plain definition: loop e, then t, then j. */
void orc_permutation(const int *ids, int T, int k, int E, int *counts, int *offsets, int *perm)
{
    int pos = 0;
    for (int e = 0; e < E; e++) {
        offsets[e] = pos;
        for (int t = 0; t < T; t++)
            for (int j = 0; j < k; j++)
                if (ids[t * k + j] == e) perm[pos++] = t * k + j;
        counts[e] = pos - offsets[e];
    }
    offsets[E] = pos;
}

/* The optional cut of a token's picks to cumulative weight p (the README's
 * K3_TOPP run-time option: drop the low-weight tail of the top-k and
 * renormalise). ids/w hold the k picks in selection order. In weight order
 * (larger first, equal weights: lower id first) a pick is kept while the sum
 * of the weights before it is below p times the total; the kept weights are
 * scaled back to the total. The kept picks stay in selection order at the
 * front; the dropped slots become id -1, weight 0. Returns the number kept.
 * *margin (optional) = the smallest |before - p * total| / total over the
 * picks after the first in weight order: how far the cut is from moving. */
int orc_topp_cut(int *ids, double *w, int k, double p, double *margin)
{
    int order[64], keep[64];
    double total = 0.0;
    for (int j = 0; j < k; j++) {
        order[j] = j;
        total += w[j];
    }
    for (int a = 1; a < k; a++)   /* insertion sort by (w desc, id asc) */
        for (int b = a; b > 0; b--) {
            const int x = order[b - 1], y = order[b];
            const int swap = w[y] > w[x] || (w[y] == w[x] && ids[y] < ids[x]);
            if (!swap) break;
            order[b - 1] = y;
            order[b] = x;
        }
    double before = 0.0, kept = 0.0, mg = INFINITY;
    for (int r = 0; r < k; r++) {
        const int j = order[r];
        keep[j] = total <= 0.0 || before < p * total;
        if (r > 0 && total > 0.0) {
            const double d = fabs(before - p * total) / total;
            if (d < mg) mg = d;
        }
        if (keep[j]) kept += w[j];
        before += w[j];
    }
    int tmp_ids[64];
    double tmp_w[64];
    int m = 0;
    for (int j = 0; j < k; j++)
        if (keep[j]) {
            tmp_ids[m] = ids[j];
            tmp_w[m] = kept > 0.0 ? w[j] * (total / kept) : w[j];
            m++;
        }
    for (int j = 0, n = m; j < k; j++)
        if (!keep[j]) {
            tmp_ids[n] = -1;
            tmp_w[n] = 0.0;
            n++;
        }
    memcpy(ids, tmp_ids, sizeof(int) * (size_t)k);
    memcpy(w, tmp_w, sizeof(double) * (size_t)k);
    if (margin) *margin = mg;
    return m;
}

/* ------------------------------------------------------------------------ */
/* The layer (README section 9, k3_moe; colibri "Stable LatentMoE")          */
/* ------------------------------------------------------------------------ */

typedef struct {
    int hidden, latent, n_experts, topk, moe_inter, shared_inter;
    int renorm;
    double rms_eps, situ_b1, situ_b2, routed_scale;
    double topp;   /* > 0: the cumulative-weight cut of the picks (0: off) */
} orc_cfg;

typedef struct {
    const uint16_t *router_w;   /* [E, H] bf16 */
    const float *router_bias;   /* [E] fp32 (may be NULL) */
    const uint16_t *down_w;     /* [L, H] bf16 */
    const uint16_t *up_w;       /* [H, L] bf16 */
    const uint16_t *latent_gain;/* [L] bf16 (NULL: no latent norm) */
    const uint16_t *sh_w1;      /* [S, H] bf16 (gate) */
    const uint16_t *sh_w3;      /* [S, H] bf16 (up) */
    const uint16_t *sh_w2;      /* [H, S] bf16 */
    const uint8_t *w1p, *w1s;   /* [E][I][L/2], [E][I][L/32] */
    const uint8_t *w3p, *w3s;   /* [E][I][L/2], [E][I][L/32] */
    const uint8_t *w2p, *w2s;   /* [E][L][I/2], [E][L][I/32] */
} orc_layer;

/* Optional per-token intermediates (each NULL or sized for `nrows` tokens). */
typedef struct {
    int *ids;         /* [nrows, k] */
    double *w;        /* [nrows, k] */
    double *margin;   /* [nrows] */
    double *z;        /* [nrows, L]  latent down projection */
    double *acc;      /* [nrows, L]  weighted sum of expert outputs */
    double *nrm;      /* [nrows, L]  RMSNorm(acc) */
    double *shared;   /* [nrows, S]  SiTU of the shared experts */
    double *h;        /* [nrows, k, I]  SiTU output of each picked expert */
} orc_trace;

/* One token of the layer:
 *  1. route on the full-width x;            2. z = down . x;
 *  3. acc = sum_j w_j * W2_e(SiTU(W1_e z, W3_e z)) over the picked experts;
 *  4. n = RMSNorm(acc) with the latent gain (aggregate first, then norm);
 *  5. y = up . n;
 *  6. y += Ws2 . SiTU(Ws1 x, Ws3 x): the shared experts read the ORIGINAL x
 *     and are added unweighted. */
static void orc_layer_token(const orc_cfg *c, const orc_layer *lw, const uint16_t *xrow,
                            double *y, int r, const orc_trace *tr)
{
    const int H = c->hidden, L = c->latent, E = c->n_experts, K = c->topk;
    const int I = c->moe_inter, S = c->shared_inter;
    const size_t per1 = (size_t)I * (size_t)(L / 2), per1s = (size_t)I * (size_t)(L / ORC_GROUP);
    const size_t per2 = (size_t)L * (size_t)(I / 2), per2s = (size_t)L * (size_t)(I / ORC_GROUP);

    double *x = (double *)malloc(sizeof(double) * (size_t)H);
    double *z = (double *)malloc(sizeof(double) * (size_t)L);
    double *acc = (double *)calloc((size_t)L, sizeof(double));
    double *g = (double *)malloc(sizeof(double) * (size_t)(I > S ? I : S));
    double *u = (double *)malloc(sizeof(double) * (size_t)(I > S ? I : S));
    double *a = (double *)malloc(sizeof(double) * (size_t)(I > S ? I : S));
    double *eo = (double *)malloc(sizeof(double) * (size_t)(L > H ? L : H));
    double *gain = (double *)malloc(sizeof(double) * (size_t)L);
    int *ids = (int *)malloc(sizeof(int) * (size_t)K);
    double *w = (double *)malloc(sizeof(double) * (size_t)K);
    double margin;

    for (int i = 0; i < H; i++) x[i] = orc_bf16(xrow[i]);

    /* 1. router on the full width */
    orc_router_token(ids, w, NULL, NULL, &margin, x, lw->router_w, lw->router_bias,
                     H, E, K, c->renorm, c->routed_scale);
    if (c->topp > 0.0) {   /* optional cut of the weight tail */
        double mt;
        orc_topp_cut(ids, w, K, c->topp, &mt);
        if (mt < margin) margin = mt;
    }
    /* 2. latent down projection */
    orc_bf16_matvec(z, x, lw->down_w, H, L);
    /* 3. routed experts in the latent */
    for (int j = 0; j < K; j++) {
        const int e = ids[j];
        if (e < 0) continue;   /* dropped by the cut */
        orc_mxfp4_matvec(g, z, lw->w1p + (size_t)e * per1, lw->w1s + (size_t)e * per1s, L, I);
        orc_mxfp4_matvec(u, z, lw->w3p + (size_t)e * per1, lw->w3s + (size_t)e * per1s, L, I);
        for (int i = 0; i < I; i++) a[i] = orc_situ(g[i], u[i], c->situ_b1, c->situ_b2);
        if (tr && tr->h) memcpy(tr->h + ((size_t)r * (size_t)K + (size_t)j) * (size_t)I, a, sizeof(double) * (size_t)I);
        orc_mxfp4_matvec(eo, a, lw->w2p + (size_t)e * per2, lw->w2s + (size_t)e * per2s, I, L);
        for (int i = 0; i < L; i++) acc[i] += w[j] * eo[i];
    }
    if (tr && tr->acc) memcpy(tr->acc + (size_t)r * (size_t)L, acc, sizeof(double) * (size_t)L);
    /* 4. norm the aggregate */
    if (lw->latent_gain) {
        for (int i = 0; i < L; i++) gain[i] = orc_bf16(lw->latent_gain[i]);
        orc_rmsnorm(acc, acc, gain, L, c->rms_eps);
    }
    if (tr && tr->nrm) memcpy(tr->nrm + (size_t)r * (size_t)L, acc, sizeof(double) * (size_t)L);
    /* 5. back up to full width */
    orc_bf16_matvec(y, acc, lw->up_w, L, H);
    /* 6. shared experts on the original x, unweighted */
    orc_bf16_matvec(g, x, lw->sh_w1, H, S);
    orc_bf16_matvec(u, x, lw->sh_w3, H, S);
    for (int i = 0; i < S; i++) a[i] = orc_situ(g[i], u[i], c->situ_b1, c->situ_b2);
    if (tr && tr->shared) memcpy(tr->shared + (size_t)r * (size_t)S, a, sizeof(double) * (size_t)S);
    orc_bf16_matvec(eo, a, lw->sh_w2, S, H);
    for (int i = 0; i < H; i++) y[i] += eo[i];

    if (tr) {
        if (tr->ids) memcpy(tr->ids + (size_t)r * (size_t)K, ids, sizeof(int) * (size_t)K);
        if (tr->w) memcpy(tr->w + (size_t)r * (size_t)K, w, sizeof(double) * (size_t)K);
        if (tr->margin) tr->margin[r] = margin;
        if (tr->z) memcpy(tr->z + (size_t)r * (size_t)L, z, sizeof(double) * (size_t)L);
    }
    free(x); free(z); free(acc); free(g); free(u); free(a); free(eo); free(gain); free(ids); free(w);
}

/* The layer on a subset of tokens: rows[r] (r < nrows) indexes x [T, H] bf16;
 * y is [nrows, H] fp64. rows == NULL means all T tokens (nrows = T).
 * Tokens are independent, so they are spread over OpenMP threads; each token's
 * arithmetic is unchanged, so the result does not depend on the thread count. */
void orc_layer_forward(const orc_cfg *c, const orc_layer *lw, const uint16_t *x, int T,
                       const int *rows, int nrows, double *y, const orc_trace *tr)
{
    if (!rows) nrows = T;
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < nrows; r++) {
        const int t = rows ? rows[r] : r;
        orc_layer_token(c, lw, x + (size_t)t * (size_t)c->hidden,
                        y + (size_t)r * (size_t)c->hidden, r, tr);
    }
}

/* The model's dense feed-forward layer (layer 0 of the pages' 93: a plain
 * dense FFN of width dense_inter = 33792, kimi-k3-in-c README Part II, the
 * K3Cfg "first_dense"/"dense_inter" fields) in the form of every other MLP of
 * the model: y = W2 . SiTU(W1 x, W3 x), bf16 weights W1, W3 [F, H] and W2
 * [H, F], the SiTU-GLU of section 9. x [T, H] bf16, y [T, H] fp64; tokens are
 * independent (OpenMP over tokens, each token's arithmetic unchanged). */
void orc_dense_ffn(double *y, const uint16_t *x, int T, const uint16_t *W1, const uint16_t *W3,
                   const uint16_t *W2, int H, int F, double b1, double b2)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < T; t++) {
        double *xv = (double *)malloc(sizeof(double) * (size_t)H);
        double *g = (double *)malloc(sizeof(double) * (size_t)F);
        double *u = (double *)malloc(sizeof(double) * (size_t)F);
        for (int i = 0; i < H; i++) xv[i] = orc_bf16(x[(size_t)t * (size_t)H + (size_t)i]);
        orc_bf16_matvec(g, xv, W1, H, F);
        orc_bf16_matvec(u, xv, W3, H, F);
        for (int i = 0; i < F; i++) g[i] = orc_situ(g[i], u[i], b1, b2);
        orc_bf16_matvec(y + (size_t)t * (size_t)H, g, W2, F, H);
        free(xv); free(g); free(u);
    }
}

/* Router only, for all T tokens (ids, weights and margins). */
void orc_route(const orc_cfg *c, const orc_layer *lw, const uint16_t *x, int T,
               int *ids, double *w, double *margin, double *sc_out, double *ch_out)
{
    const int H = c->hidden, E = c->n_experts, K = c->topk;
#pragma omp parallel for schedule(dynamic, 4)
    for (int t = 0; t < T; t++) {
        double *xd = (double *)malloc(sizeof(double) * (size_t)H);
        for (int i = 0; i < H; i++) xd[i] = orc_bf16(x[(size_t)t * (size_t)H + (size_t)i]);
        orc_router_token(ids + (size_t)t * (size_t)K, w + (size_t)t * (size_t)K,
                         sc_out ? sc_out + (size_t)t * (size_t)E : NULL,
                         ch_out ? ch_out + (size_t)t * (size_t)E : NULL,
                         margin ? margin + t : NULL, xd, lw->router_w, lw->router_bias,
                         H, E, K, c->renorm, c->routed_scale);
        if (c->topp > 0.0) {
            double mt;
            orc_topp_cut(ids + (size_t)t * (size_t)K, w + (size_t)t * (size_t)K, K, c->topp, &mt);
            if (margin && mt < margin[t]) margin[t] = mt;
        }
        free(xd);
    }
}

/* Glue between stacked layers: x_next = RMSNorm(y) with unit gain, per token.
 * (The pages stack layers through AttnRes, which is not part of this layer;
 * the stacked workload uses this plain norm instead.) */
void orc_chain_glue(double *out, const double *y, int T, int H, double eps)
{
    for (int t = 0; t < T; t++)
        orc_rmsnorm(out + (size_t)t * (size_t)H, y + (size_t)t * (size_t)H, NULL, H, eps);
}

int orc_group_size(void) { return ORC_GROUP; }

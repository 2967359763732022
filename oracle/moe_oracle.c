/*
 * moe_oracle.c -- plain CPU oracle of the routed mixture-of-experts forward
 * for small decode / verify / prefill sub-chunks (rows = 1..8).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file's shared library.  The product
 * path (the CUDA library and its Python binding) never calls it, and this
 * file shares no code, header, table or constant with the CUDA path.
 *
 * What it computes (the per-row definition; every floating-point step in
 * fp64 unless stated):
 *   page "Function forward_moe" (its summary and the note on the shared
 *   expert) and page "metrale_model_layers/layers/moe/forward_token_major.rs"
 *   (MoeLayer::forward_token_major_decode, from the router through
 *   moe_weighted_sum_blend_prefill): router gate projection -> top-k
 *   (softmax, or sigmoid with
 *   a per-expert correction bias and routed_scaling_factor) -> per selected
 *   (row, slot) expert: gate and up projections, SiLU(gate)*up, down
 *   projection -> routing-weighted sum over the slots -> plus the shared
 *   expert, blended through sigmoid(x . shared_expert_gate).
 *   The union of the selected experts (page "Function forward_moe", the
 *   RETRACTED and WIDENED notes) is reported as a separate result: the union sweep reaches
 *   the per-row result exactly, so the oracle computes per row.
 *
 * Readings of points the pages leave open:
 *   - NVFP4 matrix [N][K]: packed bytes [N][K/2], low nibble = even input
 *     index; E4M3 (OCP "FN": bias 7, no infinity, S.1111.111 = NaN) scales
 *     [N][K/16], one per 16 contiguous inputs; one fp32 scale2 per matrix.
 *     A weight is (float)e2m1 * (float)e4m3 * scale2 evaluated in fp32 (the
 *     first product is exact, the multiply by scale2 rounds once).
 *   - FP8 and BF16 experts (the other expert formats page
 *     "forward_token_major.rs" names; it routes them to another path and
 *     gives neither layout): FP8 matrix [N][K] = one E4M3 code per weight,
 *     row-major, and one fp32 scale2 per matrix; BF16 matrix [N][K] = one
 *     bfloat16 per weight, row-major, little-endian, times scale2.  A weight
 *     is (float)decode(code) * scale2 in fp32 (one rounding).  The router,
 *     the shared-expert gate vector and everything after the projections are
 *     the same for every expert format.
 *   - top-k order: selection key descending, ties to the lower expert id.
 *     The selection decision is taken on keys rounded to fp32, the precision
 *     of the CUDA kernel's logits; softmax selects on the logit itself
 *     (softmax is strictly increasing in the logit), sigmoid scoring selects
 *     on sigmoid(logit) + bias.
 *   - sigmoid scoring: the weights use the unbiased sigmoid, normalised over
 *     the selected slots when norm_topk_prob, then times
 *     routed_scaling_factor.  Softmax scoring has no scaling factor.
 *   - the union is the first occurrences of the ids scanned in row-major
 *     (row, slot) order; rowmask[u] is the set of rows that selected union[u].
 *   - the weighted sum runs in slot order 0..top_k-1.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Number formats                                                           */
/* ------------------------------------------------------------------------ */

/* FP4 E2M1 (OCP Microscaling formats, FP4 element type): 1 sign bit,
 * 2 exponent bits (bias 1), 1 mantissa bit; exponent field 0 is subnormal. */
double orc_e2m1(int code)
{
    int sign = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -mag : mag;
}

/* FP8 E4M3 "FN" (OCP 8-bit floating point): bias 7, subnormals for exponent
 * field 0, no infinities, S.1111.111 is NaN. */
double orc_e4m3(int code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 15;
    int m = code & 7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp(m / 8.0, -6);
    else
        mag = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* bfloat16 bits -> value (exact). */
double orc_bf16(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* value -> nearest bfloat16 (ties to even), taken directly from the double
 * (no intermediate rounding to float). */
uint16_t orc_round_bf16(double v)
{
    if (isnan(v))
        return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);                 /* a = f * 2^e, f in [0.5, 1) */
    int qexp = e - 8;             /* 8 significant bits */
    if (qexp < -133)              /* quantum of the bfloat16 subnormals */
        qexp = -133;
    double q = ldexp(nearbyint(ldexp(a, -qexp)), qexp);
    if (q > 0x1.FEp127)           /* beyond the largest finite bfloat16 */
        return sign | 0x7F80;
    float f = (float)q;           /* exact: q has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

/* Expert (or router) matrix formats. */
enum { ORC_FMT_NVFP4 = 0, ORC_FMT_FP8 = 1, ORC_FMT_BF16 = 2 };

typedef struct {
    const uint8_t *packed; /* NVFP4 [N][K/2]; FP8 [N][K]; BF16 [N][2K] bytes */
    const uint8_t *scales; /* NVFP4 [N][K/16]; unused by FP8 and BF16 */
    float scale2;
    int fmt;               /* ORC_FMT_* */
} orc_mat;

/* Dequantised weight [n][k] of an NVFP4 matrix with K inputs, as fp32. */
float orc_nvfp4_elem(const orc_mat *m, int K, int n, int k)
{
    uint8_t byte = m->packed[(size_t)n * (size_t)(K / 2) + (size_t)(k / 2)];
    int code = (k & 1) ? (byte >> 4) : (byte & 15);
    float q = (float)orc_e2m1(code);
    float s = (float)orc_e4m3(m->scales[(size_t)n * (size_t)(K / 16) + (size_t)(k / 16)]);
    float qs = q * s;
    return qs * m->scale2;
}

/* Dequantised weight [n][k] of a matrix of any format, as fp32. */
float orc_mat_elem(const orc_mat *m, int K, int n, int k)
{
    const size_t i = (size_t)n * (size_t)K + (size_t)k;
    if (m->fmt == ORC_FMT_FP8) {
        float q = (float)orc_e4m3(m->packed[i]);
        return q * m->scale2;
    }
    if (m->fmt == ORC_FMT_BF16) {
        uint16_t bits = (uint16_t)(m->packed[2 * i] | ((unsigned)m->packed[2 * i + 1] << 8));
        float q = (float)orc_bf16(bits);
        return q * m->scale2;
    }
    return orc_nvfp4_elem(m, K, n, k);
}

/* Row n of a matrix, dequantised to fp64 (from the fp32 weights). */
static void mat_row(const orc_mat *m, int K, int n, double *row)
{
    for (int k = 0; k < K; ++k)
        row[k] = (double)orc_mat_elem(m, K, n, k);
}

/* ------------------------------------------------------------------------ */
/* Layer description                                                         */
/* ------------------------------------------------------------------------ */

typedef struct {
    int hidden;         /* H */
    int num_experts;    /* E */
    int top_k;          /* k */
    int moe_inter;      /* I */
    int shared_inter;   /* Is */
    int scoring;        /* 0 = softmax, 1 = sigmoid + correction bias */
    int norm_topk_prob;
    double routed_scaling_factor;
    int router_nvfp4;   /* 0 = bf16 router [E][H], 1 = NVFP4 router */
    int has_shared;     /* 0 = no shared expert */
    int shared_gated;   /* 1 = sigmoid(x . gs) blend, 0 = plain add */
} orc_cfg;

typedef struct {
    const uint16_t *router_bf16;  /* [E][H] */
    orc_mat router_fp4;        /* [E][H] */
    const float *bias;            /* [E], sigmoid scoring */
    const orc_mat *gate;       /* [E] descriptors, each [I][H] */
    const orc_mat *up;         /* [E] descriptors, each [I][H] */
    const orc_mat *down;       /* [E] descriptors, each [H][I] */
    orc_mat sh_gate;           /* [Is][H] */
    orc_mat sh_up;             /* [Is][H] */
    orc_mat sh_down;           /* [H][Is] */
    const uint16_t *sh_gate_vec;  /* [H] bf16 shared_expert_gate */
} orc_weights;

/* ------------------------------------------------------------------------ */
/* Router                                                                    */
/* ------------------------------------------------------------------------ */

/* logits[r][e] = sum_h x[r][h] * Wr[e][h]  (forward_ep.rs and
 * forward_token_major.rs: the gate projection, dense_gemv / dense_gemm for a
 * bf16 router, w4a16_decode_gemv / w4a16_gemm for an NVFP4 router). */
void orc_router_logits(const orc_cfg *c, const orc_weights *w,
                       const uint16_t *x, int rows, double *logits)
{
    const int H = c->hidden, E = c->num_experts;
    double *xr = malloc(sizeof(double) * (size_t)H);
    double *wr = malloc(sizeof(double) * (size_t)H);
    for (int r = 0; r < rows; ++r) {
        for (int h = 0; h < H; ++h)
            xr[h] = orc_bf16(x[(size_t)r * H + h]);
        for (int e = 0; e < E; ++e) {
            if (c->router_nvfp4)
                mat_row(&w->router_fp4, H, e, wr);
            else
                for (int h = 0; h < H; ++h)
                    wr[h] = orc_bf16(w->router_bf16[(size_t)e * H + h]);
            double acc = 0.0;
            for (int h = 0; h < H; ++h)
                acc += xr[h] * wr[h];
            logits[(size_t)r * E + e] = acc;
        }
    }
    free(xr);
    free(wr);
}

/* ------------------------------------------------------------------------ */
/* Top-k                                                                     */
/* ------------------------------------------------------------------------ */

/* The k largest keys, in descending key order; equal keys go to the lower
 * expert id.  Plain repeated selection, O(k*E). */
void orc_topk(const double *key, int E, int k, int32_t *ids)
{
    char *taken = calloc((size_t)E, 1);
    for (int j = 0; j < k; ++j) {
        int best = -1;
        for (int e = 0; e < E; ++e) {
            if (taken[e])
                continue;
            if (best < 0 || key[e] > key[best])
                best = e;   /* strict '>' keeps the lower id on ties */
        }
        taken[best] = 1;
        ids[j] = best;
    }
    free(taken);
}

static double sigmoid64(double z) { return 1.0 / (1.0 + exp(-z)); }

/* Scores, selection and routing weights of one row (forward_ep.rs:
 * moe_topk_softmax with norm_topk_prob; forward_token_major.rs:
 * moe_topk_sigmoid_batched with correction bias, norm_topk_prob and
 * routed_scaling_factor, else moe_topk_softmax_batched). */
void orc_topk_row(const orc_cfg *c, const orc_weights *w, const double *logit,
                  int32_t *ids, double *wts)
{
    const int E = c->num_experts, k = c->top_k;
    double *score = malloc(sizeof(double) * (size_t)E);
    double *key = malloc(sizeof(double) * (size_t)E);
    if (c->scoring == 0) {
        double mx = logit[0];
        for (int e = 1; e < E; ++e)
            if (logit[e] > mx)
                mx = logit[e];
        double z = 0.0;
        for (int e = 0; e < E; ++e)
            z += exp(logit[e] - mx);
        for (int e = 0; e < E; ++e) {
            score[e] = exp(logit[e] - mx) / z;
            key[e] = (double)(float)logit[e];
        }
    } else {
        for (int e = 0; e < E; ++e) {
            score[e] = sigmoid64(logit[e]);
            key[e] = (double)(float)(score[e] + (double)w->bias[e]);
        }
    }
    orc_topk(key, E, k, ids);
    double sum = 0.0;
    for (int j = 0; j < k; ++j)
        sum += score[ids[j]];
    for (int j = 0; j < k; ++j) {
        double v = score[ids[j]];
        if (c->norm_topk_prob)
            v /= sum;
        if (c->scoring == 1)
            v *= c->routed_scaling_factor;
        wts[j] = v;
    }
    free(score);
    free(key);
}

/* Router + top-k for all rows.  logits may be NULL. */
void orc_route(const orc_cfg *c, const orc_weights *w, const uint16_t *x,
               int rows, double *logits, int32_t *ids, double *wts)
{
    const int E = c->num_experts, k = c->top_k;
    double *lg = logits ? logits : malloc(sizeof(double) * (size_t)rows * E);
    orc_router_logits(c, w, x, rows, lg);
    for (int r = 0; r < rows; ++r)
        orc_topk_row(c, w, lg + (size_t)r * E, ids + (size_t)r * k, wts + (size_t)r * k);
    if (!logits)
        free(lg);
}

/* ------------------------------------------------------------------------ */
/* Union of the selected experts                                             */
/* ------------------------------------------------------------------------ */

/* First occurrences of ids[rows][k] in row-major order.  Returns U and fills
 * uni[U], slot2u[rows][k] (union index of every (row, slot)) and rowmask[U]
 * (bit r set when row r selected uni[u]). */
int orc_union(const int32_t *ids, int rows, int k, int32_t *uni,
              uint8_t *slot2u, uint32_t *rowmask)
{
    int U = 0;
    for (int p = 0; p < rows * k; ++p) {
        int found = -1;
        for (int u = 0; u < U; ++u)
            if (uni[u] == ids[p]) {
                found = u;
                break;
            }
        if (found < 0) {
            found = U;
            uni[U] = ids[p];
            rowmask[U] = 0;
            ++U;
        }
        slot2u[p] = (uint8_t)found;
        rowmask[found] |= (uint32_t)(1u << (p / k));
    }
    return U;
}

/* ------------------------------------------------------------------------ */
/* Expert MLP                                                                */
/* ------------------------------------------------------------------------ */

static double silu64(double z) { return z / (1.0 + exp(-z)); }

/* y = Wd . (silu(Wg . x) * (Wu . x)); Wg, Wu [I][H], Wd [H][I]
 * (forward_token_major.rs: moe_expert_gate_up_shared_prefill, then
 * moe_expert_silu_down_shared_prefill, with the packed / scale / scale2
 * triplet of every expert matrix). */
void orc_expert_mlp(int H, int I, const orc_mat *g, const orc_mat *u,
                    const orc_mat *d, const double *x, double *y)
{
    double *hbuf = malloc(sizeof(double) * (size_t)I);
    double *row = malloc(sizeof(double) * (size_t)(H > I ? H : I));
    for (int i = 0; i < I; ++i) {
        double gs = 0.0, us = 0.0;
        mat_row(g, H, i, row);
        for (int h = 0; h < H; ++h)
            gs += row[h] * x[h];
        mat_row(u, H, i, row);
        for (int h = 0; h < H; ++h)
            us += row[h] * x[h];
        hbuf[i] = silu64(gs) * us;
    }
    for (int o = 0; o < H; ++o) {
        mat_row(d, I, o, row);
        double acc = 0.0;
        for (int i = 0; i < I; ++i)
            acc += row[i] * hbuf[i];
        y[o] = acc;
    }
    free(hbuf);
    free(row);
}

/* ------------------------------------------------------------------------ */
/* Whole layer                                                               */
/* ------------------------------------------------------------------------ */

typedef struct {
    const orc_cfg *c;
    const orc_weights *w;
    const double *x;       /* [rows][H] */
    const int32_t *ids;    /* [rows][k] */
    int rows;
    int ntask;             /* rows * (k + has_shared) */
    double *y;             /* [ntask][H] */
    int tid, nthreads;
} orc_job;

static void *orc_worker(void *arg)
{
    orc_job *j = arg;
    const orc_cfg *c = j->c;
    const int H = c->hidden, k = c->top_k;
    const int per_row = k + (c->has_shared ? 1 : 0);
    for (int t = j->tid; t < j->ntask; t += j->nthreads) {
        int r = t / per_row, s = t % per_row;
        const double *xr = j->x + (size_t)r * H;
        double *y = j->y + (size_t)t * H;
        if (s < k) {
            int e = j->ids[(size_t)r * k + s];
            orc_expert_mlp(H, c->moe_inter, &j->w->gate[e], &j->w->up[e],
                           &j->w->down[e], xr, y);
        } else {
            orc_expert_mlp(H, c->shared_inter, &j->w->sh_gate, &j->w->sh_up,
                           &j->w->sh_down, xr, y);
        }
    }
    return NULL;
}

/* The whole routed MoE layer for `rows` token rows.
 * out[r][o]      = sum_{j<k} wts[r][j] * y_{r,j}[o] + gate_r * ys_r[o]  (fp64)
 * out_bf16[r][o] = out rounded to bfloat16 (may be NULL)
 * ids / wts / logits receive the routing (logits may be NULL).
 * (forward_token_major.rs: moe_weighted_sum_blend_prefill takes the expert
 * outputs, the routing weights, the shared expert's output, the input and
 * shared_expert_gate.weight.)
 * The (row, slot) expert evaluations run on `nthreads` POSIX threads; the
 * result does not depend on nthreads. */
static void forward_experts_and_blend(const orc_cfg *c, const orc_weights *w,
                                      const uint16_t *x, int rows, int nthreads,
                                      const int32_t *ids, const double *wts,
                                      double *out, uint16_t *out_bf16)
{
    const int H = c->hidden, k = c->top_k;
    const int per_row = k + (c->has_shared ? 1 : 0);
    const int ntask = rows * per_row;
    if (nthreads < 1)
        nthreads = 1;

    double *xd = malloc(sizeof(double) * (size_t)rows * H);
    for (size_t i = 0; i < (size_t)rows * H; ++i)
        xd[i] = orc_bf16(x[i]);
    double *y = malloc(sizeof(double) * (size_t)ntask * H);

    orc_job *jobs = malloc(sizeof(orc_job) * (size_t)nthreads);
    pthread_t *th = malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int t = 0; t < nthreads; ++t) {
        orc_job j = {c, w, xd, ids, rows, ntask, y, t, nthreads};
        jobs[t] = j;
    }
    for (int t = 1; t < nthreads; ++t)
        pthread_create(&th[t], NULL, orc_worker, &jobs[t]);
    orc_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        pthread_join(th[t], NULL);

    for (int r = 0; r < rows; ++r) {
        double gate = 0.0;
        if (c->has_shared) {
            if (c->shared_gated) {
                double dot = 0.0;
                for (int h = 0; h < H; ++h)
                    dot += xd[(size_t)r * H + h] * orc_bf16(w->sh_gate_vec[h]);
                gate = sigmoid64(dot);
            } else {
                gate = 1.0;
            }
        }
        for (int o = 0; o < H; ++o) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j)
                acc += wts[(size_t)r * k + j] * y[((size_t)r * per_row + j) * H + o];
            if (c->has_shared)
                acc += gate * y[((size_t)r * per_row + k) * H + o];
            out[(size_t)r * H + o] = acc;
            if (out_bf16)
                out_bf16[(size_t)r * H + o] = orc_round_bf16(acc);
        }
    }
    free(jobs);
    free(th);
    free(y);
    free(xd);
}

void orc_forward(const orc_cfg *c, const orc_weights *w, const uint16_t *x,
                 int rows, int nthreads, double *out, uint16_t *out_bf16,
                 int32_t *ids, double *wts, double *logits)
{
    orc_route(c, w, x, rows, logits, ids, wts);
    forward_experts_and_blend(c, w, x, rows, nthreads, ids, wts, out, out_bf16);
}

/* ------------------------------------------------------------------------ */
/* The layer at caller-given experts                                         */
/* ------------------------------------------------------------------------ */

/* Routing weights of caller-given experts sel[0..k-1] of one row (distinct
 * ids in [0, E)), from the same scores the top-k uses (forward_ep.rs /
 * forward_token_major.rs: moe_topk_softmax(_batched) with norm_topk_prob,
 * moe_topk_sigmoid_batched with routed_scaling_factor): softmax over all E
 * logits, or the unbiased sigmoid; normalised over the k given experts when
 * norm_topk_prob; times routed_scaling_factor for sigmoid scoring.  With sel
 * equal to the row's top-k this is exactly the top-k's weights; it exists
 * to evaluate a row whose selection was decided elsewhere (a near tie that
 * an fp32 router resolved the other way). */
void orc_weights_for_ids(const orc_cfg *c, const double *logit,
                         const int32_t *sel, double *wsel)
{
    const int E = c->num_experts, k = c->top_k;
    double *p = malloc(sizeof(double) * (size_t)E);
    if (c->scoring == 0) {
        double top = logit[0];
        for (int e = 1; e < E; ++e)
            top = logit[e] > top ? logit[e] : top;
        double part = 0.0;
        for (int e = 0; e < E; ++e)
            part += exp(logit[e] - top);
        for (int e = 0; e < E; ++e)
            p[e] = exp(logit[e] - top) / part;
    } else {
        for (int e = 0; e < E; ++e)
            p[e] = 1.0 / (1.0 + exp(-logit[e]));
    }
    double tot = 0.0;
    for (int j = 0; j < k; ++j)
        tot += p[sel[j]];
    for (int j = 0; j < k; ++j) {
        double v = p[sel[j]];
        v = c->norm_topk_prob ? v / tot : v;
        wsel[j] = c->scoring == 1 ? v * c->routed_scaling_factor : v;
    }
    free(p);
}

/* The whole layer with the experts of every row given by the caller
 * (sel[rows][k], in slot order) instead of chosen by the top-k: the router
 * logits, the weights of orc_weights_for_ids, then the same expert MLPs,
 * weighted sum and shared-expert blend as orc_forward.  wsel receives the
 * weights; logits may be NULL. */
void orc_forward_ids(const orc_cfg *c, const orc_weights *w, const uint16_t *x,
                     int rows, const int32_t *sel, int nthreads, double *out,
                     uint16_t *out_bf16, double *wsel, double *logits)
{
    const int E = c->num_experts, k = c->top_k;
    double *lg = logits ? logits : malloc(sizeof(double) * (size_t)rows * E);
    orc_router_logits(c, w, x, rows, lg);
    for (int r = 0; r < rows; ++r)
        orc_weights_for_ids(c, lg + (size_t)r * E, sel + (size_t)r * k,
                            wsel + (size_t)r * k);
    forward_experts_and_blend(c, w, x, rows, nthreads, sel, wsel, out, out_bf16);
    if (!logits)
        free(lg);
}

int orc_abi_version(void) { return 1; }

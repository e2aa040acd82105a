/*
 * moe_oracle.c -- plain CPU statement of the MoE token-dispatch layer.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline / reference arm may load this
 * library.  It shares no source, header, table or helper with the CUDA
 * path; the two meet only at the seeded inputs.
 *
 * What it computes (one MoE layer, exactly, in fp64):
 *
 *   route  : per token, the k experts with the largest router logit
 *            (ties -> lower expert index), their softmax probability over
 *            all E logits, optionally renormalised over the k chosen.
 *            ("switchyard" page, 02 Kernels and dispatch, "Route and sort";
 *             "dispatch" README, Architecture, "Router / top-k gating".)
 *   permute: a stable counting sort of the slots s = t*k + j by expert,
 *            with an exclusive prefix-sum offset table; shared experts
 *            follow as groups that hold every token in order.
 *            ("switchyard" page, "Route and sort": rows sorted by expert
 *             with a prefix scan.)
 *   layer  : y[t] = sum_j w[t,j] * FFN_{id[t,j]}(x[t]) + sum_s FFN_{E+s}(x[t])
 *            (+ residual[t]), FFN_e(v) = Wd_e (silu(Wg_e v) * (Wu_e v)),
 *            silu(z) = z / (1 + exp(-z)).
 *            ("switchyard" page, "One launch for all experts": grouped GEMM
 *             with SwiGLU; "dispatch" README, Stack: shared + routed
 *             experts.)
 *   capacity: the dropping variant.  Routed expert e serves at most C of
 *            its slots, the first C in slot order (token-major: first come,
 *            first served); the other slots are dropped and add nothing to
 *            their token's output (the kept weights are not renormalised).
 *            Shared experts are never capped.  ("switchyard" page, 03 Load
 *            balance, "What dropping tokens costs": capacity limits drop the
 *            tokens an expert has no room for.)
 *   w8     : symmetric per-output-channel int8 weight-only quantisation,
 *            scale = max|row| / 127 (fp32), q = clamp(rint(W/scale), +-127);
 *            dequantised weight = (float)q * scale (fp32 product).
 *            ("dispatch" README, phase 5a: self-computed per-channel int8
 *             weight-only quantisation.)
 *
 * Arithmetic: bf16 weight values and activations are widened exactly and
 * every sum, product, exp and division is done in double.  Nothing is
 * rounded to bf16 in between.  Loops are the definition's loops; the only
 * parallelism is an OpenMP loop over independent tokens, which does not
 * change any token's arithmetic.
 *
 * Return codes: 0 ok, 1 bad argument, 2 bad input value (expert id out of
 * range, non-finite logit).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_OK 0
#define OR_BAD_ARG 1
#define OR_BAD_VALUE 2

/* exact widening of a bf16 bit pattern (the top 16 bits of an fp32) */
static double bf16_value(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* ---------------------------------------------------------------- route */

/* Expert a ranks before expert b: a larger logit, or an equal logit and a
 * lower index. */
static int ranks_before(const float *L, int a, int b) {
    return L[a] > L[b] || (L[a] == L[b] && a < b);
}

int oracle_route(const float *logits, int64_t T, int E, int k, int renormalize,
                 int32_t *ids, double *w) {
    if (!logits || !ids || !w || T < 0 || E < 1 || k < 1 || k > E) return OR_BAD_ARG;
    char *taken = (char *)malloc((size_t)E);
    if (!taken) return OR_BAD_ARG;
    int rc = OR_OK;
    for (int64_t t = 0; t < T && rc == OR_OK; ++t) {
        const float *L = logits + t * E;
        for (int e = 0; e < E; ++e)
            if (!isfinite(L[e])) rc = OR_BAD_VALUE;   /* NaN or +-inf: no softmax */
        if (rc != OR_OK) break;
        memset(taken, 0, (size_t)E);
        /* selection: k times, the best expert not yet taken */
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || ranks_before(L, e, best))) best = e;
            taken[best] = 1;
            ids[t * k + j] = best;
        }
        /* softmax over all E logits */
        double mx = L[0];
        for (int e = 1; e < E; ++e)
            if (L[e] > mx) mx = L[e];
        double den = 0.0;
        for (int e = 0; e < E; ++e) den += exp((double)L[e] - mx);
        double sel = 0.0;
        for (int j = 0; j < k; ++j) {
            double p = exp((double)L[ids[t * k + j]] - mx) / den;
            w[t * k + j] = p;
            sel += p;
        }
        if (renormalize)
            for (int j = 0; j < k; ++j) w[t * k + j] /= sel;
    }
    free(taken);
    return rc;
}

/* -------------------------------------------------------------- permute */

int oracle_permute(const int32_t *ids, int64_t T, int E, int S, int k, int32_t *offsets,
                   int32_t *sorted_slot, int32_t *row_of_slot) {
    if (!ids || !offsets || T < 0 || E < 1 || S < 0 || k < 1) return OR_BAD_ARG;
    const int64_t n = T * k;
    if (n > 0 && (!sorted_slot || !row_of_slot)) return OR_BAD_ARG;
    int64_t *count = (int64_t *)calloc((size_t)E, sizeof(int64_t));
    int64_t *next = (int64_t *)calloc((size_t)E, sizeof(int64_t));
    if (!count || !next) { free(count); free(next); return OR_BAD_ARG; }
    int rc = OR_OK;
    for (int64_t s = 0; s < n; ++s) {
        int32_t e = ids[s];
        if (e < 0 || e >= E) { rc = OR_BAD_VALUE; break; }
        count[e] += 1;
    }
    if (rc == OR_OK) {
        /* exclusive prefix sum: routed groups, then S shared groups of T rows */
        offsets[0] = 0;
        for (int e = 0; e < E; ++e) offsets[e + 1] = (int32_t)(offsets[e] + count[e]);
        for (int s = 0; s < S; ++s) offsets[E + s + 1] = (int32_t)(offsets[E + s] + T);
        for (int e = 0; e < E; ++e) next[e] = offsets[e];
        /* stable placement: slots in ascending order */
        for (int64_t s = 0; s < n; ++s) {
            int64_t r = next[ids[s]]++;
            sorted_slot[r] = (int32_t)s;
            row_of_slot[s] = (int32_t)r;
        }
    }
    free(count);
    free(next);
    return rc;
}

/* The dropping variant: expert e keeps its first `capacity` slots in slot
 * order.  Layout: the kept routed rows by expert ([0, kept)), then the S
 * shared groups of T rows.  sorted_slot[r] for r >= kept is -1; a dropped
 * slot's row_of_slot is -2; *dropped = number of dropped slots. */
int oracle_permute_capped(const int32_t *ids, int64_t T, int E, int S, int k, int64_t capacity,
                          int32_t *offsets, int32_t *sorted_slot, int32_t *row_of_slot,
                          int64_t *dropped) {
    if (!ids || !offsets || !dropped || T < 0 || E < 1 || S < 0 || k < 1 || capacity < 0)
        return OR_BAD_ARG;
    const int64_t n = T * k;
    if (n > 0 && (!sorted_slot || !row_of_slot)) return OR_BAD_ARG;
    int64_t *count = (int64_t *)calloc((size_t)E, sizeof(int64_t));
    int64_t *seen = (int64_t *)calloc((size_t)E, sizeof(int64_t));
    if (!count || !seen) { free(count); free(seen); return OR_BAD_ARG; }
    int rc = OR_OK;
    for (int64_t s = 0; s < n; ++s) {
        int32_t e = ids[s];
        if (e < 0 || e >= E) { rc = OR_BAD_VALUE; break; }
        count[e] += 1;
    }
    if (rc == OR_OK) {
        offsets[0] = 0;
        for (int e = 0; e < E; ++e) {
            const int64_t kept = count[e] < capacity ? count[e] : capacity;
            offsets[e + 1] = (int32_t)(offsets[e] + kept);
        }
        for (int s = 0; s < S; ++s) offsets[E + s + 1] = (int32_t)(offsets[E + s] + T);
        for (int64_t r = 0; r < n; ++r) sorted_slot[r] = -1;
        int64_t drops = 0;
        for (int64_t s = 0; s < n; ++s) {
            const int32_t e = ids[s];
            const int64_t rank = seen[e]++;          /* earlier slots of expert e */
            if (rank < capacity) {
                const int64_t r = offsets[e] + rank;
                sorted_slot[r] = (int32_t)s;
                row_of_slot[s] = (int32_t)r;
            } else {
                row_of_slot[s] = -2;
                drops += 1;
            }
        }
        *dropped = drops;
    }
    free(count);
    free(seen);
    return rc;
}

/* ------------------------------------------------------------ expert FFN */

/* h[i] = silu(sum_k Wg[i,k] x[k]) * (sum_k Wu[i,k] x[k]); Wg = rows 0..I-1 of
 * the [2I, H] gate/up block, Wu = rows I..2I-1. */
void oracle_expert_hidden(const double *x, const uint16_t *w_gu, int H, int I, double *h) {
    for (int i = 0; i < I; ++i) {
        const uint16_t *wg = w_gu + (int64_t)i * H;
        const uint16_t *wu = w_gu + (int64_t)(I + i) * H;
        double g = 0.0, u = 0.0;
        for (int c = 0; c < H; ++c) {
            g += bf16_value(wg[c]) * x[c];
            u += bf16_value(wu[c]) * x[c];
        }
        h[i] = silu(g) * u;
    }
}

/* y[n] = sum_i Wd[n,i] h[i]  with Wd the [H, I] down block */
void oracle_expert_down(const double *h, const uint16_t *w_down, int H, int I, double *y) {
    for (int n = 0; n < H; ++n) {
        const uint16_t *wd = w_down + (int64_t)n * I;
        double acc = 0.0;
        for (int i = 0; i < I; ++i) acc += bf16_value(wd[i]) * h[i];
        y[n] = acc;
    }
}

/* Same two steps with int8 weights dequantised as (float)q * scale[row]. */
static double dq(int8_t q, float scale) { return (double)((float)q * scale); }

void oracle_expert_hidden_w8(const double *x, const int8_t *q_gu, const float *s_gu, int H,
                             int I, double *h) {
    for (int i = 0; i < I; ++i) {
        const int8_t *qg = q_gu + (int64_t)i * H;
        const int8_t *qu = q_gu + (int64_t)(I + i) * H;
        double g = 0.0, u = 0.0;
        for (int c = 0; c < H; ++c) {
            g += dq(qg[c], s_gu[i]) * x[c];
            u += dq(qu[c], s_gu[I + i]) * x[c];
        }
        h[i] = silu(g) * u;
    }
}

void oracle_expert_down_w8(const double *h, const int8_t *q_down, const float *s_down, int H,
                           int I, double *y) {
    for (int n = 0; n < H; ++n) {
        const int8_t *qd = q_down + (int64_t)n * I;
        double acc = 0.0;
        for (int i = 0; i < I; ++i) acc += dq(qd[i], s_down[n]) * h[i];
        y[n] = acc;
    }
}

/* ----------------------------------------------------------------- layer */

typedef struct {
    const uint16_t *w_gu, *w_down;           /* bf16 weights, or NULL */
    const int8_t *q_gu, *q_down;             /* int8 weights, or NULL */
    const float *s_gu, *s_down;              /* their per-row scales */
} weights_t;

static void expert_ffn(const weights_t *W, int e, const double *x, int H, int I, double *h,
                       double *y) {
    if (W->w_gu) {
        oracle_expert_hidden(x, W->w_gu + (int64_t)e * 2 * I * H, H, I, h);
        oracle_expert_down(h, W->w_down + (int64_t)e * H * I, H, I, y);
    } else {
        oracle_expert_hidden_w8(x, W->q_gu + (int64_t)e * 2 * I * H, W->s_gu + (int64_t)e * 2 * I,
                                H, I, h);
        oracle_expert_down_w8(h, W->q_down + (int64_t)e * H * I, W->s_down + (int64_t)e * H, H,
                              I, y);
    }
}

/* x: [T, H] fp32 (x_is_f32) or bf16 bits.  ids/w: [T, k] routing.
 * tokens: optional list of ntok token indices to evaluate (NULL: all T, in
 * order).  y: [ntok or T, H] fp64. */
static int layer_impl(const void *x, int x_is_f32, const int32_t *ids, const double *w,
                      int64_t T, int H, int E, int S, int k, int I, const weights_t *W,
                      const uint16_t *residual, const int64_t *tokens, int64_t ntok, double *y,
                      int nthreads, const unsigned char *keep) {
    if (!x || !ids || !w || !y || T < 0 || H < 1 || E < 1 || S < 0 || k < 1 || I < 1)
        return OR_BAD_ARG;
    const int64_t nout = tokens ? ntok : T;
    for (int64_t o = 0; o < nout; ++o) {
        int64_t t = tokens ? tokens[o] : o;
        if (t < 0 || t >= T) return OR_BAD_ARG;
        for (int j = 0; j < k; ++j)
            if (ids[t * k + j] < 0 || ids[t * k + j] >= E) return OR_BAD_VALUE;
    }
    int bad = 0;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t o = 0; o < nout; ++o) {
        const int64_t t = tokens ? tokens[o] : o;
        double *xv = (double *)malloc(sizeof(double) * (size_t)H);
        double *h = (double *)malloc(sizeof(double) * (size_t)I);
        double *fe = (double *)malloc(sizeof(double) * (size_t)H);
        double *yt = y + o * H;
        if (!xv || !h || !fe) {
            bad = 1;
        } else {
            for (int c = 0; c < H; ++c)
                xv[c] = x_is_f32 ? (double)((const float *)x)[t * H + c]
                                 : bf16_value(((const uint16_t *)x)[t * H + c]);
            for (int c = 0; c < H; ++c) yt[c] = 0.0;
            for (int j = 0; j < k; ++j) {
                if (keep && !keep[t * k + j]) continue;      /* dropped slot */
                expert_ffn(W, ids[t * k + j], xv, H, I, h, fe);
                for (int c = 0; c < H; ++c) yt[c] += w[t * k + j] * fe[c];
            }
            for (int s = 0; s < S; ++s) {
                expert_ffn(W, E + s, xv, H, I, h, fe);
                for (int c = 0; c < H; ++c) yt[c] += fe[c];
            }
            if (residual)
                for (int c = 0; c < H; ++c) yt[c] += bf16_value(residual[t * H + c]);
        }
        free(xv);
        free(h);
        free(fe);
    }
    (void)nthreads;
    return bad ? OR_BAD_ARG : OR_OK;
}

int oracle_moe_layer(const void *x, int x_is_f32, const int32_t *ids, const double *w, int64_t T,
                     int H, int E, int S, int k, int I, const uint16_t *w_gu,
                     const uint16_t *w_down, const uint16_t *residual, const int64_t *tokens,
                     int64_t ntok, double *y, int nthreads) {
    if (!w_gu || !w_down) return OR_BAD_ARG;
    weights_t W = {w_gu, w_down, NULL, NULL, NULL, NULL};
    return layer_impl(x, x_is_f32, ids, w, T, H, E, S, k, I, &W, residual, tokens, ntok, y,
                      nthreads, NULL);
}

int oracle_moe_layer_w8(const void *x, int x_is_f32, const int32_t *ids, const double *w,
                        int64_t T, int H, int E, int S, int k, int I, const int8_t *q_gu,
                        const float *s_gu, const int8_t *q_down, const float *s_down,
                        const uint16_t *residual, const int64_t *tokens, int64_t ntok, double *y,
                        int nthreads) {
    if (!q_gu || !s_gu || !q_down || !s_down) return OR_BAD_ARG;
    weights_t W = {NULL, NULL, q_gu, q_down, s_gu, s_down};
    return layer_impl(x, x_is_f32, ids, w, T, H, E, S, k, I, &W, residual, tokens, ntok, y,
                      nthreads, NULL);
}

/* The layer with capacity-limited experts: slot s = t*k + j is kept when
 * fewer than `capacity` earlier slots (in slot order) chose the same expert;
 * a dropped slot contributes nothing. */
int oracle_moe_layer_capped(const void *x, int x_is_f32, const int32_t *ids, const double *w,
                            int64_t T, int H, int E, int S, int k, int I, int64_t capacity,
                            const uint16_t *w_gu, const uint16_t *w_down,
                            const uint16_t *residual, const int64_t *tokens, int64_t ntok,
                            double *y, int nthreads) {
    if (!w_gu || !w_down || !ids || capacity < 0 || T < 0 || E < 1 || k < 1) return OR_BAD_ARG;
    const int64_t n = T * k;
    unsigned char *keep = (unsigned char *)malloc((size_t)(n > 0 ? n : 1));
    int64_t *seen = (int64_t *)calloc((size_t)E, sizeof(int64_t));
    if (!keep || !seen) { free(keep); free(seen); return OR_BAD_ARG; }
    int rc = OR_OK;
    for (int64_t s = 0; s < n; ++s) {
        const int32_t e = ids[s];
        if (e < 0 || e >= E) { rc = OR_BAD_VALUE; break; }
        keep[s] = seen[e] < capacity;
        seen[e] += 1;
    }
    if (rc == OR_OK) {
        weights_t W = {w_gu, w_down, NULL, NULL, NULL, NULL};
        rc = layer_impl(x, x_is_f32, ids, w, T, H, E, S, k, I, &W, residual, tokens, ntok, y,
                        nthreads, keep);
    }
    free(keep);
    free(seen);
    return rc;
}

/* ------------------------------------------------------------- quantise */

/* Per row n of a [rows, K] bf16 matrix: scale[n] = max|W[n,:]| / 127 in fp32
 * (1 for an all-zero row), q = clamp(rint(W / scale), -127, 127) with the
 * fp32 quotient rounded half to even. */
int oracle_quantize_w8(const uint16_t *w, int64_t rows, int64_t K, int8_t *q, float *scale) {
    if (!w || !q || !scale || rows < 0 || K < 1) return OR_BAD_ARG;
    for (int64_t n = 0; n < rows; ++n) {
        float amax = 0.0f;
        for (int64_t c = 0; c < K; ++c) {
            float v = fabsf((float)bf16_value(w[n * K + c]));
            if (v > amax) amax = v;
        }
        float s = amax > 0.0f ? amax / 127.0f : 1.0f;
        scale[n] = s;
        for (int64_t c = 0; c < K; ++c) {
            float r = rintf((float)bf16_value(w[n * K + c]) / s);
            if (r > 127.0f) r = 127.0f;
            if (r < -127.0f) r = -127.0f;
            q[n * K + c] = (int8_t)r;
        }
    }
    return OR_OK;
}

/* -------------------------------------------------------- router logits */

/* logits[t,e] = sum_c x[t,c] * Wr[e,c] (+ bias[e]) in fp64; x, Wr bf16. */
int oracle_router_logits(const uint16_t *x, const uint16_t *w_r, const float *bias, int64_t T,
                         int H, int E, double *logits) {
    if (!x || !w_r || !logits || T < 0 || H < 1 || E < 1) return OR_BAD_ARG;
    for (int64_t t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int c = 0; c < H; ++c)
                acc += bf16_value(x[t * H + c]) * bf16_value(w_r[(int64_t)e * H + c]);
            logits[t * E + e] = acc + (bias ? (double)bias[e] : 0.0);
        }
    return OR_OK;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

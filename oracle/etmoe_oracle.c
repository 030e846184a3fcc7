/*
 * etmoe_oracle.c -- plain, slow, CPU oracle of the Event-Tensor MoE hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test-suite, the smoke check and the bench's
 * CPU-baseline leg do.  It shares no code, header or constant with the CUDA
 * path.
 *
 * Sources (all restated in my own words):
 *  - "Prompt Boundary-Aware Scheduling with Event Tensors for Dynamic Kernels"
 *    (AI Post Transformers episode summary): the method changes *when* tiled
 *    tasks run -- split-K summation gated by events, a symbolic batch size,
 *    MoE routing whose counters come from the router output -- never *what*
 *    the layer computes.  So every function below is the plain definition of
 *    the layer, written out with loops.
 *  - "Megakernels ch. 5 - Event Tensor et le dynamisme", section 5.1 (MoE
 *    routing: tokens per expert depend on the data) and section 5.5
 *    obstacle 1 (counter targets that depend on the routing).
 *
 * Readings where the pages are silent (each one is listed in the design
 * notes of the repository):
 *  R1 Router logits are fp32 and use one fixed summation order (32 strided
 *     partial sums, then a halving tree), so that routing is reproducible
 *     bit for bit on any machine.  Products of two bf16 values are exact in
 *     fp32, so fma and multiply-then-add agree.
 *  R2 Top-k orders experts by (logit descending, expert index ascending);
 *     -0.0 and +0.0 tie.  Gate weights are the softmax over the k selected
 *     logits, i.e. full softmax, top-k, renormalise.
 *  R3 Within one expert, routed rows are in ascending token order.
 *  R4 The expert FFN is SwiGLU: h = silu(x Wg^T) * (x Wu^T), y = h Wd^T;
 *     h and y are stored as bf16 (rounded once from the fp64 value).
 *  R5 The combine is out[t] = bf16(sum_j w[t,j] y[t,j]).
 *  R6 RMSNorm: xhat = bf16(x / sqrt(mean(x^2) + eps) * gamma), no residual.
 *  R14 The fused MoE block routes x_hat, runs the routed experts and a shared
 *     SwiGLU expert on x_hat and adds the residual:
 *     out = bf16(x + sum_j w_j y_j + y_s), one rounding of the fp64 sum.
 *  R15 In the block, x_hat feeds the (bit-exact) routing, so it is defined in
 *     fp32 with one fixed order, like R1: ss = sum of x^2 in the R1 order
 *     (32 strided partial sums, halving tree), r = 1 / sqrt(ss / H + eps),
 *     x_hat = bf16((x * r) * gamma); each step one IEEE-rounded fp32 op.
 *
 * Precision: every accumulation except R1 is fp64; each stored bf16 value is
 * rounded once, round-to-nearest-even, from the fp64 value.
 *
 * Parity pins: every function here is checked by tests/test_oracle_*.py
 * against brute force, closed forms, invariants or library routines.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* bf16 <-> float <-> double, IEEE round-to-nearest-even               */
/* ------------------------------------------------------------------ */

float eto_bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

uint16_t eto_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) /* NaN: keep it quiet */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb; /* ties go to the even bf16 */
    return (uint16_t)(u >> 16);
}

/* double -> float rounding to odd, so that a following float -> bf16 RNE
 * equals a single double -> bf16 RNE (float keeps 16 more bits than bf16). */
static float f64_to_f32_round_odd(double d) {
    float f = (float)d;
    if (isnan(d) || isinf(f) || (double)f == d) return f;
    uint32_t u;
    memcpy(&u, &f, 4);
    if (fabs((double)f) > fabs(d)) u -= 1u; /* step back toward zero */
    u |= 1u;                                 /* sticky bit */
    memcpy(&f, &u, 4);
    return f;
}

uint16_t eto_f64_to_bf16(double d) { return eto_f32_to_bf16(f64_to_f32_round_odd(d)); }

static inline double bf(uint16_t b) { return (double)eto_bf16_to_f32(b); }

/* ------------------------------------------------------------------ */
/* tiny parallel-for over [0, n) with pthreads                         */
/* ------------------------------------------------------------------ */

typedef void (*range_fn)(void* ctx, int64_t begin, int64_t end);
typedef struct {
    range_fn fn;
    void* ctx;
    int64_t begin, end;
} range_job;

static void* range_thread(void* p) {
    range_job* j = (range_job*)p;
    j->fn(j->ctx, j->begin, j->end);
    return NULL;
}

static void parallel_for(int64_t n, int nthreads, range_fn fn, void* ctx) {
    if (n <= 0) return;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > n) nthreads = (int)n;
    if (nthreads == 1) {
        fn(ctx, 0, n);
        return;
    }
    pthread_t th[256];
    range_job jobs[256];
    int started[256];
    int64_t chunk = (n + nthreads - 1) / nthreads;
    for (int i = 0; i < nthreads; ++i) {
        jobs[i].fn = fn;
        jobs[i].ctx = ctx;
        jobs[i].begin = (int64_t)i * chunk;
        jobs[i].end = jobs[i].begin + chunk < n ? jobs[i].begin + chunk : n;
        started[i] = 0;
        if (jobs[i].begin >= jobs[i].end) continue;
        if (pthread_create(&th[i], NULL, range_thread, &jobs[i]) == 0)
            started[i] = 1;
        else
            range_thread(&jobs[i]); /* could not spawn: run inline */
    }
    for (int i = 0; i < nthreads; ++i)
        if (started[i]) pthread_join(th[i], NULL);
}

/* ------------------------------------------------------------------ */
/* R1: router logits in the fixed fp32 order                          */
/* ------------------------------------------------------------------ */

/* One logit: lane l (0..31) sums x[h]*w[h] over h = l, l+32, l+64, ...
 * ascending, starting from +0.0f; then for off = 16, 8, 4, 2, 1 the partial
 * of lane l becomes p[l] + p[l+off] for every l < off; the logit is p[0],
 * plus the bias (one fp32 add) when there is one.  xs/ws are strides in
 * elements between consecutive h. */
float eto_router_logit_one(const uint16_t* x, int64_t xs, const uint16_t* w, int64_t ws,
                           int H, const float* bias_e) {
    float p[32];
    for (int l = 0; l < 32; ++l) p[l] = 0.0f;
    for (int h = 0; h < H; ++h) {
        float prod = eto_bf16_to_f32(x[(int64_t)h * xs]) * eto_bf16_to_f32(w[(int64_t)h * ws]);
        p[h % 32] = p[h % 32] + prod;
    }
    for (int off = 16; off >= 1; off /= 2)
        for (int l = 0; l < off; ++l) p[l] = p[l] + p[l + off];
    float L = p[0];
    if (bias_e) L = L + *bias_e;
    return L;
}

typedef struct {
    const uint16_t *x, *wr;
    const float* bias;
    int H, E;
    float* logits;
} logits_ctx;

static void logits_range(void* c, int64_t b, int64_t e) {
    logits_ctx* k = (logits_ctx*)c;
    for (int64_t t = b; t < e; ++t)
        for (int ex = 0; ex < k->E; ++ex)
            k->logits[t * k->E + ex] = eto_router_logit_one(
                k->x + t * k->H, 1, k->wr + ex, k->E, k->H, k->bias ? k->bias + ex : NULL);
}

/* x bf16 [T,H]; wr bf16 [H,E] (as the router weight is given: hidden-major);
 * bias fp32 [E] or NULL; logits fp32 [T,E]. */
void eto_router_logits(const uint16_t* x, const uint16_t* wr, const float* bias, int T, int H,
                       int E, float* logits, int nthreads) {
    logits_ctx c = {x, wr, bias, H, E, logits};
    parallel_for(T, nthreads, logits_range, &c);
}

/* ------------------------------------------------------------------ */
/* R2: top-k selection and renormalised softmax gate weights          */
/* ------------------------------------------------------------------ */

/* a ranks before b when its logit is larger, or equal with a lower index */
static int ranks_before(float La, int a, float Lb, int b) {
    if (La > Lb) return 1;
    if (La < Lb) return 0;
    return a < b;
}

/* logits fp32 [T,E] -> idx int32 [T,k] (slot j = j-th in rank order),
 * w fp32 [T,k] = softmax over the k selected logits (fp64, stored fp32). */
void eto_topk_gate(const float* logits, int T, int E, int k, int32_t* idx, float* w) {
    int* taken = (int*)calloc((size_t)E, sizeof(int));
    for (int t = 0; t < T; ++t) {
        const float* L = logits + (int64_t)t * E;
        for (int e = 0; e < E; ++e) taken[e] = 0;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || ranks_before(L[e], e, L[best], best)) best = e;
            }
            taken[best] = 1;
            idx[(int64_t)t * k + j] = best;
        }
        double L0 = L[idx[(int64_t)t * k]];
        double z = 0.0;
        for (int j = 0; j < k; ++j) z += exp((double)L[idx[(int64_t)t * k + j]] - L0);
        for (int j = 0; j < k; ++j)
            w[(int64_t)t * k + j] = (float)(exp((double)L[idx[(int64_t)t * k + j]] - L0) / z);
    }
    free(taken);
}

/* ------------------------------------------------------------------ */
/* R3: per-expert counts, offsets, stable permutation (dispatch)       */
/* ------------------------------------------------------------------ */

/* cnt[e] = number of (t,j) routed to e; off = exclusive prefix sum of cnt
 * (E+1 entries); perm[off[e] + r] = t*k + j where r is the rank of t among
 * the tokens routed to e, ascending t; pos is the inverse of perm. */
void eto_dispatch(const int32_t* idx, int T, int E, int k, int32_t* cnt, int32_t* off,
                  int32_t* perm, int32_t* pos) {
    for (int e = 0; e < E; ++e) cnt[e] = 0;
    for (int64_t i = 0; i < (int64_t)T * k; ++i) cnt[idx[i]] += 1;
    off[0] = 0;
    for (int e = 0; e < E; ++e) off[e + 1] = off[e] + cnt[e];
    int32_t* fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int64_t i = (int64_t)t * k + j;
            int e = idx[i];
            int32_t p = off[e] + fill[e]++;
            if (perm) perm[p] = (int32_t)i;
            if (pos) pos[i] = p;
        }
    free(fill);
}

/* ------------------------------------------------------------------ */
/* R4: one expert's SwiGLU FFN on one row                              */
/* ------------------------------------------------------------------ */

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* xrow bf16 [H]; wg, wu bf16 [F,H]; wd bf16 [H,F] (out-features major,
 * like a Linear weight).  h_out bf16 [F] or NULL; y_out bf16 [H]. */
void eto_swiglu_row(const uint16_t* xrow, const uint16_t* wg, const uint16_t* wu,
                    const uint16_t* wd, int H, int F, uint16_t* h_out, uint16_t* y_out) {
    uint16_t* hb = (uint16_t*)malloc((size_t)F * sizeof(uint16_t));
    double* xd = (double*)malloc((size_t)H * sizeof(double));
    for (int i = 0; i < H; ++i) xd[i] = bf(xrow[i]);
    for (int f = 0; f < F; ++f) {
        const uint16_t* g_row = wg + (int64_t)f * H;
        const uint16_t* u_row = wu + (int64_t)f * H;
        double g = 0.0, u = 0.0;
        for (int i = 0; i < H; ++i) {
            g += xd[i] * bf(g_row[i]);
            u += xd[i] * bf(u_row[i]);
        }
        hb[f] = eto_f64_to_bf16(silu(g) * u);
    }
    for (int o = 0; o < H; ++o) {
        const uint16_t* d_row = wd + (int64_t)o * F;
        double y = 0.0;
        for (int f = 0; f < F; ++f) y += bf(hb[f]) * bf(d_row[f]);
        y_out[o] = eto_f64_to_bf16(y);
    }
    if (h_out) memcpy(h_out, hb, (size_t)F * sizeof(uint16_t));
    free(xd);
    free(hb);
}

/* ------------------------------------------------------------------ */
/* The MoE layer                                                       */
/* ------------------------------------------------------------------ */

typedef struct {
    const uint16_t *x, *wg, *wu, *wd;
    const int32_t* idx;
    const float* w;
    const int32_t* tokens; /* which tokens to produce, or NULL = all */
    int H, F, k;
    uint16_t* out;
} moe_ctx;

static void moe_rows(void* c, int64_t b, int64_t e) {
    moe_ctx* m = (moe_ctx*)c;
    uint16_t* y = (uint16_t*)malloc((size_t)m->H * sizeof(uint16_t));
    double* acc = (double*)malloc((size_t)m->H * sizeof(double));
    const int64_t ew = (int64_t)m->F * m->H; /* elements per expert matrix */
    for (int64_t r = b; r < e; ++r) {
        int64_t t = m->tokens ? m->tokens[r] : r;
        for (int i = 0; i < m->H; ++i) acc[i] = 0.0;
        for (int j = 0; j < m->k; ++j) {
            int ex = m->idx[t * m->k + j];
            eto_swiglu_row(m->x + t * m->H, m->wg + ex * ew, m->wu + ex * ew, m->wd + ex * ew,
                           m->H, m->F, NULL, y);
            double wj = (double)m->w[t * m->k + j];
            for (int i = 0; i < m->H; ++i) acc[i] += wj * bf(y[i]);
        }
        for (int i = 0; i < m->H; ++i) m->out[r * m->H + i] = eto_f64_to_bf16(acc[i]);
    }
    free(acc);
    free(y);
}

/* Full layer.  x bf16 [T,H]; wr bf16 [H,E]; bias fp32 [E] or NULL;
 * wg, wu bf16 [E,F,H]; wd bf16 [E,H,F].
 * Routing (idx [T,k], w [T,k], cnt [E], off [E+1], perm [T*k], pos [T*k])
 * is produced for all T tokens; any of those outputs may be NULL.
 * out bf16 gets one row per produced token: tokens[0..n_tokens) when tokens
 * is non-NULL (sampled check), else all T rows. */
int eto_moe_layer(const uint16_t* x, const uint16_t* wr, const float* bias, const uint16_t* wg,
                  const uint16_t* wu, const uint16_t* wd, int T, int H, int F, int E, int k,
                  const int32_t* tokens, int n_tokens, uint16_t* out, int32_t* idx_out,
                  float* w_out, int32_t* cnt_out, int32_t* off_out, int32_t* perm_out,
                  int32_t* pos_out, int nthreads) {
    if (T < 0 || H <= 0 || F <= 0 || E <= 0 || k <= 0 || k > E) return 1;
    float* logits = (float*)malloc(((size_t)T * E + 1) * sizeof(float));
    int32_t* idx = (int32_t*)malloc(((size_t)T * k + 1) * sizeof(int32_t));
    float* w = (float*)malloc(((size_t)T * k + 1) * sizeof(float));
    eto_router_logits(x, wr, bias, T, H, E, logits, nthreads);
    eto_topk_gate(logits, T, E, k, idx, w);
    if (cnt_out || off_out || perm_out || pos_out) {
        int32_t* cnt = (int32_t*)malloc((size_t)E * sizeof(int32_t));
        int32_t* off = (int32_t*)malloc((size_t)(E + 1) * sizeof(int32_t));
        eto_dispatch(idx, T, E, k, cnt, off, perm_out, pos_out);
        if (cnt_out) memcpy(cnt_out, cnt, (size_t)E * sizeof(int32_t));
        if (off_out) memcpy(off_out, off, (size_t)(E + 1) * sizeof(int32_t));
        free(cnt);
        free(off);
    }
    if (idx_out) memcpy(idx_out, idx, (size_t)T * k * sizeof(int32_t));
    if (w_out) memcpy(w_out, w, (size_t)T * k * sizeof(float));
    if (out) {
        moe_ctx c = {x, wg, wu, wd, idx, w, tokens, H, F, k, out};
        parallel_for(tokens ? n_tokens : T, nthreads, moe_rows, &c);
    }
    free(logits);
    free(idx);
    free(w);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Split-K GEMM: Y = bf16( sum_s X[:,K_s] Wt[:,K_s]^T )                */
/* ------------------------------------------------------------------ */

typedef struct {
    const uint16_t *X, *Wt;
    const int32_t* rows;
    int N, K, split;
    uint16_t* Y;
} splitk_ctx;

static void splitk_rows(void* c, int64_t b, int64_t e) {
    splitk_ctx* s = (splitk_ctx*)c;
    int64_t ks = s->K / s->split;
    double* xd = (double*)malloc((size_t)s->K * sizeof(double));
    for (int64_t r = b; r < e; ++r) {
        int64_t m = s->rows ? s->rows[r] : r;
        for (int i = 0; i < s->K; ++i) xd[i] = bf(s->X[m * s->K + i]);
        for (int n = 0; n < s->N; ++n) {
            const uint16_t* wrow = s->Wt + (int64_t)n * s->K;
            double total = 0.0;
            for (int sp = 0; sp < s->split; ++sp) { /* partial of chunk sp */
                double part = 0.0;
                for (int64_t i = sp * ks; i < (sp + 1) * ks; ++i) part += xd[i] * bf(wrow[i]);
                total += part;
            }
            s->Y[r * s->N + n] = eto_f64_to_bf16(total);
        }
    }
    free(xd);
}

/* X bf16 [M,K]; Wt bf16 [N,K] (the weight transposed: K contiguous);
 * split must divide K.  Y bf16 gets one row per produced row: rows[0..n_rows)
 * when rows is non-NULL, else all M. */
int eto_splitk_gemm(const uint16_t* X, const uint16_t* Wt, int M, int N, int K, int split,
                    const int32_t* rows, int n_rows, uint16_t* Y, int nthreads) {
    if (split <= 0 || K % split != 0 || M < 0 || N <= 0) return 1;
    splitk_ctx c = {X, Wt, rows, N, K, split, Y};
    parallel_for(rows ? n_rows : M, nthreads, splitk_rows, &c);
    return 0;
}

/* ------------------------------------------------------------------ */
/* R6 RMSNorm and the dense dependent MLP chain                        */
/* ------------------------------------------------------------------ */

void eto_rmsnorm_row(const uint16_t* x, const uint16_t* gamma, double eps, int H, uint16_t* xhat) {
    double ss = 0.0;
    for (int i = 0; i < H; ++i) ss += bf(x[i]) * bf(x[i]);
    double r = 1.0 / sqrt(ss / H + eps);
    for (int i = 0; i < H; ++i) xhat[i] = eto_f64_to_bf16(bf(x[i]) * r * bf(gamma[i]));
}

typedef struct {
    const uint16_t *x, *gamma, *wg, *wu, *wd;
    double eps;
    const int32_t* rows;
    int H, F;
    uint16_t* out;
} mlp_ctx;

static void mlp_rows(void* c, int64_t b, int64_t e) {
    mlp_ctx* m = (mlp_ctx*)c;
    uint16_t* xhat = (uint16_t*)malloc((size_t)m->H * sizeof(uint16_t));
    for (int64_t r = b; r < e; ++r) {
        int64_t row = m->rows ? m->rows[r] : r;
        eto_rmsnorm_row(m->x + row * m->H, m->gamma, m->eps, m->H, xhat);
        eto_swiglu_row(xhat, m->wg, m->wu, m->wd, m->H, m->F, NULL, m->out + r * m->H);
    }
    free(xhat);
}

/* x bf16 [B,H]; gamma bf16 [H]; wg, wu bf16 [F,H]; wd bf16 [H,F];
 * out bf16 one row per produced row (rows[] or all B). */
int eto_mlp_chain(const uint16_t* x, const uint16_t* gamma, float eps, const uint16_t* wg,
                  const uint16_t* wu, const uint16_t* wd, int B, int H, int F,
                  const int32_t* rows, int n_rows, uint16_t* out, int nthreads) {
    if (B < 0 || H <= 0 || F <= 0) return 1;
    mlp_ctx c = {x, gamma, wg, wu, wd, (double)eps, rows, H, F, out};
    parallel_for(rows ? n_rows : B, nthreads, mlp_rows, &c);
    return 0;
}

/* ------------------------------------------------------------------ */
/* The fused MoE block (R14): x_hat = RMSNorm(x) * gamma, routed MoE   */
/* on x_hat, a shared SwiGLU expert on x_hat, residual add:            */
/*   out = bf16( x + sum_j w_j * y_j + y_s )  (fp64 sum, one rounding)  */
/* ------------------------------------------------------------------ */

/* R15: x_hat of one row in fp32, fixed order.  x^2 is exact in fp32 (a bf16
 * square), so the R1 sum of x*x is the fixed-order sum of squares. */
void eto_rmsnorm_row_f32(const uint16_t* x, const uint16_t* gamma, float eps, int H,
                         uint16_t* xhat) {
    float p[32];
    for (int l = 0; l < 32; ++l) p[l] = 0.0f;
    for (int h = 0; h < H; ++h) {
        const float v = eto_bf16_to_f32(x[h]);
        p[h % 32] = p[h % 32] + v * v;
    }
    for (int off = 16; off >= 1; off /= 2)
        for (int l = 0; l < off; ++l) p[l] = p[l] + p[l + off];
    const float ms = p[0] / (float)H;
    const float r = 1.0f / sqrtf(ms + eps);
    for (int h = 0; h < H; ++h)
        xhat[h] = eto_f32_to_bf16((eto_bf16_to_f32(x[h]) * r) * eto_bf16_to_f32(gamma[h]));
}

typedef struct {
    const uint16_t *x, *xhat, *wg, *wu, *wd, *sg, *su, *sd;
    const int32_t* idx;
    const float* w;
    const int32_t* tokens;
    int H, F, Fs, k;
    uint16_t* out;
} block_ctx;

static void block_rows(void* c, int64_t b, int64_t e) {
    block_ctx* m = (block_ctx*)c;
    uint16_t* y = (uint16_t*)malloc((size_t)m->H * sizeof(uint16_t));
    double* acc = (double*)malloc((size_t)m->H * sizeof(double));
    const int64_t ew = (int64_t)m->F * m->H;
    for (int64_t r = b; r < e; ++r) {
        int64_t t = m->tokens ? m->tokens[r] : r;
        const uint16_t* xh = m->xhat + t * m->H;
        for (int i = 0; i < m->H; ++i) acc[i] = bf(m->x[t * m->H + i]);  /* the residual */
        for (int j = 0; j < m->k; ++j) {                                  /* routed experts */
            int ex = m->idx[t * m->k + j];
            eto_swiglu_row(xh, m->wg + ex * ew, m->wu + ex * ew, m->wd + ex * ew, m->H, m->F,
                           NULL, y);
            double wj = (double)m->w[t * m->k + j];
            for (int i = 0; i < m->H; ++i) acc[i] += wj * bf(y[i]);
        }
        if (m->Fs > 0) {                                                  /* shared expert */
            eto_swiglu_row(xh, m->sg, m->su, m->sd, m->H, m->Fs, NULL, y);
            for (int i = 0; i < m->H; ++i) acc[i] += bf(y[i]);
        }
        for (int i = 0; i < m->H; ++i) m->out[r * m->H + i] = eto_f64_to_bf16(acc[i]);
    }
    free(acc);
    free(y);
}

typedef struct {
    const uint16_t *x, *gamma;
    float eps;
    int H;
    uint16_t* xhat;
} norm_ctx;

static void norm_rows_range(void* c, int64_t b, int64_t e) {
    norm_ctx* m = (norm_ctx*)c;
    for (int64_t r = b; r < e; ++r)
        eto_rmsnorm_row_f32(m->x + r * m->H, m->gamma, m->eps, m->H, m->xhat + r * m->H);
}

/* x bf16 [T,H]; gamma bf16 [H]; routed weights as in eto_moe_layer; shared
 * expert sg, su bf16 [Fs,H], sd bf16 [H,Fs] (Fs = 0: none, pointers ignored).
 * Routing outputs as in eto_moe_layer (routing of x_hat); out bf16 one row per
 * produced token (tokens[] or all T); xhat_out bf16 [T,H] or NULL. */
int eto_moe_block(const uint16_t* x, const uint16_t* gamma, float eps, const uint16_t* wr,
                  const float* bias, const uint16_t* wg, const uint16_t* wu, const uint16_t* wd,
                  const uint16_t* sg, const uint16_t* su, const uint16_t* sd, int T, int H, int F,
                  int Fs, int E, int k, const int32_t* tokens, int n_tokens, uint16_t* out,
                  uint16_t* xhat_out, int32_t* idx_out, float* w_out, int32_t* cnt_out,
                  int32_t* perm_out, int nthreads) {
    if (T < 0 || H <= 0 || F <= 0 || Fs < 0 || E <= 0 || k <= 0 || k > E) return 1;
    uint16_t* xhat = (uint16_t*)malloc(((size_t)T * H + 1) * sizeof(uint16_t));
    norm_ctx nc = {x, gamma, eps, H, xhat};
    parallel_for(T, nthreads, norm_rows_range, &nc);
    int32_t* idx = (int32_t*)malloc(((size_t)T * k + 1) * sizeof(int32_t));
    float* w = (float*)malloc(((size_t)T * k + 1) * sizeof(float));
    int32_t* cnt = (int32_t*)malloc((size_t)E * sizeof(int32_t));
    int32_t* off = (int32_t*)malloc((size_t)(E + 1) * sizeof(int32_t));
    int rc = eto_moe_layer(xhat, wr, bias, wg, wu, wd, T, H, F, E, k, NULL, 0, NULL, idx, w, cnt,
                           off, perm_out, NULL, nthreads);
    if (rc == 0 && out) {
        block_ctx c = {x, xhat, wg, wu, wd, sg, su, sd, idx, w, tokens, H, F, Fs, k, out};
        parallel_for(tokens ? n_tokens : T, nthreads, block_rows, &c);
    }
    if (idx_out) memcpy(idx_out, idx, (size_t)T * k * sizeof(int32_t));
    if (w_out) memcpy(w_out, w, (size_t)T * k * sizeof(float));
    if (cnt_out) memcpy(cnt_out, cnt, (size_t)E * sizeof(int32_t));
    if (xhat_out) memcpy(xhat_out, xhat, (size_t)T * H * sizeof(uint16_t));
    free(off);
    free(cnt);
    free(w);
    free(idx);
    free(xhat);
    return rc;
}

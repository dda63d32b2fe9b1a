/*
 * oracle.c -- plain, slow, obviously-correct fp32 CPU oracle for Lookahead
 * Decoding (Fu, Bailis, Stoica, Zhang 2024, "Break the Sequential Dependency
 * of LLM Inference Using Lookahead Decoding").
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this library.  It shares no code, header, table or
 * constant with the CUDA library: it is written from the method's definition.
 *
 * What it computes
 *  - G-oracle: plain greedy decoding of a Llama-style decoder (the baseline
 *    the summary's "Summary" paragraph says each step of which is bound by
 *    memory bandwidth).  Its output is the definition of the right answer:
 *    the summary states that lookahead decoding keeps the output exactly the
 *    same.
 *  - LA-oracle: lookahead decoding, step by step: a lookahead branch over a
 *    2D window of W columns x (N-1) levels, an n-gram pool keyed on the first
 *    token holding up to G (N-1)-grams per key, and a verification branch,
 *    all evaluated in one forward pass per step under one attention mask
 *    ("Summary" paragraph and "Key points", tuning knobs W, N, G).
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  R1 window init from a splitmix64 stream (Vigna's published definition);
 *  R2 row order: row 0 = current token c at P; lookahead row (l,j) =
 *     1 + l*W + j at P+1+j+l; verification row (g,i) = 1 + W(N-1) + g(N-1) + i
 *     at P+1+i;
 *  R3 mask: row 0 sees {0}; (l,j) sees {0} u {(0,j'): j'<=j} u {(l',j):
 *     1<=l'<=l}; (g,i) sees {0} u {(g,i'): i'<=i}; every row also sees the
 *     cache [0,P) and itself;
 *  R3' (variant "diagonal levels", om_ctrl_set_variant): each level is one
 *     Jacobi iterate over the same positions: (l,j) at P+1+j sees {0} u
 *     {(l,j'): j'<=j}; the new last level is the Jacobi update (argmax of
 *     row 0, then the argmax of the last level's row j-1 at column j); the
 *     n-grams run along diagonals: key win[0][j], value (win[1][j+1], ...,
 *     win[N-2][j+N-2], argmax of row (N-2,j+N-2)) for j = 0..W-N+1;
 *  R5 verify: longest candidate prefix equal to the model's argmaxes, ties to
 *     the lowest g, plus one bonus token;
 *  R6 harvest: for j ascending, key win[0][j], value (win[1..N-2][j],
 *     argmax of row (N-2,j)); present -> no-op, else append, evicting the
 *     oldest when G entries are held (FIFO);
 *  R7 window: drop level 0, shift up, new last level = argmaxes of the last
 *     level's rows;
 *  R8 commit KV of row 0 and of the accepted candidate rows;
 *  R9 optional prompt pre-seed: insert (prompt[i], prompt[i+1..i+N-1]) for
 *     i ascending ("Key points": prompt n-grams in the pool help).
 *  R10 sampling verification (the summary says the method supports sampling
 *     and keeps the output distribution; it gives no algorithm, so this one
 *     is designed here): temperature softmax p = softmax(z / tau) of a row
 *     (exponentials in fp32 by om_exp_neg, as exact integer weights: see
 *     om_sample_weight);
 *     at each candidate level the distinct candidate tokens v are tried in
 *     candidate order, v accepted with probability p(v) / (1 - mass of the
 *     tokens already rejected at this level); if none is accepted, the token
 *     is drawn from p restricted to the tokens not rejected.  Each emitted
 *     token is then distributed exactly as p of its row (the acceptance
 *     probabilities telescope), so the emitted sequence has the distribution
 *     of plain ancestral sampling.  The lookahead branch keeps using argmaxes.
 *     Top-k and top-p (optional; the summary says several sampling schemes
 *     are supported): p is first restricted to the top_k tokens by weight
 *     (ties to the lower index), then to the smallest leading set of those,
 *     in the same order, holding at least top_p of their weight, and
 *     renormalised; the rule is unchanged, so each emitted token then
 *     follows the restricted p (keep_top_k, keep_top_p).
 *
 * Model (M1-M3): h = x + Wo*Attn(RMSNorm(x)); y = h + Wd*(silu(Wg n) . Wu n),
 * n = RMSNorm(h); RMSNorm(x) = x / sqrt(mean(x^2) + eps) * w (Zhang and
 * Sennrich 2019, cited by the pages); rotate-half RoPE, angle
 * pos * theta^(-2i/hd), table computed in double and rounded to float;
 * softmax over visible keys in ascending position order; GQA head map
 * h -> h / (H/Hkv); greedy argmax = lowest index of the maximum.
 * All dot products accumulate in ascending index order in fp32.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define OM_EXPORT __attribute__((visibility("default")))

typedef struct om_model {
    int n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn, vocab;
    float rms_eps, rope_theta;
    const float* emb;        /* [vocab][d_model] */
    const float* final_norm; /* [d_model] */
    const float* lm_head;    /* [vocab][d_model] */
    const float* const* attn_norm; /* per layer [d_model] */
    const float* const* wq;        /* per layer [H*hd][d_model] */
    const float* const* wk;        /* per layer [Hkv*hd][d_model] */
    const float* const* wv;        /* per layer [Hkv*hd][d_model] */
    const float* const* wo;        /* per layer [d_model][H*hd] */
    const float* const* ffn_norm;  /* per layer [d_model] */
    const float* const* wg;        /* per layer [ffn][d_model] */
    const float* const* wu;        /* per layer [ffn][d_model] */
    const float* const* wd;        /* per layer [d_model][ffn] */
} om_model;

/* ---------------------------------------------------------------- sequence */

typedef struct om_seq {
    const om_model* m;
    int max_seq, d_kv;
    float* kc;   /* [L][max_seq][d_kv] rotated keys */
    float* vc;   /* [L][max_seq][d_kv] */
    float* cosb; /* [max_seq][hd/2] */
    float* sinb;
    int cap_rows, last_T;
    float* sk;   /* [L][cap_rows][d_kv] keys of the last step's rows */
    float* sv;
} om_seq;

OM_EXPORT om_seq* om_seq_new(const om_model* m, int max_seq)
{
    om_seq* s = (om_seq*)calloc(1, sizeof(om_seq));
    if (!s) return NULL;
    s->m = m;
    s->max_seq = max_seq;
    s->d_kv = m->n_kv_heads * m->head_dim;
    size_t n = (size_t)m->n_layers * max_seq * s->d_kv;
    s->kc = (float*)calloc(n, sizeof(float));
    s->vc = (float*)calloc(n, sizeof(float));
    int half = m->head_dim / 2;
    s->cosb = (float*)malloc(sizeof(float) * (size_t)max_seq * half);
    s->sinb = (float*)malloc(sizeof(float) * (size_t)max_seq * half);
    if (!s->kc || !s->vc || !s->cosb || !s->sinb) return NULL;
    for (int p = 0; p < max_seq; p++)
        for (int i = 0; i < half; i++) {
            double ang = (double)p * pow((double)m->rope_theta, -2.0 * i / (double)m->head_dim);
            s->cosb[(size_t)p * half + i] = (float)cos(ang);
            s->sinb[(size_t)p * half + i] = (float)sin(ang);
        }
    return s;
}

OM_EXPORT void om_seq_free(om_seq* s)
{
    if (!s) return;
    free(s->kc); free(s->vc); free(s->cosb); free(s->sinb); free(s->sk); free(s->sv);
    free(s);
}

OM_EXPORT int om_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads of the parallel loops that follow (results do not depend on it:
 * every parallel loop is over independent output elements). */
OM_EXPORT void om_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

OM_EXPORT void om_rope_table(const om_seq* s, float* cos_out, float* sin_out)
{
    size_t n = (size_t)s->max_seq * (s->m->head_dim / 2);
    memcpy(cos_out, s->cosb, n * sizeof(float));
    memcpy(sin_out, s->sinb, n * sizeof(float));
}

static float dot(const float* a, const float* b, int n)
{
    float acc = 0.0f;
    for (int i = 0; i < n; i++) acc += a[i] * b[i];
    return acc;
}

static void rmsnorm(const float* x, const float* w, int d, float eps, float* out)
{
    float ss = 0.0f;
    for (int i = 0; i < d; i++) ss += x[i] * x[i];
    float r = 1.0f / sqrtf(ss / (float)d + eps);
    for (int i = 0; i < d; i++) out[i] = x[i] * r * w[i];
}

/* rotate-half RoPE of one head vector at position pos */
static void rope(float* v, int hd, const float* cosb, const float* sinb, int pos)
{
    int half = hd / 2;
    for (int i = 0; i < half; i++) {
        float c = cosb[(size_t)pos * half + i], s = sinb[(size_t)pos * half + i];
        float x1 = v[i], x2 = v[i + half];
        v[i] = x1 * c - x2 * s;
        v[i + half] = x2 * c + x1 * s;
    }
}

/* rotate one head vector in place with the sequence's table (exported so the
 * tests can check the rotation's relative-position property directly) */
OM_EXPORT void om_rope(const om_seq* s, float* v, int pos)
{
    rope(v, s->m->head_dim, s->cosb, s->sinb, pos);
}

/* visible in-step rows of each row, sorted by (position, index) */
static void visible_order(int T, const int* pos, const unsigned char* vis, int* order, int* nvis)
{
    for (int r = 0; r < T; r++) {
        int n = 0;
        for (int c = 0; c < T; c++) {
            if (!vis[(size_t)r * T + c]) continue;
            int k = n++;
            while (k > 0 && pos[order[(size_t)r * T + k - 1]] > pos[c]) {
                order[(size_t)r * T + k] = order[(size_t)r * T + k - 1];
                k--;
            }
            order[(size_t)r * T + k] = c;
        }
        nvis[r] = n;
    }
}

/* Softmax attention of one query head vector over the cache rows [0,P)
 * (row j at kc + j*kv_stride) followed by the visible step rows order[0..nvis)
 * (row c at ks + c*step_stride), in ascending position order: scores
 * q.k / sqrt(hd), subtract the max, expf, sum, then the weighted V sum
 * divided by the sum. */
static void attend_row(const float* qh, const float* kc, const float* vc, int kv_stride, int P, const float* ks,
                       const float* vs, int step_stride, const int* order, int nvis, int hd, float* out)
{
    const float scale_div = sqrtf((float)hd);
    int nk = P + nvis;
    float* sc = (float*)malloc(sizeof(float) * (size_t)(nk > 0 ? nk : 1));
    for (int j = 0; j < P; j++) sc[j] = dot(qh, kc + (size_t)j * kv_stride, hd) / scale_div;
    for (int t = 0; t < nvis; t++) sc[P + t] = dot(qh, ks + (size_t)order[t] * step_stride, hd) / scale_div;
    float mx = -INFINITY;
    for (int j = 0; j < nk; j++)
        if (sc[j] > mx) mx = sc[j];
    float sum = 0.0f;
    for (int j = 0; j < nk; j++) {
        sc[j] = expf(sc[j] - mx);
        sum += sc[j];
    }
    for (int e = 0; e < hd; e++) {
        float acc = 0.0f;
        for (int j = 0; j < P; j++) acc += sc[j] * vc[(size_t)j * kv_stride + e];
        for (int t = 0; t < nvis; t++) acc += sc[P + t] * vs[(size_t)order[t] * step_stride + e];
        out[e] = acc / sum;
    }
    free(sc);
}

/*
 * One layer's masked attention on its own (the lookahead step's attention
 * with given q, k, v): q [T][H][hd], k_cache/v_cache [Hkv][max_seq][hd]
 * (positions [0,P)), k_step/v_step [T][Hkv][hd], vis [T][T] (row r sees step
 * row c), pos [T].  out [T][H][hd].  Query head h uses KV head h/(H/Hkv).
 */
OM_EXPORT int om_attention(int T, int H, int Hkv, int hd, int max_seq, int P, const float* q, const float* k_cache,
                           const float* v_cache, const float* k_step, const float* v_step, const unsigned char* vis,
                           const int* pos, float* out)
{
    if (T <= 0 || H % Hkv || P < 0 || P > max_seq) return -1;
    int* order = (int*)malloc(sizeof(int) * (size_t)T * T);
    int* nvis = (int*)malloc(sizeof(int) * T);
    if (!order || !nvis) return -1;
    visible_order(T, pos, vis, order, nvis);
    const int grp = H / Hkv;
    #pragma omp parallel for collapse(2) schedule(dynamic)
    for (int r = 0; r < T; r++)
        for (int h = 0; h < H; h++) {
            int kvh = h / grp;
            attend_row(q + ((size_t)r * H + h) * hd, k_cache + (size_t)kvh * max_seq * hd,
                       v_cache + (size_t)kvh * max_seq * hd, hd, P, k_step + (size_t)kvh * hd,
                       v_step + (size_t)kvh * hd, Hkv * hd, order + (size_t)r * T, nvis[r], hd,
                       out + ((size_t)r * H + h) * hd);
        }
    free(order);
    free(nvis);
    return 0;
}

static float silu(float z) { return z / (1.0f + expf(-z)); }

static int argmax_row(const float* x, int n)
{
    int best = 0;
    for (int i = 1; i < n; i++)
        if (x[i] > x[best]) best = i;
    return best;
}

/*
 * One forward pass over T rows (tokens tok[r] at positions pos[r]).  Row r
 * attends to the cache [0,P) and to every in-step row s with
 * vis[r*T+s] != 0, in ascending position order.  The step rows' keys and
 * values are kept for om_commit.  logits (T x V) and argmax (T) may be NULL.
 * Returns 0, or -1 on bad arguments / allocation failure.
 */
OM_EXPORT int om_step_forward(om_seq* s, int P, int T, const int* tok, const int* pos,
                              const unsigned char* vis, float* logits, int* amax)
{
    const om_model* m = s->m;
    const int L = m->n_layers, d = m->d_model, H = m->n_heads, Hkv = m->n_kv_heads;
    const int hd = m->head_dim, F = m->ffn, V = m->vocab, dq = H * hd, dkv = s->d_kv;
    const int grp = H / Hkv;
    if (T <= 0 || P < 0) return -1;
    for (int r = 0; r < T; r++)
        if (pos[r] < 0 || pos[r] >= s->max_seq || tok[r] < 0 || tok[r] >= V) return -1;
    if (T > s->cap_rows) {
        free(s->sk); free(s->sv);
        s->sk = (float*)malloc(sizeof(float) * (size_t)L * T * dkv);
        s->sv = (float*)malloc(sizeof(float) * (size_t)L * T * dkv);
        if (!s->sk || !s->sv) return -1;
        s->cap_rows = T;
    }
    s->last_T = T;
    float* x = (float*)malloc(sizeof(float) * (size_t)T * d);
    float* xn = (float*)malloc(sizeof(float) * (size_t)T * d);
    float* q = (float*)malloc(sizeof(float) * (size_t)T * dq);
    float* att = (float*)malloc(sizeof(float) * (size_t)T * dq);
    float* act = (float*)malloc(sizeof(float) * (size_t)T * F);
    int* order = (int*)malloc(sizeof(int) * (size_t)T * T);
    int* nvis = (int*)malloc(sizeof(int) * T);
    if (!x || !xn || !q || !att || !act || !order || !nvis) return -1;

    visible_order(T, pos, vis, order, nvis);

    for (int r = 0; r < T; r++)
        memcpy(x + (size_t)r * d, m->emb + (size_t)tok[r] * d, sizeof(float) * d);

    for (int l = 0; l < L; l++) {
        float* skl = s->sk + (size_t)l * s->cap_rows * dkv;
        float* svl = s->sv + (size_t)l * s->cap_rows * dkv;
        const float* kcl = s->kc + (size_t)l * s->max_seq * dkv;
        const float* vcl = s->vc + (size_t)l * s->max_seq * dkv;

        for (int r = 0; r < T; r++)
            rmsnorm(x + (size_t)r * d, m->attn_norm[l], d, m->rms_eps, xn + (size_t)r * d);
        #pragma omp parallel for collapse(2) schedule(static)
        for (int r = 0; r < T; r++)
            for (int o = 0; o < dq + 2 * dkv; o++) {
                const float* xr = xn + (size_t)r * d;
                if (o < dq) q[(size_t)r * dq + o] = dot(m->wq[l] + (size_t)o * d, xr, d);
                else if (o < dq + dkv) skl[(size_t)r * dkv + (o - dq)] = dot(m->wk[l] + (size_t)(o - dq) * d, xr, d);
                else svl[(size_t)r * dkv + (o - dq - dkv)] = dot(m->wv[l] + (size_t)(o - dq - dkv) * d, xr, d);
            }
        for (int r = 0; r < T; r++) {
            for (int h = 0; h < H; h++) rope(q + (size_t)r * dq + h * hd, hd, s->cosb, s->sinb, pos[r]);
            for (int h = 0; h < Hkv; h++) rope(skl + (size_t)r * dkv + h * hd, hd, s->cosb, s->sinb, pos[r]);
        }

        /* attention: row r, head h over cache [0,P) then visible step rows */
        #pragma omp parallel for collapse(2) schedule(dynamic)
        for (int r = 0; r < T; r++)
            for (int h = 0; h < H; h++) {
                int kvh = h / grp;
                attend_row(q + (size_t)r * dq + h * hd, kcl + kvh * hd, vcl + kvh * hd, dkv, P, skl + kvh * hd,
                           svl + kvh * hd, dkv, order + (size_t)r * T, nvis[r], hd, att + (size_t)r * dq + h * hd);
            }

        #pragma omp parallel for collapse(2) schedule(static)
        for (int r = 0; r < T; r++)
            for (int o = 0; o < d; o++)
                x[(size_t)r * d + o] = x[(size_t)r * d + o] + dot(m->wo[l] + (size_t)o * dq, att + (size_t)r * dq, dq);

        for (int r = 0; r < T; r++)
            rmsnorm(x + (size_t)r * d, m->ffn_norm[l], d, m->rms_eps, xn + (size_t)r * d);
        #pragma omp parallel for collapse(2) schedule(static)
        for (int r = 0; r < T; r++)
            for (int f = 0; f < F; f++) {
                const float* xr = xn + (size_t)r * d;
                float g = dot(m->wg[l] + (size_t)f * d, xr, d);
                float u = dot(m->wu[l] + (size_t)f * d, xr, d);
                act[(size_t)r * F + f] = silu(g) * u;
            }
        #pragma omp parallel for collapse(2) schedule(static)
        for (int r = 0; r < T; r++)
            for (int o = 0; o < d; o++)
                x[(size_t)r * d + o] = x[(size_t)r * d + o] + dot(m->wd[l] + (size_t)o * F, act + (size_t)r * F, F);
    }

    if (logits || amax) {
        for (int r = 0; r < T; r++)
            rmsnorm(x + (size_t)r * d, m->final_norm, d, m->rms_eps, xn + (size_t)r * d);
        float* lg = logits ? logits : (float*)malloc(sizeof(float) * (size_t)T * V);
        #pragma omp parallel for collapse(2) schedule(static)
        for (int r = 0; r < T; r++)
            for (int v = 0; v < V; v++)
                lg[(size_t)r * V + v] = dot(m->lm_head + (size_t)v * d, xn + (size_t)r * d, d);
        if (amax)
            for (int r = 0; r < T; r++) amax[r] = argmax_row(lg + (size_t)r * V, V);
        if (!logits) free(lg);
    }
    free(x); free(xn); free(q); free(att); free(act); free(order); free(nvis);
    return 0;
}

/* Copy the keys/values of the last step's rows rows[0..n-1] to cache
 * positions P..P+n-1 of every layer. */
OM_EXPORT int om_commit(om_seq* s, int P, int n, const int* rows)
{
    if (P < 0 || P + n > s->max_seq) return -1;
    const int L = s->m->n_layers, dkv = s->d_kv;
    for (int i = 0; i < n; i++)
        if (rows[i] < 0 || rows[i] >= s->last_T) return -1;
    for (int l = 0; l < L; l++)
        for (int i = 0; i < n; i++) {
            memcpy(s->kc + ((size_t)l * s->max_seq + P + i) * dkv, s->sk + ((size_t)l * s->cap_rows + rows[i]) * dkv,
                   sizeof(float) * dkv);
            memcpy(s->vc + ((size_t)l * s->max_seq + P + i) * dkv, s->sv + ((size_t)l * s->cap_rows + rows[i]) * dkv,
                   sizeof(float) * dkv);
        }
    return 0;
}

/* Causal prefill of toks[0..n-1] at positions P0.. one token at a time. */
OM_EXPORT int om_prefill(om_seq* s, int P0, const int* toks, int n)
{
    for (int t = 0; t < n; t++) {
        int p = P0 + t;
        unsigned char one = 1;
        int row = 0;
        if (om_step_forward(s, p, 1, toks + t, &p, &one, NULL, NULL)) return -1;
        if (om_commit(s, p, 1, &row)) return -1;
    }
    return 0;
}

/* ------------------------------------------------------------------ greedy */

/* G-oracle: greedy decoding.  Prefills prompt[0..len-2], then emits max_new
 * tokens, each the argmax of the forward of the current token at P.
 * logits_out (max_new x V) may be NULL. */
OM_EXPORT int om_greedy(const om_model* m, const int* prompt, int len, int max_new, int max_seq,
                        int* out, float* logits_out)
{
    if (len < 1 || len - 1 + max_new > max_seq) return -1;
    om_seq* s = om_seq_new(m, max_seq);
    if (!s) return -1;
    int rc = om_prefill(s, 0, prompt, len - 1);
    int c = prompt[len - 1], P = len - 1;
    for (int t = 0; t < max_new && !rc; t++) {
        unsigned char one = 1;
        int a, row = 0;
        rc = om_step_forward(s, P, 1, &c, &P, &one, logits_out ? logits_out + (size_t)t * m->vocab : NULL, &a);
        if (!rc) rc = om_commit(s, P, 1, &row);
        out[t] = a;
        c = a;
        P++;
    }
    om_seq_free(s);
    return rc;
}

/* -------------------------------------------------------------- controller */

typedef struct om_ctrl {
    int W, N, G, V;
    int diag;      /* 0: R3 (levels along columns), 1: R3' (diagonal levels) */
    int* win;      /* [N-1][W] */
    int* pool_cnt; /* [V] */
    int* pool;     /* [V][G][N-1], oldest first */
    /* snapshot of the last om_ctrl_rows call */
    int c, P, T, Gp;
    int* cands;    /* [G][N-1] */
} om_ctrl;

OM_EXPORT om_ctrl* om_ctrl_new(int W, int N, int G, int V)
{
    if (W < 0 || N < 2 || G < 0 || V < 1) return NULL;
    om_ctrl* k = (om_ctrl*)calloc(1, sizeof(om_ctrl));
    k->W = W; k->N = N; k->G = G; k->V = V;
    k->win = (int*)calloc((size_t)(N - 1) * (W > 0 ? W : 1), sizeof(int));
    k->pool_cnt = (int*)calloc(V, sizeof(int));
    k->pool = (int*)calloc((size_t)V * (G > 0 ? G : 1) * (N - 1), sizeof(int));
    k->cands = (int*)calloc((size_t)(G > 0 ? G : 1) * (N - 1), sizeof(int));
    return k;
}

OM_EXPORT void om_ctrl_free(om_ctrl* k)
{
    if (!k) return;
    free(k->win); free(k->pool_cnt); free(k->pool); free(k->cands); free(k);
}

/* Select the mask reading: 0 = R3, 1 = R3' (diagonal levels). */
OM_EXPORT int om_ctrl_set_variant(om_ctrl* k, int diag)
{
    if (diag != 0 && diag != 1) return -1;
    k->diag = diag;
    return 0;
}

/* splitmix64 (S. Vigna): state += golden gamma, then two xor-shift-multiply
 * mixing rounds and a final xor-shift. */
OM_EXPORT uint64_t om_splitmix64(uint64_t* state)
{
    uint64_t z = (*state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* R6: insert an (N-1)-gram under key. */
OM_EXPORT void om_pool_insert(om_ctrl* k, int key, const int* val)
{
    const int n1 = k->N - 1;
    if (k->G == 0 || key < 0 || key >= k->V) return;
    int* e = k->pool + (size_t)key * k->G * n1;
    int cnt = k->pool_cnt[key];
    for (int g = 0; g < cnt; g++)
        if (memcmp(e + (size_t)g * n1, val, sizeof(int) * n1) == 0) return;
    if (cnt == k->G) {
        memmove(e, e + n1, sizeof(int) * (size_t)(k->G - 1) * n1);
        cnt--;
    }
    memcpy(e + (size_t)cnt * n1, val, sizeof(int) * n1);
    k->pool_cnt[key] = cnt + 1;
}

/* R1 window init and optional R9 prompt pre-seed; clears the pool. */
OM_EXPORT int om_ctrl_init(om_ctrl* k, const int* prompt, int len, uint64_t seed, int preseed)
{
    if (len < 1) return -1;
    memset(k->pool_cnt, 0, sizeof(int) * k->V);
    uint64_t st = seed;
    for (int l = 0; l < k->N - 1; l++)
        for (int j = 0; j < k->W; j++)
            k->win[(size_t)l * k->W + j] = prompt[om_splitmix64(&st) % (uint64_t)len];
    if (preseed)
        for (int i = 0; i + k->N - 1 < len; i++) om_pool_insert(k, prompt[i], prompt + i + 1);
    return 0;
}

OM_EXPORT int om_ctrl_rows_max(const om_ctrl* k) { return 1 + (k->W + k->G) * (k->N - 1); }

static int row_la(const om_ctrl* k, int l, int j) { return 1 + l * k->W + j; }
static int row_vf(const om_ctrl* k, int g, int i) { return 1 + k->W * (k->N - 1) + g * (k->N - 1) + i; }

/*
 * R2 + R3: the rows of the step for current token c with P cached tokens.
 * Candidates = pool[c] in insertion order (G' of them).  Writes tok, pos (T
 * entries) and vis (T*T, vis[r*T+s]) and returns T = 1 + (W+G')(N-1).
 * Buffers must hold om_ctrl_rows_max() rows.
 */
OM_EXPORT int om_ctrl_rows(om_ctrl* k, int c, int P, int* tok, int* pos, unsigned char* vis)
{
    const int W = k->W, n1 = k->N - 1;
    int Gp = (c >= 0 && c < k->V && k->G > 0) ? k->pool_cnt[c] : 0;
    k->c = c; k->P = P; k->Gp = Gp;
    if (Gp) memcpy(k->cands, k->pool + (size_t)c * k->G * n1, sizeof(int) * (size_t)Gp * n1);
    int T = 1 + (W + Gp) * n1;
    k->T = T;
    memset(vis, 0, (size_t)T * T);
    tok[0] = c; pos[0] = P; vis[0] = 1;
    for (int l = 0; l < n1; l++)
        for (int j = 0; j < W; j++) {
            int r = row_la(k, l, j);
            tok[r] = k->win[(size_t)l * W + j];
            vis[(size_t)r * T + 0] = 1;
            if (k->diag) {
                /* R3': the row's own level, columns 0..j */
                pos[r] = P + 1 + j;
                for (int jj = 0; jj <= j; jj++) vis[(size_t)r * T + row_la(k, l, jj)] = 1;
            } else {
                pos[r] = P + 1 + j + l;
                for (int jj = 0; jj <= j; jj++) vis[(size_t)r * T + row_la(k, 0, jj)] = 1;
                for (int ll = 1; ll <= l; ll++) vis[(size_t)r * T + row_la(k, ll, j)] = 1;
            }
        }
    for (int g = 0; g < Gp; g++)
        for (int i = 0; i < n1; i++) {
            int r = row_vf(k, g, i);
            tok[r] = k->cands[(size_t)g * n1 + i];
            pos[r] = P + 1 + i;
            vis[(size_t)r * T + 0] = 1;
            for (int ii = 0; ii <= i; ii++) vis[(size_t)r * T + row_vf(k, g, ii)] = 1;
        }
    return T;
}

/* R6 harvest (j ascending, from the window before the shift) and R7 window
 * shift, given the argmax of every row of the step.  Under R3' the n-gram
 * starting at column j steps one column right per level, and the new last
 * level is the Jacobi update of the last level. */
static void harvest_and_shift(om_ctrl* k, const int* amax)
{
    const int W = k->W, n1 = k->N - 1, d = k->diag;
    int* val = (int*)malloc(sizeof(int) * n1);
    const int n_grams = d ? W - (n1 - 1) : W;
    for (int j = 0; j < n_grams; j++) {
        int key = k->win[j];
        for (int l = 1; l < n1; l++) val[l - 1] = k->win[(size_t)l * W + j + d * l];
        val[n1 - 1] = amax[row_la(k, n1 - 1, j + d * (n1 - 1))];
        om_pool_insert(k, key, val);
    }
    free(val);
    for (int l = 0; l + 1 < n1; l++)
        memcpy(k->win + (size_t)l * W, k->win + (size_t)(l + 1) * W, sizeof(int) * W);
    for (int j = 0; j < W; j++) {
        int a;
        if (!d) a = amax[row_la(k, n1 - 1, j)];
        else a = (j == 0) ? amax[0] : amax[row_la(k, n1 - 1, j - 1)];
        k->win[(size_t)(n1 - 1) * W + j] = a;
    }
}

/*
 * R5-R7 after the forward of the rows built by the last om_ctrl_rows call.
 * amax: argmax of every row.  Writes the emitted tokens (m+1 of them) to emit,
 * the rows whose KV is committed (m+1, row 0 first) to rows, returns m + 1.
 * *gstar receives the chosen candidate (-1 if none).
 */
OM_EXPORT int om_ctrl_advance(om_ctrl* k, const int* amax, int* emit, int* rows, int* gstar)
{
    const int n1 = k->N - 1;
    int best_m = 0, best_g = -1;
    for (int g = 0; g < k->Gp; g++) {
        int m = 0;
        while (m < n1) {
            int expect = (m == 0) ? amax[0] : amax[row_vf(k, g, m - 1)];
            if (k->cands[(size_t)g * n1 + m] != expect) break;
            m++;
        }
        if (best_g < 0 || m > best_m) { best_m = m; best_g = g; }
    }
    emit[0] = amax[0];
    rows[0] = 0;
    for (int i = 0; i < best_m; i++) {
        emit[i + 1] = amax[row_vf(k, best_g, i)];
        rows[i + 1] = row_vf(k, best_g, i);
    }
    if (gstar) *gstar = best_g;
    harvest_and_shift(k, amax);
    return best_m + 1;
}

OM_EXPORT int om_ctrl_pool(const om_ctrl* k, int key, int* out)
{
    if (key < 0 || key >= k->V || k->G == 0) return 0;
    int cnt = k->pool_cnt[key];
    memcpy(out, k->pool + (size_t)key * k->G * (k->N - 1), sizeof(int) * (size_t)cnt * (k->N - 1));
    return cnt;
}

OM_EXPORT void om_ctrl_window(const om_ctrl* k, int* out)
{
    memcpy(out, k->win, sizeof(int) * (size_t)(k->N - 1) * k->W);
}

/* --------------------------------------------------------- sampling (R10) */

/* Uniform draw in [0,1): the top 24 bits of the next splitmix64 output. */
OM_EXPORT double om_uniform(uint64_t* rng) { return (double)(om_splitmix64(rng) >> 40) * (1.0 / 16777216.0); }

/* exp(x) for x <= 0 in fp32, the exponential of the sampling probabilities.
 * Range reduction after Cody and Waite: k = the integer nearest x log2(e),
 * t = x - k ln 2 with ln 2 split into a float and the float remainder
 * (two fused multiply-adds, so that t keeps its precision for large |x|),
 * |t| <= 0.35; e^t by its Taylor series to degree 7 (truncation below 6e-9
 * relative), by Horner's rule with fused multiply-adds; then scaled by 2^k
 * (exact).  Results below 2^-125 are flushed to 0.  Every step is a
 * correctly rounded IEEE fp32 operation, so any implementation performing
 * the same operations (the CUDA library's sampling kernels do) returns the
 * same bits. */
OM_EXPORT float om_exp_neg(float x)
{
    const float k = rintf(x * 0x1.715476p+0f); /* log2(e) */
    if (k < -125.0f) return 0.0f;
    float t = fmaf(-k, 0x1.62e430p-1f, x);  /* ln 2, float part */
    t = fmaf(-k, -0x1.05c610p-29f, t);      /* ln 2, remainder */
    float q = 0x1.a01a02p-13f;              /* 1/7! */
    q = fmaf(q, t, 0x1.6c16c2p-10f);        /* 1/6! */
    q = fmaf(q, t, 0x1.111112p-7f);         /* 1/5! */
    q = fmaf(q, t, 0x1.555556p-5f);         /* 1/4! */
    q = fmaf(q, t, 0x1.555556p-3f);         /* 1/3! */
    q = fmaf(q, t, 0.5f);
    q = fmaf(q, t, 1.0f);
    q = fmaf(q, t, 1.0f);
    return ldexpf(q, (int)k);
}

/* The sampling distribution as exact integers.  e(v) = om_exp_neg of
 * (z_v - max) / tau (an fp32 subtraction, then an fp32 division); the weight of
 * token v is E(v) = floor(e(v) 2^B) with B = 63 - ceil(log2(V + 1)), so that
 * S = sum of all E(v) < 2^63; p(v) = E(v) / S.  Every sum and comparison
 * below is exact integer arithmetic (products in 128 bits), so the result
 * does not depend on the order of the sums.  A uniform u = U / 2^24 (U the
 * top 24 bits of the next splitmix64 output):
 *  - accepts v against the mass R already rejected at a level when
 *    u (1 - R/S) < p(v), i.e. U (S - R) < E(v) 2^24;
 *  - draws from p restricted to the tokens not excluded the first token, in
 *    ascending order, whose running weight A has A 2^24 > U (S - R); the last
 *    admissible token of nonzero weight if none (cannot happen unless every
 *    admissible weight is 0). */
static int sample_bits(int V)
{
    int b = 0;
    while ((1LL << b) < (long long)V + 1) b++;
    return 63 - b;
}

OM_EXPORT uint64_t om_sample_weight(float z, float mx, float tau, int V)
{
    const float d = z - mx;
    const float e = om_exp_neg(d / tau);
    return (uint64_t)ldexpf(e, sample_bits(V));
}

/* Top-k restriction (top_k in 1..V-1; 0 or >= V keeps every token): the
 * distribution is renormalised over the top_k tokens by weight, ties to the
 * lower token index, i.e. the top_k largest keys E(v) V + (V - 1 - v) (all
 * distinct, < 2^63 since E(v) <= 2^B); the others get weight 0. */
static int cmp_desc_u64(const void* a, const void* b)
{
    const uint64_t x = *(const uint64_t*)a, y = *(const uint64_t*)b;
    return x < y ? 1 : (x > y ? -1 : 0);
}

OM_EXPORT uint64_t om_top_k_key(uint64_t E, int v, int V) { return E * (uint64_t)V + (uint64_t)(V - 1 - v); }

static void keep_top_k(uint64_t* E, int V, int top_k)
{
    if (top_k <= 0 || top_k >= V) return;
    uint64_t* key = (uint64_t*)malloc(sizeof(uint64_t) * V);
    for (int v = 0; v < V; v++) key[v] = om_top_k_key(E[v], v, V);
    qsort(key, (size_t)V, sizeof(uint64_t), cmp_desc_u64);
    const uint64_t K = key[top_k - 1];  /* the top_k-th largest key */
    for (int v = 0; v < V; v++)
        if (om_top_k_key(E[v], v, V) < K) E[v] = 0;
    free(key);
}

/* Top-p (nucleus) restriction after top-k: p24 = floor(top_p 2^24) in
 * 1..2^24 (2^24 keeps every token of nonzero weight).  In descending key
 * order, the smallest leading set whose weight A has A 2^24 >= p24 S (S the
 * total kept so far) is kept; the rest gets weight 0. */
OM_EXPORT uint32_t om_top_p24(float top_p)
{
    if (!(top_p < 1.0f)) return 1u << 24;
    const double x = (double)top_p * 16777216.0;
    return x < 1.0 ? 1u : (uint32_t)x;
}

typedef struct {
    uint64_t key;
    int v;
} keyed;

static int cmp_keyed_desc(const void* a, const void* b)
{
    const uint64_t x = ((const keyed*)a)->key, y = ((const keyed*)b)->key;
    return x < y ? 1 : (x > y ? -1 : 0);
}

static void keep_top_p(uint64_t* E, int V, uint32_t p24)
{
    if (p24 >= (1u << 24)) return;
    uint64_t S = 0;
    for (int v = 0; v < V; v++) S += E[v];
    if (S == 0) return;
    keyed* o = (keyed*)malloc(sizeof(keyed) * V);
    for (int v = 0; v < V; v++) {
        o[v].key = om_top_k_key(E[v], v, V);
        o[v].v = v;
    }
    qsort(o, (size_t)V, sizeof(keyed), cmp_keyed_desc);
    const unsigned __int128 target = (unsigned __int128)p24 * S;
    uint64_t A = 0;
    int i = 0;
    for (; i < V; i++) {
        A += E[o[i].v];
        if (((unsigned __int128)A << 24) >= target) break;
    }
    for (int j = i + 1; j < V; j++) E[o[j].v] = 0;
    free(o);
}

static uint64_t weights_tau(const float* z, int V, float tau, int top_k, uint32_t p24, uint64_t* E)
{
    float mx = z[0];
    for (int v = 1; v < V; v++)
        if (z[v] > mx) mx = z[v];
    for (int v = 0; v < V; v++) E[v] = om_sample_weight(z[v], mx, tau, V);
    keep_top_k(E, V, top_k);
    keep_top_p(E, V, p24);
    uint64_t S = 0;
    for (int v = 0; v < V; v++) S += E[v];
    return S;
}

static uint64_t uniform24(uint64_t* rng) { return om_splitmix64(rng) >> 40; }

/* U (S - R) < E 2^24 */
static int accepts(uint64_t U, uint64_t S, uint64_t R, uint64_t E)
{
    return (unsigned __int128)U * (S - R) < ((unsigned __int128)E << 24);
}

static int in_list(const int* a, int n, int x)
{
    for (int i = 0; i < n; i++)
        if (a[i] == x) return 1;
    return 0;
}

/* Draw with weights E (total S) restricted to the tokens not in
 * excl[0..ne-1] (whose weight is R), uniform U. */
static int draw_excluding(const uint64_t* E, int V, uint64_t S, const int* excl, int ne, uint64_t R, uint64_t U)
{
    const unsigned __int128 target = (unsigned __int128)U * (S - R);
    uint64_t acc = 0;
    int last = -1;
    for (int v = 0; v < V; v++) {
        if (in_list(excl, ne, v)) continue;
        if (E[v] > 0) last = v;
        acc += E[v];
        if (((unsigned __int128)acc << 24) > target) return v;
    }
    return last >= 0 ? last : 0;
}

/* n plain draws from softmax(z / tau), restricted to the top_k tokens when
 * top_k is in 1..V-1 (the primitive every sampled token goes through). */
OM_EXPORT void om_sample_logits(const float* z, int V, float tau, int top_k, float top_p, uint64_t* rng, int n,
                                int* out)
{
    uint64_t* E = (uint64_t*)malloc(sizeof(uint64_t) * V);
    const uint64_t S = weights_tau(z, V, tau, top_k, om_top_p24(top_p), E);
    for (int i = 0; i < n; i++) out[i] = draw_excluding(E, V, S, NULL, 0, 0, uniform24(rng));
    free(E);
}

/*
 * R10 + R6/R7 after the forward of the rows built by the last om_ctrl_rows
 * call.  logits: [T][V] of every row.  Verification by sampling (one uniform
 * per candidate try, one per drawn token, in the order below); the
 * lookahead branch's harvest and shift use the rows' argmaxes as in R6/R7.
 * Writes the emitted tokens and the rows whose KV is committed; returns m+1.
 */
OM_EXPORT int om_ctrl_advance_sample(om_ctrl* k, const float* logits, float tau, int top_k, float top_p,
                                     uint64_t* rng, int* emit, int* rows, int* gstar)
{
    const int V = k->V, n1 = k->N - 1, Gp = k->Gp;
    uint64_t* E = (uint64_t*)malloc(sizeof(uint64_t) * V);
    int* alive = (int*)malloc(sizeof(int) * (Gp > 0 ? Gp : 1));
    int* rej = (int*)malloc(sizeof(int) * (Gp > 0 ? Gp : 1));
    int* amax = (int*)malloc(sizeof(int) * k->T);
    for (int r = 0; r < k->T; r++) amax[r] = argmax_row(logits + (size_t)r * V, V);
    for (int g = 0; g < Gp; g++) alive[g] = 1;
    int row = 0, m = 0, g_best = -1, done = 0;
    rows[0] = 0;
    for (int i = 0; i < n1 && !done; i++) {
        const uint64_t S = weights_tau(logits + (size_t)row * V, V, tau, top_k, om_top_p24(top_p), E);
        int nrej = 0, acc_g = -1;
        uint64_t R = 0;
        for (int g = 0; g < Gp && acc_g < 0; g++) {
            if (!alive[g]) continue;
            const int v = k->cands[(size_t)g * n1 + i];
            if (in_list(rej, nrej, v)) continue;  /* a value already tried at this level */
            if (accepts(uniform24(rng), S, R, E[v])) {
                acc_g = g;
            } else {
                rej[nrej++] = v;
                R += E[v];
            }
        }
        if (acc_g < 0) {
            emit[m] = draw_excluding(E, V, S, rej, nrej, R, uniform24(rng));
            done = 1;
            break;
        }
        const int v = k->cands[(size_t)acc_g * n1 + i];
        emit[m] = v;
        for (int g = 0; g < Gp; g++)
            if (alive[g] && k->cands[(size_t)g * n1 + i] != v) alive[g] = 0;
        g_best = acc_g;  /* the lowest candidate still alive */
        row = row_vf(k, g_best, i);
        m++;
    }
    /* committed rows: row 0 and the accepted levels of the lowest candidate
     * alive at the end (every candidate alive at a level has the same
     * visible tokens there, so its rows hold the same keys and values) */
    for (int i = 0; i < m; i++) rows[i + 1] = row_vf(k, g_best, i);
    if (!done) {
        /* every level accepted: the bonus token from the last accepted row */
        const uint64_t S = weights_tau(logits + (size_t)row * V, V, tau, top_k, om_top_p24(top_p), E);
        emit[m] = draw_excluding(E, V, S, NULL, 0, 0, uniform24(rng));
    }
    if (gstar) *gstar = g_best;
    harvest_and_shift(k, amax);
    free(E); free(alive); free(rej); free(amax);
    return m + 1;
}

/* ---------------------------------------------------------------- lookahead */

/*
 * LA-oracle: lookahead decoding of max_new tokens.  steps_out receives the
 * number of steps, accept_hist (N+1 entries, may be NULL) counts steps by the
 * number of tokens they emitted.  Returns 0, or -1 on bad arguments.
 */
OM_EXPORT int om_lookahead(const om_model* m, const int* prompt, int len, int W, int N, int G,
                           uint64_t seed, int preseed, int variant, int max_new, int max_seq, int* out,
                           int* steps_out, int* accept_hist)
{
    if (len < 1 || max_new < 0) return -1;
    /* the farthest position a step touches is P + W + N - 2 */
    if (len - 1 + max_new + W + N > max_seq) return -1;
    om_ctrl* k = om_ctrl_new(W, N, G, m->vocab);
    om_seq* s = om_seq_new(m, max_seq);
    if (!k || !s || om_ctrl_set_variant(k, variant)) return -1;
    om_ctrl_init(k, prompt, len, seed, preseed);
    int rc = om_prefill(s, 0, prompt, len - 1);
    int Tmax = om_ctrl_rows_max(k);
    int* tok = (int*)malloc(sizeof(int) * Tmax);
    int* pos = (int*)malloc(sizeof(int) * Tmax);
    int* amax = (int*)malloc(sizeof(int) * Tmax);
    unsigned char* vis = (unsigned char*)malloc((size_t)Tmax * Tmax);
    int emit[64], rows[64];
    int c = prompt[len - 1], P = len - 1, n = 0, steps = 0;
    if (accept_hist) memset(accept_hist, 0, sizeof(int) * (N + 1));
    while (n < max_new && !rc) {
        int T = om_ctrl_rows(k, c, P, tok, pos, vis);
        rc = om_step_forward(s, P, T, tok, pos, vis, NULL, amax);
        if (rc) break;
        int ne = om_ctrl_advance(k, amax, emit, rows, NULL);
        rc = om_commit(s, P, ne, rows);
        for (int i = 0; i < ne && n < max_new; i++) out[n++] = emit[i];
        if (accept_hist) accept_hist[ne]++;
        P += ne;
        c = emit[ne - 1];
        steps++;
    }
    if (steps_out) *steps_out = steps;
    free(tok); free(pos); free(amax); free(vis);
    om_ctrl_free(k);
    om_seq_free(s);
    return rc;
}

/* ------------------------------------------------------ sampled decoding */

/* Plain ancestral sampling (the definition the sampled lookahead must match
 * in distribution): like om_greedy, with each token drawn from
 * softmax(logits / tau) by om_sample_logits' rule, one uniform per token from
 * the splitmix64 stream seeded with rng_seed. */
OM_EXPORT int om_sample_decode(const om_model* m, const int* prompt, int len, int max_new, int max_seq, float tau,
                               int top_k, float top_p, uint64_t rng_seed, int* out)
{
    if (len < 1 || max_new < 0 || len - 1 + max_new > max_seq || !(tau > 0.0f)) return -1;
    om_seq* s = om_seq_new(m, max_seq);
    if (!s) return -1;
    int rc = om_prefill(s, 0, prompt, len - 1);
    float* z = (float*)malloc(sizeof(float) * m->vocab);
    int c = prompt[len - 1], P = len - 1, a = 0;
    const unsigned char one = 1;
    uint64_t rng = rng_seed;
    for (int t = 0; t < max_new && !rc; t++) {
        rc = om_step_forward(s, P, 1, &c, &P, &one, z, &a);
        if (rc) break;
        const int row0 = 0;
        rc = om_commit(s, P, 1, &row0);
        om_sample_logits(z, m->vocab, tau, top_k, top_p, &rng, 1, &out[t]);
        c = out[t];
        P++;
    }
    free(z);
    om_seq_free(s);
    return rc;
}

/* Lookahead decoding with sampling verification (R10): as om_lookahead, the
 * verification drawing from softmax(logits / tau) with the splitmix64 stream
 * seeded with rng_seed. */
OM_EXPORT int om_lookahead_sample(const om_model* m, const int* prompt, int len, int W, int N, int G, uint64_t seed,
                                  int preseed, int variant, float tau, int top_k, float top_p, uint64_t rng_seed,
                                  int max_new, int max_seq, int* out, int* steps_out, int* accept_hist)
{
    if (len < 1 || max_new < 0 || !(tau > 0.0f)) return -1;
    if (len - 1 + max_new + W + N > max_seq) return -1;
    om_ctrl* k = om_ctrl_new(W, N, G, m->vocab);
    om_seq* s = om_seq_new(m, max_seq);
    if (!k || !s || om_ctrl_set_variant(k, variant)) return -1;
    om_ctrl_init(k, prompt, len, seed, preseed);
    int rc = om_prefill(s, 0, prompt, len - 1);
    int Tmax = om_ctrl_rows_max(k);
    int* tok = (int*)malloc(sizeof(int) * Tmax);
    int* pos = (int*)malloc(sizeof(int) * Tmax);
    int* amax = (int*)malloc(sizeof(int) * Tmax);
    float* logits = (float*)malloc(sizeof(float) * (size_t)Tmax * m->vocab);
    unsigned char* vis = (unsigned char*)malloc((size_t)Tmax * Tmax);
    int emit[64], rows[64];
    int c = prompt[len - 1], P = len - 1, n = 0, steps = 0;
    uint64_t rng = rng_seed;
    if (accept_hist) memset(accept_hist, 0, sizeof(int) * (N + 1));
    while (n < max_new && !rc) {
        int T = om_ctrl_rows(k, c, P, tok, pos, vis);
        rc = om_step_forward(s, P, T, tok, pos, vis, logits, amax);
        if (rc) break;
        int ne = om_ctrl_advance_sample(k, logits, tau, top_k, top_p, &rng, emit, rows, NULL);
        rc = om_commit(s, P, ne, rows);
        for (int i = 0; i < ne && n < max_new; i++) out[n++] = emit[i];
        if (accept_hist) accept_hist[ne]++;
        P += ne;
        c = emit[ne - 1];
        steps++;
    }
    if (steps_out) *steps_out = steps;
    free(tok); free(pos); free(amax); free(logits); free(vis);
    om_ctrl_free(k);
    om_seq_free(s);
    return rc;
}

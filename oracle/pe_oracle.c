/*
 * CPU oracle for the drafter forward pass of one P-EAGLE parallel-drafting round.
 *
 * TEST INFRASTRUCTURE ONLY.  This library exists to check the CUDA path: only
 * the test suite, the package's smoke check and the benchmark's CPU-baseline
 * leg load it.  It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes (P-EAGLE pages, "P-EAGLE architecture and mechanism",
 * step 2 "Parallel Drafting": every position goes through N transformer
 * layers and the language-model head in one pass, predicting t_1..t_K
 * together; "KV cache and CUDA Graphs": rejected tokens carry slot -1 and
 * write nothing to the cache).  The layer itself (fc from 2d to d, RMSNorm,
 * GQA attention with rotate-half RoPE over a paged cache, SwiGLU MLP) is the
 * drafter the workload statement names; the pages only say "N layers".
 *
 * Every value is computed from its plain definition in double precision:
 * each dot product is one sequential sum over its index, softmax subtracts
 * the maximum, nothing is blocked, fused or reordered beyond that.  Weights
 * and cache entries are read from their storage type (float32 or bf16 bit
 * patterns) and widened exactly to double.  Intermediate activations are NOT
 * rounded to the storage type.  Threads only split independent outputs.
 *
 * Parity status: the pages print no numeric example for any of these
 * functions, so every function here is "parity unpinned" by the pages; the
 * test suite pins each one to closed forms, special cases and invariants.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    int32_t n_rows;      /* rows handed to this call */
    int32_t d, n_q, n_kv, head_dim, ffn, vocab, n_layers, page_size, max_pages;
    int32_t storage;     /* 0: float32, 1: bf16 bit patterns (uint16) */
    double rms_eps, rope_theta;
    int32_t n_threads;   /* 0: all online cores */
} oc_config;

typedef struct {
    const void *fc;                 /* [d][2d] */
    const void *norm_final;         /* [d] */
    const void *lm_head;            /* [vocab][d] */
    const void *const *norm_attn;   /* [L] -> [d] */
    const void *const *wqkv;        /* [L] -> [(n_q+2n_kv)*hd][d] */
    const void *const *wo;          /* [L] -> [d][n_q*hd] */
    const void *const *norm_mlp;    /* [L] -> [d] */
    const void *const *w_gate_up;   /* [L] -> [2F][d] */
    const void *const *w_down;      /* [L] -> [d][F] */
} oc_weights;

/* ------------------------------------------------------------------ storage */

static double widen(const void *p, size_t i, int storage) {
    if (storage == 0) return (double)((const float *)p)[i];
    uint32_t u = (uint32_t)((const uint16_t *)p)[i] << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------ threads */

typedef void (*range_fn)(long begin, long end, void *ctx);
typedef struct { range_fn fn; void *ctx; long begin, end; } range_task;

static void *run_range(void *p) {
    range_task *t = (range_task *)p;
    if (t->begin < t->end) t->fn(t->begin, t->end, t->ctx);
    return NULL;
}

static int g_threads = 0;

static void parallel_for(long n, range_fn fn, void *ctx) {
    int nt = g_threads > 0 ? g_threads : (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nt < 1) nt = 1;
    if (nt > 256) nt = 256;
    if (n < nt) nt = (int)(n > 0 ? n : 1);
    pthread_t th[256];
    range_task task[256];
    for (int i = 0; i < nt; ++i) {
        task[i].fn = fn;
        task[i].ctx = ctx;
        task[i].begin = n * i / nt;
        task[i].end = n * (i + 1) / nt;
    }
    for (int i = 1; i < nt; ++i) pthread_create(&th[i], NULL, run_range, &task[i]);
    run_range(&task[0]);
    for (int i = 1; i < nt; ++i) pthread_join(th[i], NULL);
}

/* ------------------------------------------------------------------ linear: Y = X W^T */

typedef struct {
    const double *xT;   /* [in][n] : X transposed so that the row loop is contiguous */
    const void *W;      /* [out][in] storage */
    int storage, n, in_dim, out_dim;
    double *Y;          /* [n][out] */
} linear_ctx;

static void linear_range(long o0, long o1, void *p) {
    linear_ctx *c = (linear_ctx *)p;
    double *acc = (double *)malloc(sizeof(double) * (size_t)c->n);
    for (long o = o0; o < o1; ++o) {
        for (int i = 0; i < c->n; ++i) acc[i] = 0.0;
        /* Y[i][o] = sum_k X[i][k] * W[o][k], one sequential sum over k per (i, o) */
        for (int k = 0; k < c->in_dim; ++k) {
            double w = widen(c->W, (size_t)o * c->in_dim + k, c->storage);
            const double *xk = c->xT + (size_t)k * c->n;
            for (int i = 0; i < c->n; ++i) acc[i] += xk[i] * w;
        }
        for (int i = 0; i < c->n; ++i) c->Y[(size_t)i * c->out_dim + o] = acc[i];
    }
    free(acc);
}

/* Y[n][out] = X[n][in] . W[out][in]^T  (nn.Linear, no bias) */
void oc_linear(const double *X, int n, int in_dim, const void *W, int out_dim, int storage, double *Y) {
    double *xT = (double *)malloc(sizeof(double) * (size_t)n * in_dim + 8);
    for (int i = 0; i < n; ++i)
        for (int k = 0; k < in_dim; ++k) xT[(size_t)k * n + i] = X[(size_t)i * in_dim + k];
    linear_ctx c = {xT, W, storage, n, in_dim, out_dim, Y};
    parallel_for(out_dim, linear_range, &c);
    free(xT);
}

/* ------------------------------------------------------------------ elementwise ops */

/* RMSNorm: y = x / sqrt(mean(x^2) + eps) * g, row by row. */
void oc_rmsnorm(const double *x, int n, int d, const void *g, int storage, double eps, double *y) {
    for (int i = 0; i < n; ++i) {
        const double *xi = x + (size_t)i * d;
        double ss = 0.0;
        for (int j = 0; j < d; ++j) ss += xi[j] * xi[j];
        double inv = 1.0 / sqrt(ss / d + eps);
        for (int j = 0; j < d; ++j) y[(size_t)i * d + j] = xi[j] * inv * widen(g, (size_t)j, storage);
    }
}

/* Rotate-half rotary embedding of one head vector v[hd] at position pos:
 * pair (i, i + hd/2) rotated by angle pos * theta^(-2i/hd). */
void oc_rope(double *v, int hd, int pos, double theta) {
    int half = hd / 2;
    for (int i = 0; i < half; ++i) {
        double ang = (double)pos * pow(theta, -2.0 * i / hd);
        double c = cos(ang), s = sin(ang);
        double x1 = v[i], x2 = v[i + half];
        v[i] = x1 * c - x2 * s;
        v[i + half] = x2 * c + x1 * s;
    }
}

double oc_silu(double x) { return x / (1.0 + exp(-x)); }

/* Single-head softmax attention of query q over T keys/values:
 * out = sum_t softmax_t(q.k_t * scale) v_t.  K and V rows have stride hd. */
void oc_attend(const double *q, const double *K, const double *V, int T, int hd, double scale, double *out) {
    double *s = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    double m = -INFINITY;
    for (int t = 0; t < T; ++t) {
        double dot = 0.0;
        for (int e = 0; e < hd; ++e) dot += q[e] * K[(size_t)t * hd + e];
        s[t] = dot * scale;
        if (s[t] > m) m = s[t];
    }
    double l = 0.0;
    for (int t = 0; t < T; ++t) {
        s[t] = exp(s[t] - m);
        l += s[t];
    }
    for (int e = 0; e < hd; ++e) {
        double o = 0.0;
        for (int t = 0; t < T; ++t) o += s[t] * V[(size_t)t * hd + e];
        out[e] = T > 0 ? o / l : 0.0;
    }
    free(s);
}

/* ------------------------------------------------------------------ paged cache view */

/* This round's cache writes, kept in double: (slot, row) sorted by slot, values per row. */
typedef struct { int64_t slot; int32_t row; } slot_entry;

static int slot_cmp(const void *a, const void *b) {
    const slot_entry *x = (const slot_entry *)a, *y = (const slot_entry *)b;
    if (x->slot != y->slot) return x->slot < y->slot ? -1 : 1;
    return x->row < y->row ? -1 : (x->row > y->row);
}

/* Row whose write this round landed on `slot` (the last such row), or -1. */
static int written_row(const slot_entry *w, int nw, int64_t slot) {
    int lo = 0, hi = nw - 1, found = -1;
    while (lo <= hi) {
        int mid = (lo + hi) / 2;
        if (w[mid].slot < slot) lo = mid + 1;
        else if (w[mid].slot > slot) hi = mid - 1;
        else { found = mid; lo = mid + 1; }
    }
    return found < 0 ? -1 : w[found].row;
}

typedef struct {
    const oc_config *cfg;
    const double *q;          /* [n][n_q*hd], post-RoPE */
    const double *knew, *vnew;/* [n][n_kv*hd] this round's values */
    const slot_entry *w; int nw;
    const void *kc, *vc;      /* cache of this layer, storage type */
    const int32_t *position, *seq, *block_table;
    double *out;              /* [n][n_q*hd] */
    int err;
} attn_ctx;

static void attn_range(long i0, long i1, void *p) {
    attn_ctx *c = (attn_ctx *)p;
    const oc_config *cfg = c->cfg;
    int hd = cfg->head_dim, nkv = cfg->n_kv, group = cfg->n_q / cfg->n_kv, ps = cfg->page_size;
    for (long it = i0; it < i1; ++it) {
        int r = (int)(it / cfg->n_q), h = (int)(it % cfg->n_q);
        int g = h / group;                       /* GQA: q head h reads kv head h / (n_q/n_kv) */
        int T = c->position[r] + 1;              /* positions 0..p of the row's sequence */
        double *K = (double *)malloc(sizeof(double) * (size_t)T * hd);
        double *V = (double *)malloc(sizeof(double) * (size_t)T * hd);
        for (int t = 0; t < T; ++t) {
            int pi = t / ps;
            int32_t page = pi < cfg->max_pages ? c->block_table[(size_t)c->seq[r] * cfg->max_pages + pi] : -1;
            if (page < 0) { c->err = 1; page = 0; }
            int64_t slot = (int64_t)page * ps + t % ps;
            int wr = written_row(c->w, c->nw, slot);
            for (int e = 0; e < hd; ++e) {
                if (wr >= 0) {
                    K[(size_t)t * hd + e] = c->knew[(size_t)wr * nkv * hd + (size_t)g * hd + e];
                    V[(size_t)t * hd + e] = c->vnew[(size_t)wr * nkv * hd + (size_t)g * hd + e];
                } else {
                    size_t off = ((size_t)slot * nkv + g) * hd + e;
                    K[(size_t)t * hd + e] = widen(c->kc, off, cfg->storage);
                    V[(size_t)t * hd + e] = widen(c->vc, off, cfg->storage);
                }
            }
        }
        oc_attend(c->q + (size_t)r * cfg->n_q * hd + (size_t)h * hd, K, V, T, hd, 1.0 / sqrt((double)hd),
                  c->out + (size_t)r * cfg->n_q * hd + (size_t)h * hd);
        free(K);
        free(V);
    }
}

/* ------------------------------------------------------------------ forward */

/*
 * One drafter pass over n_rows rows.
 *   x0[n][2d]        concat(emb(token), hidden) per row
 *   position[n]      RoPE position and causal bound of each row
 *   slot[n]          cache slot written by the row (-1: no write)
 *   seq[n]           block-table row of the row's sequence
 *   block_table      [n_seq][max_pages] physical page ids
 *   k_cache/v_cache  [L] -> [num_pages][page][n_kv][hd], read only (this
 *                    round's writes are modelled in double on the side)
 *   draft_rows[n_draft]  rows scored by the LM head, logits[n_draft][vocab]
 *   new_k/new_v      optional [L][n][n_kv*hd]: post-RoPE k and v of every row
 *   x_out            optional [n][d]: residual stream after the last layer
 * Returns 0, or 1 when a row's causal range leaves its block table.
 */
int oc_forward(const oc_config *cfg, const oc_weights *W, const double *x0, const int32_t *position,
               const int64_t *slot, const int32_t *seq, const int32_t *block_table,
               const void *const *k_cache, const void *const *v_cache, int32_t n_draft,
               const int32_t *draft_rows, double *logits, double *new_k, double *new_v, double *x_out) {
    g_threads = cfg->n_threads;
    const int n = cfg->n_rows, d = cfg->d, hd = cfg->head_dim, st = cfg->storage;
    const int qd = cfg->n_q * hd, kvd = cfg->n_kv * hd, F = cfg->ffn;
    const int qkvd = qd + 2 * kvd;
    int err = 0;

    double *x = calloc((size_t)n * d + 1, sizeof(double));
    double *y = calloc((size_t)n * d + 1, sizeof(double));
    double *qkv = calloc((size_t)n * qkvd + 1, sizeof(double));
    double *q = calloc((size_t)n * qd + 1, sizeof(double));
    double *kn = calloc((size_t)n * kvd + 1, sizeof(double));
    double *vn = calloc((size_t)n * kvd + 1, sizeof(double));
    double *att = calloc((size_t)n * qd + 1, sizeof(double));
    double *tmp = calloc((size_t)n * d + 1, sizeof(double));
    double *gu = calloc((size_t)n * 2 * F + 1, sizeof(double));
    double *u = calloc((size_t)n * F + 1, sizeof(double));
    slot_entry *wlist = calloc((size_t)n + 1, sizeof(slot_entry));

    /* fc: x = X0 . W_fc^T  (2d -> d) */
    oc_linear(x0, n, 2 * d, W->fc, d, st, x);

    for (int l = 0; l < cfg->n_layers; ++l) {
        /* attention block (pre-norm) */
        oc_rmsnorm(x, n, d, W->norm_attn[l], st, cfg->rms_eps, y);
        oc_linear(y, n, d, W->wqkv[l], qkvd, st, qkv);
        for (int r = 0; r < n; ++r) {
            const double *src = qkv + (size_t)r * qkvd;
            memcpy(q + (size_t)r * qd, src, sizeof(double) * qd);
            memcpy(kn + (size_t)r * kvd, src + qd, sizeof(double) * kvd);
            memcpy(vn + (size_t)r * kvd, src + qd + kvd, sizeof(double) * kvd);
            for (int h = 0; h < cfg->n_q; ++h) oc_rope(q + (size_t)r * qd + (size_t)h * hd, hd, position[r], cfg->rope_theta);
            for (int g = 0; g < cfg->n_kv; ++g) oc_rope(kn + (size_t)r * kvd + (size_t)g * hd, hd, position[r], cfg->rope_theta);
        }
        /* cache write before attention, skipped for slot -1 */
        int nw = 0;
        for (int r = 0; r < n; ++r)
            if (slot[r] >= 0) { wlist[nw].slot = slot[r]; wlist[nw].row = r; ++nw; }
        qsort(wlist, (size_t)nw, sizeof(slot_entry), slot_cmp);
        if (new_k) memcpy(new_k + (size_t)l * n * kvd, kn, sizeof(double) * (size_t)n * kvd);
        if (new_v) memcpy(new_v + (size_t)l * n * kvd, vn, sizeof(double) * (size_t)n * kvd);

        attn_ctx ac = {cfg, q, kn, vn, wlist, nw, k_cache[l], v_cache[l], position, seq, block_table, att, 0};
        parallel_for((long)n * cfg->n_q, attn_range, &ac);
        if (ac.err) err = 1;

        oc_linear(att, n, qd, W->wo[l], d, st, tmp);
        for (size_t i = 0; i < (size_t)n * d; ++i) x[i] += tmp[i];

        /* MLP block (pre-norm, SwiGLU) */
        oc_rmsnorm(x, n, d, W->norm_mlp[l], st, cfg->rms_eps, y);
        oc_linear(y, n, d, W->w_gate_up[l], 2 * F, st, gu);
        for (int r = 0; r < n; ++r)
            for (int f = 0; f < F; ++f)
                u[(size_t)r * F + f] = oc_silu(gu[(size_t)r * 2 * F + f]) * gu[(size_t)r * 2 * F + F + f];
        oc_linear(u, n, F, W->w_down[l], d, st, tmp);
        for (size_t i = 0; i < (size_t)n * d; ++i) x[i] += tmp[i];
    }
    if (x_out) memcpy(x_out, x, sizeof(double) * (size_t)n * d);

    /* final norm + LM head on the draft rows only */
    double *xd = calloc((size_t)n_draft * d + 1, sizeof(double));
    double *yd = calloc((size_t)n_draft * d + 1, sizeof(double));
    for (int i = 0; i < n_draft; ++i) memcpy(xd + (size_t)i * d, x + (size_t)draft_rows[i] * d, sizeof(double) * d);
    oc_rmsnorm(xd, n_draft, d, W->norm_final, st, cfg->rms_eps, yd);
    oc_linear(yd, n_draft, d, W->lm_head, cfg->vocab, st, logits);

    free(xd); free(yd);
    free(x); free(y); free(qkv); free(q); free(kn); free(vn); free(att); free(tmp); free(gu); free(u); free(wlist);
    return err;
}

/* Thread count used by the last call (0 = all cores), for reporting. */
int oc_threads_used(void) {
    int nt = g_threads > 0 ? g_threads : (int)sysconf(_SC_NPROCESSORS_ONLN);
    return nt < 1 ? 1 : (nt > 256 ? 256 : nt);
}

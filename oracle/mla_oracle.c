/*
 * MLA oracle: plain, slow, fp64 CPU implementation of weight-absorbed
 * Multi-head Latent Attention decode over a paged latent cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is compiled into liboracle.so and is
 * loaded exclusively by the test-suite, by the smoke check and by the timed
 * CPU-baseline leg of the benchmark.  The CUDA library never links, loads or
 * calls it, and it shares no code, header, table or constant with the CUDA
 * library.
 *
 * Source: "DeepSeek-V2" explainer (aiany.app), Steps 5-8, and the DeepSeek-V2
 * breakdown (edtech.ai360xpert.com), "How It Works":
 *   - Step 5: a token is cached only as its latent c (512 numbers); per-head
 *     keys and values are regenerated as k = W^UK c and v = W^UV c.
 *   - Step 6: score = q . (W^UK c) = (W^UK^T q) . c  (associativity: the key
 *     is never built; "absorbing" W^UK into the query side).
 *   - Step 7: decoupled RoPE: per head a 64-d query q^R, per token one shared
 *     64-d rotated key k^R; the content and position scores add inside the
 *     softmax.
 *   - Step 8: the cache row is 512 + 64 = 576 numbers per token per layer.
 *
 * Conventions (readings where the pages are silent):
 *   - A cache row is [c (d_c) | k^R (d_r)]; rows live in pages of `page`
 *     tokens; logical page p of sequence b is physical page block_table[b,p].
 *   - W_UK[h] and W_UV[h] are d_h x d_c, row-major: k[d] = sum_c W_UK[h][d][c] c[c].
 *   - s_j = scale * (q . k_j); softmax over the visible tokens; lse is the
 *     natural log of sum_j exp(s_j).  No visible token: o = 0, lse = -inf.
 *   - causal with Tq query tokens: the Tq new tokens are already in the cache;
 *     query t sees tokens 0 .. L_b - Tq + t (bottom-right aligned).
 *
 * Inputs are float (every bf16 value is exact in float); all arithmetic and
 * every output is double.  No blocking, no fusion: each function is the
 * definition written out, loop by loop.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Work splitting over independent (b, t, h) problems.                       */
/* ------------------------------------------------------------------------ */

typedef void (*task_fn)(void *ctx, long idx);

typedef struct {
    task_fn fn;
    void *ctx;
    long n;
    long next;
    pthread_mutex_t lock;
} pool_t;

static void *pool_worker(void *arg) {
    pool_t *p = (pool_t *)arg;
    for (;;) {
        long i;
        pthread_mutex_lock(&p->lock);
        i = p->next++;
        pthread_mutex_unlock(&p->lock);
        if (i >= p->n) break;
        p->fn(p->ctx, i);
    }
    return NULL;
}

static void run_tasks(task_fn fn, void *ctx, long n, int nthreads) {
    pool_t p;
    p.fn = fn;
    p.ctx = ctx;
    p.n = n;
    p.next = 0;
    pthread_mutex_init(&p.lock, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 512) nthreads = 512;
    if (nthreads == 1) {
        pool_worker(&p);
    } else {
        pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
        int started = 0;
        for (int i = 0; i < nthreads; ++i)
            if (pthread_create(&th[i], NULL, pool_worker, &p) == 0) ++started;
        if (started == 0) pool_worker(&p);
        for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
        free(th);
    }
    pthread_mutex_destroy(&p.lock);
}

/* Number of cache tokens query t of sequence b may look at. */
static long visible_tokens(long L, int Tq, int t, int causal) {
    if (!causal) return L;
    long n = L - (long)(Tq - 1 - t);
    return n < 0 ? 0 : n;
}

/* Address of cache row j (token j) of sequence b. */
static const float *cache_row(const float *pool, const int32_t *block_table, int b,
                              int max_pages, int page, int row_width, long j) {
    long p = block_table[(long)b * max_pages + j / page];
    return pool + (p * page + j % page) * (long)row_width;
}

/* ------------------------------------------------------------------------ */
/* Absorption (Step 6): q_abs[n,h,:d_c] = W_UK[h]^T q_nope[n,h,:],           */
/* q_abs[n,h,d_c:] = q_rope[n,h,:]  (Step 7: the position channel is passed   */
/* through, it cannot be absorbed).                                           */
/* ------------------------------------------------------------------------ */
void oracle_absorb_q(const float *q_nope, const float *q_rope, const float *w_uk,
                     int N, int H, int d_h, int d_c, int d_r, double *q_abs) {
    int D = d_c + d_r;
    for (int n = 0; n < N; ++n)
        for (int h = 0; h < H; ++h) {
            const float *qn = q_nope + ((long)n * H + h) * d_h;
            const float *W = w_uk + (long)h * d_h * d_c;
            double *out = q_abs + ((long)n * H + h) * D;
            for (int c = 0; c < d_c; ++c) {
                double acc = 0.0;
                for (int d = 0; d < d_h; ++d) acc += (double)W[(long)d * d_c + c] * (double)qn[d];
                out[c] = acc;
            }
            for (int r = 0; r < d_r; ++r) out[d_c + r] = (double)q_rope[((long)n * H + h) * d_r + r];
        }
}

/* ------------------------------------------------------------------------ */
/* Up-projection (Step 5 / Step 6): out[n,h,:] = W_UV[h] o_lat[n,h,:].        */
/* ------------------------------------------------------------------------ */
void oracle_up_proj(const double *o_lat, const float *w_uv, int N, int H, int d_h, int d_c,
                    double *out) {
    for (int n = 0; n < N; ++n)
        for (int h = 0; h < H; ++h) {
            const double *o = o_lat + ((long)n * H + h) * d_c;
            const float *W = w_uv + (long)h * d_h * d_c;
            for (int d = 0; d < d_h; ++d) {
                double acc = 0.0;
                for (int c = 0; c < d_c; ++c) acc += (double)W[(long)d * d_c + c] * o[c];
                out[((long)n * H + h) * d_h + d] = acc;
            }
        }
}

/* ------------------------------------------------------------------------ */
/* Absorbed decode (Steps 6-8): per (b, t, h)                                 */
/*   s_j   = scale * q_abs[b,t,h,:] . row_j          (576-wide dot)           */
/*   p_j   = exp(s_j - max s) / sum_k exp(s_k - max s)                        */
/*   o_lat = sum_j p_j c_j                            (c_j = row_j[:d_c])      */
/*   lse   = max s + log sum_k exp(s_k - max s)                               */
/* ------------------------------------------------------------------------ */
typedef struct {
    const float *q_abs;   /* [B,Tq,H,D] */
    const double *q_abs64;/* alternative double query (fused path) or NULL */
    const float *pool;
    const int32_t *block_table;
    const int32_t *seq_lens;
    int B, Tq, H, d_c, d_r, page, max_pages, causal;
    double scale;
    double *o_lat;        /* [B,Tq,H,d_c] */
    double *lse;          /* [B,Tq,H] */
} absorbed_ctx;

static void absorbed_task(void *vctx, long idx) {
    absorbed_ctx *c = (absorbed_ctx *)vctx;
    int D = c->d_c + c->d_r;
    int h = (int)(idx % c->H);
    int t = (int)((idx / c->H) % c->Tq);
    int b = (int)(idx / ((long)c->H * c->Tq));
    long n = visible_tokens(c->seq_lens[b], c->Tq, t, c->causal);
    double *o = c->o_lat + idx * c->d_c;
    for (int k = 0; k < c->d_c; ++k) o[k] = 0.0;
    if (n <= 0) {
        c->lse[idx] = -INFINITY;
        return;
    }
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    const float *q32 = c->q_abs ? c->q_abs + idx * D : NULL;
    const double *q64 = c->q_abs64 ? c->q_abs64 + idx * D : NULL;
    double m = -INFINITY;
    for (long j = 0; j < n; ++j) {
        const float *row = cache_row(c->pool, c->block_table, b, c->max_pages, c->page, D, j);
        double dot = 0.0;
        for (int k = 0; k < D; ++k) dot += (q64 ? q64[k] : (double)q32[k]) * (double)row[k];
        s[j] = c->scale * dot;
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (long j = 0; j < n; ++j) {
        s[j] = exp(s[j] - m);
        l += s[j];
    }
    for (long j = 0; j < n; ++j) {
        const float *row = cache_row(c->pool, c->block_table, b, c->max_pages, c->page, D, j);
        double p = s[j] / l;
        for (int k = 0; k < c->d_c; ++k) o[k] += p * (double)row[k];
    }
    c->lse[idx] = m + log(l);
    free(s);
}

void oracle_decode_absorbed(const float *q_abs, const double *q_abs64, const float *pool,
                            const int32_t *block_table, const int32_t *seq_lens, int B, int Tq,
                            int H, int d_c, int d_r, int page, int max_pages, double scale,
                            int causal, int nthreads, double *o_lat, double *lse) {
    absorbed_ctx c;
    c.q_abs = q_abs;
    c.q_abs64 = q_abs64;
    c.pool = pool;
    c.block_table = block_table;
    c.seq_lens = seq_lens;
    c.B = B;
    c.Tq = Tq;
    c.H = H;
    c.d_c = d_c;
    c.d_r = d_r;
    c.page = page;
    c.max_pages = max_pages;
    c.causal = causal;
    c.scale = scale;
    c.o_lat = o_lat;
    c.lse = lse;
    run_tasks(absorbed_task, &c, (long)B * Tq * H, nthreads);
}

/* ------------------------------------------------------------------------ */
/* Naive form (Steps 2, 5, 7): rebuild the per-head key and value of every   */
/* cached token and run ordinary multi-head attention:                        */
/*   K_j = [W_UK[h] c_j | k^R_j]   (d_h + d_r)                                */
/*   V_j =  W_UV[h] c_j            (d_h)                                      */
/*   Q   = [q_nope | q_rope]                                                  */
/*   out = softmax_j(scale * Q.K_j) V_j,  lse as above.                       */
/* ------------------------------------------------------------------------ */
typedef struct {
    const float *q_nope, *q_rope, *w_uk, *w_uv, *pool;
    const int32_t *block_table, *seq_lens;
    int B, Tq, H, d_h, d_c, d_r, page, max_pages, causal;
    double scale;
    double *out, *lse;
} naive_ctx;

static void naive_task(void *vctx, long idx) {
    naive_ctx *c = (naive_ctx *)vctx;
    int D = c->d_c + c->d_r;
    int h = (int)(idx % c->H);
    int t = (int)((idx / c->H) % c->Tq);
    int b = (int)(idx / ((long)c->H * c->Tq));
    long n = visible_tokens(c->seq_lens[b], c->Tq, t, c->causal);
    double *out = c->out + idx * c->d_h;
    for (int d = 0; d < c->d_h; ++d) out[d] = 0.0;
    if (n <= 0) {
        c->lse[idx] = -INFINITY;
        return;
    }
    const float *qn = c->q_nope + idx * c->d_h;
    const float *qr = c->q_rope + idx * c->d_r;
    const float *Wk = c->w_uk + (long)h * c->d_h * c->d_c;
    const float *Wv = c->w_uv + (long)h * c->d_h * c->d_c;
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    double *kv = (double *)malloc(sizeof(double) * (size_t)c->d_h);
    double m = -INFINITY;
    for (long j = 0; j < n; ++j) {
        const float *row = cache_row(c->pool, c->block_table, b, c->max_pages, c->page, D, j);
        /* content key k = W_UK[h] c_j */
        for (int d = 0; d < c->d_h; ++d) {
            double acc = 0.0;
            for (int k = 0; k < c->d_c; ++k) acc += (double)Wk[(long)d * c->d_c + k] * (double)row[k];
            kv[d] = acc;
        }
        double dot = 0.0;
        for (int d = 0; d < c->d_h; ++d) dot += (double)qn[d] * kv[d];
        for (int r = 0; r < c->d_r; ++r) dot += (double)qr[r] * (double)row[c->d_c + r];
        s[j] = c->scale * dot;
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (long j = 0; j < n; ++j) {
        s[j] = exp(s[j] - m);
        l += s[j];
    }
    for (long j = 0; j < n; ++j) {
        const float *row = cache_row(c->pool, c->block_table, b, c->max_pages, c->page, D, j);
        /* value v = W_UV[h] c_j */
        double p = s[j] / l;
        for (int d = 0; d < c->d_h; ++d) {
            double acc = 0.0;
            for (int k = 0; k < c->d_c; ++k) acc += (double)Wv[(long)d * c->d_c + k] * (double)row[k];
            out[d] += p * acc;
        }
    }
    c->lse[idx] = m + log(l);
    free(kv);
    free(s);
}

void oracle_decode_naive(const float *q_nope, const float *q_rope, const float *w_uk,
                         const float *w_uv, const float *pool, const int32_t *block_table,
                         const int32_t *seq_lens, int B, int Tq, int H, int d_h, int d_c, int d_r,
                         int page, int max_pages, double scale, int causal, int nthreads,
                         double *out, double *lse) {
    naive_ctx c;
    c.q_nope = q_nope;
    c.q_rope = q_rope;
    c.w_uk = w_uk;
    c.w_uv = w_uv;
    c.pool = pool;
    c.block_table = block_table;
    c.seq_lens = seq_lens;
    c.B = B;
    c.Tq = Tq;
    c.H = H;
    c.d_h = d_h;
    c.d_c = d_c;
    c.d_r = d_r;
    c.page = page;
    c.max_pages = max_pages;
    c.causal = causal;
    c.scale = scale;
    c.out = out;
    c.lse = lse;
    run_tasks(naive_task, &c, (long)B * Tq * H, nthreads);
}

/* ------------------------------------------------------------------------ */
/* Merging attention over disjoint token sets.  If o_i, lse_i are the        */
/* softmax-weighted output and log-sum-exp over token set i, the result over  */
/* the union is lse = log sum_i exp(lse_i), o = sum_i exp(lse_i - lse) o_i.   */
/* This follows from the softmax definition (the partial sums of exp(s_j)    */
/* are exp(lse_i)); sets with lse_i = -inf carry weight 0.                    */
/*   o_parts [R, M, d], lse_parts [R, M] -> o [M, d], lse [M]                 */
/* ------------------------------------------------------------------------ */
void oracle_combine(const double *o_parts, const double *lse_parts, int R, long M, int d,
                    double *o, double *lse) {
    for (long i = 0; i < M; ++i) {
        double mx = -INFINITY;
        for (int r = 0; r < R; ++r)
            if (lse_parts[(long)r * M + i] > mx) mx = lse_parts[(long)r * M + i];
        for (int k = 0; k < d; ++k) o[i * d + k] = 0.0;
        if (mx == -INFINITY) {
            lse[i] = -INFINITY;
            continue;
        }
        double tot = 0.0;
        for (int r = 0; r < R; ++r) tot += exp(lse_parts[(long)r * M + i] - mx);
        double L = mx + log(tot);
        for (int r = 0; r < R; ++r) {
            double w = exp(lse_parts[(long)r * M + i] - L);
            for (int k = 0; k < d; ++k) o[i * d + k] += w * o_parts[((long)r * M + i) * d + k];
        }
        lse[i] = L;
    }
}

/* ------------------------------------------------------------------------ */
/* Cache write for new tokens.                                               */
/* ------------------------------------------------------------------------ */

/*
 * Rotary position embedding of one vector ("DeepSeek-V2" explainer, Step 7:
 * order is encoded by turning each query and key through an angle that grows
 * in proportion to the token's position, so that a query-key score depends
 * only on their distance).  The pages give no formula; the reading taken:
 *   - coordinates (2i, 2i+1) form pair i, i = 0 .. d/2 - 1;
 *   - pair i turns counter-clockwise by pos * theta_i,
 *     theta_i = base^(-2i/d), base given by the caller (10000 by default);
 *   - out[2i]   = x[2i] cos(a) - x[2i+1] sin(a)
 *     out[2i+1] = x[2i] sin(a) + x[2i+1] cos(a),   a = pos * theta_i.
 * `pos` is a double so that tests can place a vector at any angle.
 */
void oracle_rope(const double *x, double pos, int d, double base, double *out) {
    for (int i = 0; i < d / 2; ++i) {
        const double theta = pow(base, -2.0 * (double)i / (double)d);
        const double a = pos * theta;
        const double c = cos(a), s = sin(a);
        const double x0 = x[2 * i], x1 = x[2 * i + 1];
        out[2 * i] = x0 * c - x1 * s;
        out[2 * i + 1] = x0 * s + x1 * c;
    }
}

/*
 * The cache row of each new token (explainer Step 5, the paper's equation 9:
 * the hidden vector h is projected down to the latent c = W^DKV h; Step 7:
 * the token's one shared position key is k^R = RoPE(W^KR h); Step 8: the row
 * kept per token is [c | k^R], d_c + d_r numbers) and the pool row it is
 * written to.
 *   h        [B*Tq, d_model]  the new tokens, sequence-major
 *   w_dkv    [d_c, d_model]   row-major: c[r] = sum_k w_dkv[r][k] h[k]
 *   w_kr     [d_r, d_model]   row-major, likewise for the unrotated k^R
 *   block_table [B, max_pages], seq_lens [B]: the lengths already count the
 *            Tq new tokens, so token t of sequence b has position
 *            p = seq_lens[b] - Tq + t, the same convention as the causal
 *            decode above.
 * Outputs: rows [B*Tq, d_c + d_r] (the row values, double) and slot [B*Tq],
 * the pool row block_table[b, p / page] * page + p % page, or -1 where p is
 * negative or beyond the block table, or the table entry is outside
 * [0, num_pages).
 */
void oracle_cache_append(const float *h, const float *w_dkv, const float *w_kr, const int32_t *block_table,
                         const int32_t *seq_lens, int B, int Tq, int d_model, int d_c, int d_r, int page,
                         int max_pages, int num_pages, double rope_base, double *rows, int64_t *slot) {
    const int D = d_c + d_r;
    double *kr = (double *)malloc(sizeof(double) * (size_t)(d_r > 0 ? d_r : 1));
    for (int b = 0; b < B; ++b) {
        for (int t = 0; t < Tq; ++t) {
            const long n = (long)b * Tq + t;
            const float *x = h + (size_t)n * d_model;
            double *row = rows + (size_t)n * D;
            /* c = W^DKV h */
            for (int r = 0; r < d_c; ++r) {
                double acc = 0.0;
                for (int k = 0; k < d_model; ++k) acc += (double)w_dkv[(size_t)r * d_model + k] * (double)x[k];
                row[r] = acc;
            }
            /* k^R = RoPE(W^KR h) at the token's position */
            for (int r = 0; r < d_r; ++r) {
                double acc = 0.0;
                for (int k = 0; k < d_model; ++k) acc += (double)w_kr[(size_t)r * d_model + k] * (double)x[k];
                kr[r] = acc;
            }
            const long p = (long)seq_lens[b] - Tq + t;
            oracle_rope(kr, (double)p, d_r, rope_base, row + d_c);
            /* where the row goes */
            slot[n] = -1;
            if (p >= 0 && p / page < max_pages) {
                const int32_t pg = block_table[(size_t)b * max_pages + p / page];
                if (pg >= 0 && pg < num_pages) slot[n] = (int64_t)pg * page + p % page;
            }
        }
    }
    free(kr);
}

/* ------------------------------------------------------------------------ */
/* Token-level compression of the cache.                                     */
/* ------------------------------------------------------------------------ */

/*
 * Merge blocks of m consecutive cache rows into one row each (the DeepSeek
 * page's "KV cache compression" section, the token-level compression of V4:
 * the merged key-value vector is a component-wise weighted sum of the m
 * tokens' vectors, the weights a softmax over the m tokens taken separately
 * for every component of z = W^Z x):
 *   out[g][k] = sum_i w[g*m+i][k] * rows[g*m+i][k],
 *   w[g*m+i][k] = exp(z[g*m+i][k]) / sum_j exp(z[g*m+j][k]).
 * rows, z: [n_blocks * m, D]; out: [n_blocks, D].  The softmax is taken about
 * the block's largest z of the component (which does not change it).
 */
void oracle_compress(const double *rows, const double *z, long n_blocks, int m, int D, double *out) {
    for (long g = 0; g < n_blocks; ++g) {
        for (int k = 0; k < D; ++k) {
            double mx = -INFINITY;
            for (int i = 0; i < m; ++i) {
                const double v = z[((size_t)g * m + i) * D + k];
                if (v > mx) mx = v;
            }
            double den = 0.0, num = 0.0;
            for (int i = 0; i < m; ++i) {
                const double e = exp(z[((size_t)g * m + i) * D + k] - mx);
                den += e;
                num += e * rows[((size_t)g * m + i) * D + k];
            }
            out[(size_t)g * D + k] = num / den;
        }
    }
}

/*
 * The compressed cache write: nb new compressed rows per sequence, each the
 * merge of m new tokens.  Token rows are the cache write's (c = W^DKV h,
 * k^R = RoPE(W^KR h) at the token's own position, row = [c | k^R]); their
 * weights come from z = W^Z h (w_z: [d_c + d_r, d_model], row-major).
 * seq_lens counts compressed rows and already includes the nb new ones, so
 * the j-th new row of sequence b is compressed position P = seq_lens[b] - nb + j,
 * merges the tokens at positions P*m .. P*m + m - 1 (h rows (b*nb + j)*m + i),
 * and goes to pool row block_table[b, P / page] * page + P % page (slot -1 when
 * invalid, as for the plain cache write).
 * Outputs: rows [B*nb, D] (merged), slot [B*nb].
 */
void oracle_cache_append_compressed(const float *h, const float *w_dkv, const float *w_kr, const float *w_z,
                                    const int32_t *block_table, const int32_t *seq_lens, int B, int nb, int m,
                                    int d_model, int d_c, int d_r, int page, int max_pages, int num_pages,
                                    double rope_base, double *rows, int64_t *slot) {
    const int D = d_c + d_r;
    double *tok = (double *)malloc(sizeof(double) * (size_t)m * D);
    double *zz = (double *)malloc(sizeof(double) * (size_t)m * D);
    double *kr = (double *)malloc(sizeof(double) * (size_t)(d_r > 0 ? d_r : 1));
    for (int b = 0; b < B; ++b) {
        for (int j = 0; j < nb; ++j) {
            const long P = (long)seq_lens[b] - nb + j;
            const long g = (long)b * nb + j;
            for (int i = 0; i < m; ++i) {
                const float *x = h + ((size_t)g * m + i) * d_model;
                double *row = tok + (size_t)i * D;
                for (int r = 0; r < d_c; ++r) {
                    double acc = 0.0;
                    for (int k = 0; k < d_model; ++k) acc += (double)w_dkv[(size_t)r * d_model + k] * (double)x[k];
                    row[r] = acc;
                }
                for (int r = 0; r < d_r; ++r) {
                    double acc = 0.0;
                    for (int k = 0; k < d_model; ++k) acc += (double)w_kr[(size_t)r * d_model + k] * (double)x[k];
                    kr[r] = acc;
                }
                oracle_rope(kr, (double)(P * m + i), d_r, rope_base, row + d_c);
                for (int r = 0; r < D; ++r) {
                    double acc = 0.0;
                    for (int k = 0; k < d_model; ++k) acc += (double)w_z[(size_t)r * d_model + k] * (double)x[k];
                    zz[(size_t)i * D + r] = acc;
                }
            }
            oracle_compress(tok, zz, 1, m, D, rows + (size_t)g * D);
            slot[g] = -1;
            if (P >= 0 && P / page < max_pages) {
                const int32_t pg = block_table[(size_t)b * max_pages + P / page];
                if (pg >= 0 && pg < num_pages) slot[g] = (int64_t)pg * page + P % page;
            }
        }
    }
    free(tok);
    free(zz);
    free(kr);
}

/* ------------------------------------------------------------------------ */
/* Indexer: top-k sparse decode.                                             */
/* ------------------------------------------------------------------------ */

/*
 * Index scores (the DeepSeek page's "KV cache data movement minimization"
 * section: every cached vector also has a small index vector; a decoding
 * token scores all of them, keeps the top k, and attends over those tokens
 * only).  s[b][t] = q_idx[b] . k_idx(b, t) for t < seq_lens[b], where
 * k_idx(b, t) = idx_pool[block_table[b, t / page], t % page, :] (d_idx wide);
 * entries t >= seq_lens[b] are left untouched.  scores: [B, max_len].
 */
void oracle_index_scores(const float *q_idx, const float *idx_pool, const int32_t *block_table,
                         const int32_t *seq_lens, int B, int d_idx, int page, int max_pages, long max_len,
                         double *scores) {
    for (int b = 0; b < B; ++b) {
        const long L = seq_lens[b];
        for (long t = 0; t < L && t < max_len; ++t) {
            const float *k = idx_pool + ((size_t)block_table[(size_t)b * max_pages + t / page] * page + t % page) * d_idx;
            double acc = 0.0;
            for (int d = 0; d < d_idx; ++d) acc += (double)q_idx[(size_t)b * d_idx + d] * (double)k[d];
            scores[(size_t)b * max_len + t] = acc;
        }
    }
}

/*
 * Top k of one row of n scores (the "TopK" of the indexer method): the k
 * largest, ties broken by the lower index, returned in ascending index order
 * (k >= n: every index).  A NaN score ranks below every number, -inf included.
 * A plain selection: repeatedly take the best remaining entry.  Returns the count.
 */
static int cmp_long(const void *a, const void *b) {
    const long x = *(const long *)a, y = *(const long *)b;
    return (x > y) - (x < y);
}
static int ranks_above(double a, double b) {
    if (isnan(a)) return 0;
    if (isnan(b)) return 1;
    return a > b;
}
long oracle_topk_row(const double *s, long n, long k, long *out) {
    const long take = k < n ? (k > 0 ? k : 0) : n;
    char *used = (char *)calloc((size_t)(n > 0 ? n : 1), 1);
    for (long j = 0; j < take; ++j) {
        long best = -1;
        for (long t = 0; t < n; ++t) {
            if (used[t]) continue;
            if (best < 0 || ranks_above(s[t], s[best])) best = t;  /* strict: the lowest index wins ties */
        }
        used[best] = 1;
        out[j] = best;
    }
    free(used);
    qsort(out, (size_t)take, sizeof(long), cmp_long);
    return take;
}

/*
 * The value of one FP8 E4M3 code (the OCP 8-bit floating-point format's E4M3 variant, as used
 * for low-bit caches): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field
 * 0 holds the subnormals m/8 * 2^-6; S.1111.111 is NaN and there is no infinity, so
 * S.1111.110 = 448 is the largest magnitude.
 */
double oracle_e4m3_value(uint8_t code) {
    const int sign = code >> 7, e = (code >> 3) & 0xF, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    const double mag = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/*
 * Index scores over an e4m3 index cache with one scale per cached token (the indexer of the
 * DeepSeek page's "KV cache data movement minimization" section, with its index vectors held
 * in 8 bits): s[b][t] = scale(b, t) * sum_d q_idx[b][d] * value(code(b, t, d)), where
 * code(b, t, :) = idx_codes[block_table[b, t / page], t % page, :] and scale(b, t) is the
 * scale array's entry at the same place.  Entries t >= seq_lens[b] are left untouched.
 */
void oracle_index_scores_e4m3(const float *q_idx, const uint8_t *idx_codes, const float *idx_scale,
                              const int32_t *block_table, const int32_t *seq_lens, int B, int d_idx, int page,
                              int max_pages, long max_len, double *scores) {
    for (int b = 0; b < B; ++b) {
        const long L = seq_lens[b];
        for (long t = 0; t < L && t < max_len; ++t) {
            const size_t slot = (size_t)block_table[(size_t)b * max_pages + t / page] * page + t % page;
            const uint8_t *k = idx_codes + slot * d_idx;
            double acc = 0.0;
            for (int d = 0; d < d_idx; ++d) acc += (double)q_idx[(size_t)b * d_idx + d] * oracle_e4m3_value(k[d]);
            scores[(size_t)b * max_len + t] = (double)idx_scale[slot] * acc;
        }
    }
}

/*
 * CPU oracle for block-sparse attention forward -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct statement of what the block-sparse forward
 * computes, in fp64.  Only the tests, the smoke check and the benchmark's CPU
 * baseline may load it; the product path (the CUDA library) never does, and the
 * two share no code, header, table or helper.
 *
 * Sources (page titles, with the part of each page that defines the step):
 *  [VARLEN]  "[CuTe,Flex] varlen blocksparsity", flash-attention pull request
 *            #2224, description: batched metadata *_block_cnt [B,H,num_m] and
 *            *_block_idx [B,H,num_m,num_n]; varlen metadata packed as
 *            [H,total_m_blocks] / [H,total_n_blocks] with
 *            num_m(b) = ceildiv(seqlen_q[b], tile_m), num_n(b) = ceildiv(seqlen_k[b], tile_n),
 *            total_m_blocks = sum num_m(b), total_n_blocks = sum num_m(b)*num_n(b);
 *            review thread: the metadata tuple is (mask_block_cnt, mask_block_idx,
 *            full_block_cnt, full_block_idx); cu_block_idx_offsets is the
 *            cumulative sum of num_m(b)*num_n(b); mask_mod applies to mask blocks.
 *  [LIST]    "Dense FlashAttention vs Block-Sparse Attention" (learning note on
 *            Block-Sparse-Attention), section 2: a boolean block row becomes a
 *            reversed index list padded with -1, e.g. [1,0,0,1,0,1] -> [5,3,0,-1,-1,-1].
 *  [VSA]     "[feat] VSA-256 fastpath on Blackwell via FA4 CuTe block-sparse
 *            attention" (FastVideo #1354), review: mask_mod reads a per-KV-block
 *            valid length; tokens at or past it inside the block are masked.
 *
 * Readings where the pages leave a step open (each is also listed in the design
 * notes):
 *  - a selected block is classified by the token predicate over its tile:
 *    true everywhere -> full list, true somewhere -> mask list, nowhere -> dropped;
 *  - lists are in descending block order, padded with -1 after the count;
 *  - mask kinds use sequence-local positions i (query) and j (key):
 *      causal  j <= i;  sliding window  j <= i and (i - j < window_left or j < sink_tokens);
 *      prefix  j < prefix_len or j <= i;  document  doc_id_q[q row] == doc_id_k[k row];
 *  - the result for query row i is softmax over the allowed key set A(i): every
 *    key of a full-list tile below seqlen_k, and every key of a mask-list tile
 *    that passes the token predicate; LSE is the natural log of the sum of
 *    exp(scale * q.k) over A(i); an empty A(i) gives O = 0, LSE = -inf.
 */
#include <math.h>
#include <pthread.h>
#include <stdatomic.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { KIND_NONE = 0, KIND_CAUSAL = 1, KIND_SLIDING = 2, KIND_DOCUMENT = 3, KIND_PREFIX = 4 };

typedef struct {
    int32_t B, H, D, varlen;
    int32_t num_m, num_n;          /* batched: tiles per sequence; varlen: unused / stride */
    int32_t tile_m, tile_n;
    const int32_t *cu_q, *cu_k;    /* [B+1] packed row start of each sequence */
    const int32_t *kv_valid_len;   /* [B, vl_stride] or NULL (all tokens valid) */
    int32_t vl_stride;
    int32_t kind, window_left, sink_tokens, prefix_len;
    const int32_t *doc_q, *doc_k;  /* per packed row, DOCUMENT only */
} oracle_problem;

typedef struct {
    int32_t *full_cnt, *full_idx, *mask_cnt, *mask_idx;
    int32_t *cu_total_m_blocks, *cu_block_idx_offsets; /* varlen, [B+1] */
    int32_t total_m_blocks, total_n_blocks;            /* varlen */
} oracle_meta;

static int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* ---------------------------------------------------------------- threads -- */

typedef struct {
    atomic_llong next;
    int64_t n, chunk;
    void (*fn)(void *ctx, int64_t lo, int64_t hi, void *scratch);
    void (*cleanup)(void *scratch);
    void *ctx;
} pool_t;

static void *pool_worker(void *arg) {
    pool_t *p = (pool_t *)arg;
    void *scratch = 0;
    for (;;) {
        int64_t lo = atomic_fetch_add(&p->next, p->chunk);
        if (lo >= p->n) break;
        int64_t hi = lo + p->chunk < p->n ? lo + p->chunk : p->n;
        p->fn(p->ctx, lo, hi, &scratch);
    }
    if (p->cleanup) p->cleanup(scratch);
    return 0;
}

static void parallel_for(int64_t n, int64_t chunk, int threads,
                         void (*fn)(void *, int64_t, int64_t, void *),
                         void (*cleanup)(void *), void *ctx) {
    pool_t p;
    atomic_init(&p.next, 0);
    p.n = n;
    p.chunk = chunk;
    p.fn = fn;
    p.cleanup = cleanup;
    p.ctx = ctx;
    if (threads < 1) threads = 1;
    if (threads > 512) threads = 512;
    pthread_t tid[512];
    int started = 0;
    for (int t = 1; t < threads; ++t) {
        if (pthread_create(&tid[started], 0, pool_worker, &p) != 0) break;
        ++started;
    }
    pool_worker(&p);
    for (int t = 0; t < started; ++t) pthread_join(tid[t], 0);
}

/* ------------------------------------------------------------ definitions -- */

static int32_t seqlen_q(const oracle_problem *p, int b) { return p->cu_q[b + 1] - p->cu_q[b]; }
static int32_t seqlen_k(const oracle_problem *p, int b) { return p->cu_k[b + 1] - p->cu_k[b]; }

/* Number of Q tiles and KV tiles of sequence b ([VARLEN] num_m(b), num_n(b)). */
static int64_t num_m_of(const oracle_problem *p, int b) { return cdiv(seqlen_q(p, b), p->tile_m); }
static int64_t num_n_of(const oracle_problem *p, int b) { return cdiv(seqlen_k(p, b), p->tile_n); }

/* mask_mod at sequence-local query position i and key position j. */
static int mask_mod(const oracle_problem *p, int64_t i, int64_t j, int64_t qrow, int64_t krow) {
    switch (p->kind) {
    case KIND_NONE: return 1;
    case KIND_CAUSAL: return j <= i;
    case KIND_SLIDING: return j <= i && (i - j < p->window_left || j < p->sink_tokens);
    case KIND_PREFIX: return j < p->prefix_len || j <= i;
    case KIND_DOCUMENT: return p->doc_q[qrow] == p->doc_k[krow];
    default: return 0;
    }
}

/* Token predicate of key j in KV tile n for query i of sequence b: inside the
 * sequence, allowed by mask_mod, and before the tile's valid length ([VSA]). */
static int token_ok(const oracle_problem *p, int b, int64_t n, int64_t i, int64_t j) {
    if (j >= seqlen_k(p, b)) return 0;
    if (!mask_mod(p, i, j, p->cu_q[b] + i, p->cu_k[b] + j)) return 0;
    if (p->kv_valid_len && j - n * p->tile_n >= p->kv_valid_len[(int64_t)b * p->vl_stride + n])
        return 0;
    return 1;
}

/* Where the count and the index list of row (b, h, m) live ([VARLEN]). */
static void row_location(const oracle_problem *p, const oracle_meta *mt, int b, int h, int64_t m,
                         int64_t *cnt_at, int64_t *idx_at) {
    if (!p->varlen) {
        *cnt_at = ((int64_t)b * p->H + h) * p->num_m + m;
        *idx_at = *cnt_at * p->num_n;
    } else {
        *cnt_at = (int64_t)h * mt->total_m_blocks + mt->cu_total_m_blocks[b] + m;
        *idx_at = (int64_t)h * mt->total_n_blocks + mt->cu_block_idx_offsets[b] + m * num_n_of(p, b);
    }
}

/* [VARLEN]: cu_total_m_blocks[b+1] = sum over b' <= b of num_m(b');
 *           cu_block_idx_offsets[b+1] = sum over b' <= b of num_m(b') * num_n(b'). */
int oracle_varlen_offsets(const oracle_problem *p, oracle_meta *mt) {
    int64_t cm = 0, cn = 0;
    mt->cu_total_m_blocks[0] = 0;
    mt->cu_block_idx_offsets[0] = 0;
    for (int b = 0; b < p->B; ++b) {
        if (seqlen_q(p, b) < 0 || seqlen_k(p, b) < 0) return 1;
        cm += num_m_of(p, b);
        cn += num_m_of(p, b) * num_n_of(p, b);
        if (cm > INT32_MAX || cn > INT32_MAX) return 1;
        mt->cu_total_m_blocks[b + 1] = (int32_t)cm;
        mt->cu_block_idx_offsets[b + 1] = (int32_t)cn;
    }
    mt->total_m_blocks = (int32_t)cm;
    mt->total_n_blocks = (int32_t)cn;
    return 0;
}

/* ------------------------------------------------------------- metadata -- */

typedef struct {
    const oracle_problem *p;
    const uint8_t *map;
    oracle_meta *mt;
    int64_t rows_per_bh;   /* batched only */
} meta_ctx;

/* One row (b, h, m): classify every selected KV tile by evaluating the token
 * predicate over all (query, key) pairs of the tile, then write both lists in
 * descending block order with -1 padding ([LIST]). */
static void meta_row(const oracle_problem *p, const uint8_t *map, oracle_meta *mt, int b, int h,
                     int64_t m) {
    int64_t cnt_at, idx_at;
    row_location(p, mt, b, h, m, &cnt_at, &idx_at);
    int64_t nn = p->varlen ? num_n_of(p, b) : p->num_n;
    int64_t i_lo = m * p->tile_m, i_hi = i_lo + p->tile_m;
    if (i_hi > seqlen_q(p, b)) i_hi = seqlen_q(p, b);
    int32_t nf = 0, nm = 0;
    for (int64_t n = nn - 1; n >= 0; --n) {
        if (!map[idx_at + n]) continue;
        int some = 0, all = 1;
        for (int64_t i = i_lo; i < i_hi; ++i)
            for (int64_t j = n * p->tile_n; j < (n + 1) * p->tile_n; ++j) {
                if (token_ok(p, b, n, i, j)) some = 1;
                else all = 0;
            }
        if (some && all) mt->full_idx[idx_at + nf++] = (int32_t)n;
        else if (some) mt->mask_idx[idx_at + nm++] = (int32_t)n;
    }
    for (int64_t e = nf; e < nn; ++e) mt->full_idx[idx_at + e] = -1;
    for (int64_t e = nm; e < nn; ++e) mt->mask_idx[idx_at + e] = -1;
    mt->full_cnt[cnt_at] = nf;
    mt->mask_cnt[cnt_at] = nm;
}

static void meta_chunk(void *vctx, int64_t lo, int64_t hi, void *scratch) {
    (void)scratch;
    meta_ctx *c = (meta_ctx *)vctx;
    const oracle_problem *p = c->p;
    for (int64_t r = lo; r < hi; ++r) {
        if (!p->varlen) {
            int64_t bh = r / p->num_m, m = r % p->num_m;
            meta_row(p, c->map, c->mt, (int)(bh / p->H), (int)(bh % p->H), m);
        } else {
            /* rows enumerated as h * total_m + packed m */
            int h = (int)(r / c->mt->total_m_blocks);
            int64_t pm = r % c->mt->total_m_blocks;
            int b = 0;
            while (c->mt->cu_total_m_blocks[b + 1] <= pm) ++b;
            meta_row(p, c->map, c->mt, b, h, pm - c->mt->cu_total_m_blocks[b]);
        }
    }
}

int oracle_build_meta(const oracle_problem *p, const uint8_t *map, oracle_meta *mt, int threads) {
    if (p->tile_m <= 0 || p->tile_n <= 0 || p->B <= 0 || p->H <= 0) return 1;
    int64_t rows;
    if (p->varlen) {
        if (oracle_varlen_offsets(p, mt)) return 1;
        rows = (int64_t)p->H * mt->total_m_blocks;
    } else {
        for (int b = 0; b < p->B; ++b)
            if (num_m_of(p, b) != p->num_m || num_n_of(p, b) != p->num_n) return 1;
        rows = (int64_t)p->B * p->H * p->num_m;
    }
    meta_ctx c = {p, map, mt, 0};
    parallel_for(rows, 4, threads, meta_chunk, 0, &c);
    return 0;
}

/* -------------------------------------------------------------- forward -- */

typedef struct {
    const oracle_problem *p;
    const oracle_meta *mt;
    const uint16_t *q, *k, *v;
    double scale;
    const int32_t *tok, *head;
    double *o, *lse;
} fwd_ctx;

typedef struct {
    int64_t cap;
    int64_t *keys;
    double *s;
} fwd_scratch;

static double bf16_to_double(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Query row `tok` (packed row index), head h.  Builds A(i) from the lists, then
 * a two-pass softmax in fp64: the maximum first, then the sum. */
static void fwd_row(const fwd_ctx *c, int32_t tok, int32_t h, double *o, double *lse,
                    fwd_scratch *sc) {
    const oracle_problem *p = c->p;
    const int D = p->D, H = p->H;
    int b = 0;
    while (p->cu_q[b + 1] <= tok) ++b;
    int64_t i = tok - p->cu_q[b];
    int64_t m = i / p->tile_m;
    int64_t cnt_at, idx_at;
    row_location(p, c->mt, b, h, m, &cnt_at, &idx_at);
    int32_t nf = c->mt->full_cnt[cnt_at], nm = c->mt->mask_cnt[cnt_at];
    int64_t need = ((int64_t)nf + nm) * p->tile_n;
    if (need > sc->cap) {
        free(sc->keys);
        free(sc->s);
        sc->cap = need;
        sc->keys = (int64_t *)malloc(sizeof(int64_t) * (size_t)need);
        sc->s = (double *)malloc(sizeof(double) * (size_t)need);
    }
    int64_t nk = 0, sk = seqlen_k(p, b);
    for (int32_t e = 0; e < nf; ++e) {
        int64_t n = c->mt->full_idx[idx_at + e];
        for (int64_t j = n * p->tile_n; j < (n + 1) * p->tile_n && j < sk; ++j) sc->keys[nk++] = j;
    }
    for (int32_t e = 0; e < nm; ++e) {
        int64_t n = c->mt->mask_idx[idx_at + e];
        for (int64_t j = n * p->tile_n; j < (n + 1) * p->tile_n; ++j)
            if (token_ok(p, b, n, i, j)) sc->keys[nk++] = j;
    }
    if (nk == 0) {
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        *lse = -INFINITY;
        return;
    }
    const uint16_t *qi = c->q + ((int64_t)tok * H + h) * D;
    double mx = -INFINITY;
    for (int64_t t = 0; t < nk; ++t) {
        const uint16_t *kj = c->k + ((int64_t)(p->cu_k[b] + sc->keys[t]) * H + h) * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += bf16_to_double(qi[d]) * bf16_to_double(kj[d]);
        sc->s[t] = c->scale * dot;
        if (sc->s[t] > mx) mx = sc->s[t];
    }
    double sum = 0.0;
    for (int64_t t = 0; t < nk; ++t) sum += exp(sc->s[t] - mx);
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    for (int64_t t = 0; t < nk; ++t) {
        double w = exp(sc->s[t] - mx) / sum;
        const uint16_t *vj = c->v + ((int64_t)(p->cu_k[b] + sc->keys[t]) * H + h) * D;
        for (int d = 0; d < D; ++d) o[d] += w * bf16_to_double(vj[d]);
    }
    *lse = mx + log(sum);
}

static void fwd_scratch_free(void *s) {
    fwd_scratch *sc = (fwd_scratch *)s;
    if (!sc) return;
    free(sc->keys);
    free(sc->s);
    free(sc);
}

static void fwd_chunk(void *vctx, int64_t lo, int64_t hi, void *scratch) {
    fwd_ctx *c = (fwd_ctx *)vctx;
    fwd_scratch **sp = (fwd_scratch **)scratch;
    if (!*sp) *sp = (fwd_scratch *)calloc(1, sizeof(fwd_scratch));
    for (int64_t r = lo; r < hi; ++r)
        fwd_row(c, c->tok[r], c->head[r], c->o + r * c->p->D, c->lse + r, *sp);
}

/* Forward for an explicit list of (packed query row, head) pairs.  Outputs are
 * O[r, :D] and LSE[r] in fp64.  Returns 0 on success. */
int oracle_fwd_rows(const oracle_problem *p, const oracle_meta *mt, const uint16_t *q,
                    const uint16_t *k, const uint16_t *v, double scale, int64_t nrows,
                    const int32_t *tok, const int32_t *head, double *o, double *lse,
                    int threads) {
    for (int64_t r = 0; r < nrows; ++r)
        if (tok[r] < 0 || tok[r] >= p->cu_q[p->B] || head[r] < 0 || head[r] >= p->H) return 1;
    fwd_ctx c = {p, mt, q, k, v, scale, tok, head, o, lse};
    parallel_for(nrows, 8, threads, fwd_chunk, fwd_scratch_free, &c);
    return 0;
}


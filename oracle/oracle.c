/*
 * Oracle for batched decode attention over a paged KV cache with shared
 * prefixes.  TEST INFRASTRUCTURE ONLY: it is loaded by the tests, by the smoke
 * check and by the benchmark's CPU-baseline leg, never by the library.  It
 * shares no code, header or table with the CUDA path.
 *
 * What it computes is the plain definition, with no split, merge or
 * de-duplication:
 *
 *   "continuous-batching" page (guijiagi.com), section on PagedAttention,
 *   attention computation: for each request, collect the K/V of all its
 *   tokens through its block table, keep the first num_tokens of them, then
 *   scores = q K^T / sqrt(head_dim), weights = softmax(scores), out = weights V.
 *
 * The shared-prefix split of BatchLLM (papercache.org, section 2.2, Eq. 1)
 * reaches the same result exactly (up to rounding order); it is checked here
 * only through the split-plus-merge invariant tests, not used.
 *
 * Readings of what the pages leave open (each listed in the design notes):
 *  - the token list of request r is its prefix chain, root level first, then
 *    its own suffix; each level occupies ceil(P/B) block-table columns
 *    starting at a block boundary ("segment addressing"), the suffix starts at
 *    the next column;
 *  - q head h reads KV head h / (Hq/Hkv) (contiguous GQA grouping);
 *  - the decode token's own K/V is part of the suffix; no causal mask;
 *  - LSE is the natural log of sum(exp(scaled score)).
 *
 * Chunked prefill (oracle_attention_chunked): BatchLLM (papercache.org,
 * sections 2 and 6, chunked prefill / SplitFuse) mixes prefill chunks with
 * decode tokens in one token batch.  Reading: a request's chunk of n queries
 * is the last n tokens of its token list, and query i of the chunk attends to
 * the tokens up to and including its own position (the causal mask of a
 * decoder), i.e. the first n_tok - n + i + 1 tokens.  A decode request is a
 * chunk of one query and sees every token, as above.
 *
 * Arithmetic: inputs are widened exactly to double (bf16 -> fp32 -> double);
 * everything after that is double.  OpenMP spreads the (request, q head)
 * pairs over threads; each pair is computed independently, so the result
 * does not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int32_t num_req, num_groups, num_q_heads, num_kv_heads, head_dim, block_size;
    int32_t max_blocks_per_req, num_pool_blocks;
    int32_t dtype; /* 0: fp32, 1: bf16 stored as uint16 bit patterns */
    double scale;
    const void* q;              /* [R][Hq][d] */
    const void* pool;           /* [nb][2][Hkv][B][d], index 0 = K, 1 = V */
    const int32_t* block_table; /* [R][max_blocks_per_req] */
    const int32_t* group_of_req;/* [R], -1 = none */
    const int32_t* group_parent;/* [num_groups] or NULL */
    const int32_t* prefix_len;  /* [num_groups] */
    const int32_t* suffix_len;  /* [R] */
} oracle_problem;

enum { OR_OK = 0, OR_BAD_ARG = -1, OR_BAD_BLOCK = -2, OR_BAD_GROUP = -3, OR_EMPTY = -4 };

static double widen(const void* base, int dtype, size_t idx) {
    if (dtype == 0) return (double)((const float*)base)[idx];
    uint32_t u = (uint32_t)((const uint16_t*)base)[idx] << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Prefix chain of request r, root first.  Returns its length, or -1 if the
 * chain is malformed (bad id or longer than num_groups, i.e. a cycle). */
static int chain_of(const oracle_problem* p, int r, int32_t* out) {
    int32_t tmp[64];
    int n = 0;
    int32_t g = p->group_of_req[r];
    while (g >= 0) {
        if (g >= p->num_groups || n >= 64 || n > p->num_groups) return -1;
        tmp[n++] = g;
        g = p->group_parent ? p->group_parent[g] : -1;
    }
    for (int i = 0; i < n; ++i) out[i] = tmp[n - 1 - i];
    return n;
}

/* Number of tokens request r attends to, or a negative error. */
long long oracle_num_tokens(const oracle_problem* p, int r) {
    int32_t ch[64];
    int n = chain_of(p, r, ch);
    if (n < 0) return OR_BAD_GROUP;
    long long t = p->suffix_len[r];
    for (int i = 0; i < n; ++i) t += p->prefix_len[ch[i]];
    return t;
}

/* Physical (block, slot) of every token of request r, in order.  Returns the
 * token count, or a negative error.  `blk` and `slot` hold `cap` entries. */
static long long token_map(const oracle_problem* p, int r, int32_t* blk, int32_t* slot,
                           long long cap) {
    int32_t ch[64];
    int n = chain_of(p, r, ch);
    if (n < 0) return OR_BAD_GROUP;
    const int B = p->block_size;
    const int32_t* row = p->block_table + (size_t)r * p->max_blocks_per_req;
    long long col = 0, t = 0;
    for (int lv = 0; lv <= n; ++lv) {
        long long len = (lv < n) ? p->prefix_len[ch[lv]] : p->suffix_len[r];
        if (len < 0) return OR_BAD_ARG;
        for (long long j = 0; j < len; ++j) {
            long long c = col + j / B;
            if (c >= p->max_blocks_per_req || t >= cap) return OR_BAD_BLOCK;
            int32_t b = row[c];
            if (b < 0 || b >= p->num_pool_blocks) return OR_BAD_BLOCK;
            blk[t] = b;
            slot[t] = (int32_t)(j % B);
            ++t;
        }
        col += (len + B - 1) / B;
    }
    return t;
}

static size_t pool_index(const oracle_problem* p, int32_t b, int kv, int h, int32_t s, int e) {
    return ((((size_t)b * 2 + kv) * p->num_kv_heads + h) * p->block_size + s) *
               (size_t)p->head_dim + e;
}

/* Dense copy of the K and V rows request r reads for KV head kvh, widened to
 * double: K, V are [n][d].  Returns n or a negative error. */
long long oracle_gather_kv(const oracle_problem* p, int r, int kvh, double* K, double* V,
                           long long cap) {
    long long n = oracle_num_tokens(p, r);
    if (n < 0) return n;
    if (n > cap) return OR_BAD_ARG;
    int32_t* blk = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n ? n : 1));
    int32_t* slot = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n ? n : 1));
    long long m = token_map(p, r, blk, slot, n);
    if (m >= 0) {
        const int d = p->head_dim;
        for (long long t = 0; t < m; ++t)
            for (int e = 0; e < d; ++e) {
                K[t * d + e] = widen(p->pool, p->dtype, pool_index(p, blk[t], 0, kvh, slot[t], e));
                V[t * d + e] = widen(p->pool, p->dtype, pool_index(p, blk[t], 1, kvh, slot[t], e));
            }
    }
    free(blk);
    free(slot);
    return m;
}

/* Attention of q row `qrow` of `q` ([rows][Hq][d]), head h, over the first n
 * tokens of a request's token map, from the definition. */
static int attend_one(const oracle_problem* p, const void* q, long long qrow, int h,
                      const int32_t* blk, const int32_t* slot, long long n, double* s,
                      double* out, double* lse) {
    const int d = p->head_dim;
    const int kvh = h / (p->num_q_heads / p->num_kv_heads);
    const size_t qoff = ((size_t)qrow * p->num_q_heads + h) * d;
    double m = -INFINITY;
    for (long long t = 0; t < n; ++t) {
        double acc = 0.0;
        for (int e = 0; e < d; ++e)
            acc += widen(q, p->dtype, qoff + e) *
                   widen(p->pool, p->dtype, pool_index(p, blk[t], 0, kvh, slot[t], e));
        s[t] = acc * p->scale;
        if (s[t] > m) m = s[t];
    }
    double z = 0.0;
    for (long long t = 0; t < n; ++t) {
        s[t] = exp(s[t] - m);
        z += s[t];
    }
    for (int e = 0; e < d; ++e) out[e] = 0.0;
    for (long long t = 0; t < n; ++t) {
        double w = s[t] / z;
        for (int e = 0; e < d; ++e)
            out[e] += w * widen(p->pool, p->dtype, pool_index(p, blk[t], 1, kvh, slot[t], e));
    }
    *lse = m + log(z);
    return OR_OK;
}

/* Attention output and LSE for the requests listed in `req` (all requests when
 * req == NULL, n_req ignored).  out: [n][Hq][d] double, lse: [n][Hq] double.
 * nthreads <= 0 uses the OpenMP default.  Returns 0 or a negative error. */
int oracle_attention(const oracle_problem* p, const int32_t* req, int n_req, double* out,
                     double* lse, int nthreads) {
    if (!p || p->num_q_heads <= 0 || p->num_kv_heads <= 0 ||
        p->num_q_heads % p->num_kv_heads || p->head_dim <= 0 || p->block_size <= 0)
        return OR_BAD_ARG;
    const int n = req ? n_req : p->num_req;
    const int Hq = p->num_q_heads, d = p->head_dim;
    int status = OR_OK;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
#pragma omp parallel
    {
        long long cap = 0;
        int32_t *blk = NULL, *slot = NULL;
        double* s = NULL;
        int cur = -1;
        long long ntok = 0;
#pragma omp for schedule(dynamic, 4)
        for (long long i = 0; i < (long long)n * Hq; ++i) {
            int k = (int)(i / Hq), h = (int)(i % Hq);
            int r = req ? req[k] : k;
            if (r < 0 || r >= p->num_req) {
#pragma omp atomic write
                status = OR_BAD_ARG;
                continue;
            }
            if (r != cur) {
                long long need = oracle_num_tokens(p, r);
                if (need <= 0) {
#pragma omp atomic write
                    status = need < 0 ? (int)need : OR_EMPTY;
                    cur = -1;
                    continue;
                }
                if (need > cap) {
                    free(blk); free(slot); free(s);
                    cap = need;
                    blk = (int32_t*)malloc(sizeof(int32_t) * (size_t)cap);
                    slot = (int32_t*)malloc(sizeof(int32_t) * (size_t)cap);
                    s = (double*)malloc(sizeof(double) * (size_t)cap);
                }
                ntok = token_map(p, r, blk, slot, cap);
                if (ntok < 0) {
#pragma omp atomic write
                    status = (int)ntok;
                    cur = -1;
                    continue;
                }
                cur = r;
            }
            attend_one(p, p->q, r, h, blk, slot, ntok, s, out + ((size_t)k * Hq + h) * d,
                       lse + (size_t)k * Hq + h);
        }
        free(blk); free(slot); free(s);
    }
    return status;
}

/* Chunked prefill.  Request r has q_len[r] >= 1 queries; q is [Q][Hq][d] with
 * Q = sum q_len, request r's queries at rows off_r .. off_r + q_len[r] - 1
 * (off_r = sum of q_len over the earlier requests).  Query i of request r
 * attends to the first n_tok(r) - q_len[r] + i + 1 tokens of r's token list.
 * out: [Q][Hq][d] double, lse: [Q][Hq] double.  Returns 0 or a negative
 * error (OR_BAD_ARG when a chunk is longer than its request's token list). */
int oracle_attention_chunked(const oracle_problem* p, const int32_t* q_len, const void* q,
                             double* out, double* lse, int nthreads) {
    if (!p || !q_len || !q || p->num_q_heads <= 0 || p->num_kv_heads <= 0 ||
        p->num_q_heads % p->num_kv_heads || p->head_dim <= 0 || p->block_size <= 0)
        return OR_BAD_ARG;
    const int R = p->num_req, Hq = p->num_q_heads, d = p->head_dim;
    long long Q = 0;
    for (int r = 0; r < R; ++r) {
        if (q_len[r] < 1) return OR_BAD_ARG;
        Q += q_len[r];
    }
    int32_t* req_of = (int32_t*)malloc(sizeof(int32_t) * (size_t)(Q ? Q : 1));
    int32_t* idx_of = (int32_t*)malloc(sizeof(int32_t) * (size_t)(Q ? Q : 1));
    long long k = 0;
    for (int r = 0; r < R; ++r)
        for (int i = 0; i < q_len[r]; ++i, ++k) {
            req_of[k] = r;
            idx_of[k] = i;
        }
    int status = OR_OK;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
#pragma omp parallel
    {
        long long cap = 0;
        int32_t *blk = NULL, *slot = NULL;
        double* s = NULL;
        int cur = -1;
        long long ntok = 0;
#pragma omp for schedule(dynamic, 4)
        for (long long i = 0; i < Q * Hq; ++i) {
            const long long row = i / Hq;
            const int h = (int)(i % Hq), r = req_of[row];
            if (r != cur) {
                long long need = oracle_num_tokens(p, r);
                if (need < q_len[r]) {
#pragma omp atomic write
                    status = need < 0 ? (int)need : OR_BAD_ARG;
                    cur = -1;
                    continue;
                }
                if (need > cap) {
                    free(blk); free(slot); free(s);
                    cap = need;
                    blk = (int32_t*)malloc(sizeof(int32_t) * (size_t)cap);
                    slot = (int32_t*)malloc(sizeof(int32_t) * (size_t)cap);
                    s = (double*)malloc(sizeof(double) * (size_t)cap);
                }
                ntok = token_map(p, r, blk, slot, cap);
                if (ntok < 0) {
#pragma omp atomic write
                    status = (int)ntok;
                    cur = -1;
                    continue;
                }
                cur = r;
            }
            const long long nvis = ntok - q_len[r] + idx_of[row] + 1;
            attend_one(p, q, row, h, blk, slot, nvis, s, out + ((size_t)row * Hq + h) * d,
                       lse + (size_t)row * Hq + h);
        }
        free(blk); free(slot); free(s);
    }
    free(req_of);
    free(idx_of);
    return status;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * CPU oracle for paged-KV append, paged grouped-query-attention decode and
 * paged prefill.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline / reference legs use it.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * What it computes, and where that comes from:
 *   - forge-engine README, "What it implements" table, row "KV cache": the
 *     KV cache is a pool of fixed-size blocks handed out to sequences.
 *   - "Make the Engine Talk", section 1.2 (the `stream` loop): each decode
 *     pass runs the model on one new token and the cache grows by that
 *     token; section 1.3: attention is grouped-query attention.
 *   - Everything the pages leave open (formula, layout, head grouping,
 *     masking) follows the plainest reading:
 *       out[b,h,:] = sum_t softmax_t(scale * q[b,h,:] . K_b[t,:]) * V_b[t,:]
 *     over the positions t < context_lens[b], with query head h reading KV
 *     head h / (Hq/Hkv), and K_b[t] found at
 *       k_cache[block_tables[b][t / BS], h_kv, t % BS, :].
 *
 * The decode is written the slow, obvious way: gather the sequence's K and V
 * into contiguous fp64 arrays (the contiguous per-layer cache of "Make the
 * Engine Talk", section 1.2), take fp64 dot products, subtract the maximum,
 * exponentiate with libm `exp`, normalise.  bf16 inputs convert to fp64
 * exactly.  No blocking, no online softmax, no splits.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG (-1)
#define ORACLE_ERR_BLOCK (-2)
#define ORACLE_ERR_LEN (-3)
#define ORACLE_ERR_SLOT (-4)
#define ORACLE_ERR_NOMEM (-5)

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_bits_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Append: for every sequence b whose slot is non-negative, copy the new
 * token's K and V rows (all KV heads) into block slot/BS, offset slot%BS.
 * A negative slot means "no token for this row".  Plain bit copies in
 * sequence order.  Returns ORACLE_ERR_SLOT (and copies nothing further) on a
 * slot beyond the pool.
 */
int oracle_paged_kv_append(const uint16_t *k_new, const uint16_t *v_new,
                           const int64_t *slot_mapping, uint16_t *k_cache,
                           uint16_t *v_cache, int B, int Hkv, int D, int NB,
                           int BS) {
    if (B < 0 || Hkv <= 0 || D <= 0 || NB < 0 || BS <= 0) return ORACLE_ERR_ARG;
    for (int b = 0; b < B; ++b) {
        int64_t slot = slot_mapping[b];
        if (slot < 0) continue;
        if (slot >= (int64_t)NB * BS) return ORACLE_ERR_SLOT;
        int64_t blk = slot / BS;
        int64_t off = slot % BS;
        for (int h = 0; h < Hkv; ++h) {
            size_t src = ((size_t)b * Hkv + h) * (size_t)D;
            size_t dst = (((size_t)blk * Hkv + h) * BS + off) * (size_t)D;
            memcpy(k_cache + dst, k_new + src, (size_t)D * sizeof(uint16_t));
            memcpy(v_cache + dst, v_new + src, (size_t)D * sizeof(uint16_t));
        }
    }
    return ORACLE_OK;
}

/*
 * RMSNorm of each row of x ([rows, D], bf16 bits) with weight w ([D], bf16
 * bits; NULL = all ones), in fp64:  y = x / sqrt(mean(x^2) + eps) * w.
 * ("Make the Engine Talk", 1.3: RMSNorm is one of the forward pass's
 * mechanisms; here it is applied per attention head to q and k.)
 */
void oracle_rmsnorm(const uint16_t *x, const uint16_t *w, double eps, double *y, int rows, int D) {
    for (int r = 0; r < rows; ++r) {
        double ss = 0.0;
        for (int d = 0; d < D; ++d) {
            double v = bf16_bits_to_double(x[(size_t)r * D + d]);
            ss += v * v;
        }
        double inv = 1.0 / sqrt(ss / D + eps);
        for (int d = 0; d < D; ++d) {
            double wd = w ? bf16_bits_to_double(w[d]) : 1.0;
            y[(size_t)r * D + d] = bf16_bits_to_double(x[(size_t)r * D + d]) * inv * wd;
        }
    }
}

/*
 * Rotary position embedding, rotate-half form, in place on fp64 rows
 * ([rows, D]) at positions pos[r] ("Make the Engine Talk", 1.3: rotary
 * position embeddings).  For i < D/2, with angle a = pos * theta^(-2i/D):
 *   y[i]       = x[i] cos a - x[i+D/2] sin a
 *   y[i+D/2]   = x[i+D/2] cos a + x[i] sin a
 */
void oracle_rope(double *x, const int64_t *pos, double theta, int rows, int D) {
    const int h = D / 2;
    for (int r = 0; r < rows; ++r) {
        double *row = x + (size_t)r * D;
        for (int i = 0; i < h; ++i) {
            double a = (double)pos[r] * pow(theta, -2.0 * i / D);
            double c = cos(a), s = sin(a);
            double x1 = row[i], x2 = row[i + h];
            row[i] = x1 * c - x2 * s;
            row[i + h] = x2 * c + x1 * s;
        }
    }
}

typedef struct {
    const uint16_t *q, *k_cache, *v_cache;
    const int32_t *block_tables, *context_lens;
    double scale;
    double *out;
    int B, Hq, Hkv, D, NB, BS, MB;
    int max_len;
    int next_item; /* shared work counter over (b, h) */
    int status;
} decode_job;

/* One (sequence, query head) output row, by the definition above. */
static int decode_one(const decode_job *j, int b, int h, double *K, double *V,
                      double *s) {
    const int D = j->D, BS = j->BS, Hkv = j->Hkv;
    const int G = j->Hq / j->Hkv;
    const int g = h / G; /* contiguous groups of G query heads share KV head g */
    const int L = j->context_lens[b];
    double *o = j->out + ((size_t)b * j->Hq + h) * (size_t)D;

    if (L <= 0) {
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        return ORACLE_OK;
    }
    if (L > j->MB * BS) return ORACLE_ERR_LEN;

    /* gather this sequence's first L tokens of KV head g into contiguous rows */
    for (int t = 0; t < L; ++t) {
        int32_t blk = j->block_tables[(size_t)b * j->MB + t / BS];
        if (blk < 0 || blk >= j->NB) return ORACLE_ERR_BLOCK;
        size_t row = (((size_t)blk * Hkv + g) * BS + (size_t)(t % BS)) * (size_t)D;
        for (int d = 0; d < D; ++d) {
            K[(size_t)t * D + d] = bf16_bits_to_double(j->k_cache[row + d]);
            V[(size_t)t * D + d] = bf16_bits_to_double(j->v_cache[row + d]);
        }
    }

    /* scaled logits */
    const uint16_t *qrow = j->q + ((size_t)b * j->Hq + h) * (size_t)D;
    double m = -INFINITY;
    for (int t = 0; t < L; ++t) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d)
            acc += bf16_bits_to_double(qrow[d]) * K[(size_t)t * D + d];
        s[t] = j->scale * acc;
        if (s[t] > m) m = s[t];
    }

    /* softmax weights and the weighted sum of values */
    double den = 0.0;
    for (int t = 0; t < L; ++t) {
        s[t] = exp(s[t] - m);
        den += s[t];
    }
    /* numerators: for every d the sum runs over t in ascending order */
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    for (int t = 0; t < L; ++t)
        for (int d = 0; d < D; ++d) o[d] += s[t] * V[(size_t)t * D + d];
    for (int d = 0; d < D; ++d) o[d] /= den;
    return ORACLE_OK;
}

static void *decode_worker(void *arg) {
    decode_job *j = (decode_job *)arg;
    size_t n = (size_t)(j->max_len > 0 ? j->max_len : 1);
    double *K = (double *)malloc(n * (size_t)j->D * sizeof(double));
    double *V = (double *)malloc(n * (size_t)j->D * sizeof(double));
    double *s = (double *)malloc(n * sizeof(double));
    if (!K || !V || !s) {
        __atomic_store_n(&j->status, ORACLE_ERR_NOMEM, __ATOMIC_RELAXED);
    } else {
        const int items = j->B * j->Hq;
        for (;;) {
            int it = __atomic_fetch_add(&j->next_item, 1, __ATOMIC_RELAXED);
            if (it >= items) break;
            int rc = decode_one(j, it / j->Hq, it % j->Hq, K, V, s);
            if (rc != ORACLE_OK) __atomic_store_n(&j->status, rc, __ATOMIC_RELAXED);
        }
    }
    free(K);
    free(V);
    free(s);
    return NULL;
}

/*
 * Decode attention for every (b, h).  `out` is fp64 [B, Hq, D].  `nthreads`
 * <= 1 runs on the calling thread; otherwise (b, h) rows are shared out to
 * that many POSIX threads.  Layouts (all dense, row-major):
 *   q [B, Hq, D] bf16 bits; k_cache, v_cache [NB, Hkv, BS, D] bf16 bits;
 *   block_tables [B, MB] int32; context_lens [B] int32.
 */
int oracle_paged_gqa_decode(const uint16_t *q, const uint16_t *k_cache,
                            const uint16_t *v_cache, const int32_t *block_tables,
                            const int32_t *context_lens, double scale, double *out,
                            int B, int Hq, int Hkv, int D, int NB, int BS, int MB,
                            int nthreads) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || BS <= 0 ||
        MB < 0 || NB < 0)
        return ORACLE_ERR_ARG;
    decode_job j;
    j.q = q;
    j.k_cache = k_cache;
    j.v_cache = v_cache;
    j.block_tables = block_tables;
    j.context_lens = context_lens;
    j.scale = scale;
    j.out = out;
    j.B = B;
    j.Hq = Hq;
    j.Hkv = Hkv;
    j.D = D;
    j.NB = NB;
    j.BS = BS;
    j.MB = MB;
    j.next_item = 0;
    j.status = ORACLE_OK;
    j.max_len = 0;
    for (int b = 0; b < B; ++b)
        if (context_lens[b] > j.max_len) j.max_len = context_lens[b];
    if (j.max_len > MB * BS) return ORACLE_ERR_LEN;

    if (nthreads <= 1) {
        decode_worker(&j);
        return j.status;
    }
    pthread_t *tids = (pthread_t *)malloc((size_t)nthreads * sizeof(pthread_t));
    if (!tids) return ORACLE_ERR_NOMEM;
    int started = 0;
    for (int i = 0; i < nthreads; ++i) {
        if (pthread_create(&tids[i], NULL, decode_worker, &j) != 0) break;
        ++started;
    }
    if (started == 0) decode_worker(&j);
    for (int i = 0; i < started; ++i) pthread_join(tids[i], NULL);
    free(tids);
    return j.status;
}

/*
 * Paged prefill (causal attention of a chunk of new query tokens).
 *
 * "Make the Engine Talk", 1.2: the prefill runs one forward pass over all
 * prompt tokens at once and fills the KV cache; forge-engine README, "What it
 * implements": prefill and decode are separate engine paths over the same
 * paged cache.  The chunk's K/V is already in the cache (written by the
 * append), so for sequence b with n_b = query_start[b+1] - query_start[b]
 * query tokens and context length L_b (the chunk included), query token i
 * sits at position p = L_b - n_b + i and attends to positions t <= p:
 *   out[query_start[b] + i, h, :] =
 *       sum_{t <= p} softmax_t(scale * q . K_b[t]) V_b[t]
 * with the same head grouping and cache addressing as the decode (which is
 * the n_b = 1 case).  n_b = 0 produces nothing; n_b > L_b is an error.
 */
typedef struct {
    const uint16_t *q, *k_cache, *v_cache;
    const int32_t *block_tables, *context_lens, *query_start;
    double scale;
    double *out;
    int B, Hq, Hkv, D, NB, BS, MB;
    int max_len;
    int next_item; /* shared work counter over (b, h) */
    int status;
} prefill_job;

/* All query tokens of one (sequence, query head). */
static int prefill_one(const prefill_job *j, int b, int h, double *K, double *V, double *s) {
    const int D = j->D, BS = j->BS, Hkv = j->Hkv;
    const int G = j->Hq / j->Hkv;
    const int g = h / G;
    const int L = j->context_lens[b];
    const int q0 = j->query_start[b];
    const int n = j->query_start[b + 1] - q0;
    if (n <= 0) return n == 0 ? ORACLE_OK : ORACLE_ERR_ARG;
    if (n > L) return ORACLE_ERR_LEN;
    if (L > j->MB * BS) return ORACLE_ERR_LEN;

    /* gather the sequence's L tokens of KV head g into contiguous rows */
    for (int t = 0; t < L; ++t) {
        int32_t blk = j->block_tables[(size_t)b * j->MB + t / BS];
        if (blk < 0 || blk >= j->NB) return ORACLE_ERR_BLOCK;
        size_t row = (((size_t)blk * Hkv + g) * BS + (size_t)(t % BS)) * (size_t)D;
        for (int d = 0; d < D; ++d) {
            K[(size_t)t * D + d] = bf16_bits_to_double(j->k_cache[row + d]);
            V[(size_t)t * D + d] = bf16_bits_to_double(j->v_cache[row + d]);
        }
    }

    for (int i = 0; i < n; ++i) {
        const int p = L - n + i; /* this query token's position */
        const uint16_t *qrow = j->q + ((size_t)(q0 + i) * j->Hq + h) * (size_t)D;
        double *o = j->out + ((size_t)(q0 + i) * j->Hq + h) * (size_t)D;
        double m = -INFINITY;
        for (int t = 0; t <= p; ++t) {
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += bf16_bits_to_double(qrow[d]) * K[(size_t)t * D + d];
            s[t] = j->scale * acc;
            if (s[t] > m) m = s[t];
        }
        double den = 0.0;
        for (int t = 0; t <= p; ++t) {
            s[t] = exp(s[t] - m);
            den += s[t];
        }
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        for (int t = 0; t <= p; ++t)
            for (int d = 0; d < D; ++d) o[d] += s[t] * V[(size_t)t * D + d];
        for (int d = 0; d < D; ++d) o[d] /= den;
    }
    return ORACLE_OK;
}

static void *prefill_worker(void *arg) {
    prefill_job *j = (prefill_job *)arg;
    size_t n = (size_t)(j->max_len > 0 ? j->max_len : 1);
    double *K = (double *)malloc(n * (size_t)j->D * sizeof(double));
    double *V = (double *)malloc(n * (size_t)j->D * sizeof(double));
    double *s = (double *)malloc(n * sizeof(double));
    if (!K || !V || !s) {
        __atomic_store_n(&j->status, ORACLE_ERR_NOMEM, __ATOMIC_RELAXED);
    } else {
        const int items = j->B * j->Hq;
        for (;;) {
            int it = __atomic_fetch_add(&j->next_item, 1, __ATOMIC_RELAXED);
            if (it >= items) break;
            int rc = prefill_one(j, it / j->Hq, it % j->Hq, K, V, s);
            if (rc != ORACLE_OK) __atomic_store_n(&j->status, rc, __ATOMIC_RELAXED);
        }
    }
    free(K);
    free(V);
    free(s);
    return NULL;
}

/*
 * Prefill for every sequence.  q and out are packed by query_start ([B+1],
 * query_start[0] = 0, non-decreasing): q [T, Hq, D] bf16 bits, out [T, Hq, D]
 * fp64 with T = query_start[B].  Other layouts as in the decode.  nthreads as
 * in the decode.
 */
int oracle_paged_prefill(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                         const int32_t *block_tables, const int32_t *context_lens,
                         const int32_t *query_start, double scale, double *out, int B, int Hq,
                         int Hkv, int D, int NB, int BS, int MB, int nthreads) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || BS <= 0 || MB < 0 || NB < 0)
        return ORACLE_ERR_ARG;
    if (B > 0 && query_start[0] != 0) return ORACLE_ERR_ARG;
    for (int b = 0; b < B; ++b)
        if (query_start[b + 1] < query_start[b]) return ORACLE_ERR_ARG;
    prefill_job j;
    j.q = q;
    j.k_cache = k_cache;
    j.v_cache = v_cache;
    j.block_tables = block_tables;
    j.context_lens = context_lens;
    j.query_start = query_start;
    j.scale = scale;
    j.out = out;
    j.B = B;
    j.Hq = Hq;
    j.Hkv = Hkv;
    j.D = D;
    j.NB = NB;
    j.BS = BS;
    j.MB = MB;
    j.next_item = 0;
    j.status = ORACLE_OK;
    j.max_len = 0;
    for (int b = 0; b < B; ++b)
        if (context_lens[b] > j.max_len) j.max_len = context_lens[b];
    if (j.max_len > MB * BS) return ORACLE_ERR_LEN;

    if (nthreads <= 1) {
        prefill_worker(&j);
        return j.status;
    }
    pthread_t *tids = (pthread_t *)malloc((size_t)nthreads * sizeof(pthread_t));
    if (!tids) return ORACLE_ERR_NOMEM;
    int started = 0;
    for (int i = 0; i < nthreads; ++i) {
        if (pthread_create(&tids[i], NULL, prefill_worker, &j) != 0) break;
        ++started;
    }
    if (started == 0) prefill_worker(&j);
    for (int i = 0; i < started; ++i) pthread_join(tids[i], NULL);
    free(tids);
    return j.status;
}

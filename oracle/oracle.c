/*
 * CPU oracle for paged-KV decode attention -- TEST INFRASTRUCTURE ONLY.
 *
 * This file is the slow, plain, obviously-correct statement of what the
 * paged-attention path computes.  It shares no code, header, table or helper
 * with the CUDA library; only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may build, load or call it.  The product path
 * never routes through it.
 *
 * Sources (the pages on vLLM / PagedAttention):
 *   - "vLLM PagedAttention chuyen sau" (locionic.com), section "Tuong tu phan
 *     trang bo nho ao": the KV cache of a sequence is cut into fixed-size
 *     logical blocks; each maps to a physical block; a per-sequence block
 *     table maps logical block index -> physical block index.
 *   - same page, section "Co che PagedAttention", steps 1-3: look the
 *     physical blocks up in the block table, gather K and V from them, then
 *     run standard attention on the gathered data.
 *   - same page, section "Chunked Prefill", mechanism step 3: the KV cache of
 *     each chunk accumulates into the sequence's blocks.
 *   - same page, section "Luu tru tien to tu dong (APC)", mechanism step 3:
 *     copy-on-write duplicates a shared block before a sequence diverges.
 *
 * Readings where the pages are silent (the pages give no layout, dtype rule
 * or head grouping; these are the readings the whole project uses):
 *   - pool layout [num_blocks][num_kv_heads][block_size][head_dim], row-major;
 *     token slot t lives in block t / block_size at offset t % block_size;
 *   - query head h reads KV head h / (num_heads / num_kv_heads);
 *   - "standard attention" = softmax(scale * q.K^T) V, computed here in fp64
 *     as max-subtracted exponentials, sum, weighted sum, divide;
 *   - context length 0 gives an all-zero output row;
 *   - a negative slot in slot_mapping means "padding, write nothing".
 *
 * Element storage is 16-bit (IEEE binary16 or bfloat16); values are decoded
 * to double by the two functions below, written from the formats'
 * definitions.  All arithmetic is fp64; nothing is blocked, fused or
 * reordered beyond the textbook formulas.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F16 0
#define ORACLE_BF16 1

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 10) & 0x1f;
    int frac = bits & 0x3ff;
    double mag;
    if (expo == 0)
        mag = ldexp((double)frac, -24);                 /* subnormal: frac * 2^-24 */
    else if (expo == 31)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + frac), expo - 25);  /* (1 + frac/1024) * 2^(expo-15) */
    return sign ? -mag : mag;
}

/* bfloat16 is the upper half of an IEEE binary32: 1 sign, 8 exponent (bias
 * 127), 7 fraction bits. */
double oracle_bf16_to_f64(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 7) & 0xff;
    int frac = bits & 0x7f;
    double mag;
    if (expo == 0)
        mag = ldexp((double)frac, -133);                /* subnormal: frac * 2^-133 */
    else if (expo == 255)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(128 + frac), expo - 134);  /* (1 + frac/128) * 2^(expo-127) */
    return sign ? -mag : mag;
}

static double decode_elem(uint16_t bits, int dtype)
{
    return dtype == ORACLE_BF16 ? oracle_bf16_to_f64(bits) : oracle_f16_to_f64(bits);
}

/* Offset (in elements) of row (physical block, kv head, in-block offset). */
static size_t pool_row(long blk, int kvh, int off, int num_kv_heads, int block_size, int head_dim)
{
    return (((size_t)blk * num_kv_heads + kvh) * block_size + off) * head_dim;
}

/*
 * Cache write: each new token i whose slot_mapping[i] >= 0 has its K and V
 * rows (all kv heads) copied bit for bit into block slot/bs, offset slot%bs.
 * Slots past the pool are skipped and counted.  Returns that count.
 * key, value: [T][Hkv][D]; caches: [NB][Hkv][bs][D].
 */
int oracle_reshape_and_cache(const uint16_t *key, const uint16_t *value,
                             uint16_t *k_cache, uint16_t *v_cache,
                             const int64_t *slot_mapping, int num_tokens,
                             int num_kv_heads, int head_dim, int block_size, int num_blocks)
{
    int bad = 0;
    for (int i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0)
            continue;
        if (slot >= (int64_t)num_blocks * block_size) {
            ++bad;
            continue;
        }
        long blk = (long)(slot / block_size);
        int off = (int)(slot % block_size);
        for (int h = 0; h < num_kv_heads; ++h) {
            size_t src = ((size_t)i * num_kv_heads + h) * head_dim;
            size_t dst = pool_row(blk, h, off, num_kv_heads, block_size, head_dim);
            memcpy(k_cache + dst, key + src, (size_t)head_dim * sizeof(uint16_t));
            memcpy(v_cache + dst, value + src, (size_t)head_dim * sizeof(uint16_t));
        }
    }
    return bad;
}

/*
 * Copy-on-write block copy: for each valid (src, dst) pair the whole K block
 * and V block of src (all kv heads) are copied to dst.  A pair is valid when
 * both ids are in the pool, src != dst, no other pair has the same dst, and
 * dst is nobody's src; invalid pairs are skipped and counted.  Under these
 * rules the result does not depend on the order of the pairs.
 */
int oracle_copy_blocks(uint16_t *k_cache, uint16_t *v_cache, const int64_t *pairs, int num_pairs,
                       int num_kv_heads, int head_dim, int block_size, int num_blocks)
{
    size_t blk_elems = (size_t)num_kv_heads * block_size * head_dim;
    int bad = 0;
    for (int i = 0; i < num_pairs; ++i) {
        int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        int ok = src >= 0 && src < num_blocks && dst >= 0 && dst < num_blocks && src != dst;
        for (int j = 0; ok && j < num_pairs; ++j) {
            if (j != i && pairs[2 * j + 1] == dst)
                ok = 0;
            if (pairs[2 * j] == dst)
                ok = 0;
        }
        if (!ok) {
            ++bad;
            continue;
        }
        memcpy(k_cache + (size_t)dst * blk_elems, k_cache + (size_t)src * blk_elems,
               blk_elems * sizeof(uint16_t));
        memcpy(v_cache + (size_t)dst * blk_elems, v_cache + (size_t)src * blk_elems,
               blk_elems * sizeof(uint16_t));
    }
    return bad;
}

/*
 * Gather: rows 0..n-1 of one sequence's K (or V) for one kv head, through the
 * block table, into a contiguous [n][D] fp64 array.  Returns -1 if a table
 * entry is outside the pool.
 */
static int gather_rows(double *dst, const uint16_t *pool, const int32_t *table, int n,
                       int kvh, int num_kv_heads, int head_dim, int block_size, int num_blocks,
                       int dtype)
{
    for (int j = 0; j < n; ++j) {
        int32_t blk = table[j / block_size];
        if (blk < 0 || blk >= num_blocks)
            return -1;
        const uint16_t *row = pool + pool_row(blk, kvh, j % block_size, num_kv_heads, block_size, head_dim);
        for (int d = 0; d < head_dim; ++d)
            dst[(size_t)j * head_dim + d] = decode_elem(row[d], dtype);
    }
    return 0;
}

/*
 * Textbook single-query softmax attention over contiguous fp64 K, V:
 *   z_j = scale * sum_d q_d K[j][d];  p_j = exp(z_j - max z);
 *   out_d = sum_j p_j V[j][d] / sum_j p_j.
 * n == 0 gives zeros.  z and out are caller buffers of n and D doubles.
 */
static void attend_one(double *out, const double *q, const double *K, const double *V, int n,
                       int head_dim, double scale, double *z)
{
    for (int d = 0; d < head_dim; ++d)
        out[d] = 0.0;
    if (n <= 0)
        return;
    double zmax = -INFINITY;
    for (int j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d)
            dot += q[d] * K[(size_t)j * head_dim + d];
        z[j] = scale * dot;
        if (z[j] > zmax)
            zmax = z[j];
    }
    double denom = 0.0;
    for (int j = 0; j < n; ++j) {
        z[j] = exp(z[j] - zmax);
        denom += z[j];
    }
    for (int j = 0; j < n; ++j)
        for (int d = 0; d < head_dim; ++d)
            out[d] += z[j] * V[(size_t)j * head_dim + d];
    for (int d = 0; d < head_dim; ++d)
        out[d] /= denom;
}

/* ------------------------------------------------------------------ decode */

struct decode_args {
    double *out;
    const uint16_t *query, *k_cache, *v_cache;
    const int32_t *block_tables, *context_lens;
    int max_blocks_per_seq, num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks;
    double scale;
    int dtype, stride, first;
    int err;
};

static void *decode_worker(void *p)
{
    struct decode_args *a = (struct decode_args *)p;
    int D = a->head_dim, G = a->num_heads / a->num_kv_heads;
    int items = a->num_seqs * a->num_kv_heads;
    for (int it = a->first; it < items; it += a->stride) {
        int s = it / a->num_kv_heads, kvh = it % a->num_kv_heads;
        int L = a->context_lens[s];
        if (L < 0 || L > a->max_blocks_per_seq * a->block_size) {
            a->err = -1;
            continue;
        }
        size_t n = L > 0 ? (size_t)L : 1;
        double *K = malloc(n * D * sizeof(double));
        double *V = malloc(n * D * sizeof(double));
        double *z = malloc(n * sizeof(double));
        double *q = malloc((size_t)D * sizeof(double));
        const int32_t *table = a->block_tables + (size_t)s * a->max_blocks_per_seq;
        /* steps 1 and 2 of the paged-attention mechanism: look up and gather */
        if (gather_rows(K, a->k_cache, table, L, kvh, a->num_kv_heads, D, a->block_size, a->num_blocks, a->dtype) ||
            gather_rows(V, a->v_cache, table, L, kvh, a->num_kv_heads, D, a->block_size, a->num_blocks, a->dtype)) {
            a->err = -1;
        } else {
            /* step 3: standard attention, once per query head of the group */
            for (int h = kvh * G; h < (kvh + 1) * G; ++h) {
                const uint16_t *qrow = a->query + ((size_t)s * a->num_heads + h) * D;
                for (int d = 0; d < D; ++d)
                    q[d] = decode_elem(qrow[d], a->dtype);
                attend_one(a->out + ((size_t)s * a->num_heads + h) * D, q, K, V, L, D, a->scale, z);
            }
        }
        free(K);
        free(V);
        free(z);
        free(q);
    }
    return NULL;
}

/*
 * Single-query decode attention over the paged cache.
 *   out [B][Hq][D] fp64; query [B][Hq][D]; block_tables [B][MB] int32;
 *   context_lens [B] int32 (tokens already in the cache, new token included).
 * Work is spread over num_threads POSIX threads by (sequence, kv head).
 * Returns 0, or -1 if a length or table entry is out of range.
 */
int oracle_decode(double *out, const uint16_t *query, const uint16_t *k_cache, const uint16_t *v_cache,
                  const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
                  int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                  int num_blocks, double scale, int dtype, int num_threads)
{
    if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0)
        return -2;
    if (num_threads < 1)
        num_threads = 1;
    struct decode_args *args = calloc((size_t)num_threads, sizeof(*args));
    pthread_t *tid = calloc((size_t)num_threads, sizeof(pthread_t));
    for (int t = 0; t < num_threads; ++t) {
        struct decode_args a = {out, query, k_cache, v_cache, block_tables, context_lens,
                                max_blocks_per_seq, num_seqs, num_heads, num_kv_heads, head_dim,
                                block_size, num_blocks, scale, dtype, num_threads, t, 0};
        args[t] = a;
    }
    for (int t = 1; t < num_threads; ++t)
        pthread_create(&tid[t], NULL, decode_worker, &args[t]);
    decode_worker(&args[0]);
    int err = args[0].err;
    for (int t = 1; t < num_threads; ++t) {
        pthread_join(tid[t], NULL);
        if (args[t].err)
            err = args[t].err;
    }
    free(args);
    free(tid);
    return err;
}

/* --------------------------------------------------------- chunked prefill */

struct prefill_args {
    double *out;
    const uint16_t *query, *k_cache, *v_cache;
    const int32_t *block_table;
    int prefix_len, chunk_len, num_heads, num_kv_heads, head_dim, block_size, num_blocks;
    double scale;
    int dtype, stride, first;
    int err;
};

static void *prefill_worker(void *p)
{
    struct prefill_args *a = (struct prefill_args *)p;
    int D = a->head_dim, G = a->num_heads / a->num_kv_heads;
    int n = a->prefix_len + a->chunk_len;
    size_t nn = n > 0 ? (size_t)n : 1;
    double *K = malloc(nn * D * sizeof(double));
    double *V = malloc(nn * D * sizeof(double));
    double *z = malloc(nn * sizeof(double));
    double *q = malloc((size_t)D * sizeof(double));
    for (int kvh = a->first; kvh < a->num_kv_heads; kvh += a->stride) {
        if (gather_rows(K, a->k_cache, a->block_table, n, kvh, a->num_kv_heads, D, a->block_size, a->num_blocks, a->dtype) ||
            gather_rows(V, a->v_cache, a->block_table, n, kvh, a->num_kv_heads, D, a->block_size, a->num_blocks, a->dtype)) {
            a->err = -1;
            continue;
        }
        for (int i = 0; i < a->chunk_len; ++i) {
            /* query row i sits at position prefix_len + i and sees keys 0..prefix_len + i */
            int visible = a->prefix_len + i + 1;
            for (int h = kvh * G; h < (kvh + 1) * G; ++h) {
                const uint16_t *qrow = a->query + ((size_t)i * a->num_heads + h) * D;
                for (int d = 0; d < D; ++d)
                    q[d] = decode_elem(qrow[d], a->dtype);
                attend_one(a->out + ((size_t)i * a->num_heads + h) * D, q, K, V, visible, D, a->scale, z);
            }
        }
    }
    free(K);
    free(V);
    free(z);
    free(q);
    return NULL;
}

/*
 * Attention of one prompt chunk over the sequence's paged cache, causal:
 * query row i (position prefix_len + i) attends to keys 0 .. prefix_len + i.
 * The chunk's own K/V must already be in the cache.
 *   out [C][Hq][D] fp64; query [C][Hq][D]; block_table [>= ceil((P+C)/bs)].
 */
int oracle_prefill_chunk(double *out, const uint16_t *query, const uint16_t *k_cache,
                         const uint16_t *v_cache, const int32_t *block_table, int prefix_len,
                         int chunk_len, int num_heads, int num_kv_heads, int head_dim,
                         int block_size, int num_blocks, double scale, int dtype, int num_threads)
{
    if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || prefix_len < 0 || chunk_len < 0)
        return -2;
    if (num_threads < 1)
        num_threads = 1;
    struct prefill_args *args = calloc((size_t)num_threads, sizeof(*args));
    pthread_t *tid = calloc((size_t)num_threads, sizeof(pthread_t));
    for (int t = 0; t < num_threads; ++t) {
        struct prefill_args a = {out, query, k_cache, v_cache, block_table, prefix_len, chunk_len,
                                 num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                                 dtype, num_threads, t, 0};
        args[t] = a;
    }
    for (int t = 1; t < num_threads; ++t)
        pthread_create(&tid[t], NULL, prefill_worker, &args[t]);
    prefill_worker(&args[0]);
    int err = args[0].err;
    for (int t = 1; t < num_threads; ++t) {
        pthread_join(tid[t], NULL);
        if (args[t].err)
            err = args[t].err;
    }
    free(args);
    free(tid);
    return err;
}

/*
 * pa_oracle.c: plain, slow fp64 CPU oracle for the paged KV-cache hot path.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the bench's CPU-baseline /
 * reference leg load this library. The CUDA library never calls it, and it shares no code,
 * header, table or helper with the CUDA library.
 *
 * What it computes, and where the pages state it:
 *
 *   store   "nano-vLLM Part 4", section 3 (prefill/decode table, row "K/V work": write K/V for
 *           every new token) and the per-rank tensors list (slot mappings); the smzdm nano-vLLM
 *           deep dive, "Attention" paragraph (store_kvcache writes each new K and V row to its
 *           physical position). Each new token's K and V rows are copied bit for bit to the
 *           pool slot its slot_mapping entry names; a negative entry means "do not store".
 *
 *   decode  "nano-vLLM Part 4", section 3 (decode: one already-sampled token per sequence,
 *           attention over cached history through a block table); "mini-vLLM" (one token per
 *           sequence attending to that sequence's cached keys and values; grouped-query
 *           attention). For sequence i and query head h, with G = Hq / Hkv and kv head g = h / G:
 *               s_j = scale * sum_d q[i,h,d] * K_j[d]              for 0 <= j < ctx_i
 *               o[i,h,:] = sum_j exp(s_j - max s) V_j / sum_j exp(s_j - max s)
 *           where row j lives in physical block block_tables[i][j / bs], offset j % bs.
 *
 *   prefill "nano-vLLM Part 4", section 3 (prefill: variable-length attention with an optional
 *           prefix block table); the smzdm deep dive (cu_seqlens mark sequence boundaries; the
 *           prefix cache is in use when cu_seqlens_k exceeds cu_seqlens_q); "mini-vLLM"
 *           (several prompts concatenated, each attending causally to itself). For sequence s
 *           with q_len new rows and k_len = P + q_len keys, new row r sits at position P + r and
 *           sees keys 0 .. P + r (all k_len keys when not causal). Keys and values come from the
 *           pool through block_tables[s] when a block table is given, else from the packed k, v
 *           rows cu_seqlens_k[s] .. cu_seqlens_k[s+1].
 *
 * Readings where the pages are silent: pool layout [num_blocks, block_size, Hkv, D]; slot =
 * block * block_size + offset; int32 indices; q-head h uses kv-head h / (Hq / Hkv); the decode
 * token is already stored and counted in ctx; causal rows are aligned to the end of the keys; a
 * sequence with no keys gets a zero output row.
 *
 * All arithmetic is in double. Values are decoded from their 16-bit storage bits exactly.
 * Every function returns 0 on success or a negative code for inputs outside the contract;
 * it never aborts.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F16 0
#define ORACLE_BF16 1

#define ORACLE_OK 0
#define ORACLE_ERR_ARG (-1)     /* bad size or dtype */
#define ORACLE_ERR_SLOT (-2)    /* slot outside the pool, or two tokens to one slot */
#define ORACLE_ERR_TABLE (-3)   /* a needed block-table entry outside [0, num_blocks) */
#define ORACLE_ERR_LENGTH (-4)  /* a context longer than its table, or k_len < q_len */
#define ORACLE_ERR_NOMEM (-5)

/* IEEE 754 binary16 bits to double. Layout: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits. Exponent 0 holds subnormals (fraction * 2^-24); exponent 31 holds inf and NaN. */
double oracle_f16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, -24);
    else if (e == 31)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexp((double)(0x400 | f), e - 15 - 10);
    return sign ? -mag : mag;
}

/* bfloat16 bits to double. bfloat16 is the upper half of an IEEE binary32: 1 sign bit, 8 exponent
 * bits (bias 127), 7 fraction bits. Exponent 0 holds subnormals (fraction * 2^-133). */
double oracle_bf16_to_double(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, -126 - 7);
    else if (e == 255)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexp((double)(0x80 | f), e - 127 - 7);
    return sign ? -mag : mag;
}

static double to_double(uint16_t bits, int dtype)
{
    return dtype == ORACLE_BF16 ? oracle_bf16_to_double(bits) : oracle_f16_to_double(bits);
}

/* Vectorised decode of n storage words, for the tests' checks of the two functions above. */
void oracle_bits_to_double(const uint16_t *bits, double *out, long long n, int dtype)
{
    for (long long i = 0; i < n; ++i)
        out[i] = to_double(bits[i], dtype);
}

static void set_threads(int threads)
{
#ifdef _OPENMP
    if (threads > 0)
        omp_set_num_threads(threads);
#else
    (void)threads;
#endif
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------------------------ */
/* store                                                                                      */
/* ------------------------------------------------------------------------------------------ */

int oracle_store_kv(const uint16_t *k, const uint16_t *v, uint16_t *k_cache, uint16_t *v_cache,
                    const int32_t *slot_mapping, int T, int num_blocks, int block_size, int Hkv,
                    int D)
{
    if (T < 0 || num_blocks < 0 || block_size < 1 || Hkv < 1 || D < 1)
        return ORACLE_ERR_ARG;
    const long long num_slots = (long long)num_blocks * block_size;
    const size_t row = (size_t)Hkv * D; /* elements of one token in one pool */

    /* two tokens aimed at one slot have no defined result: refuse them */
    unsigned char *seen = calloc(num_slots > 0 ? (size_t)num_slots : 1, 1);
    if (!seen)
        return ORACLE_ERR_NOMEM;
    for (int t = 0; t < T; ++t) {
        long long s = slot_mapping[t];
        if (s < 0)
            continue;
        if (s >= num_slots || seen[s]) {
            free(seen);
            return ORACLE_ERR_SLOT;
        }
        seen[s] = 1;
    }
    free(seen);

    for (int t = 0; t < T; ++t) {
        long long s = slot_mapping[t];
        if (s < 0)
            continue;
        memcpy(k_cache + (size_t)s * row, k + (size_t)t * row, row * sizeof(uint16_t));
        memcpy(v_cache + (size_t)s * row, v + (size_t)t * row, row * sizeof(uint16_t));
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* attention of one query row over n keys                                                     */
/* ------------------------------------------------------------------------------------------ */

/* Where key/value row j of one sequence lives, for one kv head. */
typedef struct {
    const uint16_t *k_cache, *v_cache; /* pool, or NULL when rows come packed */
    const int32_t *table;              /* this sequence's block-table row */
    const uint16_t *k, *v;             /* packed rows, used when k_cache is NULL */
    long long first;                   /* packed row index of key 0 */
    int block_size, Hkv, D, g;
} key_source;

static const uint16_t *key_row(const key_source *src, int j, const uint16_t *base_pool,
                               const uint16_t *base_packed)
{
    if (src->k_cache) {
        long long block = src->table[j / src->block_size];
        long long slot = block * src->block_size + j % src->block_size;
        return base_pool + ((size_t)slot * src->Hkv + src->g) * src->D;
    }
    return base_packed + ((size_t)(src->first + j) * src->Hkv + src->g) * src->D;
}

/* out[0..D) = softmax_j(scale * q . K_j) weighted sum of V_j over j < n; zeros when n == 0.
 * s is scratch for n scores. */
static void attend_one(double *out, const uint16_t *q, const key_source *src, int n, double scale,
                       int dtype, double *s)
{
    const int D = src->D;
    for (int d = 0; d < D; ++d)
        out[d] = 0.0;
    if (n <= 0)
        return;

    double m = -INFINITY;
    for (int j = 0; j < n; ++j) {
        const uint16_t *kr = key_row(src, j, src->k_cache, src->k);
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += to_double(q[d], dtype) * to_double(kr[d], dtype);
        s[j] = scale * dot;
        if (s[j] > m)
            m = s[j];
    }
    double z = 0.0;
    for (int j = 0; j < n; ++j) {
        s[j] = exp(s[j] - m);
        z += s[j];
    }
    for (int j = 0; j < n; ++j) {
        const uint16_t *vr = key_row(src, j, src->v_cache, src->v);
        for (int d = 0; d < D; ++d)
            out[d] += s[j] * to_double(vr[d], dtype);
    }
    for (int d = 0; d < D; ++d)
        out[d] /= z;
}

static int table_ok(const int32_t *table, int n, int block_size, int num_blocks)
{
    int used = (n + block_size - 1) / block_size;
    for (int b = 0; b < used; ++b)
        if (table[b] < 0 || table[b] >= num_blocks)
            return 0;
    return 1;
}

/* ------------------------------------------------------------------------------------------ */
/* decode                                                                                     */
/* ------------------------------------------------------------------------------------------ */

int oracle_decode(double *out, const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                  const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
                  int B, int Hq, int Hkv, int D, int block_size, int num_blocks, double scale,
                  int dtype, int threads)
{
    if (B < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv || D < 1 || block_size < 1 || num_blocks < 0 ||
        max_blocks_per_seq < 0 || (dtype != ORACLE_F16 && dtype != ORACLE_BF16))
        return ORACLE_ERR_ARG;
    const int G = Hq / Hkv;
    int max_ctx = 0;
    for (int i = 0; i < B; ++i) {
        int n = context_lens[i];
        if (n < 0 || (long long)n > (long long)max_blocks_per_seq * block_size)
            return ORACLE_ERR_LENGTH;
        if (!table_ok(block_tables + (size_t)i * max_blocks_per_seq, n, block_size, num_blocks))
            return ORACLE_ERR_TABLE;
        if (n > max_ctx)
            max_ctx = n;
    }

    set_threads(threads);
    int failed = 0;
#pragma omp parallel
    {
        double *s = malloc(sizeof(double) * (size_t)(max_ctx > 0 ? max_ctx : 1));
        if (!s) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (long long w = 0; w < (long long)B * Hq; ++w) {
            if (!s)
                continue;
            int i = (int)(w / Hq), h = (int)(w % Hq);
            key_source src = {k_cache, v_cache, block_tables + (size_t)i * max_blocks_per_seq,
                              NULL, NULL, 0, block_size, Hkv, D, h / G};
            attend_one(out + ((size_t)i * Hq + h) * D, q + ((size_t)i * Hq + h) * D, &src,
                       context_lens[i], scale, dtype, s);
        }
        free(s);
    }
    return failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* varlen prefill                                                                             */
/* ------------------------------------------------------------------------------------------ */

int oracle_prefill(double *out, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                   const uint16_t *k_cache, const uint16_t *v_cache, const int32_t *cu_seqlens_q,
                   const int32_t *cu_seqlens_k, int S, const int32_t *block_tables,
                   int max_blocks_per_seq, int Hq, int Hkv, int D, int block_size, int num_blocks,
                   double scale, int causal, int dtype, int threads)
{
    if (S < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv || D < 1 || block_size < 1 || num_blocks < 0 ||
        (dtype != ORACLE_F16 && dtype != ORACLE_BF16))
        return ORACLE_ERR_ARG;
    if (block_tables && (!k_cache || !v_cache))
        return ORACLE_ERR_ARG;
    if (!block_tables && (!k || !v))
        return ORACLE_ERR_ARG;
    const int G = Hq / Hkv;
    int max_k = 0;
    for (int s = 0; s < S; ++s) {
        int ql = cu_seqlens_q[s + 1] - cu_seqlens_q[s];
        int kl = cu_seqlens_k[s + 1] - cu_seqlens_k[s];
        if (ql < 0 || kl < ql)
            return ORACLE_ERR_LENGTH;
        if (block_tables) {
            if ((long long)kl > (long long)max_blocks_per_seq * block_size)
                return ORACLE_ERR_LENGTH;
            if (!table_ok(block_tables + (size_t)s * max_blocks_per_seq, kl, block_size,
                          num_blocks))
                return ORACLE_ERR_TABLE;
        }
        if (kl > max_k)
            max_k = kl;
    }

    set_threads(threads);
    int failed = 0;
    for (int s = 0; s < S; ++s) {
        const int ql = cu_seqlens_q[s + 1] - cu_seqlens_q[s];
        const int kl = cu_seqlens_k[s + 1] - cu_seqlens_k[s];
        const int P = kl - ql; /* keys cached before this step's rows */
#pragma omp parallel
        {
            double *sc = malloc(sizeof(double) * (size_t)(max_k > 0 ? max_k : 1));
            if (!sc) {
#pragma omp atomic write
                failed = 1;
            }
#pragma omp for schedule(dynamic, 4)
            for (long long w = 0; w < (long long)ql * Hq; ++w) {
                if (!sc)
                    continue;
                int r = (int)(w / Hq), h = (int)(w % Hq);
                long long row = (long long)cu_seqlens_q[s] + r;
                key_source src = {block_tables ? k_cache : NULL,
                                  block_tables ? v_cache : NULL,
                                  block_tables ? block_tables + (size_t)s * max_blocks_per_seq
                                               : NULL,
                                  k, v, cu_seqlens_k[s], block_size, Hkv, D, h / G};
                int n = causal ? P + r + 1 : kl;
                attend_one(out + ((size_t)row * Hq + h) * D, q + ((size_t)row * Hq + h) * D,
                           &src, n, scale, dtype, sc);
            }
            free(sc);
        }
    }
    return failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

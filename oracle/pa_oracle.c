/*
 * pa_oracle.c -- float64 CPU oracle for paged-attention decode.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent checker of the
 * CUDA path: only the test suite, the smoke check and the benchmark's CPU
 * baseline may build, load or call it.  It shares no header, helper, table
 * or constant with the CUDA library, and the library never calls it.
 *
 * What it computes (plain definitions, no blocking or fusion):
 *
 *  oracle_paged_decode   -- the definition of decode attention over a
 *      block-tabled cache:  out[b,h,:] = softmax(scale * q[b,h,:] . K_b^T) V_b
 *      where K_b / V_b are the first seq_lens[b] tokens of sequence b,
 *      token t living in physical block block_tables[b][t / block_size],
 *      slot t % block_size, and query head h reads kv head h / (H / Hkv).
 *      Sources: "paged_attention_v2_triton.py" commit page, online-softmax
 *      fix (the compound partial and the softmax it reproduces);
 *      "docs" commit page, GQA grid paragraph (query heads of one group share
 *      one kv head); "qwen3_6_scripts/paged_attn.py" commit page, pre-gather
 *      paragraph (context K/V gathered by block ids).
 *
 *  oracle_partition_partials -- the method's own steps for one (seq, head):
 *      the sequence is cut into partitions of partition_size tokens; inside a
 *      partition, tiles of tile_size tokens are folded with the alpha/beta
 *      online-softmax update of the "paged_attention_v2_triton.py" commit
 *      page (online-softmax fix):
 *          p     = exp(s - m_ij)          l_ij  = sum(p)
 *          m_new = max(m_i, m_ij)          alpha = exp(m_i - m_new)
 *          beta  = exp(m_ij - m_new)       l_new = alpha*l_i + beta*l_ij
 *          acc   = acc*(alpha*l_i/l_new) + (p*beta/l_new) @ V
 *      giving the partial (max_score, exp_sum, weighted_v) of the "docs"
 *      commit page (compound type paragraph), with weighted_v normalised.
 *
 *  oracle_combine_lse / oracle_combine_fold -- the second pass that merges
 *      the partials of one (seq, head): a log-sum-exp reduce
 *      (M = max m_p, w_p = l_p exp(m_p - M), out = sum w_p acc_p / sum w_p),
 *      and the same alpha/beta rule applied partition by partition.  The
 *      "docs" commit page calls this the Phase 2 reduce over partitions.
 *
 *  oracle_prefix_attention -- chunked-prefill ("prefix") attention: sequence
 *      b already has context_lens[b] tokens in the paged cache and brings a
 *      chunk of q_len_b new tokens (rows query_start_loc[b] .. [b+1]-1 of q,
 *      k_new, v_new).  Chunk token i attends to every context token and to
 *      chunk tokens 0..i (causal inside the chunk):
 *          out = softmax(scale * q . [K_ctx ; K_new[0..i]]^T) [V_ctx ; V_new[0..i]]
 *      Source: "qwen3_6_scripts/paged_attn.py" commit page, prefix-path
 *      paragraphs (online softmax over the pre-gathered paged context, then
 *      over the current chunk with the same update).
 *
 * fp16 inputs are widened to double exactly (IEEE 754 binary16 decode written
 * from the format's definition below); all arithmetic is double.
 *
 * Return codes: 0 ok, -1 bad argument, -2 block id out of range,
 * -3 seq_len out of range.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits.  exponent 0 -> subnormal  (-1)^s * f * 2^-24,
 * exponent 31 -> inf (f == 0) or NaN, otherwise (-1)^s * (1024 + f) * 2^(e-25). */
double oracle_half_to_double(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 10) & 0x1f;
    int frac = bits & 0x3ff;
    double mag;
    if (expo == 0)
        mag = ldexp((double)frac, -24);
    else if (expo == 31)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + frac), expo - 25);
    return sign ? -mag : mag;
}

/* All 65536 binary16 values widened by oracle_half_to_double, filled once so
 * that full-size checks finish in seconds; every lookup returns exactly what
 * the function above returns. */
static double g_half_table[1 << 16];
static int g_half_table_ready = 0;

static void fill_half_table(void)
{
    if (g_half_table_ready) return;
    for (int i = 0; i < (1 << 16); ++i) g_half_table[i] = oracle_half_to_double((uint16_t)i);
    g_half_table_ready = 1;
}

#define H2D(bits) (g_half_table[(bits)])

typedef struct {
    const uint16_t *q, *k_cache, *v_cache;
    const int32_t *block_tables, *seq_lens;
    int num_seqs, max_blocks_per_seq, num_heads, num_kv_heads, head_dim, block_size;
    long long num_blocks;
    double scale;
} oracle_problem;

static int check_problem(const oracle_problem* P)
{
    if (!P->q || !P->k_cache || !P->v_cache || !P->block_tables || !P->seq_lens) return -1;
    if (P->num_seqs < 0 || P->num_heads <= 0 || P->num_kv_heads <= 0 || P->head_dim <= 0 ||
        P->block_size <= 0 || P->max_blocks_per_seq < 0 || P->num_blocks < 0)
        return -1;
    if (P->num_heads % P->num_kv_heads) return -1;
    return 0;
}

/* Address of element d of token t of sequence b for kv head g in a cache laid
 * out [num_blocks][num_kv_heads][block_size][head_dim]; NULL when the block
 * id is out of range. */
static const uint16_t* token_row(const oracle_problem* P, const uint16_t* cache, int b, int g, int t)
{
    int logical_block = t / P->block_size;
    int slot = t % P->block_size;
    int32_t phys = P->block_tables[(long long)b * P->max_blocks_per_seq + logical_block];
    if (phys < 0 || (long long)phys >= P->num_blocks) return NULL;
    long long row = ((long long)phys * P->num_kv_heads + g) * P->block_size + slot;
    return cache + row * P->head_dim;
}

static int check_seq(const oracle_problem* P, int b)
{
    int L = P->seq_lens[b];
    if (L < 0 || (long long)L > (long long)P->max_blocks_per_seq * P->block_size) return -3;
    return 0;
}

/* score s_t = scale * sum_d q[d] * k_t[d] for every token of sequence b. */
static int scores_of(const oracle_problem* P, int b, int h, double* s)
{
    int G = P->num_heads / P->num_kv_heads;
    int g = h / G;
    int L = P->seq_lens[b];
    const uint16_t* qv = P->q + ((long long)b * P->num_heads + h) * P->head_dim;
    for (int t = 0; t < L; ++t) {
        const uint16_t* k = token_row(P, P->k_cache, b, g, t);
        if (!k) return -2;
        double dot = 0.0;
        for (int d = 0; d < P->head_dim; ++d)
            dot += H2D(qv[d]) * H2D(k[d]);
        s[t] = P->scale * dot;
    }
    return 0;
}

/* The definition, for one (seq, head): out = sum_t e^{s_t - M} v_t / sum_t e^{s_t - M}. */
static int decode_one(const oracle_problem* P, int b, int h, double* out, double* s)
{
    int G = P->num_heads / P->num_kv_heads;
    int g = h / G;
    int L = P->seq_lens[b];
    int D = P->head_dim;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (L == 0) return 0; /* empty sequence: output is zero */
    int rc = scores_of(P, b, h, s);
    if (rc) return rc;
    double M = -INFINITY;
    for (int t = 0; t < L; ++t)
        if (s[t] > M) M = s[t];
    double denom = 0.0;
    for (int t = 0; t < L; ++t) {
        double w = exp(s[t] - M);
        const uint16_t* v = token_row(P, P->v_cache, b, g, t);
        denom += w;
        for (int d = 0; d < D; ++d) out[d] += w * H2D(v[d]);
    }
    for (int d = 0; d < D; ++d) out[d] /= denom;
    return 0;
}

static oracle_problem make_problem(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                   const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                                   int max_blocks_per_seq, int num_heads, int num_kv_heads, int head_dim,
                                   int block_size, long long num_blocks, double scale)
{
    oracle_problem P;
    fill_half_table();
    P.q = q; P.k_cache = k_cache; P.v_cache = v_cache;
    P.block_tables = block_tables; P.seq_lens = seq_lens;
    P.num_seqs = num_seqs; P.max_blocks_per_seq = max_blocks_per_seq;
    P.num_heads = num_heads; P.num_kv_heads = num_kv_heads; P.head_dim = head_dim;
    P.block_size = block_size; P.num_blocks = num_blocks; P.scale = scale;
    return P;
}

/* out: double [num_seqs][num_heads][head_dim].  threads <= 0: library default. */
int oracle_paged_decode(double* out, const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                        const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                        int max_blocks_per_seq, int num_heads, int num_kv_heads, int head_dim,
                        int block_size, long long num_blocks, double scale, int threads)
{
    oracle_problem P = make_problem(q, k_cache, v_cache, block_tables, seq_lens, num_seqs,
                                    max_blocks_per_seq, num_heads, num_kv_heads, head_dim,
                                    block_size, num_blocks, scale);
    if (!out || check_problem(&P)) return -1;
    int max_len = 0;
    for (int b = 0; b < num_seqs; ++b) {
        if (check_seq(&P, b)) return -3;
        if (seq_lens[b] > max_len) max_len = seq_lens[b];
    }
    long long pairs = (long long)num_seqs * num_heads;
    int status = 0;
    (void)threads;
#ifdef _OPENMP
    int nt = threads > 0 ? threads : omp_get_max_threads();
#pragma omp parallel num_threads(nt)
#endif
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
        int local = s ? 0 : -1;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (long long i = 0; i < pairs; ++i) {
            int b = (int)(i / num_heads), h = (int)(i % num_heads);
            int rc = s ? decode_one(&P, b, h, out + i * head_dim, s) : -1;
            if (rc) local = rc;
        }
        free(s);
        if (local) {
#ifdef _OPENMP
#pragma omp critical
#endif
            status = local;
        }
    }
    return status;
}

/* One (seq, head) of the definition; used for sampled checks at full size. */
int oracle_paged_decode_one(double* out, const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                            const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                            int max_blocks_per_seq, int num_heads, int num_kv_heads, int head_dim,
                            int block_size, long long num_blocks, double scale, int b, int h)
{
    oracle_problem P = make_problem(q, k_cache, v_cache, block_tables, seq_lens, num_seqs,
                                    max_blocks_per_seq, num_heads, num_kv_heads, head_dim,
                                    block_size, num_blocks, scale);
    if (!out || check_problem(&P) || b < 0 || b >= num_seqs || h < 0 || h >= num_heads) return -1;
    if (check_seq(&P, b)) return -3;
    int L = seq_lens[b];
    double* s = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    if (!s) return -1;
    int rc = decode_one(&P, b, h, out, s);
    free(s);
    return rc;
}

/* The method's first pass for one (seq b, head h): for each partition p of
 * partition_size tokens, fold tiles of tile_size tokens with the alpha/beta
 * rule.  Writes n = ceil(L / partition_size) partials:
 *   m_out[p] = running max score, l_out[p] = exp-sum relative to it,
 *   acc_out[p*D + d] = weighted V, normalised by l_out[p].
 * Returns n (>= 0) or a negative error code. */
int oracle_partition_partials(double* m_out, double* l_out, double* acc_out, const uint16_t* q,
                              const uint16_t* k_cache, const uint16_t* v_cache, const int32_t* block_tables,
                              const int32_t* seq_lens, int num_seqs, int max_blocks_per_seq, int num_heads,
                              int num_kv_heads, int head_dim, int block_size, long long num_blocks,
                              double scale, int b, int h, int partition_size, int tile_size)
{
    oracle_problem P = make_problem(q, k_cache, v_cache, block_tables, seq_lens, num_seqs,
                                    max_blocks_per_seq, num_heads, num_kv_heads, head_dim,
                                    block_size, num_blocks, scale);
    if (check_problem(&P) || b < 0 || b >= num_seqs || h < 0 || h >= num_heads) return -1;
    if (partition_size <= 0 || tile_size <= 0) return -1;
    if (check_seq(&P, b)) return -3;
    int G = num_heads / num_kv_heads, g = h / G, D = head_dim;
    int L = seq_lens[b];
    int n = (L + partition_size - 1) / partition_size;
    double* s = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    double* pv = (double*)malloc(sizeof(double) * (size_t)D);
    double* p_tile = (double*)malloc(sizeof(double) * (size_t)tile_size);
    if (!s || !pv || !p_tile) { free(s); free(pv); free(p_tile); return -1; }
    int rc = scores_of(&P, b, h, s);
    if (rc) { free(s); free(pv); free(p_tile); return rc; }

    for (int part = 0; part < n; ++part) {
        int t0 = part * partition_size;
        int t1 = t0 + partition_size < L ? t0 + partition_size : L;
        double m_i = -INFINITY, l_i = 0.0;
        double* acc = acc_out + (long long)part * D;
        for (int d = 0; d < D; ++d) acc[d] = 0.0;
        for (int a = t0; a < t1; a += tile_size) {
            int e = a + tile_size < t1 ? a + tile_size : t1;
            /* p = exp(s - m_ij), l_ij = sum(p): probabilities relative to the tile max */
            double m_ij = -INFINITY;
            for (int t = a; t < e; ++t)
                if (s[t] > m_ij) m_ij = s[t];
            double l_ij = 0.0;
            for (int t = a; t < e; ++t) {
                p_tile[t - a] = exp(s[t] - m_ij);
                l_ij += p_tile[t - a];
            }
            /* m_new, alpha (old accumulator), beta (new tile), l_new */
            double m_new = m_i > m_ij ? m_i : m_ij;
            double alpha = exp(m_i - m_new); /* m_i = -inf on the first tile gives 0 */
            double beta = exp(m_ij - m_new);
            double l_new = alpha * l_i + beta * l_ij;
            /* (p @ V) for this tile */
            for (int d = 0; d < D; ++d) pv[d] = 0.0;
            for (int t = a; t < e; ++t) {
                const uint16_t* v = token_row(&P, P.v_cache, b, g, t);
                if (!v) { free(s); free(pv); free(p_tile); return -2; }
                for (int d = 0; d < D; ++d) pv[d] += p_tile[t - a] * H2D(v[d]);
            }
            /* acc = acc * (alpha * l_i / l_new) + (beta / l_new) * (p @ V) */
            double keep = alpha * l_i / l_new;
            double take = beta / l_new;
            for (int d = 0; d < D; ++d) acc[d] = acc[d] * keep + take * pv[d];
            m_i = m_new;
            l_i = l_new;
        }
        m_out[part] = m_i;
        l_out[part] = l_i;
    }
    free(s); free(pv); free(p_tile);
    return n;
}

/* Second pass, log-sum-exp form: M = max_p m_p, w_p = l_p e^{m_p - M},
 * out = sum_p w_p acc_p / sum_p w_p.  n == 0 gives a zero output. */
int oracle_combine_lse(double* out, const double* m, const double* l, const double* acc, int n, int head_dim)
{
    if (!out || n < 0 || head_dim <= 0) return -1;
    for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
    if (n == 0) return 0;
    double M = -INFINITY;
    for (int p = 0; p < n; ++p)
        if (m[p] > M) M = m[p];
    double W = 0.0;
    for (int p = 0; p < n; ++p) {
        double w = l[p] * exp(m[p] - M);
        W += w;
        for (int d = 0; d < head_dim; ++d) out[d] += w * acc[(long long)p * head_dim + d];
    }
    for (int d = 0; d < head_dim; ++d) out[d] /= W;
    return 0;
}

/* Second pass, sequential form: the alpha/beta rule applied with each
 * partition's (m_p, l_p, acc_p) in the role of a tile. */
int oracle_combine_fold(double* out, const double* m, const double* l, const double* acc, int n, int head_dim)
{
    if (!out || n < 0 || head_dim <= 0) return -1;
    for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
    double m_i = -INFINITY, l_i = 0.0;
    for (int p = 0; p < n; ++p) {
        double m_new = m_i > m[p] ? m_i : m[p];
        double alpha = exp(m_i - m_new);
        double beta = exp(m[p] - m_new);
        double l_new = alpha * l_i + beta * l[p];
        double keep = alpha * l_i / l_new;
        double take = beta * l[p] / l_new;
        for (int d = 0; d < head_dim; ++d) out[d] = out[d] * keep + take * acc[(long long)p * head_dim + d];
        m_i = m_new;
        l_i = l_new;
    }
    return 0;
}


/* Chunked-prefill attention, the definition, for one (new token, head).
 * tok indexes the packed new tokens; its sequence b is the one whose
 * [query_start_loc[b], query_start_loc[b+1]) range holds it. */
static int prefix_one(double* out, double* s, const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                      const oracle_problem* P, const int32_t* context_lens, const int32_t* query_start_loc,
                      int b, int tok, int h)
{
    int G = P->num_heads / P->num_kv_heads, g = h / G, D = P->head_dim;
    int C = context_lens[b];
    int i = tok - query_start_loc[b];
    const uint16_t* qv = q + ((long long)tok * P->num_heads + h) * D;
    int n = C + i + 1;
    for (int t = 0; t < n; ++t) {
        const uint16_t* k;
        if (t < C) {
            k = token_row(P, P->k_cache, b, g, t);
            if (!k) return -2;
        } else {
            k = k_new + ((long long)(query_start_loc[b] + (t - C)) * P->num_kv_heads + g) * D;
        }
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += H2D(qv[d]) * H2D(k[d]);
        s[t] = P->scale * dot;
    }
    double M = -INFINITY;
    for (int t = 0; t < n; ++t)
        if (s[t] > M) M = s[t];
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    double denom = 0.0;
    for (int t = 0; t < n; ++t) {
        double w = exp(s[t] - M);
        const uint16_t* v = t < C ? token_row(P, P->v_cache, b, g, t)
                                  : v_new + ((long long)(query_start_loc[b] + (t - C)) * P->num_kv_heads + g) * D;
        denom += w;
        for (int d = 0; d < D; ++d) out[d] += w * H2D(v[d]);
    }
    for (int d = 0; d < D; ++d) out[d] /= denom;
    return 0;
}

static int check_prefix(const oracle_problem* P, const int32_t* context_lens, const int32_t* query_start_loc,
                        int num_tokens, int* max_keys)
{
    if (!context_lens || !query_start_loc || num_tokens < 0) return -1;
    if (query_start_loc[0] != 0 || query_start_loc[P->num_seqs] != num_tokens) return -1;
    *max_keys = 1;
    for (int b = 0; b < P->num_seqs; ++b) {
        int C = context_lens[b], ql = query_start_loc[b + 1] - query_start_loc[b];
        if (ql < 0) return -1;
        if (C < 0 || (long long)C > (long long)P->max_blocks_per_seq * P->block_size) return -3;
        if (C + ql > *max_keys) *max_keys = C + ql;
    }
    return 0;
}

/* out: double [num_tokens][num_heads][head_dim]. */
int oracle_prefix_attention(double* out, const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                            const uint16_t* k_cache, const uint16_t* v_cache, const int32_t* block_tables,
                            const int32_t* context_lens, const int32_t* query_start_loc, int num_seqs,
                            int num_tokens, int max_blocks_per_seq, int num_heads, int num_kv_heads, int head_dim,
                            int block_size, long long num_blocks, double scale, int threads)
{
    oracle_problem P = make_problem(q, k_cache, v_cache, block_tables, context_lens, num_seqs, max_blocks_per_seq,
                                    num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale);
    if (!out || !k_new || !v_new || check_problem(&P)) return -1;
    int max_keys = 1;
    int rc = check_prefix(&P, context_lens, query_start_loc, num_tokens, &max_keys);
    if (rc) return rc;
    long long rows = (long long)num_tokens * num_heads;
    int status = 0;
    (void)threads;
#ifdef _OPENMP
    int nt = threads > 0 ? threads : omp_get_max_threads();
#pragma omp parallel num_threads(nt)
#endif
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)max_keys);
        int local = s ? 0 : -1;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
        for (long long r = 0; r < rows; ++r) {
            int tok = (int)(r / num_heads), h = (int)(r % num_heads);
            int b = 0;
            while (b + 1 < num_seqs && query_start_loc[b + 1] <= tok) ++b;
            int e = s ? prefix_one(out + r * head_dim, s, q, k_new, v_new, &P, context_lens, query_start_loc, b,
                                   tok, h)
                      : -1;
            if (e) local = e;
        }
        free(s);
        if (local) {
#ifdef _OPENMP
#pragma omp critical
#endif
            status = local;
        }
    }
    return status;
}

/* One (new token, head) of the definition, for sampled checks at full size. */
int oracle_prefix_attention_one(double* out, const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                                const uint16_t* k_cache, const uint16_t* v_cache, const int32_t* block_tables,
                                const int32_t* context_lens, const int32_t* query_start_loc, int num_seqs,
                                int num_tokens, int max_blocks_per_seq, int num_heads, int num_kv_heads,
                                int head_dim, int block_size, long long num_blocks, double scale, int tok, int h)
{
    oracle_problem P = make_problem(q, k_cache, v_cache, block_tables, context_lens, num_seqs, max_blocks_per_seq,
                                    num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale);
    if (!out || !k_new || !v_new || check_problem(&P) || tok < 0 || tok >= num_tokens || h < 0 || h >= num_heads)
        return -1;
    int max_keys = 1;
    int rc = check_prefix(&P, context_lens, query_start_loc, num_tokens, &max_keys);
    if (rc) return rc;
    int b = 0;
    while (b + 1 < num_seqs && query_start_loc[b + 1] <= tok) ++b;
    double* s = (double*)malloc(sizeof(double) * (size_t)max_keys);
    if (!s) return -1;
    rc = prefix_one(out, s, q, k_new, v_new, &P, context_lens, query_start_loc, b, tok, h);
    free(s);
    return rc;
}

/*
 * oracle.c -- plain fp64 CPU reference for paged decode attention and the
 * KV-cache append.
 *
 * TEST INFRASTRUCTURE. Only the test-suite, the package smoke check and the
 * CPU-baseline leg of the benchmark load this file's library. No product code
 * path links or calls it, and it shares no code with the CUDA library: it has
 * its own bf16 decoding, its own block-table gather and its own softmax.
 *
 * What it computes (definitions, written out with no blocking or fusion):
 *
 *  - Paged KV cache: K and V are each [num_blocks][block_size][num_kv_heads]
 *    [head_dim] bf16 ("LLM Inference Serving", KV-cache shape section); a
 *    sequence's block table maps logical block i (tokens 16i..16i+15) to a
 *    physical block ("ML Interview Prep, Lesson 13", section 3.5 "Paged
 *    attention"; "07 -- Inference", section 2.2 diagram A -> [0, 3, 5]).
 *
 *  - Append ("LLM Inference Serving", block-table pseudo-code: append in place
 *    into the last block's free slot): new token i goes to physical block
 *    slot/16, offset slot%16; a negative slot is padding and is skipped.
 *
 *  - Attention: PagedAttention gives exactly the attention of the sequence's
 *    logical tokens ("07 -- Inference", section 5.1: the online softmax is exact,
 *    not an approximation), so the oracle gathers the blocks into a contiguous
 *    fp64 K_s, V_s and evaluates softmax(scale * q K_s^T) V_s in fp64. With
 *    n_query_per_seq = nq, query j (0-based) of a sequence of T tokens sits at
 *    position T - nq + j and sees positions 0 .. T - nq + j (the causal mask of
 *    speculative verification: "LLM Serving: Continuous Batching &
 *    PagedAttention", section on speculative decoding mechanics). Query head qh
 *    reads kv head qh / (num_q_heads / num_kv_heads) (grouped-query attention,
 *    "ML Interview Prep, Lesson 13", section 3.3). A row that sees no token
 *    (T < nq) is defined as all zeros.
 *
 *  - Copy-on-write block copy ("ML Interview Prep, Lesson 13", section 3.5
 *    "Sharing": before a sequence writes into a block whose reference count is
 *    above 1 it gets a private copy): for each (src, dst) pair, in order, all
 *    16 token rows of physical block src are copied to block dst, in K and in
 *    V. A pair naming a block outside the pool copies nothing.
 *
 *  - Split and merge ("07 -- Inference", section 5.3 FlashDecoding): a token
 *    range gives a partial (m, l, acc) with m = max score, l = sum exp(x - m),
 *    acc = sum exp(x - m) V; partials merge with the same rescaling rule as the
 *    online softmax. These two routines are separate from the definition above
 *    so the tests can check the merge rule against it.
 *
 * Parity: pinned (dense library attention, permutation invariance, weight sums,
 * shared == copied, closed forms, the page's block-table diagram, merge algebra;
 * block copy: the copy-on-write worked example and read-back of every
 * sequence's logical tokens through a simulated pool).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the upper half of an IEEE binary32; widening it is exact. */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_kv_append(const uint16_t *k_new, const uint16_t *v_new,
                     const int64_t *slot_mapping, int64_t n_new,
                     uint16_t *k_cache, uint16_t *v_cache, int64_t num_blocks,
                     int32_t block_size, int32_t num_kv_heads, int32_t head_dim)
{
    const int64_t row = (int64_t)num_kv_heads * head_dim; /* elements per token */
    int bad = 0;
    for (int64_t i = 0; i < n_new; ++i) {
        const int64_t slot = slot_mapping[i];
        if (slot < 0)
            continue; /* padding */
        const int64_t blk = slot / block_size;
        const int64_t off = slot % block_size;
        if (blk >= num_blocks) {
            bad = 1; /* out of the pool: nothing written */
            continue;
        }
        const int64_t dst = (blk * block_size + off) * row;
        for (int64_t e = 0; e < row; ++e) {
            k_cache[dst + e] = k_new[i * row + e];
            v_cache[dst + e] = v_new[i * row + e];
        }
    }
    return bad ? -1 : 0;
}

int oracle_copy_blocks(uint16_t *k_cache, uint16_t *v_cache, int64_t num_blocks,
                       int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                       const int32_t *src, const int32_t *dst, int64_t n_pairs)
{
    const int64_t blk = (int64_t)block_size * num_kv_heads * head_dim; /* elements per block */
    int bad = 0;
    for (int64_t i = 0; i < n_pairs; ++i) {
        const int64_t a = src[i], b = dst[i];
        if (a < 0 || a >= num_blocks || b < 0 || b >= num_blocks) {
            bad = 1;
            continue;
        }
        for (int64_t e = 0; e < blk; ++e) {
            k_cache[b * blk + e] = k_cache[a * blk + e];
            v_cache[b * blk + e] = v_cache[a * blk + e];
        }
    }
    return bad ? -1 : 0;
}

/* Copy the first T tokens of (sequence s, kv head h) into contiguous fp64
 * K[T][D] and V[T][D], following the block table. Returns -1 if a block id
 * the context needs is outside the pool. */
static int gather_kv(const uint16_t *k_cache, const uint16_t *v_cache, int64_t num_blocks,
                     int32_t block_size, const int32_t *table, int32_t T,
                     int32_t num_kv_heads, int32_t head_dim, int32_t h,
                     double *K, double *V)
{
    for (int32_t t = 0; t < T; ++t) {
        const int32_t logical = t / block_size;
        const int32_t off = t % block_size;
        const int64_t phys = table[logical];
        if (phys < 0 || phys >= num_blocks)
            return -1;
        const int64_t base = ((phys * block_size + off) * num_kv_heads + h) * (int64_t)head_dim;
        for (int32_t d = 0; d < head_dim; ++d) {
            K[(int64_t)t * head_dim + d] = bf16_to_double(k_cache[base + d]);
            V[(int64_t)t * head_dim + d] = bf16_to_double(v_cache[base + d]);
        }
    }
    return 0;
}

/* Softmax weights of one query row over the visible tokens 0..lim (others 0).
 * x_t = scale * <q, K_t>; w_t = exp(x_t - max x) / sum exp(x - max x). */
static void row_weights(const double *qrow, const double *K, int32_t T, int32_t lim,
                        int32_t head_dim, double scale, double *w)
{
    double mx = -INFINITY;
    for (int32_t t = 0; t < T; ++t) {
        if (t > lim) {
            w[t] = 0.0;
            continue;
        }
        double dot = 0.0;
        for (int32_t d = 0; d < head_dim; ++d)
            dot += qrow[d] * K[(int64_t)t * head_dim + d];
        w[t] = scale * dot;
        if (w[t] > mx)
            mx = w[t];
    }
    double z = 0.0;
    for (int32_t t = 0; t <= lim && t < T; ++t) {
        w[t] = exp(w[t] - mx);
        z += w[t];
    }
    for (int32_t t = 0; t <= lim && t < T; ++t)
        w[t] /= z;
}

static int check_shapes(int32_t num_seqs, int32_t nq, int32_t num_q_heads,
                        int32_t num_kv_heads, int32_t head_dim, int32_t block_size)
{
    if (num_seqs < 0 || nq < 1 || num_kv_heads < 1 || num_q_heads < 1 || head_dim < 1 ||
        block_size < 1 || num_q_heads % num_kv_heads != 0)
        return -1;
    return 0;
}

/* T_s clamped to what the block table can hold (a longer context is invalid
 * input; both sides of the parity tests treat it as the table's capacity). */
static int32_t eff_len(const int32_t *context_lens, int32_t s, int32_t mb, int32_t block_size)
{
    int32_t T = context_lens[s];
    if (T < 0)
        T = 0;
    if ((int64_t)T > (int64_t)mb * block_size)
        T = mb * block_size;
    return T;
}

/*
 * out[(s*nq + j)][qh][d] (fp64), for every sequence s, query j, query head qh.
 * pair_mask (optional, [num_seqs][num_kv_heads]) restricts the work to the
 * selected (sequence, kv head) pairs; rows of other pairs are left untouched.
 */
int oracle_paged_attention(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                           int64_t num_blocks, int32_t block_size,
                           const int32_t *block_tables, int32_t max_blocks_per_seq,
                           const int32_t *context_lens, int32_t num_seqs,
                           int32_t n_query_per_seq, int32_t num_q_heads, int32_t num_kv_heads,
                           int32_t head_dim, float scale, const uint8_t *pair_mask,
                           double *out, int32_t num_threads)
{
    if (check_shapes(num_seqs, n_query_per_seq, num_q_heads, num_kv_heads, head_dim, block_size))
        return -2;
    const int32_t group = num_q_heads / num_kv_heads;
    const int64_t npairs = (int64_t)num_seqs * num_kv_heads;
    int status = 0;
#ifdef _OPENMP
    if (num_threads > 0)
        omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t pair = 0; pair < npairs; ++pair) {
        const int32_t s = (int32_t)(pair / num_kv_heads);
        const int32_t h = (int32_t)(pair % num_kv_heads);
        if (pair_mask && !pair_mask[pair])
            continue;
        const int32_t T = eff_len(context_lens, s, max_blocks_per_seq, block_size);
        double *K = (double *)malloc(sizeof(double) * ((size_t)T * head_dim + 1));
        double *V = (double *)malloc(sizeof(double) * ((size_t)T * head_dim + 1));
        double *w = (double *)malloc(sizeof(double) * ((size_t)T + 1));
        double *qrow = (double *)malloc(sizeof(double) * (size_t)head_dim);
        int bad = gather_kv(k_cache, v_cache, num_blocks, block_size,
                            block_tables + (int64_t)s * max_blocks_per_seq, T,
                            num_kv_heads, head_dim, h, K, V);
        if (bad) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            status = -1;
        }
        for (int32_t j = 0; j < n_query_per_seq && !bad; ++j) {
            const int32_t lim = T - n_query_per_seq + j; /* last visible position */
            for (int32_t g = 0; g < group; ++g) {
                const int32_t qh = h * group + g;
                const int64_t row = ((int64_t)s * n_query_per_seq + j) * num_q_heads + qh;
                double *o = out + row * head_dim;
                for (int32_t d = 0; d < head_dim; ++d)
                    o[d] = 0.0;
                if (lim < 0 || T == 0)
                    continue; /* sees no token */
                for (int32_t d = 0; d < head_dim; ++d)
                    qrow[d] = bf16_to_double(q[row * head_dim + d]);
                row_weights(qrow, K, T, lim, head_dim, (double)scale, w);
                for (int32_t t = 0; t <= lim && t < T; ++t)
                    for (int32_t d = 0; d < head_dim; ++d)
                        o[d] += w[t] * V[(int64_t)t * head_dim + d];
            }
        }
        free(K);
        free(V);
        free(w);
        free(qrow);
    }
    return status;
}

/* The softmax weights of one query row (sequence s, query j, query head qh):
 * w[0..T-1], zero past the row's causal limit. Returns T, or -1 on error. */
int oracle_attention_weights(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                             int64_t num_blocks, int32_t block_size,
                             const int32_t *block_tables, int32_t max_blocks_per_seq,
                             const int32_t *context_lens, int32_t num_seqs,
                             int32_t n_query_per_seq, int32_t num_q_heads, int32_t num_kv_heads,
                             int32_t head_dim, float scale, int32_t s, int32_t j, int32_t qh,
                             double *w)
{
    if (check_shapes(num_seqs, n_query_per_seq, num_q_heads, num_kv_heads, head_dim, block_size) ||
        s < 0 || s >= num_seqs || j < 0 || j >= n_query_per_seq || qh < 0 || qh >= num_q_heads)
        return -1;
    const int32_t group = num_q_heads / num_kv_heads;
    const int32_t h = qh / group;
    const int32_t T = eff_len(context_lens, s, max_blocks_per_seq, block_size);
    const int32_t lim = T - n_query_per_seq + j;
    double *K = (double *)malloc(sizeof(double) * ((size_t)T * head_dim + 1));
    double *V = (double *)malloc(sizeof(double) * ((size_t)T * head_dim + 1));
    double *qrow = (double *)malloc(sizeof(double) * (size_t)head_dim);
    int bad = gather_kv(k_cache, v_cache, num_blocks, block_size,
                        block_tables + (int64_t)s * max_blocks_per_seq, T, num_kv_heads,
                        head_dim, h, K, V);
    if (!bad) {
        const int64_t row = ((int64_t)s * n_query_per_seq + j) * num_q_heads + qh;
        for (int32_t d = 0; d < head_dim; ++d)
            qrow[d] = bf16_to_double(q[row * head_dim + d]);
        if (lim < 0) {
            for (int32_t t = 0; t < T; ++t)
                w[t] = 0.0;
        } else {
            row_weights(qrow, K, T, lim, head_dim, (double)scale, w);
        }
    }
    free(K);
    free(V);
    free(qrow);
    return bad ? -1 : T;
}

/*
 * The partial state of one query row over the token range [t_begin, t_end)
 * intersected with its visible tokens ("07 -- Inference", section 5.3): m is the
 * largest score in the range (-inf if none), l = sum exp(x_t - m) and
 * acc[d] = sum exp(x_t - m) V_t[d] (both 0 if the range sees nothing).
 */
int oracle_partial_state(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                         int64_t num_blocks, int32_t block_size,
                         const int32_t *block_tables, int32_t max_blocks_per_seq,
                         const int32_t *context_lens, int32_t num_seqs,
                         int32_t n_query_per_seq, int32_t num_q_heads, int32_t num_kv_heads,
                         int32_t head_dim, float scale, int32_t s, int32_t j, int32_t qh,
                         int32_t t_begin, int32_t t_end, double *m_out, double *l_out,
                         double *acc)
{
    if (check_shapes(num_seqs, n_query_per_seq, num_q_heads, num_kv_heads, head_dim, block_size) ||
        s < 0 || s >= num_seqs || j < 0 || j >= n_query_per_seq || qh < 0 || qh >= num_q_heads)
        return -1;
    const int32_t group = num_q_heads / num_kv_heads;
    const int32_t h = qh / group;
    const int32_t T = eff_len(context_lens, s, max_blocks_per_seq, block_size);
    const int32_t lim = T - n_query_per_seq + j;
    double *K = (double *)malloc(sizeof(double) * ((size_t)T * head_dim + 1));
    double *V = (double *)malloc(sizeof(double) * ((size_t)T * head_dim + 1));
    double *x = (double *)malloc(sizeof(double) * ((size_t)T + 1));
    double *qrow = (double *)malloc(sizeof(double) * (size_t)head_dim);
    int bad = gather_kv(k_cache, v_cache, num_blocks, block_size,
                        block_tables + (int64_t)s * max_blocks_per_seq, T, num_kv_heads,
                        head_dim, h, K, V);
    double m = -INFINITY, l = 0.0;
    for (int32_t d = 0; d < head_dim; ++d)
        acc[d] = 0.0;
    if (!bad) {
        const int64_t row = ((int64_t)s * n_query_per_seq + j) * num_q_heads + qh;
        for (int32_t d = 0; d < head_dim; ++d)
            qrow[d] = bf16_to_double(q[row * head_dim + d]);
        int32_t lo = t_begin < 0 ? 0 : t_begin;
        int32_t hi = t_end;
        if (hi > lim + 1)
            hi = lim + 1;
        if (hi > T)
            hi = T;
        for (int32_t t = lo; t < hi; ++t) {
            double dot = 0.0;
            for (int32_t d = 0; d < head_dim; ++d)
                dot += qrow[d] * K[(int64_t)t * head_dim + d];
            x[t] = (double)scale * dot;
            if (x[t] > m)
                m = x[t];
        }
        for (int32_t t = lo; t < hi; ++t) {
            const double e = exp(x[t] - m);
            l += e;
            for (int32_t d = 0; d < head_dim; ++d)
                acc[d] += e * V[(int64_t)t * head_dim + d];
        }
    }
    *m_out = m;
    *l_out = l;
    free(K);
    free(V);
    free(x);
    free(qrow);
    return bad ? -1 : 0;
}

/* Merge n partial states (m[i], l[i], acc[i][D]) into the normalised output:
 * M = max m_i, L = sum l_i exp(m_i - M), out = sum acc_i exp(m_i - M) / L
 * (zeros if no partial saw a token). */
void oracle_merge_states(int32_t n, int32_t head_dim, const double *m, const double *l,
                         const double *acc, double *out)
{
    double M = -INFINITY;
    for (int32_t i = 0; i < n; ++i)
        if (m[i] > M)
            M = m[i];
    for (int32_t d = 0; d < head_dim; ++d)
        out[d] = 0.0;
    if (M == -INFINITY)
        return;
    double L = 0.0;
    for (int32_t i = 0; i < n; ++i) {
        if (m[i] == -INFINITY)
            continue;
        const double f = exp(m[i] - M);
        L += l[i] * f;
        for (int32_t d = 0; d < head_dim; ++d)
            out[d] += acc[(int64_t)i * head_dim + d] * f;
    }
    for (int32_t d = 0; d < head_dim; ++d)
        out[d] /= L;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------
 * FP8 (E4M3) KV cache.
 *
 * "ML Interview Prep, Lesson 13", section 3.7 (an fp8 or int8 KV cache stores
 * keys and values in 8 bits while the matmuls still run at 16 bits: twice the
 * tokens in memory, half the KV read time) and "07 -- Inference", section 4.3
 * (E4M3 for inference, largest magnitude 448; per-tensor, per-channel or
 * per-block scales). Reading: one float scale per kv head for K and one for V;
 * a stored code c of head h stands for decode(c) * scale[h].
 *
 * E4M3 ("fn" variant of the OCP 8-bit floating point format): sign bit,
 * 4 exponent bits with bias 7, 3 mantissa bits. Exponent field 0 holds the
 * subnormals m * 2^-9; S.1111.111 is NaN; there are no infinities, so the
 * largest finite magnitude is 1.75 * 2^8 = 448.
 * ---------------------------------------------------------------------- */

double oracle_e4m3_decode(uint8_t c)
{
    const int e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7)
        return NAN;
    const double v = (e == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    return (c & 0x80) ? -v : v;
}

/* Nearest E4M3 value, ties to the even code; magnitudes whose rounded value
 * exceeds 448 (and infinities) give 448 with the sign kept; NaN gives 0x7F. */
uint8_t oracle_e4m3_encode(float x)
{
    if (isnan(x))
        return 0x7F;
    const uint8_t sgn = signbit(x) ? 0x80 : 0x00;
    const double a = fabs((double)x);
    if (isinf(a))
        return sgn | 0x7E;
    int k;
    frexp(a, &k); /* a = f * 2^k, f in [0.5, 1): floor(log2 a) = k - 1 */
    int E = k - 1;
    if (a == 0.0 || E < -6) {
        /* subnormal range: grid step 2^-9; the code is the step count (8 = 2^-6) */
        const double n = nearbyint(ldexp(a, 9));
        return sgn | (uint8_t)n;
    }
    double n = nearbyint(ldexp(a, 3 - E)); /* 8 .. 16 steps of 2^(E-3) */
    if (n == 16.0) {
        E += 1;
        n = 8.0;
    }
    const int field = E + 7;
    if (field > 15 || (field == 15 && n - 8.0 > 6.0))
        return sgn | 0x7E; /* beyond 448: saturate */
    return sgn | (uint8_t)((field << 3) | (int)(n - 8.0));
}

/* The fp8 append: for every new token i with slot >= 0 and every kv head h,
 * code = encode(k_new / k_scale[h]) (bf16 widened to float, divided in float
 * with round-to-nearest), stored at block slot/16, offset slot%16; V likewise. */
int oracle_kv_append_fp8(const uint16_t *k_new, const uint16_t *v_new,
                         const int64_t *slot_mapping, int64_t n_new,
                         uint8_t *k_cache, uint8_t *v_cache, int64_t num_blocks,
                         int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                         const float *k_scale, const float *v_scale)
{
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    int bad = 0;
    for (int64_t i = 0; i < n_new; ++i) {
        const int64_t slot = slot_mapping[i];
        if (slot < 0)
            continue;
        const int64_t blk = slot / block_size;
        const int64_t off = slot % block_size;
        if (blk >= num_blocks) {
            bad = 1;
            continue;
        }
        for (int32_t h = 0; h < num_kv_heads; ++h) {
            for (int32_t d = 0; d < head_dim; ++d) {
                const int64_t src = i * row + (int64_t)h * head_dim + d;
                const int64_t dst = (blk * block_size + off) * row + (int64_t)h * head_dim + d;
                const float kx = (float)bf16_to_double(k_new[src]);
                const float vx = (float)bf16_to_double(v_new[src]);
                k_cache[dst] = oracle_e4m3_encode(kx / k_scale[h]);
                v_cache[dst] = oracle_e4m3_encode(vx / v_scale[h]);
            }
        }
    }
    return bad ? -1 : 0;
}

/* Attention over the fp8 pool: the gathered K/V are decode(code) * scale[h] in
 * fp64; everything after the gather is the bf16 definition above. */
int oracle_paged_attention_fp8(const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                               int64_t num_blocks, int32_t block_size,
                               const int32_t *block_tables, int32_t max_blocks_per_seq,
                               const int32_t *context_lens, int32_t num_seqs,
                               int32_t n_query_per_seq, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim, float scale,
                               const float *k_scale, const float *v_scale,
                               const uint8_t *pair_mask, double *out, int32_t num_threads)
{
    if (check_shapes(num_seqs, n_query_per_seq, num_q_heads, num_kv_heads, head_dim, block_size))
        return -2;
    const int32_t group = num_q_heads / num_kv_heads;
    const int64_t npairs = (int64_t)num_seqs * num_kv_heads;
    int status = 0;
#ifdef _OPENMP
    if (num_threads > 0)
        omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t pair = 0; pair < npairs; ++pair) {
        const int32_t s = (int32_t)(pair / num_kv_heads);
        const int32_t h = (int32_t)(pair % num_kv_heads);
        if (pair_mask && !pair_mask[pair])
            continue;
        const int32_t T = eff_len(context_lens, s, max_blocks_per_seq, block_size);
        double *K = (double *)malloc(sizeof(double) * ((size_t)T * head_dim + 1));
        double *V = (double *)malloc(sizeof(double) * ((size_t)T * head_dim + 1));
        double *w = (double *)malloc(sizeof(double) * ((size_t)T + 1));
        double *qrow = (double *)malloc(sizeof(double) * (size_t)head_dim);
        const int32_t *table = block_tables + (int64_t)s * max_blocks_per_seq;
        int bad = 0;
        for (int32_t t = 0; t < T && !bad; ++t) {
            const int64_t phys = table[t / block_size];
            if (phys < 0 || phys >= num_blocks) {
                bad = 1;
                break;
            }
            const int64_t base =
                ((phys * block_size + t % block_size) * num_kv_heads + h) * (int64_t)head_dim;
            for (int32_t d = 0; d < head_dim; ++d) {
                K[(int64_t)t * head_dim + d] = oracle_e4m3_decode(k_cache[base + d]) * k_scale[h];
                V[(int64_t)t * head_dim + d] = oracle_e4m3_decode(v_cache[base + d]) * v_scale[h];
            }
        }
        if (bad) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            status = -1;
        }
        for (int32_t j = 0; j < n_query_per_seq && !bad; ++j) {
            const int32_t lim = T - n_query_per_seq + j;
            for (int32_t g = 0; g < group; ++g) {
                const int32_t qh = h * group + g;
                const int64_t row = ((int64_t)s * n_query_per_seq + j) * num_q_heads + qh;
                double *o = out + row * head_dim;
                for (int32_t d = 0; d < head_dim; ++d)
                    o[d] = 0.0;
                if (lim < 0 || T == 0)
                    continue;
                for (int32_t d = 0; d < head_dim; ++d)
                    qrow[d] = bf16_to_double(q[row * head_dim + d]);
                row_weights(qrow, K, T, lim, head_dim, (double)scale, w);
                for (int32_t t = 0; t <= lim && t < T; ++t)
                    for (int32_t d = 0; d < head_dim; ++d)
                        o[d] += w[t] * V[(int64_t)t * head_dim + d];
            }
        }
        free(K);
        free(V);
        free(w);
        free(qrow);
    }
    return status;
}

/* Element-wise helpers for the tests. */
void oracle_e4m3_encode_array(const float *x, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_encode(x[i]);
}

void oracle_e4m3_decode_array(const uint8_t *c, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_decode(c[i]);
}

/* ------------------------------------------------------------------------
 * Variable query counts, tree masks (and chunked prefill through them).
 *
 * "Chapter 18", section 18.1.2 (tree-based speculative decoding: the target
 * scores every node of a candidate tree in one pass, each node attending to
 * its own ancestors) and "07 -- Inference", section 2.4 (chunked prefill: a
 * prompt processed in chunks gives the same result as one prefill). Sequence s
 * owns query rows q_start[s] .. q_start[s+1]-1 (q_len = their count) and T_s
 * cached tokens including the new ones. Without masks query j sees positions
 * 0 .. T_s - q_len + j (causal). With masks the last W = tree_len[s] positions
 * form a window: query j sees every position before T_s - W, and window
 * position i (absolute T_s - W + i) iff bit i of tree_mask[q_start[s] + j].
 * A row that sees no position is all zeros.
 * ---------------------------------------------------------------------- */

/* Weights of one row over the visible positions (vis[t] != 0), others 0. */
static void row_weights_visible(const double *qrow, const double *K, int32_t T,
                                const uint8_t *vis, int32_t head_dim, double scale, double *w)
{
    double mx = -INFINITY;
    for (int32_t t = 0; t < T; ++t) {
        if (!vis[t]) {
            w[t] = 0.0;
            continue;
        }
        double dot = 0.0;
        for (int32_t d = 0; d < head_dim; ++d)
            dot += qrow[d] * K[(int64_t)t * head_dim + d];
        w[t] = scale * dot;
        if (w[t] > mx)
            mx = w[t];
    }
    double z = 0.0;
    for (int32_t t = 0; t < T; ++t)
        if (vis[t]) {
            w[t] = exp(w[t] - mx);
            z += w[t];
        }
    for (int32_t t = 0; t < T; ++t)
        if (vis[t])
            w[t] /= z;
}

int oracle_paged_attention_varlen(const uint16_t *q, const uint16_t *k_cache,
                                  const uint16_t *v_cache, int64_t num_blocks, int32_t block_size,
                                  const int32_t *block_tables, int32_t max_blocks_per_seq,
                                  const int32_t *context_lens, int32_t num_seqs,
                                  const int32_t *q_start, const uint32_t *tree_mask,
                                  const int32_t *tree_len, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, float scale,
                                  double *out, int32_t num_threads)
{
    if (check_shapes(num_seqs, 1, num_q_heads, num_kv_heads, head_dim, block_size))
        return -2;
    for (int32_t s = 0; s < num_seqs; ++s) {
        if (q_start[s + 1] < q_start[s])
            return -2;
        if (tree_mask && (tree_len[s] < 0 || tree_len[s] > 32))
            return -2;
    }
    const int32_t group = num_q_heads / num_kv_heads;
    const int64_t npairs = (int64_t)num_seqs * num_kv_heads;
    int status = 0;
#ifdef _OPENMP
    if (num_threads > 0)
        omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t pair = 0; pair < npairs; ++pair) {
        const int32_t s = (int32_t)(pair / num_kv_heads);
        const int32_t h = (int32_t)(pair % num_kv_heads);
        const int32_t T = eff_len(context_lens, s, max_blocks_per_seq, block_size);
        const int32_t ql = q_start[s + 1] - q_start[s];
        double *K = (double *)malloc(sizeof(double) * ((size_t)T * head_dim + 1));
        double *V = (double *)malloc(sizeof(double) * ((size_t)T * head_dim + 1));
        double *w = (double *)malloc(sizeof(double) * ((size_t)T + 1));
        uint8_t *vis = (uint8_t *)malloc((size_t)T + 1);
        double *qrow = (double *)malloc(sizeof(double) * (size_t)head_dim);
        int bad = gather_kv(k_cache, v_cache, num_blocks, block_size,
                            block_tables + (int64_t)s * max_blocks_per_seq, T,
                            num_kv_heads, head_dim, h, K, V);
        if (bad) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            status = -1;
        }
        for (int32_t j = 0; j < ql && !bad; ++j) {
            const int64_t qr = (int64_t)q_start[s] + j; /* the query's row */
            int any = 0;
            for (int32_t t = 0; t < T; ++t) {
                if (tree_mask) {
                    const int32_t w0 = T - tree_len[s]; /* first window position */
                    vis[t] = (uint8_t)(t < w0 || ((tree_mask[qr] >> (t - w0)) & 1u));
                } else {
                    vis[t] = (uint8_t)(t <= T - ql + j);
                }
                any |= vis[t];
            }
            for (int32_t g = 0; g < group; ++g) {
                const int32_t qh = h * group + g;
                double *o = out + (qr * num_q_heads + qh) * head_dim;
                for (int32_t d = 0; d < head_dim; ++d)
                    o[d] = 0.0;
                if (!any)
                    continue;
                for (int32_t d = 0; d < head_dim; ++d)
                    qrow[d] = bf16_to_double(q[(qr * num_q_heads + qh) * head_dim + d]);
                row_weights_visible(qrow, K, T, vis, head_dim, (double)scale, w);
                for (int32_t t = 0; t < T; ++t)
                    if (vis[t])
                        for (int32_t d = 0; d < head_dim; ++d)
                            o[d] += w[t] * V[(int64_t)t * head_dim + d];
            }
        }
        free(K);
        free(V);
        free(w);
        free(vis);
        free(qrow);
    }
    return status;
}

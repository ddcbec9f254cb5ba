/*
 * ua_oracle.c -- plain, slow, fp64 CPU oracle for unified paged varlen attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this file's library.  It shares no
 * code with the CUDA path and is never called by the product.
 *
 * What it computes follows the problem statement of the unified kernel
 * ("[Kernel] Unified Triton kernel that doesn't distinguish between prefill +
 * decode", vLLM PR #16828, PR description, first bullet): the kernel has the
 * semantics of FlashAttention's varlen function over an arbitrary number of
 * new query tokens per sequence, with the key cache in the FlashAttention
 * layout (third bullet).  Written out, for every sequence s, query head h and new token i:
 *
 *     Lq = cu_seqlens_q[s+1] - cu_seqlens_q[s],   Lk = seqused_k[s]
 *     g  = h / (Hq / Hkv)                          (GQA: contiguous groups)
 *     limit = causal ? Lk - Lq + i + 1 : Lk        (bottom-right alignment:
 *                                                   the new tokens are the
 *                                                   last Lq of the context)
 *     for j < limit:  page = block_table[s][j / block_size],
 *                     k_j  = K[page][j % block_size][g][:],  v_j likewise
 *                     x_j  = scale * <q[t][h][:], k_j>       (fp64)
 *     out[t][h][:] = sum_j exp(x_j - max x) v_j / sum_j exp(x_j - max x)
 *
 * Non-causal mode (all Lk keys visible) answers a request in the review
 * thread of the same page, which asks for it in addition to causal mode.  The optional
 * key window [key_lo, key_hi) restricts j further; it exists so tests can
 * form split-KV partials, and ua_oracle_merge() is the log-sum-exp merge of
 * such partials.
 *
 * bf16 inputs are widened exactly (bits << 16 -> float -> double).  Every
 * product, sum and exponential is fp64.  64-bit offsets are used for every
 * cache index (the int64 indexing point of "[ROCM][KERNEL] Paged attention
 * for V1", vLLM PR #15720, review thread on static_cast).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum {
    ORACLE_OK = 0,
    ORACLE_BAD_SHAPE = 1,
    ORACLE_BAD_SEQLENS = 2,
    ORACLE_BAD_BLOCK = 3,
    ORACLE_NO_MEMORY = 4
};

static double bf16_to_f64(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * FP8 E4M3 (the OCP 8-bit format with 4 exponent bits, bias 7, and 3
 * mantissa bits, "fn": no infinities) to double, from the format's
 * definition: exponent field e = 0 is subnormal, m/8 * 2^-6; otherwise
 * (1 + m/8) * 2^(e-7); the code with e = 15 and m = 7 is NaN.  The FP8 cache
 * is the "KV cache compression" of the review thread on "[Kernel] [V1]
 * Improved performance for V1 Triton (ROCm) backend" (vLLM PR #14152), which
 * names the fp8_e4m3fn type.
 */
double ua_oracle_e4m3_to_f64(uint8_t b)
{
    const int sign = b >> 7, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Check the batch description before touching any data. */
static int check_batch(const int32_t *cu, const int32_t *seqused_k, const int32_t *block_table,
                       int num_seqs, int num_q_heads, int num_kv_heads, int head_size,
                       int block_size, int num_blocks, int bt_stride, int causal)
{
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_size <= 0 ||
        block_size <= 0 || num_blocks < 0 || bt_stride < 0)
        return ORACLE_BAD_SHAPE;
    if (num_q_heads % num_kv_heads != 0)
        return ORACLE_BAD_SHAPE;
    if (num_seqs > 0 && cu[0] != 0)
        return ORACLE_BAD_SEQLENS;
    for (int s = 0; s < num_seqs; ++s) {
        int lq = cu[s + 1] - cu[s];
        int lk = seqused_k[s];
        if (lq < 0 || lk < 0)
            return ORACLE_BAD_SEQLENS;
        if (lq > 0 && lk == 0)
            return ORACLE_BAD_SEQLENS;
        if (causal && lk < lq)
            return ORACLE_BAD_SEQLENS;
        int64_t pages = ((int64_t)lk + block_size - 1) / block_size;
        if (pages > bt_stride)
            return ORACLE_BAD_SEQLENS;
        for (int64_t p = 0; p < pages; ++p) {
            int32_t b = block_table[(int64_t)s * bt_stride + p];
            if (b < 0 || b >= num_blocks)
                return ORACLE_BAD_BLOCK;
        }
    }
    return ORACLE_OK;
}

/*
 * out: fp64 [total_q, num_q_heads, head_size]; lse: fp64 [total_q, num_q_heads]
 * (natural log of sum_j exp(x_j); -inf where no key is visible), may be NULL.
 * key_lo/key_hi: visible keys are additionally restricted to [key_lo, key_hi);
 * pass 0 and INT32_MAX for the plain operation.  Rows with no visible key get
 * out = 0 and lse = -inf (only possible with a window).
 */
/* One element of a K or V cache row: bf16 bits (kv8 = 0) or an e4m3 byte
 * times the cache's scale (kv8 = 1). */
static double cache_elem(const void *cache, int64_t idx, int kv8, double scale)
{
    if (kv8)
        return scale * ua_oracle_e4m3_to_f64(((const uint8_t *)cache)[idx]);
    return bf16_to_f64(((const uint16_t *)cache)[idx]);
}

static int attention_impl(const uint16_t *q, const void *k_cache, const void *v_cache, int kv8,
                          double k_scale, double v_scale, const int32_t *cu_seqlens_q,
                          const int32_t *seqused_k, const int32_t *block_table, int num_seqs,
                          int num_q_heads, int num_kv_heads, int head_size, int block_size,
                          int num_blocks, int block_table_stride, double softmax_scale,
                          int causal, int key_lo, int key_hi, double *out, double *lse,
                          int nthreads)
{
    int rc = check_batch(cu_seqlens_q, seqused_k, block_table, num_seqs, num_q_heads,
                         num_kv_heads, head_size, block_size, num_blocks, block_table_stride,
                         causal);
    if (rc != ORACLE_OK)
        return rc;
    const int group = num_q_heads / num_kv_heads;
    const int64_t n_pairs = (int64_t)num_seqs * num_q_heads;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t sh = 0; sh < n_pairs; ++sh) {
        const int s = (int)(sh / num_q_heads);
        const int h = (int)(sh % num_q_heads);
        const int g = h / group;
        const int lq = cu_seqlens_q[s + 1] - cu_seqlens_q[s];
        const int lk = seqused_k[s];
        if (lq == 0)
            continue;
        double *x = (double *)malloc(sizeof(double) * (size_t)(lk > 0 ? lk : 1));
        if (!x) {
            failed = 1;
            continue;
        }
        for (int i = 0; i < lq; ++i) {
            const int64_t t = (int64_t)cu_seqlens_q[s] + i;
            const uint16_t *qrow = q + (t * num_q_heads + h) * (int64_t)head_size;
            double *orow = out + (t * num_q_heads + h) * (int64_t)head_size;
            int limit = causal ? lk - lq + i + 1 : lk;
            int j0 = key_lo > 0 ? key_lo : 0;
            int j1 = key_hi < limit ? key_hi : limit;
            for (int d = 0; d < head_size; ++d)
                orow[d] = 0.0;
            if (j1 <= j0) {
                if (lse)
                    lse[t * num_q_heads + h] = -INFINITY;
                continue;
            }
            /* scores, gathering each key page by page through the block table */
            double m = -INFINITY;
            for (int j = j0; j < j1; ++j) {
                int64_t page = block_table[(int64_t)s * block_table_stride + j / block_size];
                int64_t slot = j % block_size;
                const int64_t krow = ((page * block_size + slot) * num_kv_heads + g) * (int64_t)head_size;
                double dot = 0.0;
                for (int d = 0; d < head_size; ++d)
                    dot += bf16_to_f64(qrow[d]) * cache_elem(k_cache, krow + d, kv8, k_scale);
                x[j - j0] = softmax_scale * dot;
                if (x[j - j0] > m)
                    m = x[j - j0];
            }
            /* max-subtracted softmax, then the weighted sum of values */
            double denom = 0.0;
            for (int j = j0; j < j1; ++j) {
                double w = exp(x[j - j0] - m);
                denom += w;
                int64_t page = block_table[(int64_t)s * block_table_stride + j / block_size];
                int64_t slot = j % block_size;
                const int64_t vrow = ((page * block_size + slot) * num_kv_heads + g) * (int64_t)head_size;
                for (int d = 0; d < head_size; ++d)
                    orow[d] += w * cache_elem(v_cache, vrow + d, kv8, v_scale);
            }
            for (int d = 0; d < head_size; ++d)
                orow[d] /= denom;
            if (lse)
                lse[t * num_q_heads + h] = m + log(denom);
        }
        free(x);
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

int ua_oracle_attention(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                        const int32_t *cu_seqlens_q, const int32_t *seqused_k,
                        const int32_t *block_table, int num_seqs, int num_q_heads,
                        int num_kv_heads, int head_size, int block_size, int num_blocks,
                        int block_table_stride, double softmax_scale, int causal,
                        int key_lo, int key_hi, double *out, double *lse, int nthreads)
{
    return attention_impl(q, k_cache, v_cache, 0, 1.0, 1.0, cu_seqlens_q, seqused_k, block_table,
                          num_seqs, num_q_heads, num_kv_heads, head_size, block_size, num_blocks,
                          block_table_stride, softmax_scale, causal, key_lo, key_hi, out, lse,
                          nthreads);
}

/* The same over an e4m3 cache: k = k_scale * e4m3(byte), v = v_scale * e4m3(byte). */
int ua_oracle_attention_fp8kv(const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                              double k_scale, double v_scale, const int32_t *cu_seqlens_q,
                              const int32_t *seqused_k, const int32_t *block_table, int num_seqs,
                              int num_q_heads, int num_kv_heads, int head_size, int block_size,
                              int num_blocks, int block_table_stride, double softmax_scale,
                              int causal, double *out, double *lse, int nthreads)
{
    return attention_impl(q, k_cache, v_cache, 1, k_scale, v_scale, cu_seqlens_q, seqused_k,
                          block_table, num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
                          num_blocks, block_table_stride, softmax_scale, causal, 0, 2147483647,
                          out, lse, nthreads);
}

/*
 * Log-sum-exp merge of partial results over disjoint key sets:
 *   M = max_p lse_p,  w_p = exp(lse_p - M),
 *   out = sum_p w_p out_p / sum_p w_p,  lse = M + log(sum_p w_p).
 * outs: nparts arrays of rows*head_size; lses: nparts arrays of rows.
 * Rows where every part is empty (all lse = -inf) come out as 0 / -inf.
 */
int ua_oracle_merge(int nparts, const double *const *outs, const double *const *lses,
                    int64_t rows, int head_size, double *out, double *lse)
{
    for (int64_t r = 0; r < rows; ++r) {
        double M = -INFINITY;
        for (int p = 0; p < nparts; ++p)
            if (lses[p][r] > M)
                M = lses[p][r];
        double *o = out + r * head_size;
        for (int d = 0; d < head_size; ++d)
            o[d] = 0.0;
        if (M == -INFINITY) {
            if (lse)
                lse[r] = -INFINITY;
            continue;
        }
        double wsum = 0.0;
        for (int p = 0; p < nparts; ++p) {
            if (lses[p][r] == -INFINITY)
                continue;
            double w = exp(lses[p][r] - M);
            wsum += w;
            for (int d = 0; d < head_size; ++d)
                o[d] += w * outs[p][r * head_size + d];
        }
        for (int d = 0; d < head_size; ++d)
            o[d] /= wsum;
        if (lse)
            lse[r] = M + log(wsum);
    }
    return ORACLE_OK;
}

int ua_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the paged KV store and GQA
 * paged attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may build, load or call this file.  It shares
 * no code, header, table or constant with the CUDA library and includes
 * nothing from it.
 *
 * Sources it restates (page title, section):
 *  - "核心数据结构：Req、Batch、Context" (mini-sglang handbook, core), sections
 *    "Req：请求的三个长度" and "Batch：谁来填哪个字段": a request is described by
 *    cached_len and device_len; extend_len = device_len - cached_len; the batch
 *    concatenates the requests' new tokens with no padding; positions of a
 *    request are cached_len .. device_len-1.
 *  - "Engine 与采样器" (mini-sglang handbook, engine), section "手工驱动引擎":
 *    out_loc of a request is the page-table row of that request sliced at
 *    [cached_len, device_len).
 *  - "Mini-SGLang 完整剖析", section 4.4.3 (the KV pool is one tensor per K/V
 *    and layer whose flattened view is [slots, kv_heads, head_dim]; store_kv
 *    scatters the new rows through out_loc) and section 4.6.7 (store_kv runs
 *    before the attention kernel, so the step's own K/V is attended).
 *  - "第 0 步：一个能跑的最小推理引擎", section "这份代码在做什么", the attention
 *    operator: K/V heads are repeated to the query heads with repeat_interleave
 *    (query head h reads KV head h / (HQ/HKV)), scores are q.k / sqrt(D), the
 *    t-th of T new queries sits at absolute position S-T+t and sees keys at
 *    positions <= its own, then softmax and a weighted sum of V.
 *
 * Everything is computed in double precision from the exact bf16 values; no
 * blocking, fusion or reordering beyond the definition.  K/V are gathered
 * token by token through the page table (every token's own entry).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Per-batch metadata ("Batch：谁来填哪个字段"; "手工驱动引擎").
 * For each request r, in batch order:
 *   qo_indptr[r+1] = qo_indptr[r] + extend_len[r]   (ragged concatenation)
 *   kv_len[r]      = cached_len[r] + extend_len[r]  (= device_len)
 *   positions[qo_indptr[r] + i] = cached_len[r] + i
 *   out_loc[qo_indptr[r] + i]   = page_table[row_r][cached_len[r] + i]
 * row_r = req_rows[r] (or r when req_rows is NULL). */
void oracle_metadata(const int32_t *page_table, int64_t pt_stride,
                     const int32_t *req_rows, const int32_t *cached_len,
                     const int32_t *extend_len, int32_t num_reqs,
                     int32_t *qo_indptr, int32_t *kv_len, int64_t *out_loc,
                     int32_t *positions) {
    qo_indptr[0] = 0;
    for (int32_t r = 0; r < num_reqs; ++r) {
        int64_t row = req_rows ? req_rows[r] : r;
        int32_t c = cached_len[r], e = extend_len[r];
        qo_indptr[r + 1] = qo_indptr[r] + e;
        kv_len[r] = c + e;
        for (int32_t i = 0; i < e; ++i) {
            int64_t t = (int64_t)qo_indptr[r] + i;
            positions[t] = c + i;
            out_loc[t] = page_table[row * pt_stride + c + i];
        }
    }
}

/* store_kv ("Mini-SGLang 完整剖析" 4.4.3 and the store.cu shape contract in
 * 4.9.4): for i = 0 .. num_tokens-1 in order, pool row out_loc[i] receives
 * the bit pattern of new row i, for K and for V.  row_elems = kv_heads *
 * head_dim. */
void oracle_store_kv(const uint16_t *k, const uint16_t *v, int64_t in_stride,
                     int64_t num_tokens, int64_t row_elems,
                     const int64_t *out_loc, uint16_t *k_pool,
                     uint16_t *v_pool, int64_t pool_stride) {
    for (int64_t i = 0; i < num_tokens; ++i) {
        int64_t slot = out_loc[i];
        memcpy(k_pool + slot * pool_stride, k + i * in_stride,
               (size_t)row_elems * sizeof(uint16_t));
        memcpy(v_pool + slot * pool_stride, v + i * in_stride,
               (size_t)row_elems * sizeof(uint16_t));
    }
}

/* Request that owns global query row t: the r with
 * qo_indptr[r] <= t < qo_indptr[r+1] (plain linear scan). */
static int32_t owner_of(const int32_t *qo_indptr, int32_t num_reqs, int64_t t) {
    for (int32_t r = 0; r < num_reqs; ++r)
        if (t >= qo_indptr[r] && t < qo_indptr[r + 1]) return r;
    return -1;
}

/* Paged GQA attention for selected query rows ("第 0 步" attention operator,
 * with K/V gathered through the page table as in "Mini-SGLang 完整剖析"
 * 4.6.4, token-granular entries).
 *
 * q        : [total_q, num_qo_heads, head_dim] bf16, row stride q_stride elems
 * k_pool/v_pool : [num_slots, num_kv_heads, head_dim] bf16, row stride
 *            pool_stride elems
 * rows     : the global query rows to compute (n_rows of them)
 * out      : [n_rows, num_qo_heads, head_dim] double
 *
 * For row t of request r, i = t - qo_indptr[r], p = cached_len[r] + i; for
 * every query head h, g = h / (num_qo_heads / num_kv_heads):
 *   s_j = (sum_d q[t,h,d] * K_j[g,d]) * scale      for j = 0 .. p
 *   out[t,h,:] = sum_j exp(s_j - max s) V_j[g,:] / sum_j exp(s_j - max s)
 * with K_j = k_pool[page_table[row_r][j]]. */
void oracle_paged_attention_rows(
    const uint16_t *q, int64_t q_stride, const uint16_t *k_pool,
    const uint16_t *v_pool, int64_t pool_stride, const int32_t *page_table,
    int64_t pt_stride, const int32_t *req_rows, const int32_t *cached_len,
    const int32_t *qo_indptr, int32_t num_reqs, int32_t num_qo_heads,
    int32_t num_kv_heads, int32_t head_dim, double scale, const int64_t *rows,
    int64_t n_rows, double *out) {
    const int32_t group = num_qo_heads / num_kv_heads;
    const int64_t work = n_rows * (int64_t)num_qo_heads;
#pragma omp parallel
    {
        double *s = NULL;
        int64_t s_cap = 0;
#pragma omp for schedule(dynamic, 1)
        for (int64_t w = 0; w < work; ++w) {
            int64_t n = w / num_qo_heads;
            int32_t h = (int32_t)(w % num_qo_heads);
            int64_t t = rows[n];
            int32_t r = owner_of(qo_indptr, num_reqs, t);
            double *o = out + (n * num_qo_heads + h) * (int64_t)head_dim;
            if (r < 0) {
                for (int32_t d = 0; d < head_dim; ++d) o[d] = NAN;
                continue;
            }
            int64_t row = req_rows ? req_rows[r] : r;
            int64_t p = (int64_t)cached_len[r] + (t - qo_indptr[r]);
            int32_t g = h / group;
            if (p + 1 > s_cap) {
                free(s);
                s_cap = p + 1;
                s = (double *)malloc((size_t)s_cap * sizeof(double));
            }
            const uint16_t *qh = q + t * q_stride + (int64_t)h * head_dim;
            double m = -INFINITY;
            for (int64_t j = 0; j <= p; ++j) {
                int64_t slot = page_table[row * pt_stride + j];
                const uint16_t *kj =
                    k_pool + slot * pool_stride + (int64_t)g * head_dim;
                double dot = 0.0;
                for (int32_t d = 0; d < head_dim; ++d)
                    dot += bf16_to_double(qh[d]) * bf16_to_double(kj[d]);
                s[j] = dot * scale;
                if (s[j] > m) m = s[j];
            }
            double denom = 0.0;
            for (int32_t d = 0; d < head_dim; ++d) o[d] = 0.0;
            for (int64_t j = 0; j <= p; ++j) {
                double wj = exp(s[j] - m);
                denom += wj;
                int64_t slot = page_table[row * pt_stride + j];
                const uint16_t *vj =
                    v_pool + slot * pool_stride + (int64_t)g * head_dim;
                for (int32_t d = 0; d < head_dim; ++d)
                    o[d] += wj * bf16_to_double(vj[d]);
            }
            for (int32_t d = 0; d < head_dim; ++d) o[d] /= denom;
        }
        free(s);
    }
}

/* Number of OpenMP threads the oracle runs with (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Set the number of OpenMP threads of later calls (timing on one core or on
 * all of them); no effect without OpenMP.  Changes no arithmetic: every
 * output element is computed by one thread in the same order. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    extern void omp_set_num_threads(int);
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

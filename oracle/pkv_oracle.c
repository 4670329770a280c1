/*
 * Plain float64 CPU oracle for batched attention over a paged KV cache with a
 * per-element sliding-window mask.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
 * baseline may load this file's library. It shares no code, header or table
 * with the CUDA library in paged_kv_sliding_gb300/; the two meet only through
 * the seeded inputs.
 *
 * What it computes (no blocking, no fusion, no reordering beyond the plain
 * definition):
 *
 *   for request b, query row i < qo_len_b, query head h:
 *     hk  = h / (H_qo / H_kv)                 consecutive query heads share a KV
 *                                             head (the query-head group of a KV
 *                                             head is packed into the matrix rows:
 *                                             sglang flashinfer_backend.py page,
 *                                             section should_use_tensor_core)
 *     p   = q_start_b + i, q_start_b defaulting to kv_len_b - qo_len_b
 *                                             (extend rows sit at prefix + i:
 *                                             sglang flashinfer_backend.py page,
 *                                             section _build_swa_prefix_custom_mask)
 *     key j in [0, kv_len_b) is visible iff
 *        (!causal || j <= p) && (window_left < 0 || j >= p - window_left)
 *                                             (window_left = W lets the query at p
 *                                             see [p-W, p], W+1 tokens:
 *                                             AMD flashinfer PR #234, "Sliding
 *                                             window" convention; k_abs >= q_abs -
 *                                             window: sglang flashinfer_backend.py page,
 *                                             section _build_swa_prefix_custom_mask)
 *     K/V row of key j = cache[kv_indices[kv_indptr[b] + j / P], j % P, hk, :]
 *                                             (paged "NHD" layout with kv_indptr,
 *                                             kv_indices, kv_last_page_len:
 *                                             sglang flashinfer_backend.py page,
 *                                             sections fast_prefill_plan and
 *                                             call_begin_forward)
 *     s_j = sm_scale * sum_c q[c] k_j[c]
 *     lse = ln sum_{j visible} exp(s_j)        (natural log of the scaled logits)
 *     out = sum_{j visible} exp(s_j - lse) v_j
 *   pkv_oracle_attention_ext adds the three per-layer arguments the pages pass with
 *   every attention call (flashinfer_backend.py forward_extend / forward_decode:
 *   the layer's logit soft cap, k_scale and v_scale), which the pages do not
 *   define further; the readings taken (plainest ones):
 *     s_j = cap * tanh(sm_scale * k_scale * q.k_j / cap)   (cap > 0; else no cap)
 *     out = v_scale * sum_j exp(s_j - lse) v_j           (K and V dequantised by
 *                                                          their scales)
 *   A row with no visible key has out = 0 and lse = -inf.
 *
 *   kv_len_b = (kv_indptr[b+1] - kv_indptr[b] - 1) * P + kv_last_page_len[b],
 *   or 0 for a request with no pages.
 *
 * merge_state (flashinfer_backend.py, _safe_merge_state and forward_extend's
 * ragged + paged merge): two partial states (v_a, s_a), (v_b, s_b) over disjoint
 * key sets combine to s = ln(e^s_a + e^s_b), v = (e^s_a v_a + e^s_b v_b) / e^s.
 *
 * bf16 inputs are widened to double exactly (a bf16 value is the top half of an
 * IEEE binary32); all arithmetic is double.
 *
 * 8-bit caches (pkv_oracle_attention_kv): flashinfer_backend.py names
 * torch.float8_e4m3fn and torch.float8_e5m2 as KV cache dtypes
 * (should_use_tensor_core) and passes k_scale / v_scale with every call. Each
 * byte is decoded to its exact value from the format's definition (the OCP 8-bit
 * floating point formats E4M3 and E5M2, below) and the attention above runs on
 * those values, k_scale and v_scale dequantising as stated.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define PKV_ORACLE_OK 0
#define PKV_ORACLE_BAD_ARG (-1)
#define PKV_ORACLE_BAD_PAGE (-2)

static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t word = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &word, sizeof f);
    return (double)f;
}

/*
 * E4M3: sign bit, 4 exponent bits with bias 7, 3 mantissa bits. Exponent field 0
 * holds zero and the subnormals (m/8) * 2^-6; S.1111.111 is NaN; there are no
 * infinities, so the largest finite value is 1.75 * 2^8 = 448.
 */
static double e4m3_to_double(uint8_t x)
{
    const int sign = x >> 7, e = (x >> 3) & 15, m = x & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/*
 * E5M2: sign bit, 5 exponent bits with bias 15, 2 mantissa bits (IEEE-like).
 * Exponent field 0 holds zero and the subnormals (m/4) * 2^-14; field 31 is
 * infinity (m = 0) or NaN.
 */
static double e5m2_to_double(uint8_t x)
{
    const int sign = x >> 7, e = (x >> 2) & 31, m = x & 3;
    double v;
    if (e == 31)
        v = m == 0 ? INFINITY : NAN;
    else if (e == 0)
        v = ldexp((double)m / 4.0, -14);
    else
        v = ldexp(1.0 + (double)m / 4.0, e - 15);
    return sign ? -v : v;
}

/* Element idx of a cache of kv_dtype 0 (bf16), 2 (E4M3) or 3 (E5M2). */
static double cache_elem(const void *cache, int64_t idx, int kv_dtype)
{
    if (kv_dtype == 2)
        return e4m3_to_double(((const uint8_t *)cache)[idx]);
    if (kv_dtype == 3)
        return e5m2_to_double(((const uint8_t *)cache)[idx]);
    return bf16_bits_to_double(((const uint16_t *)cache)[idx]);
}

/* Exposed for the pins: decode n 8-bit codes of format kv_dtype (2 or 3). */
int pkv_oracle_decode_fp8(int kv_dtype, const uint8_t *codes, int64_t n, double *out)
{
    if (kv_dtype != 2 && kv_dtype != 3)
        return PKV_ORACLE_BAD_ARG;
    for (int64_t i = 0; i < n; ++i)
        out[i] = kv_dtype == 2 ? e4m3_to_double(codes[i]) : e5m2_to_double(codes[i]);
    return PKV_ORACLE_OK;
}

/* Threads used by the OpenMP loop below; returns the count now in force. */
int pkv_oracle_set_threads(int n)
{
    if (n > 0)
        omp_set_num_threads(n);
    return omp_get_max_threads();
}

/* Number of valid tokens held by request b's pages. */
static int64_t request_kv_len(const int32_t *kv_indptr, const int32_t *kv_last_page_len,
                              int64_t b, int64_t page_size)
{
    int64_t n_pages = (int64_t)kv_indptr[b + 1] - (int64_t)kv_indptr[b];
    if (n_pages <= 0)
        return 0;
    return (n_pages - 1) * page_size + (int64_t)kv_last_page_len[b];
}

static int key_is_visible(int64_t j, int64_t p, int64_t window_left, int causal)
{
    if (causal && j > p)
        return 0;
    if (window_left >= 0 && j < p - window_left)
        return 0;
    return 1;
}

/* Index of the request owning global query row `row` (qo_indptr is monotone). */
static int64_t request_of_row(const int32_t *qo_indptr, int64_t batch, int64_t row)
{
    int64_t lo = 0, hi = batch; /* answer in [lo, hi) */
    while (hi - lo > 1) {
        int64_t mid = (lo + hi) / 2;
        if ((int64_t)qo_indptr[mid] <= row)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

/*
 * Attention for the selected query rows.
 *   rows == NULL: every row 0..qo_indptr[batch)-1, output row r at index r.
 *   rows != NULL: output row k holds global query row rows[k].
 * out: [n_out_rows, H_qo, d] double; lse: [n_out_rows, H_qo] double (may be NULL).
 * q: bf16 bits [total_q, H_qo, d]; caches [num_pages, P, H_kv, d]: bf16 bits
 * (kv_dtype 0) or E4M3 / E5M2 bytes (kv_dtype 2 / 3).
 * Returns 0, PKV_ORACLE_BAD_ARG, or PKV_ORACLE_BAD_PAGE (a page id outside
 * [0, num_pages) met on a visible key).
 */
/* The logit of a key from its dot product with the query row. */
static double logit_of(double dot, double scale, double cap)
{
    const double s = scale * dot;
    return cap > 0.0 ? cap * tanh(s / cap) : s;
}

int pkv_oracle_attention_kv(int64_t batch, const int32_t *qo_indptr, const int32_t *kv_indptr,
                            const int32_t *kv_indices, const int32_t *kv_last_page_len,
                            const int32_t *q_start, int64_t num_qo_heads, int64_t num_kv_heads,
                            int64_t head_dim, int64_t page_size, int64_t num_pages,
                            int64_t window_left, int causal, double sm_scale, double soft_cap,
                            double k_scale, double v_scale, const uint16_t *q, int kv_dtype,
                            const void *k_cache, const void *v_cache, const int64_t *rows,
                            int64_t n_rows, double *out, double *lse)
{
    const double scale = sm_scale * k_scale;
    if (batch < 0 || num_kv_heads <= 0 || num_qo_heads <= 0 || head_dim <= 0 || page_size <= 0)
        return PKV_ORACLE_BAD_ARG;
    if (kv_dtype != 0 && kv_dtype != 2 && kv_dtype != 3)
        return PKV_ORACLE_BAD_ARG;
    if (num_qo_heads % num_kv_heads != 0)
        return PKV_ORACLE_BAD_ARG;
    const int64_t group = num_qo_heads / num_kv_heads;
    const int64_t total_q = batch > 0 ? (int64_t)qo_indptr[batch] : 0;
    const int64_t n_out = rows ? n_rows : total_q;
    int status = PKV_ORACLE_OK;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t task = 0; task < n_out * num_qo_heads; ++task) {
        const int64_t k_out = task / num_qo_heads;
        const int64_t h = task % num_qo_heads;
        const int64_t row = rows ? rows[k_out] : k_out;
        double *o = out + (k_out * num_qo_heads + h) * head_dim;
        for (int64_t c = 0; c < head_dim; ++c)
            o[c] = 0.0;
        if (lse)
            lse[k_out * num_qo_heads + h] = -INFINITY;
        if (row < 0 || row >= total_q) {
#pragma omp atomic write
            status = PKV_ORACLE_BAD_ARG;
            continue;
        }
        const int64_t b = request_of_row(qo_indptr, batch, row);
        const int64_t i = row - (int64_t)qo_indptr[b];
        const int64_t qo_len = (int64_t)qo_indptr[b + 1] - (int64_t)qo_indptr[b];
        const int64_t kv_len = request_kv_len(kv_indptr, kv_last_page_len, b, page_size);
        const int64_t p = (q_start ? (int64_t)q_start[b] : kv_len - qo_len) + i;
        const int64_t hk = h / group;
        const uint16_t *qrow = q + (row * num_qo_heads + h) * head_dim;

        /* Pass 1: the maximum visible logit. */
        double m = -INFINITY;
        int64_t n_visible = 0;
        int bad = 0;
        for (int64_t j = 0; j < kv_len; ++j) {
            if (!key_is_visible(j, p, window_left, causal))
                continue;
            int64_t page = kv_indices[(int64_t)kv_indptr[b] + j / page_size];
            if (page < 0 || page >= num_pages) {
                bad = 1;
                break;
            }
            const int64_t krow = ((page * page_size + j % page_size) * num_kv_heads + hk) * head_dim;
            double dot = 0.0;
            for (int64_t c = 0; c < head_dim; ++c)
                dot += bf16_bits_to_double(qrow[c]) * cache_elem(k_cache, krow + c, kv_dtype);
            const double s = logit_of(dot, scale, soft_cap);
            if (s > m)
                m = s;
            ++n_visible;
        }
        if (bad) {
#pragma omp atomic write
            status = PKV_ORACLE_BAD_PAGE;
            continue;
        }
        if (n_visible == 0)
            continue; /* out 0, lse -inf */

        /* Pass 2: sum of exp(s - m) and the weighted sum of V. */
        double denom = 0.0;
        for (int64_t j = 0; j < kv_len; ++j) {
            if (!key_is_visible(j, p, window_left, causal))
                continue;
            int64_t page = kv_indices[(int64_t)kv_indptr[b] + j / page_size];
            int64_t slot = (page * page_size + j % page_size) * num_kv_heads + hk;
            const int64_t row0 = slot * head_dim;
            double dot = 0.0;
            for (int64_t c = 0; c < head_dim; ++c)
                dot += bf16_bits_to_double(qrow[c]) * cache_elem(k_cache, row0 + c, kv_dtype);
            const double s = logit_of(dot, scale, soft_cap);
            double w = exp(s - m);
            denom += w;
            for (int64_t c = 0; c < head_dim; ++c)
                o[c] += w * cache_elem(v_cache, row0 + c, kv_dtype);
        }
        for (int64_t c = 0; c < head_dim; ++c)
            o[c] = v_scale * o[c] / denom;
        if (lse)
            lse[k_out * num_qo_heads + h] = m + log(denom);
    }
    return status;
}

int pkv_oracle_attention_ext(int64_t batch, const int32_t *qo_indptr, const int32_t *kv_indptr,
                             const int32_t *kv_indices, const int32_t *kv_last_page_len,
                             const int32_t *q_start, int64_t num_qo_heads, int64_t num_kv_heads,
                             int64_t head_dim, int64_t page_size, int64_t num_pages,
                             int64_t window_left, int causal, double sm_scale, double soft_cap,
                             double k_scale, double v_scale, const uint16_t *q,
                             const uint16_t *k_cache, const uint16_t *v_cache, const int64_t *rows,
                             int64_t n_rows, double *out, double *lse)
{
    return pkv_oracle_attention_kv(batch, qo_indptr, kv_indptr, kv_indices, kv_last_page_len, q_start,
                                   num_qo_heads, num_kv_heads, head_dim, page_size, num_pages, window_left,
                                   causal, sm_scale, soft_cap, k_scale, v_scale, q, 0, k_cache, v_cache,
                                   rows, n_rows, out, lse);
}

int pkv_oracle_attention(int64_t batch, const int32_t *qo_indptr, const int32_t *kv_indptr,
                         const int32_t *kv_indices, const int32_t *kv_last_page_len,
                         const int32_t *q_start, int64_t num_qo_heads, int64_t num_kv_heads,
                         int64_t head_dim, int64_t page_size, int64_t num_pages,
                         int64_t window_left, int causal, double sm_scale, const uint16_t *q,
                         const uint16_t *k_cache, const uint16_t *v_cache, const int64_t *rows,
                         int64_t n_rows, double *out, double *lse)
{
    return pkv_oracle_attention_ext(batch, qo_indptr, kv_indptr, kv_indices, kv_last_page_len, q_start,
                                    num_qo_heads, num_kv_heads, head_dim, page_size, num_pages, window_left,
                                    causal, sm_scale, 0.0, 1.0, 1.0, q, k_cache, v_cache, rows, n_rows, out, lse);
}

/*
 * merge_state over n independent (token, head) rows of width d:
 *   s = ln(e^s_a + e^s_b), v = (e^s_a v_a + e^s_b v_b) / e^s.
 * A state with s = -inf carries no weight; two empty states give v = 0, s = -inf.
 */
int pkv_oracle_merge_state(int64_t n, int64_t d, const double *v_a, const double *s_a,
                           const double *v_b, const double *s_b, double *v_out, double *s_out)
{
    if (n < 0 || d <= 0)
        return PKV_ORACLE_BAD_ARG;
    for (int64_t r = 0; r < n; ++r) {
        double sa = s_a[r], sb = s_b[r];
        double m = sa > sb ? sa : sb;
        if (m == -INFINITY) {
            for (int64_t c = 0; c < d; ++c)
                v_out[r * d + c] = 0.0;
            s_out[r] = -INFINITY;
            continue;
        }
        double wa = exp(sa - m), wb = exp(sb - m);
        double sum = wa + wb;
        for (int64_t c = 0; c < d; ++c)
            v_out[r * d + c] = (wa * v_a[r * d + c] + wb * v_b[r * d + c]) / sum;
        s_out[r] = m + log(sum);
    }
    return PKV_ORACLE_OK;
}

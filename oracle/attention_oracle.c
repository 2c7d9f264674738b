/*
 * Plain CPU oracle for the attention forward pass (FlashAttention's output).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * What it follows: "TileLang で GPU カーネル設計を解説", §6 (FlashAttention):
 * Q, K, V and O have shape [batch, seq_len, heads, dim] (dim contiguous); the
 * output row of query i of head h in batch b is
 *
 *     O[b, i, h, :] = sum_j w_ij V[b, j, h, :],
 *     w_ij = exp(s_ij) / sum_j' exp(s_ij'),   s_ij = scale * sum_d Q[b, i, h, d] K[b, j, h, d],
 *
 * with scale = 1 / sqrt(dim), over the keys j < seq_len, or only j <= i when
 * causal (the page masks keys after the query, on equal query and key
 * lengths).  The page computes it blockwise with an online softmax; this is
 * the definition it reaches, written out: every 16-bit input decoded exactly
 * to double, in-order fp64 dot products and sums, the largest score
 * subtracted before exp (the same softmax, kept finite), no blocking.
 *
 * With abs_v set, |V| replaces V: the result is then sum_j w_ij |V[j, :]|, the
 * magnitude the tests scale their error bound by.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

int oracle_decode(const uint16_t *in, double *out, int64_t n, int dtype);

static int decode_all(const uint16_t *in, int64_t n, int dtype, double **out) {
    *out = (double *)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    if (!*out) return -1;
    return oracle_decode(in, *out, n, dtype);
}

/*
 * Q, K, V: uint16 [B, S, H, D] in `dtype` (0 fp16, 1 bf16).  out: double, one
 * row of D values per requested (b, i, h): rows == NULL means every row in
 * [B, S, H] order; otherwise rows[r] = (b * S + i) * H + h for r < nrows.
 * Returns 0, or -1 on bad arguments or allocation failure.
 */
int oracle_attention_f64(const uint16_t *Q, const uint16_t *K, const uint16_t *V, double *out, int64_t B,
                         int64_t S, int64_t H, int64_t D, int causal, int abs_v, const int64_t *rows,
                         int64_t nrows, int dtype) {
    if (B < 0 || S < 0 || H < 0 || D < 1 || (dtype != 0 && dtype != 1) || !out) return -1;
    const int64_t total = B * S * H;
    if (!rows) nrows = total;
    if (nrows == 0 || total == 0) return 0;
    double *q = NULL, *k = NULL, *v = NULL;
    const int64_t n = total * D;
    if (decode_all(Q, n, dtype, &q) || decode_all(K, n, dtype, &k) || decode_all(V, n, dtype, &v)) {
        free(q); free(k); free(v);
        return -1;
    }
    if (abs_v)
        for (int64_t t = 0; t < n; ++t) v[t] = fabs(v[t]);
    const double scale = 1.0 / sqrt((double)D);
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t row = rows ? rows[r] : r;
        if (row < 0 || row >= total) { bad = 1; continue; }
        const int64_t h = row % H, bi = row / H, i = bi % S, b = bi / S;
        const int64_t nk = causal ? i + 1 : S;
        double *s = (double *)malloc((size_t)nk * sizeof(double));
        if (!s) { bad = 1; continue; }
        const double *qi = q + row * D;
        double m = -INFINITY;
        for (int64_t j = 0; j < nk; ++j) {
            const double *kj = k + ((b * S + j) * H + h) * D;
            double dot = 0.0;
            for (int64_t d = 0; d < D; ++d) dot += qi[d] * kj[d];
            s[j] = scale * dot;
            if (s[j] > m) m = s[j];
        }
        double l = 0.0;
        for (int64_t j = 0; j < nk; ++j) {
            s[j] = exp(s[j] - m);
            l += s[j];
        }
        double *o = out + r * D;
        for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
        for (int64_t j = 0; j < nk; ++j) {
            const double *vj = v + ((b * S + j) * H + h) * D;
            for (int64_t d = 0; d < D; ++d) o[d] += s[j] * vj[d];
        }
        for (int64_t d = 0; d < D; ++d) o[d] /= l;
        free(s);
    }
    free(q); free(k); free(v);
    return bad ? -1 : 0;
}

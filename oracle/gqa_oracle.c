/*
 * gqa_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of grouped-query attention.  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg load this file's
 * library; the product path (libgqa.so and its Python binding) never does, and
 * this file shares no code, header or constant with it.
 *
 * What it computes, step by step, in the order the pages give it:
 *
 *   (1) every input element is widened to fp64 exactly (a bf16 value is the top
 *       16 bits of an fp32, so the widening is lossless);
 *   (2) K and V are expanded per group exactly as `repeat_interleave(n_rep,
 *       dim=1)` does: query head h reads KV head h / n_rep with n_rep = Hq/Hkv
 *       ("手把手教你用PyTorch实现GQA", section 1.3, class GQA; the GQA paper
 *       notes on 51969.com, "QA 相关" -> inference, `repeat_kv`; the Huawei Cloud
 *       post "多头注意力机制的代码实现（MQA和GQA）", section 5,
 *       `group_index = head_index // n_head_per_group`);
 *   (3) scores  x_t = <q, k_t>            (Huawei Cloud post, section 5: Q @ K^T)
 *   (4) scaled  x_t = x_t * scale         (same code: divide by head_size**0.5;
 *       the caller passes scale = 1/sqrt(D) unless it wants another one)
 *   (5) causal mask: a key strictly after the query position is removed
 *       (same code: triu(ones, diagonal=1) -> -inf, applied as the code
 *       intends; the printed `masked_fill` result is discarded, which is read
 *       as a slip of the page);
 *   (6) p_t = exp(x_t - max) / sum exp(x_t - max)   (softmax over keys; the
 *       max shift changes nothing mathematically and only keeps exp in range)
 *   (7) out = sum_t p_t v_t                (attention @ V)
 *
 * Decode: one query token per (b, h) attends to the first seqlens[b] rows of
 * the [B, Hkv, Lmax, D] cache (no mask inside the cache).  Prefill: q, k, v of
 * one length L; row i sees keys t <= i when causal, all L keys otherwise.
 *
 * Element types: 0 = bf16 bit patterns (uint16), 1 = fp64.  Outputs are fp64.
 *
 * FP8 cache (gqa_oracle_decode_fp8): K and V are stored as OCP FP8 E4M3 bytes
 * (sign, 4 exponent bits with bias 7, 3 mantissa bits; exponent 0 encodes
 * subnormals m/8 * 2^-6; S.1111.111 is NaN; no infinities; largest 448) with
 * one scale per (batch, KV head) for K and one for V: the real entry is the
 * decoded byte times its scale ("InputsFp8" of the gsyq.cn page on xformers,
 * "混合精度计算加速", names FP8 KV storage; the per-(sequence, KV head) scale
 * is this build's reading).  Step (1) becomes: decode the byte exactly, then
 * multiply by the scale in fp64.
 * Rows to evaluate are given as an index list so that sampled rows of a
 * full-size workload can be checked one by one.
 *
 * Return codes: 0 ok, 1 bad argument, 2 out of memory, 3 empty context (no
 * visible key: the softmax of nothing is undefined; the row is written as
 * zeros and 3 is returned after the other rows were computed).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double elem(const void *base, size_t i, int type)
{
    if (type == 1) return ((const double *)base)[i];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f; /* step (1): exact */
}

/* Exact value of an OCP FP8 E4M3 byte. */
static double e4m3_value(uint8_t byte)
{
    int sign = byte >> 7, e = (byte >> 3) & 15, m = byte & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);          /* m/8 * 2^(1-7) */
    else
        mag = ldexp((double)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
    return sign ? -mag : mag;
}

/* One query row against `nk` visible keys of one (b, h).
 * kx, vx: the expanded K/V rows of this query head, [nk, D] fp64.
 * Writes out[D].  Returns 0, or 3 if nk == 0. */
static int attend_row(const double *qrow, const double *kx, const double *vx, int nk, int D,
                      double scale, double *x, double *out)
{
    if (nk <= 0) {
        for (int d = 0; d < D; ++d) out[d] = 0.0;
        return 3;
    }
    /* (3) + (4) */
    for (int t = 0; t < nk; ++t) {
        double s = 0.0;
        for (int d = 0; d < D; ++d) s += qrow[d] * kx[(size_t)t * D + d];
        x[t] = s * scale;
    }
    /* (6) */
    double mx = -INFINITY;
    for (int t = 0; t < nk; ++t)
        if (x[t] > mx) mx = x[t];
    double den = 0.0;
    for (int t = 0; t < nk; ++t) {
        x[t] = exp(x[t] - mx);
        den += x[t];
    }
    for (int t = 0; t < nk; ++t) x[t] /= den;
    /* (7) */
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (int t = 0; t < nk; ++t)
        for (int d = 0; d < D; ++d) out[d] += x[t] * vx[(size_t)t * D + d];
    return 0;
}

/* Step (2) for one query head: gather the rows [0, n) of KV head h / n_rep of
 * batch b into dense fp64 buffers, i.e. the slice of repeat_interleave(K)
 * that query head h sees. */
static void expand_head(const void *k, const void *v, int type, int b, int h, int n_rep,
                        int Hkv, int Lcap, int D, int n, double *kx, double *vx)
{
    int j = h / n_rep;
    size_t base = (((size_t)b * Hkv + j) * Lcap) * D;
    for (size_t i = 0; i < (size_t)n * D; ++i) {
        kx[i] = elem(k, base + i, type);
        vx[i] = elem(v, base + i, type);
    }
}

/* Decode.
 *   q        [B, Hq, D]            out rows of the evaluated (b, h): [nrows, D]
 *   k, v     [B, Hkv, Lmax, D]     seqlens [B] (keys visible to batch b)
 *   rows     (b, h) int pairs, nrows of them; rows == NULL means all B*Hq in
 *            order b-major, h-minor. */
int gqa_oracle_decode(const void *q, const void *k, const void *v, int type,
                      const int32_t *seqlens, int B, int Hq, int Hkv, int D, int Lmax,
                      double scale, const int32_t *rows, int nrows, double *out)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Lmax <= 0 || Hq % Hkv != 0) return 1;
    if (type != 0 && type != 1) return 1;
    if (rows == NULL) nrows = B * Hq;
    for (int b = 0; b < B; ++b)
        if (seqlens[b] > Lmax) return 1;
    int n_rep = Hq / Hkv;
    int rc_all = 0;
#pragma omp parallel
    {
        double *kx = malloc(sizeof(double) * (size_t)Lmax * D);
        double *vx = malloc(sizeof(double) * (size_t)Lmax * D);
        double *x = malloc(sizeof(double) * (size_t)Lmax);
        double *qrow = malloc(sizeof(double) * (size_t)D);
        int oom = !(kx && vx && x && qrow);
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < nrows; ++r) {
            int rc;
            if (oom) {
                rc = 2;
            } else {
                int b = rows ? rows[2 * r] : r / Hq;
                int h = rows ? rows[2 * r + 1] : r % Hq;
                if (b < 0 || b >= B || h < 0 || h >= Hq) {
                    rc = 1;
                } else {
                    int n = seqlens[b] > 0 ? seqlens[b] : 0;
                    for (int d = 0; d < D; ++d) qrow[d] = elem(q, ((size_t)b * Hq + h) * D + d, type);
                    expand_head(k, v, type, b, h, n_rep, Hkv, Lmax, D, n, kx, vx);
                    rc = attend_row(qrow, kx, vx, n, D, scale, x, out + (size_t)r * D);
                }
            }
            if (rc) {
#pragma omp critical
                if (rc_all == 0 || rc < rc_all) rc_all = rc;
            }
        }
        free(kx); free(vx); free(x); free(qrow);
    }
    return rc_all;
}

/* Decode over an FP8 E4M3 cache (see the header).
 *   q        [B, Hq, D] of element type `type` (0 bf16 bits, 1 fp64)
 *   k8, v8   [B, Hkv, Lmax, D] E4M3 bytes; k_scale, v_scale [B * Hkv] fp64
 *   everything else as gqa_oracle_decode. */
int gqa_oracle_decode_fp8(const void *q, int type, const uint8_t *k8, const uint8_t *v8,
                          const double *k_scale, const double *v_scale, const int32_t *seqlens,
                          int B, int Hq, int Hkv, int D, int Lmax, double scale,
                          const int32_t *rows, int nrows, double *out)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Lmax <= 0 || Hq % Hkv != 0) return 1;
    if (type != 0 && type != 1) return 1;
    if (rows == NULL) nrows = B * Hq;
    for (int b = 0; b < B; ++b)
        if (seqlens[b] > Lmax) return 1;
    int n_rep = Hq / Hkv;
    int rc_all = 0;
#pragma omp parallel
    {
        double *kx = malloc(sizeof(double) * (size_t)Lmax * D);
        double *vx = malloc(sizeof(double) * (size_t)Lmax * D);
        double *x = malloc(sizeof(double) * (size_t)Lmax);
        double *qrow = malloc(sizeof(double) * (size_t)D);
        int oom = !(kx && vx && x && qrow);
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < nrows; ++r) {
            int rc;
            if (oom) {
                rc = 2;
            } else {
                int b = rows ? rows[2 * r] : r / Hq;
                int h = rows ? rows[2 * r + 1] : r % Hq;
                if (b < 0 || b >= B || h < 0 || h >= Hq) {
                    rc = 1;
                } else {
                    int n = seqlens[b] > 0 ? seqlens[b] : 0;
                    int j = h / n_rep; /* step (2): the KV head of query head h */
                    size_t base = (((size_t)b * Hkv + j) * Lmax) * D;
                    double ks = k_scale[b * Hkv + j], vs = v_scale[b * Hkv + j];
                    for (size_t i = 0; i < (size_t)n * D; ++i) {
                        kx[i] = e4m3_value(k8[base + i]) * ks; /* step (1) for an FP8 cache */
                        vx[i] = e4m3_value(v8[base + i]) * vs;
                    }
                    for (int d = 0; d < D; ++d) qrow[d] = elem(q, ((size_t)b * Hq + h) * D + d, type);
                    rc = attend_row(qrow, kx, vx, n, D, scale, x, out + (size_t)r * D);
                }
            }
            if (rc) {
#pragma omp critical
                if (rc_all == 0 || rc < rc_all) rc_all = rc;
            }
        }
        free(kx); free(vx); free(x); free(qrow);
    }
    return rc_all;
}

/* Decode over a paged cache: the cache is a pool of pages
 * [num_pages, Hkv, page_size, D]; row t of (b, j) is row t % page_size of
 * page block_table[b * max_pages + t / page_size], KV head j (the split-K
 * heuristic of the gsyq.cn page on xformers takes `page_size` and `is_paged`
 * arguments; the page layout is this build's reading).  Everything else as
 * gqa_oracle_decode; returns 5 if a needed page index is out of range. */
int gqa_oracle_decode_paged(const void *q, const void *k_pages, const void *v_pages, int type,
                            const int32_t *block_table, int num_pages, int page_size, int max_pages,
                            const int32_t *seqlens, int B, int Hq, int Hkv, int D, double scale,
                            const int32_t *rows, int nrows, double *out)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0) return 1;
    if (num_pages <= 0 || page_size <= 0 || max_pages <= 0 || (type != 0 && type != 1)) return 1;
    int Lcap = page_size * max_pages;
    if (rows == NULL) nrows = B * Hq;
    for (int b = 0; b < B; ++b)
        if (seqlens[b] > Lcap) return 1;
    int n_rep = Hq / Hkv;
    int rc_all = 0;
#pragma omp parallel
    {
        double *kx = malloc(sizeof(double) * (size_t)Lcap * D);
        double *vx = malloc(sizeof(double) * (size_t)Lcap * D);
        double *x = malloc(sizeof(double) * (size_t)Lcap);
        double *qrow = malloc(sizeof(double) * (size_t)D);
        int oom = !(kx && vx && x && qrow);
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < nrows; ++r) {
            int rc = 0;
            if (oom) {
                rc = 2;
            } else {
                int b = rows ? rows[2 * r] : r / Hq;
                int h = rows ? rows[2 * r + 1] : r % Hq;
                if (b < 0 || b >= B || h < 0 || h >= Hq) {
                    rc = 1;
                } else {
                    int n = seqlens[b] > 0 ? seqlens[b] : 0;
                    int j = h / n_rep; /* step (2) */
                    for (int t = 0; t < n && rc == 0; ++t) {
                        int page = block_table[(size_t)b * max_pages + t / page_size];
                        if (page < 0 || page >= num_pages) {
                            rc = 5;
                            break;
                        }
                        size_t base = (((size_t)page * Hkv + j) * page_size + t % page_size) * D;
                        for (int d = 0; d < D; ++d) {
                            kx[(size_t)t * D + d] = elem(k_pages, base + d, type);
                            vx[(size_t)t * D + d] = elem(v_pages, base + d, type);
                        }
                    }
                    if (rc == 0) {
                        for (int d = 0; d < D; ++d) qrow[d] = elem(q, ((size_t)b * Hq + h) * D + d, type);
                        rc = attend_row(qrow, kx, vx, n, D, scale, x, out + (size_t)r * D);
                    }
                }
            }
            if (rc) {
#pragma omp critical
                if (rc_all == 0 || rc < rc_all) rc_all = rc;
            }
        }
        free(kx); free(vx); free(x); free(qrow);
    }
    return rc_all;
}

/* Exact values of n E4M3 bytes (for tests of the decoding itself). */
void gqa_oracle_e4m3_values(const uint8_t *bytes, int n, double *out)
{
    for (int i = 0; i < n; ++i) out[i] = e4m3_value(bytes[i]);
}

/* Prefill.
 *   q, out   [B, Hq, L, D]         k, v [B, Hkv, L, D]
 *   rows     (b, h, i) int triples, nrows of them; rows == NULL means every
 *            (b, h, i) in row-major order.
 *   causal   1: row i sees keys t <= i (square mask, query i at position i);
 *            0: every row sees all L keys. */
int gqa_oracle_prefill(const void *q, const void *k, const void *v, int type,
                       int B, int L, int Hq, int Hkv, int D, int causal, double scale,
                       const int32_t *rows, int nrows, double *out)
{
    if (B <= 0 || L <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0) return 1;
    if ((causal != 0 && causal != 1) || (type != 0 && type != 1)) return 1;
    if (rows == NULL) nrows = B * Hq * L;
    int n_rep = Hq / Hkv;
    int rc_all = 0;
#pragma omp parallel
    {
        double *kx = malloc(sizeof(double) * (size_t)L * D);
        double *vx = malloc(sizeof(double) * (size_t)L * D);
        double *x = malloc(sizeof(double) * (size_t)L);
        double *qrow = malloc(sizeof(double) * (size_t)D);
        int oom = !(kx && vx && x && qrow);
        int cur_b = -1, cur_h = -1;
#pragma omp for schedule(dynamic, 16)
        for (int r = 0; r < nrows; ++r) {
            int rc;
            if (oom) {
                rc = 2;
            } else {
                int b = rows ? rows[3 * r] : r / (Hq * L);
                int h = rows ? rows[3 * r + 1] : (r / L) % Hq;
                int i = rows ? rows[3 * r + 2] : r % L;
                if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= L) {
                    rc = 1;
                } else {
                    if (b != cur_b || h != cur_h) {
                        expand_head(k, v, type, b, h, n_rep, Hkv, L, D, L, kx, vx);
                        cur_b = b;
                        cur_h = h;
                    }
                    int n = causal ? i + 1 : L; /* (5) */
                    for (int d = 0; d < D; ++d)
                        qrow[d] = elem(q, (((size_t)b * Hq + h) * L + i) * D + d, type);
                    rc = attend_row(qrow, kx, vx, n, D, scale, x, out + (size_t)r * D);
                }
            }
            if (rc) {
#pragma omp critical
                if (rc_all == 0 || rc < rc_all) rc_all = rc;
            }
        }
        free(kx); free(vx); free(x); free(qrow);
    }
    return rc_all;
}

/* Rotary position embedding of one head vector x[D] at position pos, in place
 * (the `apply_rotary_pos_emb(query_states, key_states, cos, sin)` of the GQA
 * paper notes, "QA 相关"; the pages do not spell the rotation out, and this
 * is the plainest reading of it, the Llama "rotate half" form): for
 * i < D/2, the pair (x[i], x[i + D/2]) is rotated by the angle
 * pos * base^(-2i/D). */
static void rope_row(double *x, int D, double pos, double base)
{
    int half = D / 2;
    for (int i = 0; i < half; ++i) {
        double theta = pos * pow(base, -2.0 * i / D);
        double c = cos(theta), s = sin(theta);
        double x1 = x[i], x2 = x[i + half];
        x[i] = x1 * c - x2 * s;
        x[i + half] = x2 * c + x1 * s;
    }
}

/* The step before a decode: the new token of every sequence b sits at
 * position p = seqlens[b]; its query heads and its key heads are rotated at
 * p, and its key and value heads become row p of the cache (the Huawei Cloud
 * post, sections 2 and 5: the new K, V are concatenated to the layer's cache
 * along the sequence).
 *   q [B, Hq, D], k_new, v_new [B, Hkv, D] (element type `type`)
 *   q_out [B, Hq, D], k_row, v_row [B, Hkv, D]: fp64 results (v_row = v_new)
 * Returns 0, or 4 if some seqlens[b] >= Lmax (that row is not defined). */
int gqa_oracle_rope_append(const void *q, const void *k_new, const void *v_new, int type,
                           const int32_t *seqlens, int B, int Hq, int Hkv, int D, int Lmax,
                           double base, double *q_out, double *k_row, double *v_row)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || D % 2 || Lmax <= 0 || Hq % Hkv != 0) return 1;
    if (type != 0 && type != 1) return 1;
    int rc = 0;
    for (int b = 0; b < B; ++b) {
        int p = seqlens[b] < 0 ? 0 : seqlens[b];
        if (p >= Lmax) rc = 4;
        for (int h = 0; h < Hq; ++h) {
            double *x = q_out + ((size_t)b * Hq + h) * D;
            for (int d = 0; d < D; ++d) x[d] = elem(q, ((size_t)b * Hq + h) * D + d, type);
            rope_row(x, D, (double)p, base);
        }
        for (int j = 0; j < Hkv; ++j) {
            double *x = k_row + ((size_t)b * Hkv + j) * D;
            double *y = v_row + ((size_t)b * Hkv + j) * D;
            for (int d = 0; d < D; ++d) {
                x[d] = elem(k_new, ((size_t)b * Hkv + j) * D + d, type);
                y[d] = elem(v_new, ((size_t)b * Hkv + j) * D + d, type);
            }
            rope_row(x, D, (double)p, base);
        }
    }
    return rc;
}

/* Prefill of a chunk over a cached prefix: the queries are the last Lq of
 * Lk tokens (prefix = Lk - Lq already in the cache), k, v hold all Lk
 * keys.  Causal: chunk row i is token prefix + i and sees keys
 * t <= prefix + i (the square mask of the Huawei Cloud post, section 5,
 * aligned at the bottom right, which is where a query that follows a cached
 * prefix sits); otherwise every row sees all Lk keys.
 *   q, out [B, Hq, Lq, D]    k, v [B, Hkv, Lk, D]
 *   rows   (b, h, i) triples as gqa_oracle_prefill. */
int gqa_oracle_prefill_chunk(const void *q, const void *k, const void *v, int type, int B, int Lq, int Lk,
                             int Hq, int Hkv, int D, int causal, double scale, const int32_t *rows,
                             int nrows, double *out)
{
    if (B <= 0 || Lq <= 0 || Lk < Lq || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0) return 1;
    if ((causal != 0 && causal != 1) || (type != 0 && type != 1)) return 1;
    if (rows == NULL) nrows = B * Hq * Lq;
    int n_rep = Hq / Hkv, prefix = Lk - Lq;
    int rc_all = 0;
#pragma omp parallel
    {
        double *kx = malloc(sizeof(double) * (size_t)Lk * D);
        double *vx = malloc(sizeof(double) * (size_t)Lk * D);
        double *x = malloc(sizeof(double) * (size_t)Lk);
        double *qrow = malloc(sizeof(double) * (size_t)D);
        int oom = !(kx && vx && x && qrow);
        int cur_b = -1, cur_h = -1;
#pragma omp for schedule(dynamic, 16)
        for (int r = 0; r < nrows; ++r) {
            int rc;
            if (oom) {
                rc = 2;
            } else {
                int b = rows ? rows[3 * r] : r / (Hq * Lq);
                int h = rows ? rows[3 * r + 1] : (r / Lq) % Hq;
                int i = rows ? rows[3 * r + 2] : r % Lq;
                if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= Lq) {
                    rc = 1;
                } else {
                    if (b != cur_b || h != cur_h) {
                        expand_head(k, v, type, b, h, n_rep, Hkv, Lk, D, Lk, kx, vx);
                        cur_b = b;
                        cur_h = h;
                    }
                    int n = causal ? prefix + i + 1 : Lk; /* (5), bottom-right aligned */
                    for (int d = 0; d < D; ++d)
                        qrow[d] = elem(q, (((size_t)b * Hq + h) * Lq + i) * D + d, type);
                    rc = attend_row(qrow, kx, vx, n, D, scale, x, out + (size_t)r * D);
                }
            }
            if (rc) {
#pragma omp critical
                if (rc_all == 0 || rc < rc_all) rc_all = rc;
            }
        }
        free(kx); free(vx); free(x); free(qrow);
    }
    return rc_all;
}

/*
 * Checkpoint conversion MHA -> GQA (the GQA paper notes on 51969.com, section
 * "Uptraining", figure 1, and "checkpoint 转换实验", figure 4): the key (or
 * value) projection of an H-head model is cut into its H per-head blocks
 * w[h] (rows_per_head x cols each: the head's rows of an nn.Linear weight
 * [H * rows_per_head, cols], or of its bias with cols = 1); group j of the
 * GQA model with Hkv groups takes the heads h = j*G .. j*G + G - 1 (G = H /
 * Hkv, the grouping h -> h / G of step (2)) and its block is
 *   mode 0 ("Mean", the method the notes adopt): the mean of the G blocks,
 *   mode 1 ("First", figure 4's comparison): the block of head j*G.
 * Hkv = 1 is the MHA -> MQA conversion of figure 1.  out is [Hkv][rows][cols]
 * in fp64.
 */
int gqa_oracle_meanpool_heads(const void *w, int type, int H, int Hkv, int rows, int cols, int mode,
                              double *out)
{
    if (!w || !out || H <= 0 || Hkv <= 0 || rows <= 0 || cols <= 0 || H % Hkv != 0 || (mode != 0 && mode != 1))
        return 1;
    const int G = H / Hkv;
    const size_t n = (size_t)rows * cols;
    for (int j = 0; j < Hkv; ++j) {
        for (size_t e = 0; e < n; ++e) {
            double v;
            if (mode == 1) {
                v = elem(w, (size_t)(j * G) * n + e, type);
            } else {
                double sum = 0.0;
                for (int g = 0; g < G; ++g) sum += elem(w, (size_t)(j * G + g) * n + e, type);
                v = sum / G;
            }
            out[(size_t)j * n + e] = v;
        }
    }
    return 0;
}

int gqa_oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

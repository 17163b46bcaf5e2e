/*
 * Skip-Softmax (BLASST) attention forward: the plain CPU definition.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
 * baseline use this file. The CUDA library never links, calls or includes it,
 * and it includes nothing from the CUDA library.
 *
 * Everything is scalar C in fp64. Inputs are bf16 bit patterns (uint16), widened
 * exactly to double. Nothing is blocked, fused or reordered beyond what the
 * method itself states.
 *
 * Sources (page titles and sections):
 *   "Skip-Softmax" design doc (vLLM-Omni), section "Algorithm":
 *       the running values m, l, O of the online-softmax pass; the per-tile test
 *       exp(tile_max[i] - running_max[i]) < lambda for every row i of the tile,
 *       evaluated in log space as tile_max - running_max < ln(lambda); a skipped
 *       tile contributes nothing to l and O.
 *   same page, section "From configuration to the kernel threshold":
 *       lambda = threshold_scale_factor / max_kv_len; factor 0 skips nothing.
 *   "Skip-Softmax" (docs.vllm.ai), section "The online-softmax pass":
 *       key tiles of 128; tile scores are Q . K_j^T . scale.
 *
 * Readings where the cited sections are silent:
 *   - query tiles are 128 rows by default (tile_q is a parameter for small tests);
 *   - running_max is the row maximum over the tiles already accumulated, taken
 *     before tile j; a skipped tile leaves m, l and O unchanged;
 *   - the comparison is strict (<);
 *   - keys at index >= Sk do not exist: the last tile holds only the valid keys;
 *   - query rows at index >= Sq do not exist and therefore do not vote;
 *   - key tiles are visited in ascending order for every query tile;
 *   - lse = m + ln(l) in natural log over the kept keys.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL 1
#define ORACLE_ENOMEM 2

static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Element offset of row (b, s, h) in a contiguous [B, S, H, d] tensor. */
static size_t row_offset(int b, int s, int h, int S, int H, int d)
{
    return (((size_t)b * (size_t)S + (size_t)s) * (size_t)H + (size_t)h) * (size_t)d;
}

static double dot_row(const double *x, const uint16_t *y, int d)
{
    double acc = 0.0;
    for (int t = 0; t < d; ++t)
        acc += x[t] * bf16_bits_to_double(y[t]);
    return acc;
}

/*
 * Skip-Softmax attention for a list of units. A unit is one (b, h, qt): query
 * rows qt*tile_q .. min(qt*tile_q + tile_q, Sq) - 1 of head h in batch b.
 *
 * q: [B, Sq, H, d], k and v: [B, Sk, H, d], bf16 bits.
 * units: n_units triples (b, h, qt).
 * mask_in: NULL for the free-running test; otherwise [n_units][nK] decisions to
 *          replay instead of the test (1 = skip the tile).
 * Outputs, per unit (nK = ceil(Sk / tile_k)):
 *   o      [n_units][tile_q][d]   O / l       (rows past Sq are left untouched)
 *   lse    [n_units][tile_q]      m + ln l    (natural log)
 *   mask   [n_units][nK]          1 where the tile was skipped
 *   gap    [n_units][nK]          max over rows of (tile_max - running_max);
 *                                 +inf for the first tile. The free-running
 *                                 test is gap < ln(lambda).
 *   maxp   [n_units][tile_q]      1 / l: the row's largest softmax weight, exp(m - m) / l
 *                                 ("video-attention" blog, "max_prob = 1 / l_i").
 * Any output pointer may be NULL.
 */
int oracle_skip_softmax_attn(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                             int B, int H, int Sq, int Sk, int d,
                             double scale, double factor, int tile_q, int tile_k,
                             const int32_t *units, int n_units,
                             const uint8_t *mask_in,
                             double *o, double *lse, uint8_t *mask, double *gap, double *maxp)
{
    if (!q || !k || !v || !units || B <= 0 || H <= 0 || Sq <= 0 || Sk <= 0 || d <= 0 ||
        tile_q <= 0 || tile_k <= 0 || n_units < 0 || !(factor >= 0.0) || isinf(factor))
        return ORACLE_EINVAL;

    const int nQ = (Sq + tile_q - 1) / tile_q;
    const int nK = (Sk + tile_k - 1) / tile_k;

    /* lambda = factor / max_kv_len; the test is evaluated in log space. */
    const double ln_lambda = factor > 0.0 ? log(factor / (double)Sk) : -INFINITY;

    double *qrow = malloc(sizeof(double) * (size_t)tile_q * (size_t)d);
    double *m = malloc(sizeof(double) * (size_t)tile_q);          /* running max   */
    double *l = malloc(sizeof(double) * (size_t)tile_q);          /* running denom */
    double *acc = malloc(sizeof(double) * (size_t)tile_q * (size_t)d); /* running O */
    double *s = malloc(sizeof(double) * (size_t)tile_q * (size_t)tile_k);
    double *tile_max = malloc(sizeof(double) * (size_t)tile_q);
    if (!qrow || !m || !l || !acc || !s || !tile_max) {
        free(qrow); free(m); free(l); free(acc); free(s); free(tile_max);
        return ORACLE_ENOMEM;
    }

    int rc = ORACLE_OK;
    for (int u = 0; u < n_units; ++u) {
        const int b = units[3 * u + 0], h = units[3 * u + 1], qt = units[3 * u + 2];
        if (b < 0 || b >= B || h < 0 || h >= H || qt < 0 || qt >= nQ) {
            rc = ORACLE_EINVAL;
            break;
        }
        const int r0 = qt * tile_q;
        const int nr = (Sq - r0) < tile_q ? (Sq - r0) : tile_q; /* valid query rows */

        for (int i = 0; i < nr; ++i) {
            const uint16_t *src = q + row_offset(b, r0 + i, h, Sq, H, d);
            for (int t = 0; t < d; ++t)
                qrow[(size_t)i * d + t] = bf16_bits_to_double(src[t]);
            m[i] = -INFINITY;
            l[i] = 0.0;
            for (int t = 0; t < d; ++t)
                acc[(size_t)i * d + t] = 0.0;
        }

        for (int j = 0; j < nK; ++j) {
            const int c0 = j * tile_k;
            const int nc = (Sk - c0) < tile_k ? (Sk - c0) : tile_k; /* valid keys */

            /* Scores of this tile: S_j = Q . K_j^T . scale. */
            for (int i = 0; i < nr; ++i)
                for (int c = 0; c < nc; ++c)
                    s[(size_t)i * tile_k + c] =
                        scale * dot_row(qrow + (size_t)i * d,
                                        k + row_offset(b, c0 + c, h, Sk, H, d), d);

            /* tile_max[i]: the row's largest score within the tile. */
            for (int i = 0; i < nr; ++i) {
                double mx = -INFINITY;
                for (int c = 0; c < nc; ++c)
                    if (s[(size_t)i * tile_k + c] > mx)
                        mx = s[(size_t)i * tile_k + c];
                tile_max[i] = mx;
            }

            /* The test: every row must have tile_max - running_max < ln(lambda).
             * Equivalently the largest gap over the rows must be below ln(lambda). */
            double worst = -INFINITY;
            for (int i = 0; i < nr; ++i) {
                const double g = tile_max[i] - m[i]; /* +inf while m is -inf */
                if (g > worst)
                    worst = g;
            }
            const int skip = mask_in ? (mask_in[(size_t)u * nK + j] != 0) : (worst < ln_lambda);
            if (gap)
                gap[(size_t)u * nK + j] = worst;
            if (mask)
                mask[(size_t)u * nK + j] = (uint8_t)skip;
            if (skip)
                continue; /* the tile's contribution to l and O is omitted */

            /* Online-softmax update with the tile's scores. */
            for (int i = 0; i < nr; ++i) {
                const double m_new = m[i] > tile_max[i] ? m[i] : tile_max[i];
                const double alpha = exp(m[i] - m_new); /* 0 when m was -inf */
                l[i] *= alpha;
                for (int t = 0; t < d; ++t)
                    acc[(size_t)i * d + t] *= alpha;
                for (int c = 0; c < nc; ++c) {
                    const double p = exp(s[(size_t)i * tile_k + c] - m_new);
                    const uint16_t *vr = v + row_offset(b, c0 + c, h, Sk, H, d);
                    l[i] += p;
                    for (int t = 0; t < d; ++t)
                        acc[(size_t)i * d + t] += p * bf16_bits_to_double(vr[t]);
                }
                m[i] = m_new;
            }
        }

        /* Return O / l, and the log-sum-exp of the kept scores. */
        for (int i = 0; i < nr; ++i) {
            if (o)
                for (int t = 0; t < d; ++t)
                    o[((size_t)u * tile_q + i) * d + t] = acc[(size_t)i * d + t] / l[i];
            if (lse)
                lse[(size_t)u * tile_q + i] = m[i] + log(l[i]);
            if (maxp)
                maxp[(size_t)u * tile_q + i] = 1.0 / l[i];
        }
    }

    free(qrow); free(m); free(l); free(acc); free(s); free(tile_max);
    return rc;
}

/*
 * Dense softmax attention, written as the textbook definition and independent of
 * the tiled loop above: for each requested row, materialise all Sk scores
 * s_c = scale * q . k_c, take z = sum_c exp(s_c - max), and return
 * sum_c exp(s_c - max) v_c / z and lse = max + ln z.
 *
 * rows: n_rows triples (b, h, s) with s < Sq.
 * o: [n_rows][d]; lse: [n_rows]. Either may be NULL.
 */
int oracle_dense_attn(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      int B, int H, int Sq, int Sk, int d, double scale,
                      const int32_t *rows, int n_rows, double *o, double *lse)
{
    if (!q || !k || !v || !rows || B <= 0 || H <= 0 || Sq <= 0 || Sk <= 0 || d <= 0 || n_rows < 0)
        return ORACLE_EINVAL;
    double *x = malloc(sizeof(double) * (size_t)d);
    double *sc = malloc(sizeof(double) * (size_t)Sk);
    if (!x || !sc) {
        free(x); free(sc);
        return ORACLE_ENOMEM;
    }
    int rc = ORACLE_OK;
    for (int r = 0; r < n_rows; ++r) {
        const int b = rows[3 * r + 0], h = rows[3 * r + 1], si = rows[3 * r + 2];
        if (b < 0 || b >= B || h < 0 || h >= H || si < 0 || si >= Sq) {
            rc = ORACLE_EINVAL;
            break;
        }
        const uint16_t *qr = q + row_offset(b, si, h, Sq, H, d);
        for (int t = 0; t < d; ++t)
            x[t] = bf16_bits_to_double(qr[t]);
        double mx = -INFINITY;
        for (int c = 0; c < Sk; ++c) {
            sc[c] = scale * dot_row(x, k + row_offset(b, c, h, Sk, H, d), d);
            if (sc[c] > mx)
                mx = sc[c];
        }
        double z = 0.0;
        for (int c = 0; c < Sk; ++c) {
            sc[c] = exp(sc[c] - mx); /* unnormalised softmax weight of key c */
            z += sc[c];
        }
        if (o) {
            for (int t = 0; t < d; ++t) {
                double num = 0.0;
                for (int c = 0; c < Sk; ++c)
                    num += sc[c] * bf16_bits_to_double(v[row_offset(b, c, h, Sk, H, d) + t]);
                o[(size_t)r * d + t] = num / z;
            }
        }
        if (lse)
            lse[r] = mx + log(z);
    }
    free(x);
    free(sc);
    return rc;
}

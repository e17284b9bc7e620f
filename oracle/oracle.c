/*
 * CPU oracle for the MultiTowerDIN sparse forward.  TEST INFRASTRUCTURE ONLY:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg load it.
 * It shares no code, header or constant with the CUDA library; it is a plain,
 * slow, loop-by-loop restatement of the method as the pages describe it.
 *
 * Pages (cited by title and section):
 *   [P1] "MultiTowerDIN: current state analysis" (westfly, torcheasyrec-analysis 18-01)
 *   [P2] "MultiTowerDIN: integrating DynamicEmb" (westfly, torcheasyrec-analysis 18-02)
 *
 * Steps and the passages they follow:
 *   offsets  exclusive scan of KJT lengths              [P1 s2 pipeline: SparseData(values, lengths) -> KJT]
 *   pooling  EmbeddingBag sum per (feature, sample) bag  [P1 s3 "num_buckets" block: [N,16] table per feature]
 *   query    cat of the target bags adgroup/cate/brand   [P1 s1 feature-group block; P2 s2.4 shared tables]
 *   padded   to_padded_dense(max_len) of the sequence    [P1 s4.1]
 *   attn in  cat[q, s, q-s, q*s]                        [P1 s4.2 code block]
 *   MLP      attn_mlp hidden [256, 64] then linear -> 1  [P1 s4.2 shape block; P2 s7 din_towers]
 *   mask     softmax over valid positions only           [P1 s4.2 "mask + softmax", s4.4 graph]
 *   output   weighted sum [B,1,L] @ [B,L,48] -> [B,48]   [P1 s4.4 graph]
 *   precision: lookup fp32, MLP in half precision        [P2 s3.3]
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - MLP activation: Linear+bias -> ReLU -> Linear+bias -> ReLU -> Linear(64->1)+bias.
 *   - mask value is -inf; a sample with no valid position gives the zero vector.
 *   - a sequence longer than max_len keeps its first max_len positions.
 *   - ids outside [0, rows) and negative lengths are input errors: the row
 *     contributes zero / the length counts as zero, and a flag bit is returned.
 *
 * Precision: pooled sums are fp32, left to right in bag order (the pages fix
 * the lookup at fp32).  The attention path runs in double.  With bf16_mlp=1
 * the MLP operands are rounded to bf16 the way a half-precision MLP sees them
 * (x and h1 produced in fp32 then rounded to nearest-even bf16; W1, W2 rounded
 * to bf16); accumulation stays in double.
 *
 * Flag bits returned (the library's status bits mean the same):
 *   1 id out of range, 2 negative length, 4 sequence truncated to max_len,
 *   8 lengths imply more values than the values array holds.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_ID_RANGE 1
#define OR_NEG_LENGTH 2
#define OR_SEQ_TRUNC 4
#define OR_COUNT 8

/* bf16 (stored as its upper 16 bits) -> float, exact. */
static float bf16_to_float(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round a float to the nearest bf16, ties to even; returns the float value. */
static float round_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u) { /* inf / nan: keep */
        u &= 0xffff0000u;
        if ((f != f)) u |= 0x00400000u;
    } else {
        uint32_t lsb = (u >> 16) & 1u;
        u += 0x7fffu + lsb;
        u &= 0xffff0000u;
    }
    memcpy(&f, &u, 4);
    return f;
}

/* Element (row, col) of table t as float. */
static float table_at(const void *table, int32_t dtype, int32_t D, int64_t row, int32_t col)
{
    if (dtype == 1) return bf16_to_float(((const uint16_t *)table)[row * D + col]);
    return ((const float *)table)[row * D + col];
}

/* Exclusive scan of n lengths; negative lengths count as zero (flag 2). */
int oracle_offsets(const int32_t *lengths, int64_t n, int64_t *offsets)
{
    int flags = 0;
    int64_t acc = 0;
    for (int64_t i = 0; i < n; i++) {
        offsets[i] = acc;
        int32_t l = lengths[i];
        if (l < 0) { flags |= OR_NEG_LENGTH; l = 0; }
        acc += l;
    }
    offsets[n] = acc;
    return flags;
}

/* Pool one bag into out[0..D): the fp32 sum, left to right; with mean, that
 * sum divided (fp32) by the bag's length, which counts every id of the bag
 * (EmbeddingBag mean mode). An empty bag gives 0 either way. */
static int pool_bag(const void *table, int64_t rows, int32_t dtype, int32_t D,
                    const int64_t *values, int64_t n_values, int64_t begin, int64_t end,
                    int mean, float *out)
{
    int flags = 0;
    for (int32_t d = 0; d < D; d++) out[d] = 0.0f;
    for (int64_t i = begin; i < end; i++) {
        if (i >= n_values) { flags |= OR_COUNT; continue; }
        int64_t id = values[i];
        if (id < 0 || id >= rows) { flags |= OR_ID_RANGE; continue; }
        for (int32_t d = 0; d < D; d++) out[d] += table_at(table, dtype, D, id, d);
    }
    if (mean && end > begin)
        for (int32_t d = 0; d < D; d++) out[d] = out[d] / (float)(end - begin);
    return flags;
}

/*
 * EmbeddingBag pooling over a key-major KJT.
 * tables[f]: [rows[f], D]; lengths: [F*B]; pooling: [F], 0 = sum, 1 = mean
 * (NULL: all sum); samples: which samples to produce;
 * pooled: [n_samples, F*D] float, row i is sample samples[i].
 */
int oracle_emb_bag_pool(int32_t F, int32_t D, int32_t dtype,
                        const void *const *tables, const int64_t *rows,
                        const int32_t *pooling,
                        int32_t B, const int64_t *values, int64_t n_values,
                        const int32_t *lengths,
                        const int32_t *samples, int32_t n_samples, float *pooled)
{
    int64_t nb = (int64_t)F * B;
    int64_t *off = (int64_t *)malloc((size_t)(nb + 1) * sizeof(int64_t));
    if (!off) return -1;
    int flags = oracle_offsets(lengths, nb, off);
    if (off[nb] > n_values) flags |= OR_COUNT;
    for (int32_t i = 0; i < n_samples; i++) {
        int32_t b = samples[i];
        for (int32_t f = 0; f < F; f++) {
            int64_t g = (int64_t)f * B + b;
            flags |= pool_bag(tables[f], rows[f], dtype, D, values, n_values,
                              off[g], off[g + 1], pooling && pooling[f] == 1,
                              pooled + ((int64_t)i * F + f) * D);
        }
    }
    free(off);
    return flags;
}

/*
 * The attention MLP on n rows of x [n, K1] (double):
 *   h1 = ReLU(W1 x + b1)  [N1];  h2 = ReLU(W2 h1 + b2)  [N2];  z = w3 . h2 + b3.
 * W1 [N1, K1], W2 [N2, N1] in Linear [out, in] layout.  bf16_mlp: x, W1, W2 and
 * h1 are taken as bf16 values (x must already hold bf16 values in that mode).
 */
int oracle_attn_mlp(const double *x, int64_t n, int32_t K1, int32_t N1, int32_t N2,
                    const float *W1, const float *b1, const float *W2, const float *b2,
                    const float *w3, const float *b3, int32_t bf16_mlp, double *z)
{
    double *h1 = (double *)malloc((size_t)N1 * sizeof(double));
    double *h2 = (double *)malloc((size_t)N2 * sizeof(double));
    if (!h1 || !h2) { free(h1); free(h2); return -1; }
    for (int64_t r = 0; r < n; r++) {
        const double *xr = x + r * K1;
        for (int32_t j = 0; j < N1; j++) {
            double acc = 0.0;
            for (int32_t k = 0; k < K1; k++) {
                double w = bf16_mlp ? (double)round_bf16(W1[(int64_t)j * K1 + k])
                                    : (double)W1[(int64_t)j * K1 + k];
                acc += w * xr[k];
            }
            if (bf16_mlp) {
                float v = (float)acc + b1[j];
                v = v > 0.0f ? v : 0.0f;
                h1[j] = (double)round_bf16(v);
            } else {
                double v = acc + (double)b1[j];
                h1[j] = v > 0.0 ? v : 0.0;
            }
        }
        for (int32_t j = 0; j < N2; j++) {
            double acc = 0.0;
            for (int32_t k = 0; k < N1; k++) {
                double w = bf16_mlp ? (double)round_bf16(W2[(int64_t)j * N1 + k])
                                    : (double)W2[(int64_t)j * N1 + k];
                acc += w * h1[k];
            }
            double v = acc + (double)b2[j];
            h2[j] = v > 0.0 ? v : 0.0;
        }
        double zz = (double)b3[0];
        for (int32_t j = 0; j < N2; j++) zz += (double)w3[j] * h2[j];
        z[r] = zz;
    }
    free(h1);
    free(h2);
    return 0;
}

/*
 * DIN target attention for the listed samples.
 *   padded=1: the pages' flow -- sequence padded to max_len with zeros, MLP run
 *             on every padded position, padding masked with -inf before softmax.
 *   padded=0: jagged -- the same loops over the valid positions only.
 * q_feat[3]: KJT features whose pooled bags form the query (target items).
 * seq_table[3]: table of each sequence sub-feature (shared with the query tables).
 * seq_values: [3, n_seq] key-major; seq_lengths: [B].
 * din: [n_samples, 3D]; logits / weights (nullable): [n_samples, max_len],
 * entries past the valid positions are set to -inf / 0.
 */
int oracle_din(int32_t padded, int32_t bf16_mlp,
               int32_t F, int32_t D, int32_t dtype,
               const void *const *tables, const int64_t *rows, const int32_t *pooling,
               int32_t B, const int64_t *values, int64_t n_values, const int32_t *lengths,
               const int32_t *q_feat, const int32_t *seq_table,
               const int64_t *seq_values, int64_t n_seq, const int32_t *seq_lengths,
               int32_t max_len,
               const float *W1, const float *b1, const float *W2, const float *b2,
               const float *w3, const float *b3, int32_t N1, int32_t N2,
               const int32_t *samples, int32_t n_samples,
               double *din, double *logits, double *weights)
{
    const int32_t Q = 3 * D, K1 = 4 * Q;
    int64_t nb = (int64_t)F * B;
    int64_t *off = (int64_t *)malloc((size_t)(nb + 1) * sizeof(int64_t));
    int64_t *soff = (int64_t *)malloc((size_t)(B + 1) * sizeof(int64_t));
    float *qf = (float *)malloc((size_t)Q * sizeof(float));
    double *S = (double *)malloc((size_t)max_len * Q * sizeof(double));
    double *X = (double *)malloc((size_t)max_len * K1 * sizeof(double));
    double *Z = (double *)malloc((size_t)max_len * sizeof(double));
    double *A = (double *)malloc((size_t)max_len * sizeof(double));
    int flags = 0;
    if (!off || !soff || !qf || !S || !X || !Z || !A) { flags = -1; goto done; }
    flags |= oracle_offsets(lengths, nb, off);
    if (off[nb] > n_values) flags |= OR_COUNT;
    flags |= oracle_offsets(seq_lengths, B, soff);
    if (soff[B] > n_seq) flags |= OR_COUNT;

    for (int32_t i = 0; i < n_samples; i++) {
        int32_t b = samples[i];
        double *out = din + (int64_t)i * Q;
        /* query: the pooled target bags, as the lookup produces them (fp32) */
        for (int32_t k = 0; k < 3; k++) {
            int32_t f = q_feat[k];
            int64_t g = (int64_t)f * B + b;
            flags |= pool_bag(tables[f], rows[f], dtype, D, values, n_values,
                              off[g], off[g + 1], pooling && pooling[f] == 1, qf + k * D);
        }
        int32_t L = seq_lengths[b];
        if (L < 0) L = 0;
        if (L > max_len) { flags |= OR_SEQ_TRUNC; L = max_len; }
        int32_t T = padded ? max_len : L;

        /* sequence rows: cat of the three sub-feature embeddings; zeros past L */
        for (int32_t t = 0; t < T; t++) {
            for (int32_t k = 0; k < 3; k++) {
                for (int32_t d = 0; d < D; d++) S[(int64_t)t * Q + k * D + d] = 0.0;
                if (t >= L) continue;
                int64_t j = soff[b] + t;
                if (j >= n_seq) { flags |= OR_COUNT; continue; }
                int32_t tb = seq_table[k];
                int64_t id = seq_values[(int64_t)k * n_seq + j];
                if (id < 0 || id >= rows[tb]) { flags |= OR_ID_RANGE; continue; }
                for (int32_t d = 0; d < D; d++)
                    S[(int64_t)t * Q + k * D + d] = (double)table_at(tables[tb], dtype, D, id, d);
            }
        }
        /* attention input cat[q, s, q - s, q * s] */
        for (int32_t t = 0; t < T; t++) {
            double *x = X + (int64_t)t * K1;
            for (int32_t d = 0; d < Q; d++) {
                double q = (double)qf[d], s = S[(int64_t)t * Q + d];
                if (bf16_mlp) {
                    float qf32 = qf[d], sf32 = (float)s;
                    x[d] = round_bf16(qf32);
                    x[Q + d] = round_bf16(sf32);
                    x[2 * Q + d] = round_bf16(qf32 - sf32);
                    x[3 * Q + d] = round_bf16(qf32 * sf32);
                } else {
                    x[d] = q;
                    x[Q + d] = s;
                    x[2 * Q + d] = q - s;
                    x[3 * Q + d] = q * s;
                }
            }
        }
        if (T > 0 && oracle_attn_mlp(X, T, K1, N1, N2, W1, b1, W2, b2, w3, b3, bf16_mlp, Z) != 0) {
            flags = -1;
            goto done;
        }
        /* mask, softmax over the valid positions, weighted sum of s */
        for (int32_t t = L; t < T; t++) Z[t] = -INFINITY;
        for (int32_t d = 0; d < Q; d++) out[d] = 0.0;
        if (L > 0) {
            double m = -INFINITY;
            for (int32_t t = 0; t < T; t++) if (Z[t] > m) m = Z[t];
            double l = 0.0;
            for (int32_t t = 0; t < T; t++) { A[t] = exp(Z[t] - m); l += A[t]; }
            for (int32_t t = 0; t < T; t++) A[t] /= l;
            for (int32_t t = 0; t < T; t++)
                for (int32_t d = 0; d < Q; d++) out[d] += A[t] * S[(int64_t)t * Q + d];
        } else {
            for (int32_t t = 0; t < T; t++) A[t] = 0.0;
        }
        if (logits) {
            for (int32_t t = 0; t < max_len; t++)
                logits[(int64_t)i * max_len + t] = t < L ? Z[t] : -INFINITY;
        }
        if (weights) {
            for (int32_t t = 0; t < max_len; t++)
                weights[(int64_t)i * max_len + t] = t < L ? A[t] : 0.0;
        }
    }
done:
    free(off); free(soff); free(qf); free(S); free(X); free(Z); free(A);
    return flags;
}

/*
 * The dense towers after the sparse path (MultiTowerDIN: current state
 * analysis, section 4.4 and the model config of section 7):
 *   deep tower  h = ReLU(W_d3 ReLU(W_d2 ReLU(W_d1 p + b_d1) + b_d2) + b_d3)
 *               with p the pooled deep group [256] and widths 512, 256, 128;
 *   final tower y = w_o . ReLU(W_f1 cat[h, din] + b_f1) + b_o
 *               with cat[h, din] of width 128 + 48 = 176 and W_f1 [64, 176];
 * y is the logit (the loss, binary cross entropy, applies the sigmoid).
 * Weights in Linear [out, in] layout.  pooled: [n, 256] float; din: [n, 48]
 * double; logit: [n] double.  Accumulation in double.  bf16_mlp: every
 * GEMM operand is taken as bf16 -- the inputs p, h1, h2 and cat[h, din] are
 * produced in fp32 (bias added, ReLU) and rounded to nearest-even bf16, the
 * weights W_d1, W_d2, W_d3, W_f1 rounded too; the output dot stays fp32/double.
 */
int oracle_towers(const float *pooled, const double *din, int64_t n,
                  const float *Wd1, const float *bd1, const float *Wd2, const float *bd2,
                  const float *Wd3, const float *bd3, const float *Wf1, const float *bf1,
                  const float *wo, const float *bo, int32_t bf16_mlp, double *logit)
{
    enum { P = 256, H1 = 512, H2 = 256, H3 = 128, DQ = 48, KF = H3 + DQ, HF = 64 };
    double x[H1], h1[H1], h2[H2], c[KF], hf[HF];
    for (int64_t r = 0; r < n; r++) {
        const float *pr = pooled + r * P;
        for (int32_t k = 0; k < P; k++)
            x[k] = bf16_mlp ? (double)round_bf16(pr[k]) : (double)pr[k];
        /* one Linear + ReLU layer: out[j] = ReLU(W[j,:] . in + b[j]) */
#define DENSE(W, b, in, K, out, N)                                                   \
        for (int32_t j = 0; j < (N); j++) {                                          \
            double acc = 0.0;                                                        \
            for (int32_t k = 0; k < (K); k++) {                                      \
                double w = bf16_mlp ? (double)round_bf16((W)[(int64_t)j * (K) + k])  \
                                    : (double)(W)[(int64_t)j * (K) + k];             \
                acc += w * (in)[k];                                                  \
            }                                                                        \
            if (bf16_mlp) {                                                          \
                float v = (float)acc + (b)[j];                                       \
                (out)[j] = v > 0.0f ? (double)v : 0.0;                               \
            } else {                                                                 \
                double v = acc + (double)(b)[j];                                     \
                (out)[j] = v > 0.0 ? v : 0.0;                                        \
            }                                                                        \
        }
        DENSE(Wd1, bd1, x, P, h1, H1)
        if (bf16_mlp) for (int32_t k = 0; k < H1; k++) h1[k] = (double)round_bf16((float)h1[k]);
        DENSE(Wd2, bd2, h1, H1, h2, H2)
        if (bf16_mlp) for (int32_t k = 0; k < H2; k++) h2[k] = (double)round_bf16((float)h2[k]);
        DENSE(Wd3, bd3, h2, H2, c, H3)
        for (int32_t k = 0; k < DQ; k++) c[H3 + k] = din[r * DQ + k];
        if (bf16_mlp) for (int32_t k = 0; k < KF; k++) c[k] = (double)round_bf16((float)c[k]);
        DENSE(Wf1, bf1, c, KF, hf, HF)
#undef DENSE
        double y = (double)bo[0];
        for (int32_t j = 0; j < HF; j++) y += (double)wo[j] * hf[j];
        logit[r] = y;
    }
    return 0;
}

/*
 * Plain CPU oracle for the W4A16 group-quantized matrix-vector path.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this file. It shares no code, header, table or helper
 * with the CUDA library, and the CUDA library never calls it.
 *
 * What it computes is the plain definition, written out slowly and in fp64:
 *
 *   Source: "Gemma 4 E2B on a 4 GB GPU with pure PyTorch" (ainews.gemivo.de).
 *   - The checkpoint paragraph: compressed-tensors W4A16, 4-bit weights in groups
 *     of 32 along K, 16-bit activations; each group's step is stored in bf16.
 *   - The w4gemv paragraph: the kernel reads packed 4-bit words and multiplies
 *     without making a 16-bit copy; the unpack turns a code into (code - 8)
 *     ("OR into the bits of 2^23 and subtract 2^23 + 8"), so the zero point is 8.
 *   - The "Step 2 - Keep the Vocabulary Tables in 4-Bit" paragraph: the embedding
 *     and per-layer tables are 4-bit codes with a 16-bit step per group, and the
 *     per-layer row lookup runs on the card.
 *   - The memory-read paragraph: the card's read ceiling is measured by a plain
 *     sum over memory.
 *   - The decode-attention paragraph: one key/value head serves eight query
 *     heads; each cached key and value is read once for all of them and the
 *     result is a softmax over the cached positions, then the values. The
 *     cache paragraph: full layers keep one slot per position, sliding layers a
 *     512-slot ring that records each slot's position; "Step 4 - The Model in
 *     Rust": the ring's attention keeps a slot only if its recorded position is
 *     >= 0, not after the query's position, and (with a window w) after the
 *     query's position minus w, then takes the softmax and the values.
 *
 * Readings where the pages are silent (each one is stated where it is used):
 *   R1  8 codes per uint32 along K, low nibble first: code k sits in word k/8 at
 *       bits 4*(k%8) .. 4*(k%8)+3.
 *   R2  qweight is [N][K/8] (row n = output n, PyTorch Linear orientation),
 *       scales are [N][K/group] row-major, x is [M][K], y = x * W^T is [M][N].
 *   R3  The gather output is bf16, round-to-nearest-even of the exact product.
 *   R4  Argmax is the lowest index of the largest value; -0 equals +0.
 *   R5  The read probe's result is the sum of all 32-bit words mod 2^64.
 *   R7  Hadamard rotation ("fastgemma-gemma-4-E2B" card: every linear weight is
 *       rotated along K, W' = W H^T, and a runtime fast Walsh-Hadamard
 *       transform of the activation makes the product identical): H is
 *       block-diagonal over blocks of b consecutive k, each block the Sylvester
 *       matrix H_b[i][j] = (-1)^popcount(i & j) / sqrt(b), which is symmetric and
 *       orthogonal; the rotated product is y = (x H) W'^T.
 *   R6  Attention scores are scale * (q . k) with the scale an argument (the
 *       pages' listing multiplies q by k^T and names no scale); a query with no
 *       kept slot gives a zero output.
 *
 * Parity pins: every function here is pinned by the not-gpu tests (hand-worked
 * examples with the packed words written in hex, closed forms, invariants, and
 * exact rational brute force on tiny shapes). None is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* bf16 bits -> value. bf16 is the top 16 bits of an IEEE binary32. */
static double bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* binary32 -> bf16 bits, round to nearest, ties to even (finite inputs). */
static uint16_t float_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xFFFFu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u;
    return (uint16_t)upper;
}

/* R1: the 4-bit code of column k in a packed row. */
static unsigned code_at(const uint32_t *row_words, int64_t k)
{
    uint32_t word = row_words[k / 8];
    unsigned shift = 4u * (unsigned)(k % 8);
    return (unsigned)((word >> shift) & 0xFu);
}

/* The dequantized weight w(n,k) = (code - 8) * step(n, k / group), exact in fp64. */
static double weight_at(const uint32_t *qweight, const uint16_t *scales,
                        int64_t K, int64_t group, int64_t n, int64_t k)
{
    const uint32_t *row = qweight + n * (K / 8);
    int code = (int)code_at(row, k);
    double step = bf16_to_double(scales[n * (K / group) + k / group]);
    return (double)(code - 8) * step;
}

/*
 * y[m][j] = sum_{k=0}^{K-1} x[m][k] * w(rows[j], k), ascending k, fp64;
 * absy[m][j] = sum_k |x[m][k] * w(rows[j], k)| (the tolerance scale).
 * rows == NULL means every row 0..N-1 (then nrows must equal N).
 */
void w4o_gemm_rows(double *y, double *absy,
                   const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
                   int64_t M, int64_t N, int64_t K, int64_t group,
                   const int64_t *rows, int64_t nrows)
{
    (void)N;
    for (int64_t j = 0; j < nrows; ++j) {
        int64_t n = rows ? rows[j] : j;
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0, acc_abs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double t = bf16_to_double(x[m * K + k]) *
                           weight_at(qweight, scales, K, group, n, k);
                acc += t;
                acc_abs += fabs(t);
            }
            y[m * nrows + j] = acc;
            if (absy)
                absy[m * nrows + j] = acc_abs;
        }
    }
}

/* Full product: y = x * W^T over every row. */
void w4o_gemm(double *y, double *absy,
              const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
              int64_t M, int64_t N, int64_t K, int64_t group)
{
    w4o_gemm_rows(y, absy, x, qweight, scales, M, N, K, group, NULL, N);
}

/* Dequantize rows of W to fp64 [nrows][K] (used to build dense references). */
void w4o_dequant_rows(double *w, const uint32_t *qweight, const uint16_t *scales,
                      int64_t N, int64_t K, int64_t group,
                      const int64_t *rows, int64_t nrows)
{
    (void)N;
    for (int64_t j = 0; j < nrows; ++j) {
        int64_t n = rows ? rows[j] : j;
        for (int64_t k = 0; k < K; ++k)
            w[j * K + k] = weight_at(qweight, scales, K, group, n, k);
    }
}

/*
 * R4 (greedy decoding picks the most likely token): the lowest index n with
 * y[n] == max y, comparing -0 and +0 as equal. *gap receives max - (largest
 * value at any other index), or +inf when N == 1.
 */
int64_t w4o_argmax(const double *y, int64_t N, double *gap)
{
    int64_t best = 0;
    for (int64_t n = 1; n < N; ++n)
        if (y[n] > y[best])
            best = n;
    double second = -INFINITY;
    for (int64_t n = 0; n < N; ++n)
        if (n != best && y[n] > second)
            second = y[n];
    if (gap)
        *gap = (N > 1) ? (y[best] - second) : INFINITY;
    return best;
}

/*
 * The 4-bit row gather: out[t][k] = bf16_rne((code(ids[t], k) - 8) * step).
 * The product of a 4-bit integer and a bf16 step has at most 12 significant
 * bits, so it is exact in binary32 and the only rounding is the final one (R3).
 * An id outside [0, N) gives a zero row and sets *flag to 1.
 */
void w4o_embed_gather(uint16_t *out, const int32_t *ids,
                      const uint32_t *qtable, const uint16_t *scales,
                      int64_t M, int64_t N, int64_t K, int64_t group, int32_t *flag)
{
    for (int64_t t = 0; t < M; ++t) {
        int64_t id = ids[t];
        for (int64_t k = 0; k < K; ++k) {
            if (id < 0 || id >= N) {
                out[t * K + k] = 0;
                if (flag)
                    *flag = 1;
                continue;
            }
            double v = weight_at(qtable, scales, K, group, id, k);
            out[t * K + k] = float_to_bf16_rne((float)v);
        }
    }
}

/* R5: the memory read probe's checksum, sum of uint32 words mod 2^64. */
uint64_t w4o_sum_words(const uint32_t *buf, int64_t nwords)
{
    uint64_t s = 0;
    for (int64_t i = 0; i < nwords; ++i)
        s += (uint64_t)buf[i];
    return s;
}

/* Exposed for the pins on rounding: binary32 -> bf16 bits, RNE. */
uint16_t w4o_f32_to_bf16(float f) { return float_to_bf16_rne(f); }

/*
 * Decode attention for one query token (R6), in fp64, the plain definition:
 *   s[h][t] = scale * sum_d q[h][d] * k[t][d]            for kept slots t
 *   w[h][t] = exp(s[h][t] - max_t s[h][t]) / sum_t exp(...)
 *   out[h][d] = sum_t w[h][t] * v[t][d],  absout[h][d] = sum_t w[h][t] * |v[t][d]|
 * Slot t records position kpos[t] (kpos == NULL: position t). It is kept iff
 * kpos[t] >= 0, kpos[t] <= qpos and, when window > 0, kpos[t] > qpos - window.
 * q is bf16 bits [H][D]; k and v are bf16 bits [T][D] (one key/value head).
 * s is caller scratch of T doubles.
 */
void w4o_attn_decode(double *out, double *absout, const uint16_t *q, const uint16_t *k,
                     const uint16_t *v, const int32_t *kpos, int64_t qpos, int64_t window,
                     int64_t H, int64_t T, int64_t D, double scale, double *s)
{
    for (int64_t h = 0; h < H; ++h) {
        double mx = -INFINITY;
        for (int64_t t = 0; t < T; ++t) {
            int64_t p = kpos ? (int64_t)kpos[t] : t;
            int keep = p >= 0 && p <= qpos && (window <= 0 || p > qpos - window);
            if (!keep) {
                s[t] = -INFINITY;
                continue;
            }
            double acc = 0.0;
            for (int64_t d = 0; d < D; ++d)
                acc += bf16_to_double(q[h * D + d]) * bf16_to_double(k[t * D + d]);
            s[t] = scale * acc;
            if (s[t] > mx)
                mx = s[t];
        }
        for (int64_t d = 0; d < D; ++d) {
            out[h * D + d] = 0.0;
            absout[h * D + d] = 0.0;
        }
        if (mx == -INFINITY)
            continue;
        double z = 0.0;
        for (int64_t t = 0; t < T; ++t) {
            s[t] = (s[t] == -INFINITY) ? 0.0 : exp(s[t] - mx);
            z += s[t];
        }
        for (int64_t t = 0; t < T; ++t) {
            if (s[t] == 0.0)
                continue;
            double w = s[t] / z;
            for (int64_t d = 0; d < D; ++d) {
                double vv = bf16_to_double(v[t * D + d]);
                out[h * D + d] += w * vv;
                absout[h * D + d] += w * fabs(vv);
            }
        }
    }
}

/*
 * R7: xr[m][k] = sum_j x[m][j] * H_b[j mod b][k mod b] over the block of k, in
 * fp64, by the definition (no butterflies): b must be a power of two dividing K.
 */
void w4o_hadamard_rows(double *xr, const uint16_t *x, int64_t M, int64_t K, int64_t b)
{
    const double norm = 1.0 / sqrt((double)b);
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t k = 0; k < K; ++k) {
            const int64_t blk = k - k % b, kk = k % b;
            double acc = 0.0;
            for (int64_t j = 0; j < b; ++j) {
                const int sign = __builtin_popcountll((unsigned long long)(j & kk)) & 1;
                const double v = bf16_to_double(x[m * K + blk + j]);
                acc += sign ? -v : v;
            }
            xr[m * K + k] = acc * norm;
        }
    }
}

/* w4o_gemm_rows with an fp64 activation (the rotated x of R7). */
void w4o_gemm_rows_xf64(double *y, double *absy,
                        const double *x, const uint32_t *qweight, const uint16_t *scales,
                        int64_t M, int64_t N, int64_t K, int64_t group,
                        const int64_t *rows, int64_t nrows)
{
    (void)N;
    for (int64_t j = 0; j < nrows; ++j) {
        int64_t n = rows ? rows[j] : j;
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0, acc_abs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double t = x[m * K + k] * weight_at(qweight, scales, K, group, n, k);
                acc += t;
                acc_abs += fabs(t);
            }
            y[m * nrows + j] = acc;
            if (absy)
                absy[m * nrows + j] = acc_abs;
        }
    }
}

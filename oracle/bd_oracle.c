/*
 * BitDelta oracle: a plain, slow, fp64 CPU restatement of what the GPU path
 * computes.  TEST INFRASTRUCTURE ONLY: tests, the smoke check and the CPU
 * baseline leg of the benchmark call it; the product library never links,
 * loads or calls it, and it shares no source with the GPU path.
 *
 * Source of the method: the blog page "BitDelta : servir 14 modèles Zen depuis
 * un seul cluster GPU" (Hanzo blog, 2026-02-28; the same text is mirrored in
 * Thai, Traditional Chinese and Japanese).  Citations below name its sections:
 *   [math]  "Le fondement mathématique"  -- delta, 1-bit approximation, alpha
 *   [serve] "Architecture de service"    -- on-the-fly reconstruction, the
 *           conceptual fused_bitdelta_linear listing (unpack to {-1,+1},
 *           W_eff = W_base + alpha * unpacked, then a plain linear)
 *   [infra] "Détails d'infrastructure"   -- 8 sign bits per byte, fp32 alpha,
 *           4096x4096 -> 4096x512 packed
 *
 * Readings where the page leaves a step open (each listed in the design notes):
 *   - bit order inside a byte is not printed: bit i of byte c of row j holds
 *     the sign of element k = 8c + i (least significant bit = lowest d_in).
 *   - sign(0) is not printed; the listing says the unpacked values are only
 *     -1 and +1, so Delta >= 0 (including -0.0) maps to bit 1 -> +1.
 *   - alpha is "one per matrix" in [math] and "one per output dimension" in
 *     [infra]; both are supported: scalar mode = mean|Delta| over the matrix,
 *     per-row mode = mean|Delta| over row j.
 *   - "int8" storage is read as raw bytes (uint8 here, so shifts never sign
 *     extend); the byte values are identical.
 *
 * All arithmetic is fp64, except bdo_weff_bf16, which produces the stored
 * bf16 W_eff and therefore takes the rounding decisions the reading fixes
 * (fp32 sum, one rounding to bf16).  bf16 inputs arrive as their 16-bit patterns
 * (uint16) and widen exactly.  Sums are plain left-to-right loops: no
 * blocking, no reassociation.  Rows of independent outputs may run on
 * separate OpenMP threads; that changes no sum.
 *
 * Layouts (row-major): W_base, W_ft [n_out, n_in]; bits [n_out, n_in/8];
 * x [m, n_in]; y [m, n_out]; alpha [1] (scalar) or [n_out] (per-row).
 */
#include <stdint.h>
#include <string.h>
#include <math.h>

static double bf16_to_f64(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* [math] Delta = W_ft - W_base, element-wise.  Exact in fp64 for bf16 data. */
void bdo_delta(const uint16_t *w_base, const uint16_t *w_ft, int64_t count,
               double *delta)
{
    for (int64_t i = 0; i < count; ++i)
        delta[i] = bf16_to_f64(w_ft[i]) - bf16_to_f64(w_base[i]);
}

/* [math] sign(Delta) at one bit per element; [infra] eight bits per byte.
 * Byte c of row j = sum over i in 0..7 of bit(j, 8c+i) * 2^i, with
 * bit = 1 iff Delta >= 0. */
void bdo_sign_bits(const uint16_t *w_base, const uint16_t *w_ft,
                   int64_t n_out, int64_t n_in, uint8_t *bits)
{
    const int64_t bytes_per_row = n_in / 8;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n_out; ++j) {
        for (int64_t c = 0; c < bytes_per_row; ++c) {
            unsigned byte = 0;
            for (int i = 0; i < 8; ++i) {
                const int64_t e = j * n_in + 8 * c + i;
                const double d = bf16_to_f64(w_ft[e]) - bf16_to_f64(w_base[e]);
                if (d >= 0.0)
                    byte |= 1u << i;
            }
            bits[j * bytes_per_row + c] = (uint8_t)byte;
        }
    }
}

/* [math] alpha = (1/n) * ||Delta||_1 = mean |Delta_ij| over the matrix
 * (mode 0, one value), or [infra] one value per output row (mode 1):
 * alpha_j = (1/n_in) * sum_k |Delta_jk|.  Returned in fp64; storage in fp32
 * is the caller's rounding. */
void bdo_alpha(const uint16_t *w_base, const uint16_t *w_ft, int64_t n_out,
               int64_t n_in, int mode, double *alpha)
{
    if (mode == 1) {
#pragma omp parallel for schedule(static)
        for (int64_t j = 0; j < n_out; ++j) {
            double s = 0.0;
            for (int64_t k = 0; k < n_in; ++k) {
                const int64_t e = j * n_in + k;
                s += fabs(bf16_to_f64(w_ft[e]) - bf16_to_f64(w_base[e]));
            }
            alpha[j] = s / (double)n_in;
        }
    } else {
        double s = 0.0;
        const int64_t count = n_out * n_in;
        for (int64_t e = 0; e < count; ++e)
            s += fabs(bf16_to_f64(w_ft[e]) - bf16_to_f64(w_base[e]));
        alpha[0] = s / (double)count;
    }
}

/* [serve] unpack_bits: bit 1 -> +1, bit 0 -> -1 (the listing's {-1, +1}). */
void bdo_unpack_signs(const uint8_t *bits, int64_t n_out, int64_t n_in,
                      int8_t *signs)
{
    const int64_t bytes_per_row = n_in / 8;
    for (int64_t j = 0; j < n_out; ++j)
        for (int64_t k = 0; k < n_in; ++k) {
            const unsigned byte = bits[j * bytes_per_row + k / 8];
            signs[j * n_in + k] = ((byte >> (k % 8)) & 1u) ? (int8_t)1 : (int8_t)-1;
        }
}

static double alpha_of_row(const float *alpha, int mode, int64_t j)
{
    return (double)(mode == 1 ? alpha[j] : alpha[0]);
}

static double sign_at(const uint8_t *bits, int64_t bytes_per_row, int64_t j,
                      int64_t k)
{
    const unsigned byte = bits[j * bytes_per_row + k / 8];
    return ((byte >> (k % 8)) & 1u) ? 1.0 : -1.0;
}

/* [serve] W_eff = W_base + alpha * sign, built from the stored form
 * (bf16 W_base, packed bits, fp32 alpha) in fp64. */
void bdo_weff(const uint16_t *w_base, const uint8_t *bits, const float *alpha,
              int mode, int64_t n_out, int64_t n_in, double *w_eff)
{
    const int64_t bpr = n_in / 8;
    for (int64_t j = 0; j < n_out; ++j) {
        const double a = alpha_of_row(alpha, mode, j);
        for (int64_t k = 0; k < n_in; ++k)
            w_eff[j * n_in + k] =
                bf16_to_f64(w_base[j * n_in + k]) + a * sign_at(bits, bpr, j, k);
    }
}

/* Round an fp32 value to the nearest bf16, ties to the even significand (the
 * standard IEEE rounding, done on the bit pattern: add just under half an
 * ulp of the kept part, plus its lowest kept bit, and truncate).  Finite
 * inputs only, which is all this file produces. */
static uint16_t f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* [serve] with reading R5: the bf16 W_eff a standard matmul would consume
 * ("Profil de latence" reads decode as a standard matmul).  The sum
 * W_base + alpha * sign is formed in fp32 (alpha * (+-1) is exact, the add
 * rounds once to nearest even) and then rounded once, to nearest even, to
 * bf16. */
void bdo_weff_bf16(const uint16_t *w_base, const uint8_t *bits, const float *alpha,
                   int mode, int64_t n_out, int64_t n_in, uint16_t *w_eff)
{
    const int64_t bpr = n_in / 8;
    for (int64_t j = 0; j < n_out; ++j) {
        const float a = mode == 1 ? alpha[j] : alpha[0];
        for (int64_t k = 0; k < n_in; ++k) {
            const float w = (float)bf16_to_f64(w_base[j * n_in + k]);
            const float s = (float)sign_at(bits, bpr, j, k);
            const float v = w + a * s;
            w_eff[j * n_in + k] = f32_to_bf16_rne(v);
        }
    }
}

/* One output of the fused linear: y[t, j] = sum_k x[t, k] * W_eff[j, k]
 * ([serve]: linear(x, w_eff) = x . W_eff^T), plus the magnitude sum
 * sum_k |x[t, k]| * |W_eff[j, k]| that scales the rounding tolerance. */
static void one_output(const uint16_t *x_row, const uint16_t *wb_row,
                       const uint8_t *bits_row, double a, int64_t n_in,
                       double *y, double *mag)
{
    double s = 0.0, m = 0.0;
    for (int64_t k = 0; k < n_in; ++k) {
        const double sg = ((bits_row[k / 8] >> (k % 8)) & 1u) ? 1.0 : -1.0;
        const double w = bf16_to_f64(wb_row[k]) + a * sg;
        const double xv = bf16_to_f64(x_row[k]);
        s += xv * w;
        m += fabs(xv) * fabs(w);
    }
    *y = s;
    *mag = m;
}

/* Full fused linear, every output.  y, mag: [m, n_out] fp64. */
void bdo_linear(const uint16_t *x, int64_t m, const uint16_t *w_base,
                const uint8_t *bits, const float *alpha, int mode,
                int64_t n_out, int64_t n_in, double *y, double *mag)
{
    const int64_t bpr = n_in / 8;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n_out; ++j) {
        const double a = alpha_of_row(alpha, mode, j);
        for (int64_t t = 0; t < m; ++t)
            one_output(x + t * n_in, w_base + j * n_in, bits + j * bpr, a, n_in,
                       &y[t * n_out + j], &mag[t * n_out + j]);
    }
}

/* Selected outputs only: for i < count, (t, j) = (ts[i], js[i]). */
void bdo_linear_sampled(const uint16_t *x, const uint16_t *w_base,
                        const uint8_t *bits, const float *alpha, int mode,
                        int64_t n_out, int64_t n_in, const int64_t *ts,
                        const int64_t *js, int64_t count, double *y, double *mag)
{
    const int64_t bpr = n_in / 8;
    (void)n_out;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; ++i) {
        const int64_t t = ts[i], j = js[i];
        one_output(x + t * n_in, w_base + j * n_in, bits + j * bpr,
                   alpha_of_row(alpha, mode, j), n_in, &y[i], &mag[i]);
    }
}

/* Multi-tenant form ([serve]: many variants over one shared W_base; each
 * token t uses the delta (bits, alpha) of its own variant ids[t]).
 * Returns -1 (and writes nothing) if an id is outside [0, n_var). */
int bdo_linear_grouped(const uint16_t *x, const int32_t *ids, int64_t m,
                       const uint16_t *w_base, const uint8_t *const *bits_v,
                       const float *const *alpha_v, const int32_t *modes_v,
                       int32_t n_var, int64_t n_out, int64_t n_in, double *y,
                       double *mag)
{
    const int64_t bpr = n_in / 8;
    for (int64_t t = 0; t < m; ++t)
        if (ids[t] < 0 || ids[t] >= n_var)
            return -1;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n_out; ++j) {
        for (int64_t t = 0; t < m; ++t) {
            const int32_t v = ids[t];
            one_output(x + t * n_in, w_base + j * n_in, bits_v[v] + j * bpr,
                       alpha_of_row(alpha_v[v], modes_v[v], j), n_in,
                       &y[t * n_out + j], &mag[t * n_out + j]);
        }
    }
    return 0;
}

/* Selected outputs of the multi-tenant form. */
int bdo_linear_grouped_sampled(const uint16_t *x, const int32_t *ids,
                               const uint16_t *w_base,
                               const uint8_t *const *bits_v,
                               const float *const *alpha_v,
                               const int32_t *modes_v, int32_t n_var,
                               int64_t n_out, int64_t n_in, const int64_t *ts,
                               const int64_t *js, int64_t count, double *y,
                               double *mag)
{
    const int64_t bpr = n_in / 8;
    (void)n_out;
    for (int64_t i = 0; i < count; ++i)
        if (ids[ts[i]] < 0 || ids[ts[i]] >= n_var)
            return -1;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; ++i) {
        const int64_t t = ts[i], j = js[i];
        const int32_t v = ids[t];
        one_output(x + t * n_in, w_base + j * n_in, bits_v[v] + j * bpr,
                   alpha_of_row(alpha_v[v], modes_v[v], j), n_in, &y[i], &mag[i]);
    }
    return 0;
}

/* [infra] packed storage: eight signs per byte -> n_out * n_in / 8 bytes. */
int64_t bdo_packed_bytes(int64_t n_out, int64_t n_in)
{
    return n_out * (n_in / 8);
}

/*
 * ct_oracle.c -- plain, slow, single-threaded CPU oracle for the FP8
 * cast-transpose path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library includes, links
 * or calls this file; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load it.  It shares no code, header or table with the CUDA
 * sources.
 *
 * What it computes, and where that comes from:
 *   - "[PyTorch] cuda graph support", transpose-cache discussion, the
 *     DbiasCastTranspose example: db = dy.sum(dim=0) next to a cast-transpose
 *     of dy that yields an FP8 tensor together with its transpose.
 *   - "[PyTorch] Refactor FP8 workspaces in linear modules", Motivations
 *     (first and second bullet): the FP8 tensor keeps a private copy of the
 *     scale-inverse that matches the scale its bytes were cast with; a scale
 *     update kernel recomputes the scales from the amax history; the
 *     infinite-scale case (amax too tiny) must be handled.
 *   - The FP8 formats E4M3 ("fn": no infinities, one NaN pattern per sign)
 *     and E5M2 (IEEE-like) follow the OCP 8-bit floating point specification
 *     (OFP8) and Micikevicius et al., "FP8 Formats for Deep Learning" (2022),
 *     table 1: exponent bias 7 / 15, largest normal 448 / 57344.
 *   - Delayed scaling: amax over a sliding window of the last L amaxes,
 *     scale = (fp8_max / amax) / 2^margin, kept when amax is 0 or the new
 *     scale is not finite, scale_inv = 1 / scale.
 *
 * Readings taken where the sources are silent (each listed in the design
 * notes): products are one IEEE fp32 multiply, round-to-nearest-even; the FP8
 * encode rounds to nearest, ties to even, and saturates (overflow and +-Inf go
 * to +-max); NaN encodes to the canonical positive NaN 0x7F; zero and values
 * that round to zero keep their sign; no flush-to-zero anywhere; amax is the
 * largest |x| by IEEE magnitude bit pattern (NaN above Inf, so NaN
 * propagates); db is accumulated in double and rounded once to fp32.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -shared -fPIC
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_E4M3 0
#define ORACLE_E5M2 1

/* ---- FP8 format parameters (OFP8 / Micikevicius et al. table 1) ---------- */
typedef struct {
    int mbits;        /* stored mantissa bits                        */
    int ebits;        /* exponent bits                               */
    int bias;         /* exponent bias                               */
    float maxval;     /* largest finite magnitude                    */
    int maxcode;      /* its 7-bit magnitude code                    */
} fp8_format;

static fp8_format format_of(int fmt)
{
    fp8_format f;
    if (fmt == ORACLE_E5M2) {
        f.mbits = 2; f.ebits = 5; f.bias = 15;
        f.maxval = 57344.0f;   /* 1.75 * 2^15, code S.11110.11 */
        f.maxcode = 0x7B;
    } else {
        f.mbits = 3; f.ebits = 4; f.bias = 7;
        f.maxval = 448.0f;     /* 1.75 * 2^8, code S.1111.110  */
        f.maxcode = 0x7E;
    }
    return f;
}

/* Value of an FP8 code, from the field definitions.  E4M3: S.1111.111 is
 * NaN, no infinities.  E5M2: exponent field all ones is Inf (mantissa 0) or
 * NaN.  Subnormals: mantissa * 2^(1 - bias - mbits). */
float oracle_fp8_decode(uint8_t code, int fmt)
{
    const fp8_format f = format_of(fmt);
    const int sign = code >> 7;
    const int efield = (code >> f.mbits) & ((1 << f.ebits) - 1);
    const int mant = code & ((1 << f.mbits) - 1);
    const int emax_field = (1 << f.ebits) - 1;
    float v;
    if (fmt == ORACLE_E4M3 && efield == emax_field && mant == (1 << f.mbits) - 1)
        return NAN;
    if (fmt == ORACLE_E5M2 && efield == emax_field) {
        if (mant != 0) return NAN;
        return sign ? -INFINITY : INFINITY;
    }
    if (efield == 0)
        v = ldexpf((float)mant, 1 - f.bias - f.mbits);
    else
        v = ldexpf((float)((1 << f.mbits) + mant), efield - f.bias - f.mbits);
    return sign ? -v : v;
}

/* Round an fp32 value to the FP8 grid: nearest, ties to even, saturating. */
uint8_t oracle_fp8_encode(float p, int fmt)
{
    const fp8_format f = format_of(fmt);
    const int emin = 1 - f.bias;          /* exponent of the smallest normal */
    uint8_t sign;
    float a, spacing, n;
    int e, E, mag;

    if (isnan(p)) return 0x7F;
    sign = signbit(p) ? 0x80 : 0x00;
    a = fabsf(p);
    if (a >= f.maxval) return (uint8_t)(sign | f.maxcode);   /* incl. +-Inf */
    if (a == 0.0f) return sign;

    /* a = m * 2^e with m in [0.5, 1): the binade of a is 2^(e-1). Below the
     * normal range the grid spacing stays that of the smallest binade. */
    (void)frexpf(a, &e);
    E = e - 1;
    if (E < emin) E = emin;
    spacing = ldexpf(1.0f, E - f.mbits);
    n = rintf(a / spacing);   /* division by a power of two is exact; rintf
                                 rounds half to even in the default mode   */
    if (n == 0.0f) return sign;
    /* Codes are monotone in magnitude: binade E contributes
     * (E + bias) << mbits, plus the offset of n inside the binade.  For
     * E == emin this reduces to mag = n, which also covers subnormals, and
     * n == 2^(mbits+1) carries into the next binade. */
    mag = ((E + f.bias) << f.mbits) + (int)n - (1 << f.mbits);
    if (mag > f.maxcode) mag = f.maxcode;
    return (uint8_t)(sign | mag);
}

void oracle_fp8_encode_array(const float* p, int64_t count, int fmt, uint8_t* out)
{
    for (int64_t i = 0; i < count; ++i) out[i] = oracle_fp8_encode(p[i], fmt);
}

void oracle_fp8_decode_array(const uint8_t* c, int64_t count, int fmt, float* out)
{
    for (int64_t i = 0; i < count; ++i) out[i] = oracle_fp8_decode(c[i], fmt);
}

/* bf16 is the top half of an fp32: widening is exact. */
static float bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint32_t f32_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

static float f32_from_bits(uint32_t u)
{
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Largest |x| under the IEEE magnitude order of bit patterns (NaN > Inf >
 * finite), max-merged into *amax_io, whose value must be >= 0 or NaN. */
static void merge_amax(const uint16_t* x, int64_t count, float* amax_io)
{
    uint32_t best = f32_bits(*amax_io) & 0x7FFFFFFFu;
    for (int64_t i = 0; i < count; ++i) {
        uint32_t mag = ((uint32_t)x[i] << 16) & 0x7FFFFFFFu;
        if (mag > best) best = mag;
    }
    *amax_io = f32_from_bits(best);
}

/* amax alone: max-merge of max |x| into *amax_io (as in the cast below). */
void oracle_amax(const uint16_t* x, int64_t count, float* amax_io)
{
    merge_amax(x, count, amax_io);
}

/* Cast + transpose + amax + scale-inverse of one row-major bf16 matrix.
 *   q[i*cols + j]  = encode(bf16(x[i,j]) * scale)
 *   qt[j*rows + i] = q[i*cols + j]
 *   *amax_io       = max(*amax_io, max |x|)
 *   *scale_inv_out = 1 / scale
 * ("[PyTorch] cuda graph support": cast_transpose(dy) returns an FP8 tensor
 * with its transpose cached; "[PyTorch] Refactor FP8 workspaces in linear
 * modules", Motivations: the tensor's own scale-inverse.)  q or qt may be
 * NULL to skip that output (plain cast / transpose-only checks). */
void oracle_cast_transpose(const uint16_t* x, int64_t rows, int64_t cols,
                           float scale, int fmt, uint8_t* q, uint8_t* qt,
                           float* amax_io, float* scale_inv_out)
{
    for (int64_t i = 0; i < rows; ++i) {
        for (int64_t j = 0; j < cols; ++j) {
            float product = bf16_value(x[i * cols + j]) * scale;
            uint8_t code = oracle_fp8_encode(product, fmt);
            if (q) q[i * cols + j] = code;
            if (qt) qt[j * rows + i] = code;
        }
    }
    if (amax_io) merge_amax(x, rows * cols, amax_io);
    if (scale_inv_out) *scale_inv_out = 1.0f / scale;
}

/* Column sum of the unscaled bf16 values: db[j] = sum_i x[i,j], accumulated
 * in double, rounded once to fp32 ("[PyTorch] cuda graph support",
 * DbiasCastTranspose: db = dy.sum(dim=0)). */
void oracle_dbias(const uint16_t* x, int64_t rows, int64_t cols, float* db)
{
    for (int64_t j = 0; j < cols; ++j) {
        double s = 0.0;
        for (int64_t i = 0; i < rows; ++i) s += (double)bf16_value(x[i * cols + j]);
        db[j] = (float)s;
    }
}

/* fp32 -> bf16 by the IEEE rule, written out: the two bf16 values that
 * bracket |f| are its truncation to 8 significand bits and the next one up
 * (past the largest finite bf16, that next one stands for 2^128, i.e. the
 * overflow to Inf); the nearer one wins, a tie goes to the even significand.
 * The distances are exact in double.  NaN gives the canonical quiet NaN
 * 0x7FFF (reading: the pages never round a NaN db; the choice follows the
 * hardware conversion's canonical NaN).  Used for a bf16 db: the fp32 column
 * sum rounded once more, to bf16. */
uint16_t oracle_f32_to_bf16(float f)
{
    const uint32_t u = f32_bits(f);
    const uint32_t sign = u & 0x80000000u, mag = u & 0x7FFFFFFFu;
    if (mag > 0x7F800000u) return 0x7FFF;                       /* NaN */
    if (mag == 0x7F800000u) return (uint16_t)((sign | mag) >> 16); /* +-Inf */
    const uint32_t lo = mag & 0xFFFF0000u;                       /* truncation */
    const uint32_t hi = lo + 0x10000u;                           /* next bf16 up */
    const double a = (double)f32_from_bits(mag);
    const double vlo = (double)f32_from_bits(lo);
    const double vhi = hi == 0x7F800000u ? ldexp(1.0, 128) : (double)f32_from_bits(hi);
    const double dlo = a - vlo, dhi = vhi - a;
    uint32_t pick;
    if (dlo < dhi) pick = lo;
    else if (dhi < dlo) pick = hi;
    else pick = ((lo >> 16) & 1u) ? hi : lo;                     /* tie: even */
    return (uint16_t)((sign | pick) >> 16);
}

void oracle_f32_to_bf16_array(const float* f, int64_t count, uint16_t* out)
{
    for (int64_t i = 0; i < count; ++i) out[i] = oracle_f32_to_bf16(f[i]);
}

/* Byte transpose of an FP8 matrix: out[j*rows + i] = in[i*cols + j]
 * (the transpose-cache fill, "[PyTorch] Refactor FP8 workspaces in linear
 * modules", the lazy transpose caching bullet). */
void oracle_fp8_transpose(const uint8_t* in, int64_t rows, int64_t cols, uint8_t* out)
{
    for (int64_t i = 0; i < rows; ++i)
        for (int64_t j = 0; j < cols; ++j)
            out[j * rows + i] = in[i * cols + j];
}

/* Delayed-scaling update for n tensors ("[PyTorch] Refactor FP8 workspaces
 * in linear modules", Motivations: the scale update kernel and the
 * infinite-scale case; "[PyTorch] cuda graph support", feature list: amaxes
 * reduced within the current iteration).
 *
 * hist is [L, n] row-major; row 0 holds the amax of the step that just ran.
 * For each tensor i:
 *   a      = max over the L rows (NaN propagates)
 *   s_new  = (fp8_max / a) / 2^margin                 (fp32, two roundings)
 *   scale  = s_new, unless a is not > 0, a is not finite or s_new is not
 *            finite, in which case the old scale is kept
 *   scale_inv = 1 / scale
 *   then the window slides: row r takes row r-1 (r = L-1 .. 1), row 0 := 0.
 * With most_recent != 0, a is row 0 alone (the "most recent" amax rule).
 */
void oracle_amax_and_scale_update_algo(float* hist, float* scale, float* scale_inv,
                                       int L, int n, int fmt, int margin, int most_recent)
{
    const float fp8_max = format_of(fmt).maxval;
    const float two_pow_margin = ldexpf(1.0f, margin);
    for (int i = 0; i < n; ++i) {
        float a = hist[i];
        for (int r = 1; r < L && !most_recent; ++r) {
            float v = hist[(int64_t)r * n + i];
            if (isnan(a)) break;
            if (isnan(v) || v > a) a = v;
        }
        float s = scale[i];
        if (a > 0.0f && isfinite(a)) {
            float candidate = (fp8_max / a) / two_pow_margin;
            if (isfinite(candidate)) s = candidate;
        }
        scale[i] = s;
        scale_inv[i] = 1.0f / s;
        for (int r = L - 1; r >= 1; --r)
            hist[(int64_t)r * n + i] = hist[(int64_t)(r - 1) * n + i];
        hist[i] = 0.0f;
    }
}

/* The update with the window maximum (most_recent = 0). */
void oracle_amax_and_scale_update(float* hist, float* scale, float* scale_inv,
                                  int L, int n, int fmt, int margin)
{
    oracle_amax_and_scale_update_algo(hist, scale, scale_inv, L, n, fmt, margin, 0);
}

/*
 * Oracle number codecs — TEST INFRASTRUCTURE ONLY.
 *
 * Plain scalar definitions of the four encodings the MoE layer uses, in
 * double precision.  Only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark may load this file's library; the product path never
 * does.  It shares no code with the CUDA library.
 *
 * Sources (web pages on MiMo-V2.6):
 *  - "MiMo V2.6 Pro and Flash architecture teardown" (kgptalkie), section
 *    "Why Are the V2.6 Files Half the Size of V2.5?", table row "Routed
 *    experts": MXFP4 = two 4-bit values per U8 byte, one 8-bit scale per 32
 *    values; 4.25 bits per expert weight.
 *  - vLLM recipe "XiaomiMiMo/MiMo-V2.6-Pro-RL", section "Overview": weights
 *    are computed as block-wise FP8 e4m3.
 * The pages do not spell out the bit layouts; they name the public OCP
 * Microscaling (MX) v1.0 element types (E2M1 values, E8M0 shared scale) and
 * the OFP8 E4M3 ("e4m3fn": no infinities, one NaN pattern per sign) type,
 * whose definitions are written out below.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

/* E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit.
 * exponent field 0 is subnormal: magnitude = m * 0.5;
 * otherwise magnitude = (1 + m/2) * 2^(e-1).  Negative zero exists. */
double orc_e2m1_decode(uint32_t code)
{
    uint32_t s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
    double mag = (e == 0) ? 0.5 * (double)m : (1.0 + 0.5 * (double)m) * ldexp(1.0, (int)e - 1);
    return s ? -mag : mag;
}

/* E8M0: an unsigned biased exponent, value 2^(b-127); 0xFF is NaN. */
double orc_e8m0_decode(uint32_t b)
{
    if ((b & 0xFFu) == 0xFFu) return NAN;
    return ldexp(1.0, (int)(b & 0xFFu) - 127);
}

/* E4M3 (e4m3fn): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits.
 * exponent field 0: subnormal m * 2^-9.  S.1111.111 is NaN; no infinity.
 * Largest finite magnitude 1.75 * 2^8 = 448. */
double orc_e4m3_decode(uint32_t b)
{
    uint32_t s = (b >> 7) & 1u, e = (b >> 3) & 15u, m = b & 7u;
    double mag;
    if (e == 15u && m == 7u) return NAN;
    if (e == 0) mag = (double)m * ldexp(1.0, -9);
    else mag = (1.0 + (double)m / 8.0) * ldexp(1.0, (int)e - 7);
    return s ? -mag : mag;
}

/* Round-to-nearest-even of a non-negative double to an integer.  rint()
 * uses the current rounding mode, which is round-to-nearest-even by default;
 * that default is never changed in this library. */
static double rne(double a) { return rint(a); }

/* E4M3 encoding with round-to-nearest-even and saturation to +-448
 * ("satfinite": anything beyond the largest finite value becomes it). */
uint32_t orc_e4m3_encode(double v)
{
    uint32_t s = signbit(v) ? 0x80u : 0u;
    double a = fabs(v);
    if (isnan(v)) return 0x7Fu;
    if (a >= 448.0) return s | 0x7Eu;
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: quantum 2^-9; n == 8 is the smallest normal (code 8) */
        double n = rne(a * 512.0);
        return s | (uint32_t)n;
    }
    int p;
    (void)frexp(a, &p);          /* a = f * 2^p, f in [0.5, 1) */
    int E = p - 1;               /* a in [2^E, 2^(E+1)), E >= -6 */
    double n = rne(ldexp(a, 3 - E));   /* a / 2^(E-3), in [8, 16] */
    if (n >= 16.0) { E += 1; n = 8.0; }
    uint32_t code = ((uint32_t)(E + 7) << 3) | ((uint32_t)n - 8u);
    if (code > 0x7Eu) code = 0x7Eu;
    return s | code;
}

/* bfloat16 (1 sign, 8 exponent bits, 7 mantissa bits) from double with one
 * rounding step, to nearest, ties to even; overflow goes to infinity. */
uint32_t orc_bf16_encode(double v)
{
    uint32_t s = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (isnan(v)) return 0x7FC0u;
    if (isinf(v)) return s | 0x7F80u;
    if (a == 0.0) return s;
    int p;
    (void)frexp(a, &p);
    int E = p - 1;
    if (E < -126) {
        double n = rne(ldexp(a, 133));              /* quantum 2^-133 */
        return s | (uint32_t)n;                     /* n == 128 is the smallest normal */
    }
    double n = rne(ldexp(a, 7 - E));               /* in [128, 256] */
    if (n >= 256.0) { E += 1; n = 128.0; }
    if (E > 127) return s | 0x7F80u;
    return s | ((uint32_t)(E + 127) << 7) | ((uint32_t)n - 128u);
}

double orc_bf16_decode(uint32_t b)
{
    union { uint32_t u; float f; } c;
    c.u = (b & 0xFFFFu) << 16;
    return (double)c.f;
}

/* Shared power-of-two exponent of one activation block for e4m3: the
 * smallest integer e with amax <= 448 * 2^e, clamped to [-127, 127]; an
 * all-zero block takes e = 0.  With amax = f * 2^p (f in [0.5, 1)) and
 * 448 = 0.875 * 2^9 this is p - 9 when f <= 0.875 and p - 8 otherwise. */
int orc_act_block_exponent(double amax)
{
    if (!(amax > 0.0)) return 0;
    int p;
    double f = frexp(amax, &p);
    int e = (f <= 0.875) ? p - 9 : p - 8;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

/* Per-token 1 x blk activation quantisation of one row of n values
 * (n a multiple of blk): for each block, the power-of-two scale above, stored
 * as an E8M0 byte (e + 127), and e4m3(v / 2^e) with round-to-nearest-even and
 * saturation.  Division by a power of two is exact, so the codes do not
 * depend on the precision the values arrive in. */
void orc_act_quant_row(const double* v, int n, int blk, uint8_t* q, uint8_t* scale)
{
    for (int b = 0; b < n / blk; ++b) {
        double amax = 0.0;
        for (int i = 0; i < blk; ++i) {
            double a = fabs(v[b * blk + i]);
            if (a > amax) amax = a;
        }
        int e = orc_act_block_exponent(amax);
        scale[b] = (uint8_t)(e + 127);
        for (int i = 0; i < blk; ++i)
            q[b * blk + i] = (uint8_t)orc_e4m3_encode(ldexp(v[b * blk + i], -e));
    }
}

/* The fp32-scale variant of the same 1 x blk quantisation (the "dynamic
 * activation scheme" read as a per-block fp32 scale): each value is taken
 * at fp32 (the precision the activations are computed in), the block scale
 * is s = amax / 448 divided in fp32, and the code is e4m3 (round to nearest
 * even, saturating) of the fp32 quotient v / s.  An all-zero block stores
 * s = 0 and zero codes.  Dequantised value: e4m3(q) * s. */
void orc_act_quant_row_f32s(const double* v, int n, int blk, uint8_t* q, float* scale)
{
    for (int b = 0; b < n / blk; ++b) {
        float amax = 0.0f;
        for (int i = 0; i < blk; ++i) {
            const float a = fabsf((float)v[b * blk + i]);
            if (a > amax) amax = a;
        }
        const float sc = amax / 448.0f;
        scale[b] = sc;
        for (int i = 0; i < blk; ++i) {
            const float x = (float)v[b * blk + i];
            q[b * blk + i] = amax > 0.0f ? (uint8_t)orc_e4m3_encode((double)(x / sc)) : (uint8_t)0;
        }
    }
}

void orc_act_quant_rows_f32s(const double* v, size_t rows, int n, int blk, uint8_t* q, float* scale)
{
    for (size_t r = 0; r < rows; ++r)
        orc_act_quant_row_f32s(v + r * (size_t)n, n, blk, q + r * (size_t)n, scale + r * (size_t)(n / blk));
}

/* E2M1 code of one value already divided by its block scale, round to
 * nearest with ties to the even code, saturating at +-6. */
uint32_t orc_e2m1_encode(double v)
{
    static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    uint32_t s = signbit(v) ? 8u : 0u;
    double a = fabs(v);
    if (a >= 6.0) return s | 7u;
    uint32_t best = 0;
    for (uint32_t c = 1; c < 8; ++c) {
        double dc = fabs(a - mag[c]), db = fabs(a - mag[best]);
        if (dc < db || (dc == db && (c & 1u) == 0u)) best = c;
    }
    return s | best;
}

/* OCP MX v1.0 quantisation of one row of K values to MXFP4: per 32-block the
 * shared exponent X = floor(log2(amax)) - 2 (2 = the largest E2M1 exponent),
 * clamped to [-127, 127], stored as the E8M0 byte X + 127 (an all-zero block
 * stores 127); each value becomes the E2M1 code of v / 2^X.  Codes are packed
 * two per byte, element 2i in the low nibble and 2i+1 in the high nibble. */
void orc_mxfp4_quant_row(const double* w, int K, uint8_t* packed, uint8_t* scale)
{
    for (int b = 0; b < K / 32; ++b) {
        double amax = 0.0;
        for (int i = 0; i < 32; ++i) {
            double a = fabs(w[b * 32 + i]);
            if (a > amax) amax = a;
        }
        int X = 0;
        if (amax > 0.0) {
            int p;
            (void)frexp(amax, &p);       /* floor(log2(amax)) = p - 1 */
            X = p - 1 - 2;
            if (X < -127) X = -127;
            if (X > 127) X = 127;
        }
        scale[b] = (uint8_t)(X + 127);
        for (int i = 0; i < 32; i += 2) {
            uint32_t lo = amax > 0.0 ? orc_e2m1_encode(ldexp(w[b * 32 + i], -X)) : 0u;
            uint32_t hi = amax > 0.0 ? orc_e2m1_encode(ldexp(w[b * 32 + i + 1], -X)) : 0u;
            packed[(b * 32 + i) / 2] = (uint8_t)(lo | (hi << 4));
        }
    }
}

/* ---- array forms used from Python ---- */

void orc_e4m3_decode_array(const uint8_t* b, size_t n, double* out)
{
    for (size_t i = 0; i < n; ++i) out[i] = orc_e4m3_decode(b[i]);
}

void orc_e4m3_encode_array(const double* v, size_t n, uint8_t* out)
{
    for (size_t i = 0; i < n; ++i) out[i] = (uint8_t)orc_e4m3_encode(v[i]);
}

void orc_bf16_encode_array(const double* v, size_t n, uint16_t* out)
{
    for (size_t i = 0; i < n; ++i) out[i] = (uint16_t)orc_bf16_encode(v[i]);
}

void orc_act_quant_rows(const double* v, size_t rows, int n, int blk, uint8_t* q, uint8_t* scale)
{
    for (size_t r = 0; r < rows; ++r)
        orc_act_quant_row(v + r * (size_t)n, n, blk, q + r * (size_t)n, scale + r * (size_t)(n / blk));
}

void orc_mxfp4_quant_rows(const double* w, size_t rows, int K, uint8_t* packed, uint8_t* scale)
{
    for (size_t r = 0; r < rows; ++r)
        orc_mxfp4_quant_row(w + r * (size_t)K, K, packed + r * (size_t)(K / 2), scale + r * (size_t)(K / 32));
}

/* MXFP4 rows -> exact doubles: element k of row r is
 * E2M1(nibble k) * E8M0(scale[k / 32]); nibble k is the low nibble of byte
 * k/2 for even k and the high nibble for odd k. */
void orc_mxfp4_decode_rows(const uint8_t* packed, const uint8_t* scale, size_t rows, int K, double* out)
{
    double e2m1[16];
    for (uint32_t c = 0; c < 16; ++c) e2m1[c] = orc_e2m1_decode(c);
#pragma omp parallel for schedule(static)
    for (long long r = 0; r < (long long)rows; ++r) {
        const uint8_t* pr = packed + (size_t)r * (size_t)(K / 2);
        const uint8_t* sr = scale + (size_t)r * (size_t)(K / 32);
        double* o = out + (size_t)r * (size_t)K;
        for (int b = 0; b < K / 32; ++b) {
            double sc = orc_e8m0_decode(sr[b]);
            for (int k = b * 32; k < b * 32 + 32; ++k) {
                uint32_t byte = pr[k / 2];
                uint32_t code = (k & 1) ? (byte >> 4) : (byte & 15u);
                o[k] = e2m1[code] * sc;
            }
        }
    }
}

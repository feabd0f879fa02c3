/*
 * Seeded synthetic inputs for the MoE layer (shared by the tests, the smoke
 * check and the benchmark; holds none of the layer's own arithmetic).
 *
 * Random numbers: SplitMix64 (Steele, Lea & Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014) used as a counter-based
 * generator: draw i of stream s under seed z is mix64(key(z, s) + (i+1)*G),
 * G = 0x9E3779B97F4A7C15, so any element can be generated independently and
 * the result does not depend on the number of threads.
 *
 * Normal deviates: inverse-CDF lookup with linear interpolation in a table of
 * standard-normal quantiles supplied by the caller.
 *
 * Expert weights are drawn in fp32 and stored as MXFP4 with the OCP MX v1.0
 * rule (shared exponent floor(log2(amax)) - 2 per 32 values, E2M1 codes by
 * round-to-nearest with ties to the even code, saturating at 6), packed two
 * codes per byte with the first element in the low nibble - or, for the fp8
 * expert format, as e4m3 codes with one fp32 scale (amax / 448) per 128 x
 * 128 block.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ull

static inline uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream)
{
    return mix64(mix64(seed * GOLDEN + 0x632BE59BD9B4E019ull) ^ (stream * 0xD1B54A32D192ED03ull + 1));
}

static inline uint64_t draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GOLDEN); }

/* inverse-CDF normal from a 64-bit draw; table has n_tab+1 quantiles at
 * p = j / n_tab (end points clamped by the caller) */
static inline float normal_from(uint64_t r, const float* tab, int n_tab)
{
    double u = (double)(r >> 11) * (1.0 / 9007199254740992.0); /* [0, 1) */
    double pos = u * n_tab;
    int j = (int)pos;
    double f = pos - j;
    return (float)(tab[j] + f * (tab[j + 1] - tab[j]));
}

static inline uint16_t f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

void syn_normal_bf16(uint64_t seed, uint64_t stream, float sigma, size_t n, uint16_t* out,
                     const float* tab, int n_tab)
{
    uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (long long i = 0; i < (long long)n; ++i)
        out[i] = f32_to_bf16_rne(sigma * normal_from(draw(key, (uint64_t)i), tab, n_tab));
}

void syn_normal_f32(uint64_t seed, uint64_t stream, float sigma, size_t n, float* out,
                    const float* tab, int n_tab)
{
    uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (long long i = 0; i < (long long)n; ++i)
        out[i] = sigma * normal_from(draw(key, (uint64_t)i), tab, n_tab);
}

static inline uint32_t e2m1_code(float a_signed)
{
    /* magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6: the code is the number of
     * midpoints (.25, .75, 1.25, 1.75, 2.5, 3.5, 5) below the value, where a
     * value on a midpoint goes to the even code (> for midpoints above an
     * even code, >= for those above an odd one); saturates at code 7 */
    uint32_t s = signbit(a_signed) ? 8u : 0u;
    float a = fabsf(a_signed);
    uint32_t c = (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) +
                 (uint32_t)(a >= 1.75f) + (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) +
                 (uint32_t)(a > 5.0f);
    return s | c;
}

/* one row of K fp32 values -> MXFP4 (packed K/2 bytes + K/32 scale bytes) */
static void mxfp4_row(const float* w, int K, uint8_t* packed, uint8_t* scale)
{
    for (int b = 0; b < K / 32; ++b) {
        float amax = 0.f;
        for (int i = 0; i < 32; ++i) {
            float a = fabsf(w[b * 32 + i]);
            if (a > amax) amax = a;
        }
        int X = 0;
        if (amax > 0.f) {
            int p;
            (void)frexpf(amax, &p);
            X = p - 3;
            if (X < -127) X = -127;
            if (X > 127) X = 127;
        }
        scale[b] = (uint8_t)(X + 127);
        /* 2^-X as an fp32 power of two (X in [-127, 127] keeps it normal
         * except at the clamp, where ldexpf handles it): multiplying by it is
         * exact for these magnitudes */
        float inv = ldexpf(1.0f, -X);
        for (int i = 0; i < 32; i += 2) {
            uint32_t lo = 0, hi = 0;
            if (amax > 0.f) {
                lo = e2m1_code(w[b * 32 + i] * inv);
                hi = e2m1_code(w[b * 32 + i + 1] * inv);
            }
            packed[(b * 32 + i) / 2] = (uint8_t)(lo | (hi << 4));
        }
    }
}

/* Expert weight tensor [E][rows][K] drawn N(0, sigma^2) in fp32, stored as
 * MXFP4: packed [E][rows][K/2], scale [E][rows][K/32].  Expert e, row r,
 * column c is draw r*K + c of stream (stream_base + e). */
void syn_mxfp4_experts(uint64_t seed, uint64_t stream_base, int E, int rows, int K, float sigma,
                       uint8_t* packed, uint8_t* scale, const float* tab, int n_tab)
{
#pragma omp parallel
    {
        float buf[8192];
#pragma omp for schedule(static)
        for (long long er = 0; er < (long long)E * rows; ++er) {
            int e = (int)(er / rows), r = (int)(er % rows);
            uint64_t key = stream_key(seed, stream_base + (uint64_t)e);
            for (int c0 = 0; c0 < K; c0 += 8192) {
                int n = K - c0 < 8192 ? K - c0 : 8192;
                for (int c = 0; c < n; ++c)
                    buf[c] = sigma * normal_from(draw(key, (uint64_t)r * K + c0 + c), tab, n_tab);
                mxfp4_row(buf, n, packed + (size_t)er * (K / 2) + c0 / 2, scale + (size_t)er * (K / 32) + c0 / 32);
            }
        }
    }
}

/* e4m3 (e4m3fn: bias 7, no infinities, 448 the largest finite value) code of
 * a finite fp32 value, round to nearest with ties to even, saturating at 448.
 * Used only to store synthetic fp8 expert weights. */
static uint8_t e4m3_code(float v)
{
    uint8_t sign = signbit(v) ? 0x80u : 0u;
    float a = fabsf(v);
    if (a >= 464.0f) return sign | 0x7Eu;   /* 464 rounds up past 448: saturate */
    if (a < 0.015625f) {                    /* below 2^-6: steps of 2^-9 */
        int m = (int)nearbyintf(a * 512.0f);
        return sign | (uint8_t)m;           /* m == 8 is the smallest normal, code 8 */
    }
    int p;
    (void)frexpf(a, &p);                    /* a = f * 2^p, f in [0.5, 1): exponent p - 1 */
    int e = p - 1;
    int m = (int)nearbyintf(ldexpf(a, 3 - e));   /* 8..16 */
    if (m == 16) { e += 1; m = 8; }
    if (e > 8 || (e == 8 && m > 14)) return sign | 0x7Eu;
    return sign | (uint8_t)(((e + 7) << 3) | (m - 8));
}

/* Expert weight tensor [E][rows][K] drawn as syn_mxfp4_experts draws it and
 * stored in the fp8 block format: per 128 x 128 block an fp32 scale
 * amax / 448 and e4m3 codes of w / scale; q [E][rows][K], scale
 * [E][rows/128][K/128] (rows and K multiples of 128). */
void syn_fp8_experts(uint64_t seed, uint64_t stream_base, int E, int rows, int K, float sigma, uint8_t* q,
                     float* scale, const float* tab, int n_tab)
{
    const int RB = rows / 128, KB = K / 128;
#pragma omp parallel for schedule(static)
    for (long long eb = 0; eb < (long long)E * RB; ++eb) {
        int e = (int)(eb / RB), rb = (int)(eb % RB);
        uint64_t key = stream_key(seed, stream_base + (uint64_t)e);
        static __thread float blk[128 * 128];
        for (int kb = 0; kb < KB; ++kb) {
            float amax = 0.0f;
            for (int r = 0; r < 128; ++r)
                for (int c = 0; c < 128; ++c) {
                    float w = sigma * normal_from(draw(key, (uint64_t)(rb * 128 + r) * K + kb * 128 + c), tab, n_tab);
                    blk[r * 128 + c] = w;
                    if (fabsf(w) > amax) amax = fabsf(w);
                }
            float sc = amax / 448.0f;
            scale[((size_t)e * RB + rb) * KB + kb] = sc;
            for (int r = 0; r < 128; ++r)
                for (int c = 0; c < 128; ++c)
                    q[((size_t)e * rows + rb * 128 + r) * K + kb * 128 + c] =
                        amax > 0.0f ? e4m3_code(blk[r * 128 + c] / sc) : 0;
        }
    }
}

/* fp32 view of the same draws (for checking the packing on small cases) */
void syn_expert_f32(uint64_t seed, uint64_t stream_base, int E, int rows, int K, float sigma,
                    float* out, const float* tab, int n_tab)
{
#pragma omp parallel for schedule(static)
    for (long long er = 0; er < (long long)E * rows; ++er) {
        int e = (int)(er / rows), r = (int)(er % rows);
        uint64_t key = stream_key(seed, stream_base + (uint64_t)e);
        for (int c = 0; c < K; ++c)
            out[(size_t)er * K + c] = sigma * normal_from(draw(key, (uint64_t)r * K + c), tab, n_tab);
    }
}

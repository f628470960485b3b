/* Bulk synthetic-input generation for MLA prefill attention (host, OpenMP).
 *
 * Counter-based draws: draw j (j = 0, 1, ...) of the stream keyed
 * (seed, tensor, row) is output j+1 of a SplitMix64 generator (Steele, Lea,
 * Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014) whose
 * state starts at key(seed, tensor, row); uniforms take the top 53 bits.
 * Normals come from Box-Muller on draw pairs (2i, 2i+1).
 *
 * Storage encoders: IEEE bfloat16 round-to-nearest-even (single rounding from
 * double) and OCP e4m3fn (bias 7, max 448, no infinities) round-to-nearest-even
 * with saturation. Nothing here computes attention; the Python module
 * mla_prefill_attention_gb300.inputs wraps these loops.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ull

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

uint64_t gen_stream_key(uint64_t seed, uint64_t tensor, uint64_t row) {
    uint64_t k0 = mix64(seed + GAMMA);
    uint64_t k1 = mix64((k0 ^ tensor) + GAMMA);
    return mix64((k1 ^ row) + GAMMA);
}

static inline double u01(uint64_t key, uint64_t j) {
    return (double)(mix64(key + (j + 1) * GAMMA) >> 11) * 0x1.0p-53;
}

uint16_t gen_bf16_rne(double x) {
    if (isnan(x)) return 0x7FC0;
    double a = fabs(x);
    uint16_t s = signbit(x) ? 0x8000 : 0;
    if (a < 0x1.0p-126) {                       /* bf16 subnormal range */
        double m = nearbyint(a * 0x1.0p133);    /* multiple of 2^-133, RNE */
        return (uint16_t)(s | (uint16_t)m);     /* m <= 128: 128 is 2^-126 (exp field 1) */
    }
    uint64_t b;
    memcpy(&b, &a, 8);
    uint64_t lsb = (b >> 45) & 1;
    b = (b + ((1ull << 44) - 1) + lsb) & ~((1ull << 45) - 1);
    double r;
    memcpy(&r, &b, 8);
    if (r >= 0x1.0p128) return (uint16_t)(s | 0x7F80);
    float f = (float)r;                          /* exact: 8 significant bits */
    uint32_t fb;
    memcpy(&fb, &f, 4);
    return (uint16_t)(s | (fb >> 16));
}

uint8_t gen_e4m3_rne(double y) {
    uint8_t s = signbit(y) ? 0x80 : 0;
    double a = fabs(y);
    if (!(a < 448.0)) a = 448.0;                 /* saturate (also maps NaN to max) */
    if (a < 0x1.0p-6) {                          /* subnormal step 2^-9 */
        double m = nearbyint(a * 0x1.0p9);       /* 0..8; 8 is the smallest normal */
        return (uint8_t)(s | (uint8_t)m);
    }
    int e;
    frexp(a, &e);                                /* a = f*2^e, f in [0.5,1) */
    double step = ldexp(1.0, e - 4);             /* 2^(floor(log2 a) - 3) */
    double q = nearbyint(a / step) * step;
    if (q > 448.0) q = 448.0;
    double fr = frexp(q, &e);
    int ef = e - 1 + 7;
    int m = (int)nearbyint((fr * 2.0 - 1.0) * 8.0);
    return (uint8_t)(s | (uint8_t)((ef << 3) | m));
}

void gen_uniform(uint64_t seed, uint64_t tensor, const uint64_t *rows, int64_t n_rows,
                 int64_t n, double *out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n_rows; ++r) {
        uint64_t key = gen_stream_key(seed, tensor, rows[r]);
        for (int64_t j = 0; j < n; ++j) out[r * n + j] = u01(key, (uint64_t)j);
    }
}

static void normal_row(uint64_t key, int64_t n, double *z) {
    for (int64_t j = 0; j < n; j += 2) {
        double u1 = 1.0 - u01(key, (uint64_t)j);
        double u2 = u01(key, (uint64_t)j + 1);
        double r = sqrt(-2.0 * log(u1));
        double t = 2.0 * M_PI * u2;
        z[j] = r * cos(t);
        if (j + 1 < n) z[j + 1] = r * sin(t);
    }
}

void gen_normal_f64(uint64_t seed, uint64_t tensor, const uint64_t *rows, int64_t n_rows,
                    int64_t n, double *out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n_rows; ++r)
        normal_row(gen_stream_key(seed, tensor, rows[r]), n, out + r * n);
}

void gen_normal_bf16(uint64_t seed, uint64_t tensor, const uint64_t *rows, int64_t n_rows,
                     int64_t n, uint16_t *out) {
#pragma omp parallel
    {
        double z[1024];
#pragma omp for schedule(static)
        for (int64_t r = 0; r < n_rows; ++r) {
            for (int64_t c0 = 0; c0 < n; c0 += 1024) {
                /* draws are per column index, so a row is produced in 1024-wide pieces */
                int64_t c1 = c0 + 1024 < n ? c0 + 1024 : n;
                uint64_t key = gen_stream_key(seed, tensor, rows[r]);
                for (int64_t j = c0; j < c1; j += 2) {
                    double u1 = 1.0 - u01(key, (uint64_t)j);
                    double u2 = u01(key, (uint64_t)j + 1);
                    double rr = sqrt(-2.0 * log(u1));
                    double t = 2.0 * M_PI * u2;
                    z[j - c0] = rr * cos(t);
                    if (j + 1 < c1) z[j + 1 - c0] = rr * sin(t);
                }
                for (int64_t j = c0; j < c1; ++j) out[r * n + j] = gen_bf16_rne(z[j - c0]);
            }
        }
    }
}

/* N(0,1) rows of width n (n <= 1024) quantised per row: scale = absmax/448
 * (1 for an all-zero row), codes = e4m3(x / scale). */
void gen_latent_e4m3(uint64_t seed, uint64_t tensor, const uint64_t *rows, int64_t n_rows,
                     int64_t n, uint8_t *codes, float *scales) {
#pragma omp parallel
    {
        double z[1024];
#pragma omp for schedule(static)
        for (int64_t r = 0; r < n_rows; ++r) {
            normal_row(gen_stream_key(seed, tensor, rows[r]), n, z);
            double amax = 0.0;
            for (int64_t j = 0; j < n; ++j) amax = fmax(amax, fabs(z[j]));
            float sc = amax > 0.0 ? (float)(amax / 448.0) : 1.0f;
            scales[r] = sc;
            for (int64_t j = 0; j < n; ++j) codes[r * n + j] = gen_e4m3_rne(z[j] / (double)sc);
        }
    }
}

/* Integers uniform on {lo..hi}, stored as e4m3 codes. */
void gen_int_e4m3(uint64_t seed, uint64_t tensor, const uint64_t *rows, int64_t n_rows,
                  int64_t n, int32_t lo, int32_t hi, uint8_t *out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n_rows; ++r) {
        uint64_t key = gen_stream_key(seed, tensor, rows[r]);
        for (int64_t j = 0; j < n; ++j) {
            double v = lo + floor(u01(key, (uint64_t)j) * (double)(hi - lo + 1));
            out[r * n + j] = gen_e4m3_rne(v);
        }
    }
}

void gen_encode_bf16(const double *x, int64_t n, uint16_t *out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = gen_bf16_rne(x[i]);
}

void gen_encode_e4m3(const double *x, int64_t n, uint8_t *out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = gen_e4m3_rne(x[i]);
}

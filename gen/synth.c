/*
 * Seeded synthetic inputs shared by the CPU oracle and the CUDA path.
 *
 * This module only DRAWS inputs: weights, caches, recurrent states, token ids
 * and page permutations. It implements none of the verify-step arithmetic.
 * The one transformation it applies is the Q4 weight quantiser, because the
 * model's weights are stored in that format: quantising a random-init matrix
 * is how the input file is made, the step itself only ever dequantises.
 *
 * Every value is a pure function of (seed, tensor id, element index), so the
 * output does not depend on the thread count, and it is bit-identical on x86
 * and Arm (integer hashing plus IEEE-754 double arithmetic; build with
 * -ffp-contract=off so no fused multiply-add changes a rounding).
 *
 * Random numbers: SplitMix64 (Steele, Lea, Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014; the 64-bit finaliser
 * constants of Vigna's reference code). The n-th output of a SplitMix64
 * stream seeded with s is mix64(s + (n+1)*0x9E3779B97F4A7C15).
 *
 * Normal deviates: the Box-Muller transform (Box and Muller, "A note on the
 * generation of random normal deviates", Ann. Math. Statist. 1958): the two
 * 32-bit halves of one 64-bit draw give u1, u2 in (0, 1) and
 * z = sqrt(-2 ln u1) cos(2 pi u2), a standard normal deviate (tails to about
 * 6.8 sigma). ln and cos are evaluated here by fixed series in plain IEEE
 * double arithmetic, not by the C library, so every platform produces the
 * same bits: ln(m 2^e) = e ln 2 + 2 atanh((m-1)/(m+1)) for m in [1, 2), and
 * cos by its Taylor series after reducing the angle to [-pi, pi].
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <pthread.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Base of the stream for one tensor: first SplitMix64 output seeded with
 * seed*2^32 + id. */
static inline uint64_t stream_base(uint64_t seed, uint64_t id) {
    return mix64((seed << 32) + id + GOLDEN);
}

/* idx-th output of the SplitMix64 stream whose state starts at base. */
static inline uint64_t draw(uint64_t base, uint64_t idx) {
    return mix64(base + (idx + 1) * GOLDEN);
}

static const double LN2 = 0.69314718055994530942;
static const double TWO_PI = 6.28318530717958647692;
static const double PI_ = 3.14159265358979323846;

/* ln x for x in (0, 1]: x = m 2^e with m in [1, 2) (exact, frexp), then
 * ln m = 2 atanh(s), s = (m-1)/(m+1) <= 1/3, summed to s^41. */
static double ln_series(double x) {
    int e;
    double m = frexp(x, &e); /* x = m 2^e, m in [0.5, 1) */
    m *= 2.0;
    e -= 1;
    const double t = (m - 1.0) / (m + 1.0), t2 = t * t;
    double term = t, sum = 0.0;
    for (int k = 1; k <= 41; k += 2) {
        sum += term / (double)k;
        term *= t2;
    }
    return (double)e * LN2 + 2.0 * sum;
}

/* cos a for a in [0, 2 pi): reduced to [-pi, pi], Taylor series to a^40. */
static double cos_series(double a) {
    if (a > PI_) a -= TWO_PI;
    const double a2 = a * a;
    double term = 1.0, sum = 1.0;
    for (int n = 1; n <= 20; ++n) {
        term *= -a2 / (double)((2 * n - 1) * (2 * n));
        sum += term;
    }
    return sum;
}

static inline double normal_from(uint64_t h) {
    const double u1 = ((double)(h >> 32) + 0.5) * (1.0 / 4294967296.0);
    const double u2 = ((double)(h & 0xFFFFFFFFu) + 0.5) * (1.0 / 4294967296.0);
    return sqrt(-2.0 * ln_series(u1)) * cos_series(TWO_PI * u2);
}

/* Uniform double in [0, 1) with 53 random bits. */
static inline double uniform_from(uint64_t h) {
    return (double)(h >> 11) * (1.0 / 9007199254740992.0);
}

/* IEEE binary64 -> binary16, round to nearest even, with subnormals. */
static uint16_t f64_to_f16(double x) {
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(x)) return sign | 0x7e00;
    if (a >= 65520.0) return sign | 0x7c00;
    if (a < 0x1p-14) { /* subnormal range: ulp 2^-24 */
        double q = rint(a * 0x1p24);
        return sign | (uint16_t)q; /* q == 1024 is the smallest normal */
    }
    int e;
    frexp(a, &e); /* a in [2^(e-1), 2^e) */
    double q = rint(ldexp(a, 11 - e)); /* in [1024, 2048] */
    if (q >= 2048.0) { q = 1024.0; e += 1; }
    int ef = (e - 1) + 15;
    if (ef >= 31) return sign | 0x7c00;
    return sign | (uint16_t)((ef << 10) | ((int)q - 1024));
}

static double f16_to_f64(uint16_t h) {
    int e = (h >> 10) & 0x1f, m = h & 0x3ff;
    double v;
    if (e == 0) v = ldexp((double)m, -24);
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = ldexp((double)(m + 1024), e - 25);
    return (h & 0x8000) ? -v : v;
}

static inline double clampd(double v, double lo, double hi) {
    return v < lo ? lo : (v > hi ? hi : v);
}

/*
 * Q4 super-block (256 weights, 144 bytes):
 *   [0:2]  d    (binary16)      [2:4] dmin (binary16)
 *   [4:16] 96-bit little-endian field: sub-block scale sc_j (6 bits) at bit
 *          6j, sub-block min m_j (6 bits) at bit 48+6j, j = 0..7
 *   [16:144] codes: sub-block j in bytes 16+16j .. 16+16j+15; element i of
 *          the sub-block is the low nibble of byte (i mod 16) for i < 16 and
 *          the high nibble for i >= 16.
 * A weight dequantises to d*sc_j*q - dmin*m_j.
 * Quantiser: per sub-block lo = min(0, min w), hi = max w,
 *   s_j = (hi-lo)/15, mu_j = -lo; d = f16(max s_j / 63), dmin = f16(max mu_j/63);
 *   sc_j = clamp(rne(s_j/d), 0, 63), m_j = clamp(rne(mu_j/dmin), 0, 63);
 *   q = clamp(rne((w + dmin*m_j)/(d*sc_j)), 0, 15), 0 where d*sc_j == 0.
 */
static void quantize_q4_block(const double* w, uint8_t* out) {
    double s[8], mu[8], smax = 0.0, mumax = 0.0;
    for (int j = 0; j < 8; ++j) {
        double lo = 0.0, hi = w[32 * j];
        for (int i = 0; i < 32; ++i) {
            double v = w[32 * j + i];
            if (v < lo) lo = v;
            if (v > hi) hi = v;
        }
        s[j] = (hi - lo) / 15.0;
        mu[j] = -lo;
        if (s[j] > smax) smax = s[j];
        if (mu[j] > mumax) mumax = mu[j];
    }
    uint16_t dh = f64_to_f16(smax / 63.0), mh = f64_to_f16(mumax / 63.0);
    double d = f16_to_f64(dh), dmin = f16_to_f64(mh);
    int sc[8], m[8];
    for (int j = 0; j < 8; ++j) {
        sc[j] = d > 0.0 ? (int)clampd(rint(s[j] / d), 0.0, 63.0) : 0;
        m[j] = dmin > 0.0 ? (int)clampd(rint(mu[j] / dmin), 0.0, 63.0) : 0;
    }
    memset(out, 0, 144);
    out[0] = dh & 0xff; out[1] = dh >> 8;
    out[2] = mh & 0xff; out[3] = mh >> 8;
    uint8_t field[12] = {0};
    for (int j = 0; j < 8; ++j) {
        for (int b = 0; b < 6; ++b) {
            int bs = 6 * j + b, bm = 48 + 6 * j + b;
            if ((sc[j] >> b) & 1) field[bs >> 3] |= (uint8_t)(1u << (bs & 7));
            if ((m[j] >> b) & 1) field[bm >> 3] |= (uint8_t)(1u << (bm & 7));
        }
    }
    memcpy(out + 4, field, 12);
    for (int j = 0; j < 8; ++j) {
        double denom = d * (double)sc[j];
        double off = dmin * (double)m[j];
        for (int i = 0; i < 32; ++i) {
            int q = 0;
            if (denom > 0.0) q = (int)clampd(rint((w[32 * j + i] + off) / denom), 0.0, 15.0);
            uint8_t* byte = out + 16 + 16 * j + (i & 15);
            *byte |= (uint8_t)(i < 16 ? q : (q << 4));
        }
    }
}

/* ---------------------------------------------------------------- threads */

typedef struct {
    int64_t begin, end;
    void (*fn)(void* ctx, int64_t b, int64_t e);
    void* ctx;
} task_t;

static void* run_task(void* p) {
    task_t* t = (task_t*)p;
    t->fn(t->ctx, t->begin, t->end);
    return 0;
}

static void parallel_for(int64_t n, int nthreads, void (*fn)(void*, int64_t, int64_t), void* ctx) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (n < 4096 || nthreads == 1) { fn(ctx, 0, n); return; }
    pthread_t th[256];
    task_t tk[256];
    for (int i = 0; i < nthreads; ++i) {
        tk[i].begin = n * i / nthreads;
        tk[i].end = n * (i + 1) / nthreads;
        tk[i].fn = fn;
        tk[i].ctx = ctx;
        pthread_create(&th[i], 0, run_task, &tk[i]);
    }
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], 0);
}

/* ------------------------------------------------------------- Q4 matrix */

typedef struct { uint64_t base; double sigma; int64_t nsb_row; uint8_t* out; } q4_ctx;

static void q4_range(void* p, int64_t b, int64_t e) {
    q4_ctx* c = (q4_ctx*)p;
    double w[256];
    for (int64_t blk = b; blk < e; ++blk) {
        for (int i = 0; i < 256; ++i)
            w[i] = c->sigma * normal_from(draw(c->base, (uint64_t)blk * 256 + i));
        quantize_q4_block(w, c->out + blk * 144);
    }
}

/* n_rows x k weights ~ sigma*N(0,1), row-major, quantised to Q4 super-blocks
 * ([n_rows][k/256] x 144 bytes). Weight (r, c) uses draw index r*k + c. */
int synth_q4(uint64_t seed, uint64_t id, int64_t n_rows, int64_t k, double sigma,
             uint8_t* out, int nthreads) {
    if (k % 256 != 0 || n_rows < 0) return -1;
    q4_ctx c = { stream_base(seed, id), sigma, k / 256, out };
    parallel_for(n_rows * (k / 256), nthreads, q4_range, &c);
    return 0;
}

/* Raw fp64 weights behind synth_q4 (for tests of the quantiser). */
int synth_normal_f64(uint64_t seed, uint64_t id, int64_t n, double sigma, double* out) {
    uint64_t base = stream_base(seed, id);
    for (int64_t i = 0; i < n; ++i) out[i] = sigma * normal_from(draw(base, (uint64_t)i));
    return 0;
}

/* ------------------------------------------------------- dense fp32/fp16 */

typedef struct { uint64_t base; double mean, sigma; float* f32; uint16_t* f16; } dense_ctx;

static void f32_range(void* p, int64_t b, int64_t e) {
    dense_ctx* c = (dense_ctx*)p;
    for (int64_t i = b; i < e; ++i)
        c->f32[i] = (float)(c->mean + c->sigma * normal_from(draw(c->base, (uint64_t)i)));
}

static void f16_range(void* p, int64_t b, int64_t e) {
    dense_ctx* c = (dense_ctx*)p;
    for (int64_t i = b; i < e; ++i)
        c->f16[i] = f64_to_f16(c->mean + c->sigma * normal_from(draw(c->base, (uint64_t)i)));
}

int synth_normal_f32(uint64_t seed, uint64_t id, int64_t n, double mean, double sigma,
                     float* out, int nthreads) {
    dense_ctx c = { stream_base(seed, id), mean, sigma, out, 0 };
    parallel_for(n, nthreads, f32_range, &c);
    return 0;
}

int synth_normal_f16(uint64_t seed, uint64_t id, int64_t n, double mean, double sigma,
                     uint16_t* out, int nthreads) {
    dense_ctx c = { stream_base(seed, id), mean, sigma, 0, out };
    parallel_for(n, nthreads, f16_range, &c);
    return 0;
}

/* ------------------------------------------------------------ q8 blocks */

typedef struct { uint64_t base; int8_t* codes; uint16_t* scales; } q8_ctx;

/* Block b of 32 values: scale draw index b*33, value i uses b*33 + 1 + i.
 * The block's range A = 2 + 2u (u uniform), its binary16 scale is
 * f16(A/127), and its codes are a standard normal deviate times 127/A,
 * rounded half-even and clamped to [-127, 127]. */
static void q8_range(void* p, int64_t b, int64_t e) {
    q8_ctx* c = (q8_ctx*)p;
    for (int64_t blk = b; blk < e; ++blk) {
        double a = 2.0 + 2.0 * uniform_from(draw(c->base, (uint64_t)blk * 33));
        c->scales[blk] = f64_to_f16(a / 127.0);
        for (int i = 0; i < 32; ++i) {
            double z = normal_from(draw(c->base, (uint64_t)blk * 33 + 1 + i));
            c->codes[blk * 32 + i] = (int8_t)clampd(rint(z * 127.0 / a), -127.0, 127.0);
        }
    }
}

int synth_q8_blocks(uint64_t seed, uint64_t id, int64_t n_blocks, int8_t* codes,
                    uint16_t* scales, int nthreads) {
    q8_ctx c = { stream_base(seed, id), codes, scales };
    parallel_for(n_blocks, nthreads, q8_range, &c);
    return 0;
}

/* ------------------------------------------------------- integers */

/* Uniform integers in [0, n) by the multiply-shift map of the top 32 bits. */
int synth_uniform_int(uint64_t seed, uint64_t id, int64_t count, uint32_t n, int32_t* out) {
    uint64_t base = stream_base(seed, id);
    for (int64_t i = 0; i < count; ++i)
        out[i] = (int32_t)(((draw(base, (uint64_t)i) >> 32) * (uint64_t)n) >> 32);
    return 0;
}

/* Fisher-Yates shuffle of 0..n-1: for i = n-1 down to 1 swap i with
 * j uniform in [0, i] (draw index i). */
int synth_permutation(uint64_t seed, uint64_t id, int64_t n, int32_t* out) {
    uint64_t base = stream_base(seed, id);
    for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)i;
    for (int64_t i = n - 1; i >= 1; --i) {
        int64_t j = (int64_t)(((draw(base, (uint64_t)i) >> 32) * (uint64_t)(i + 1)) >> 32);
        int32_t t = out[i]; out[i] = out[j]; out[j] = t;
    }
    return 0;
}

/* Raw 64-bit draws (for the generator's own tests). */
int synth_raw(uint64_t seed, uint64_t id, int64_t n, uint64_t* out) {
    uint64_t base = stream_base(seed, id);
    for (int64_t i = 0; i < n; ++i) out[i] = draw(base, (uint64_t)i);
    return 0;
}

/*
 * ggq_synth.c -- seeded synthetic inputs for the block-quantized GEMV path.
 *
 * This module is the ONLY code shared by the CUDA path's tests/bench and the
 * CPU oracle.  It produces input bytes; it holds none of the decode or dot-product
 * arithmetic that the path computes:
 *
 *   - a counter-based N(0, sigma) generator (splitmix64 finaliser -> two uniforms
 *     -> Marsaglia polar method).  Every element is a pure function of
 *     (seed, stream, element index), so any row of a tensor can be regenerated
 *     alone for spot checks;
 *   - the Q8_0 block encoder, following "GGUF: The File Format...", section
 *     "How a Q8_0 block is stored" and its practice script: d = fp16(absmax/127),
 *     q = round-half-even(w / d) clipped to +-127;
 *   - a round-to-nearest Q4_K super-block encoder (256 weights, 8 sub-blocks of
 *     32 with 6-bit scale and min, fp16 d and dmin).  The pages give only the
 *     size (144 B) and the two-level idea ("What is quantization (in GGUF)");
 *     the byte layout is the de-facto one of real Q4_K files;
 *   - a Q4_0 block encoder, the Q8_0 recipe on a 4-bit grid: d = fp16(absmax/7),
 *     q = round-half-even(w / d) clipped to -8..7, stored as the code q + 8, the
 *     code of weight l (l < 16) in the low nibble of byte l and that of weight
 *     16 + l in its high nibble (the byte layout of real Q4_0 files);
 *   - a round-to-nearest Q6_K super-block encoder (256 weights, 16 sub-blocks of
 *     16 with a signed 8-bit scale each under an fp16 d; 6-bit codes q + 32 split
 *     into 4 low bits (ql) and 2 high bits (qh)).  The pages give only the size
 *     (210 B) and the k-quant idea; the byte layout is the de-facto one of real
 *     Q6_K files;
 *   - fp32 -> fp16 / bf16 round-to-nearest-even conversions (bit manipulation).
 *
 * Determinism across machines: the generator uses only IEEE basic operations
 * (+ - * / sqrt, frexp) and its own logarithm (atanh series), and the file is
 * compiled with -ffp-contract=off, so x86_64 and aarch64 produce identical bytes.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- RNG ---- */

/* splitmix64 output function (Steele, Lea, Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014; constants as published). */
static inline uint64_t mix64(uint64_t z) {
    z += 0x9e3779b97f4a7c15ULL;
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
    return z ^ (z >> 31);
}

/* uniform in (-1, 1) from the top 53 bits */
static inline double uniform_pm1(uint64_t key, uint64_t ctr) {
    uint64_t r = mix64(key ^ mix64(ctr));
    double u = (double)(r >> 11) * (1.0 / 9007199254740992.0); /* [0,1) */
    return 2.0 * u - 1.0;
}

/* natural log for s in (0, 1]: s = m * 2^e with m in [sqrt(1/2), sqrt(2)),
 * log m = 2 atanh(t), t = (m-1)/(m+1), |t| < 0.172, series to t^31. */
static double synth_log(double s) {
    int e;
    double m = frexp(s, &e); /* m in [0.5, 1) */
    if (m < 0.70710678118654752440) { m *= 2.0; e -= 1; }
    double t = (m - 1.0) / (m + 1.0);
    double t2 = t * t;
    /* atanh(t)/t = sum_k t2^k / (2k+1); t2 < 0.0295 so 13 terms reach 1e-20 */
    double p = 1.0 / 25.0;
    p = p * t2 + 1.0 / 23.0;
    p = p * t2 + 1.0 / 21.0;
    p = p * t2 + 1.0 / 19.0;
    p = p * t2 + 1.0 / 17.0;
    p = p * t2 + 1.0 / 15.0;
    p = p * t2 + 1.0 / 13.0;
    p = p * t2 + 1.0 / 11.0;
    p = p * t2 + 1.0 / 9.0;
    p = p * t2 + 1.0 / 7.0;
    p = p * t2 + 1.0 / 5.0;
    p = p * t2 + 1.0 / 3.0;
    p = p * t2 + 1.0;
    return 2.0 * t * p + (double)e * 0.69314718055994530942;
}

/* one N(0,1) draw for element `idx` of stream `key` (polar method) */
static double normal_at(uint64_t key, uint64_t idx) {
    for (uint64_t a = 0; a < 32; ++a) {
        uint64_t c = idx * 64u + 2u * a;
        double u = uniform_pm1(key, c);
        double v = uniform_pm1(key, c + 1u);
        double s = u * u + v * v;
        if (s > 0.0 && s < 1.0) {
            return u * sqrt(-2.0 * synth_log(s) / s);
        }
    }
    return 0.0; /* unreachable in practice: 0.215^32 */
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return mix64(seed ^ mix64(stream ^ 0x5851f42d4c957f2dULL));
}

/* ------------------------------------------------------- conversions ---- */

static inline uint32_t f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static inline float u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

uint16_t synth_f32_to_f16(float f) {
    uint32_t x = f2u(f);
    uint32_t sign = (x >> 16) & 0x8000u;
    uint32_t ax = x & 0x7fffffffu;
    if (ax >= 0x7f800000u) return (uint16_t)(sign | 0x7c00u | (ax > 0x7f800000u ? 0x200u : 0u));
    if (ax >= 0x477ff000u) return (uint16_t)(sign | 0x7c00u);          /* >= 65520 -> inf */
    if (ax >= 0x38800000u) {                                           /* normal half */
        uint32_t mant = ax & 0x7fffffu;
        uint32_t h = (((ax >> 23) - 112u) << 10) | (mant >> 13);
        uint32_t rem = mant & 0x1fffu;
        if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u;
        return (uint16_t)(sign | h);
    }
    if (ax < 0x33000000u) return (uint16_t)sign;                       /* <= 2^-25 -> 0 */
    {                                                                  /* subnormal half */
        uint32_t e = ax >> 23;
        uint32_t mant = (ax & 0x7fffffu) | 0x800000u;
        uint32_t shift = 126u - e;                                     /* 14..24 */
        uint32_t h = mant >> shift;
        uint32_t rem = mant & ((1u << shift) - 1u);
        uint32_t half = 1u << (shift - 1u);
        if (rem > half || (rem == half && (h & 1u))) h += 1u;
        return (uint16_t)(sign | h);
    }
}

/* fp16 -> fp32 for the encoder's own use (the encoder needs the stored d) */
static float f16_to_f32_enc(uint16_t h) {
    uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    uint32_t e = (h >> 10) & 0x1fu, m = h & 0x3ffu;
    if (e == 0) {
        float v = (float)m * 5.9604644775390625e-08f; /* m * 2^-24, exact */
        return sign ? -v : v;
    }
    if (e == 31) return u2f(sign | 0x7f800000u | (m << 13));
    return u2f(sign | ((e + 112u) << 23) | (m << 13));
}

uint16_t synth_f32_to_bf16(float f) {
    uint32_t x = f2u(f);
    if ((x & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((x >> 16) | 0x40u);
    uint32_t r = x + 0x7fffu + ((x >> 16) & 1u);
    return (uint16_t)(r >> 16);
}

/* ----------------------------------------------------------- encoders ---- */

/* Q8_0: 32 weights -> 34 bytes (fp16 d, 32 x int8) */
static void encode_q8_0_block(const float* w, uint8_t* out) {
    float amax = 0.0f;
    for (int i = 0; i < 32; ++i) { float a = fabsf(w[i]); if (a > amax) amax = a; }
    uint16_t dh = synth_f32_to_f16(amax / 127.0f);
    float d = f16_to_f32_enc(dh);
    out[0] = (uint8_t)(dh & 0xff);
    out[1] = (uint8_t)(dh >> 8);
    for (int i = 0; i < 32; ++i) {
        float q = (d == 0.0f) ? 0.0f : rintf(w[i] / d);
        if (q > 127.0f) q = 127.0f;
        if (q < -127.0f) q = -127.0f;
        out[2 + i] = (uint8_t)(int8_t)q;
    }
}

static inline float clampf(float v, float lo, float hi) { return v < lo ? lo : (v > hi ? hi : v); }

/* Q4_0: 32 weights -> 18 bytes (fp16 d, 16 bytes of 4-bit codes) */
static void encode_q4_0_block(const float* w, uint8_t* out) {
    float amax = 0.0f;
    for (int i = 0; i < 32; ++i) { float a = fabsf(w[i]); if (a > amax) amax = a; }
    uint16_t dh = synth_f32_to_f16(amax / 7.0f);
    float d = f16_to_f32_enc(dh);
    out[0] = (uint8_t)(dh & 0xff);
    out[1] = (uint8_t)(dh >> 8);
    uint8_t code[32];
    for (int i = 0; i < 32; ++i) {
        float q = (d == 0.0f) ? 0.0f : clampf(rintf(w[i] / d), -8.0f, 7.0f);
        code[i] = (uint8_t)((int)q + 8);
    }
    for (int l = 0; l < 16; ++l) out[2 + l] = (uint8_t)(code[l] | (code[16 + l] << 4));
}

/* Q4_K: 256 weights -> 144 bytes, round-to-nearest, no search */
static void encode_q4_k_block(const float* w, uint8_t* out) {
    float s[8], mn[8], smax = 0.0f, mmax = 0.0f;
    for (int j = 0; j < 8; ++j) {
        float lo = w[32 * j], hi = w[32 * j];
        for (int i = 1; i < 32; ++i) {
            float v = w[32 * j + i];
            if (v < lo) lo = v;
            if (v > hi) hi = v;
        }
        mn[j] = lo < 0.0f ? -lo : 0.0f;
        s[j] = (hi + mn[j]) / 15.0f;
        if (s[j] > smax) smax = s[j];
        if (mn[j] > mmax) mmax = mn[j];
    }
    uint16_t dh = synth_f32_to_f16(smax / 63.0f);
    uint16_t mh = synth_f32_to_f16(mmax / 63.0f);
    float d = f16_to_f32_enc(dh), dmin = f16_to_f32_enc(mh);
    int sc[8], m[8];
    for (int j = 0; j < 8; ++j) {
        sc[j] = (d == 0.0f) ? 0 : (int)clampf(rintf(s[j] / d), 0.0f, 63.0f);
        m[j] = (dmin == 0.0f) ? 0 : (int)clampf(rintf(mn[j] / dmin), 0.0f, 63.0f);
    }
    out[0] = (uint8_t)(dh & 0xff); out[1] = (uint8_t)(dh >> 8);
    out[2] = (uint8_t)(mh & 0xff); out[3] = (uint8_t)(mh >> 8);
    uint8_t* sb = out + 4;
    for (int j = 0; j < 4; ++j) {
        sb[j]     = (uint8_t)((sc[j] & 63) | ((sc[j + 4] >> 4) << 6));
        sb[j + 4] = (uint8_t)((m[j] & 63) | ((m[j + 4] >> 4) << 6));
        sb[j + 8] = (uint8_t)((sc[j + 4] & 15) | ((m[j + 4] & 15) << 4));
    }
    uint8_t q[256];
    for (int j = 0; j < 8; ++j) {
        float a = d * (float)sc[j];
        float b = dmin * (float)m[j];
        for (int i = 0; i < 32; ++i) {
            float v = (a == 0.0f) ? 0.0f : rintf((w[32 * j + i] + b) / a);
            q[32 * j + i] = (uint8_t)(int)clampf(v, 0.0f, 15.0f);
        }
    }
    uint8_t* qs = out + 16;
    for (int c = 0; c < 4; ++c)
        for (int l = 0; l < 32; ++l)
            qs[32 * c + l] = (uint8_t)(q[64 * c + l] | (q[64 * c + 32 + l] << 4));
}

/* Q6_K: 256 weights -> 210 bytes, round-to-nearest, no search.  Sub-block j
 * (weights 16j .. 16j+15) gets the scale amax_j / 31; d = fp16(max scale / 127),
 * sc_j = round(scale_j / d) in 0..127, q = round(w / (d * sc_j)) in -32..31. */
static void encode_q6_k_block(const float* w, uint8_t* out) {
    float s[16], smax = 0.0f;
    for (int j = 0; j < 16; ++j) {
        float amax = 0.0f;
        for (int i = 0; i < 16; ++i) { float a = fabsf(w[16 * j + i]); if (a > amax) amax = a; }
        s[j] = amax / 31.0f;
        if (s[j] > smax) smax = s[j];
    }
    uint16_t dh = synth_f32_to_f16(smax / 127.0f);
    float d = f16_to_f32_enc(dh);
    int sc[16];
    for (int j = 0; j < 16; ++j) sc[j] = (d == 0.0f) ? 0 : (int)clampf(rintf(s[j] / d), 0.0f, 127.0f);
    uint8_t* ql = out;
    uint8_t* qh = out + 128;
    memset(out, 0, 192);
    for (int k = 0; k < 256; ++k) {
        float a = d * (float)sc[k / 16];
        int q = (a == 0.0f) ? 0 : (int)clampf(rintf(w[k] / a), -32.0f, 31.0f);
        int u = q + 32;
        int h = k / 128, g = (k % 128) / 32, l = k % 32;
        ql[64 * h + 32 * (g & 1) + l] |= (uint8_t)((u & 15) << (4 * (g >> 1)));
        qh[32 * h + l] |= (uint8_t)((u >> 4) << (2 * g));
    }
    for (int j = 0; j < 16; ++j) out[192 + j] = (uint8_t)(int8_t)sc[j];
    out[208] = (uint8_t)(dh & 0xff);
    out[209] = (uint8_t)(dh >> 8);
}

/* ------------------------------------------------------------- API ---- */

static int g_threads = 0;
int synth_set_threads(int n) { g_threads = n; return n; }
static int nthreads(void) {
#ifdef _OPENMP
    return g_threads > 0 ? g_threads : omp_get_max_threads();
#else
    return 1;
#endif
}

void synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t first, int64_t n,
                      float sigma, float* out) {
    uint64_t key = stream_key(seed, stream);
    #pragma omp parallel for schedule(static) num_threads(nthreads()) if (n > 65536)
    for (int64_t i = 0; i < n; ++i)
        out[i] = (float)((double)sigma * normal_at(key, first + (uint64_t)i));
}

void synth_normal_bf16(uint64_t seed, uint64_t stream, uint64_t first, int64_t n,
                       float sigma, uint16_t* out) {
    uint64_t key = stream_key(seed, stream);
    #pragma omp parallel for schedule(static) num_threads(nthreads()) if (n > 65536)
    for (int64_t i = 0; i < n; ++i)
        out[i] = synth_f32_to_bf16((float)((double)sigma * normal_at(key, first + (uint64_t)i)));
}

void synth_quantize_q8_0(const float* w, int64_t n, uint8_t* out) {
    int64_t nb = n / 32;
    for (int64_t b = 0; b < nb; ++b) encode_q8_0_block(w + 32 * b, out + 34 * b);
}

void synth_quantize_q4_0(const float* w, int64_t n, uint8_t* out) {
    int64_t nb = n / 32;
    for (int64_t b = 0; b < nb; ++b) encode_q4_0_block(w + 32 * b, out + 18 * b);
}

void synth_quantize_q6_k(const float* w, int64_t n, uint8_t* out) {
    int64_t nb = n / 256;
    for (int64_t b = 0; b < nb; ++b) encode_q6_k_block(w + 256 * b, out + 210 * b);
}

void synth_quantize_q4_k(const float* w, int64_t n, uint8_t* out) {
    int64_t nb = n / 256;
    for (int64_t b = 0; b < nb; ++b) encode_q4_k_block(w + 256 * b, out + 144 * b);
}

/* Rows [row0, row0+nrows) of a rows x cols tensor whose element (r, c) is
 * sigma * N(0,1) at counter r*cols + c, encoded block by block. */
void synth_q8_0_rows(uint64_t seed, uint64_t stream, int64_t row0, int64_t nrows,
                     int64_t cols, float sigma, uint8_t* out) {
    uint64_t key = stream_key(seed, stream);
    int64_t rb = cols / 32 * 34;
    #pragma omp parallel for schedule(static) num_threads(nthreads()) if (nrows > 4)
    for (int64_t r = 0; r < nrows; ++r) {
        float w[32];
        uint64_t base = (uint64_t)(row0 + r) * (uint64_t)cols;
        for (int64_t b = 0; b < cols / 32; ++b) {
            for (int i = 0; i < 32; ++i)
                w[i] = (float)((double)sigma * normal_at(key, base + (uint64_t)(32 * b + i)));
            encode_q8_0_block(w, out + r * rb + 34 * b);
        }
    }
}

void synth_q4_0_rows(uint64_t seed, uint64_t stream, int64_t row0, int64_t nrows,
                     int64_t cols, float sigma, uint8_t* out) {
    uint64_t key = stream_key(seed, stream);
    int64_t rb = cols / 32 * 18;
    #pragma omp parallel for schedule(static) num_threads(nthreads()) if (nrows > 4)
    for (int64_t r = 0; r < nrows; ++r) {
        float w[32];
        uint64_t base = (uint64_t)(row0 + r) * (uint64_t)cols;
        for (int64_t b = 0; b < cols / 32; ++b) {
            for (int i = 0; i < 32; ++i)
                w[i] = (float)((double)sigma * normal_at(key, base + (uint64_t)(32 * b + i)));
            encode_q4_0_block(w, out + r * rb + 18 * b);
        }
    }
}

void synth_q6_k_rows(uint64_t seed, uint64_t stream, int64_t row0, int64_t nrows,
                     int64_t cols, float sigma, uint8_t* out) {
    uint64_t key = stream_key(seed, stream);
    int64_t rb = cols / 256 * 210;
    #pragma omp parallel for schedule(static) num_threads(nthreads()) if (nrows > 4)
    for (int64_t r = 0; r < nrows; ++r) {
        float w[256];
        uint64_t base = (uint64_t)(row0 + r) * (uint64_t)cols;
        for (int64_t b = 0; b < cols / 256; ++b) {
            for (int i = 0; i < 256; ++i)
                w[i] = (float)((double)sigma * normal_at(key, base + (uint64_t)(256 * b + i)));
            encode_q6_k_block(w, out + r * rb + 210 * b);
        }
    }
}

/* F32 rows: the same draws, stored as little-endian fp32 */
void synth_f32_rows(uint64_t seed, uint64_t stream, int64_t row0, int64_t nrows,
                    int64_t cols, float sigma, uint8_t* out) {
    uint64_t key = stream_key(seed, stream);
    #pragma omp parallel for schedule(static) num_threads(nthreads()) if (nrows > 4)
    for (int64_t r = 0; r < nrows; ++r) {
        uint64_t base = (uint64_t)(row0 + r) * (uint64_t)cols;
        for (int64_t c = 0; c < cols; ++c) {
            float v = (float)((double)sigma * normal_at(key, base + (uint64_t)c));
            memcpy(out + (r * cols + c) * 4, &v, 4);
        }
    }
}

void synth_q4_k_rows(uint64_t seed, uint64_t stream, int64_t row0, int64_t nrows,
                     int64_t cols, float sigma, uint8_t* out) {
    uint64_t key = stream_key(seed, stream);
    int64_t rb = cols / 256 * 144;
    #pragma omp parallel for schedule(static) num_threads(nthreads()) if (nrows > 4)
    for (int64_t r = 0; r < nrows; ++r) {
        float w[256];
        uint64_t base = (uint64_t)(row0 + r) * (uint64_t)cols;
        for (int64_t b = 0; b < cols / 256; ++b) {
            for (int i = 0; i < 256; ++i)
                w[i] = (float)((double)sigma * normal_at(key, base + (uint64_t)(256 * b + i)));
            encode_q4_k_block(w, out + r * rb + 144 * b);
        }
    }
}

void synth_f32_to_f16_array(const float* in, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = synth_f32_to_f16(in[i]);
}

void synth_f32_to_bf16_array(const float* in, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = synth_f32_to_bf16(in[i]);
}

uint64_t synth_mix64(uint64_t z) { return mix64(z); }

/*
 * ggq_oracle.c -- CPU oracle for the block-quantized dequantize + GEMV path.
 *
 * TEST INFRASTRUCTURE.  Only tests/, __graft_entry__.smoke() and bench.py's
 * CPU-baseline / reference leg may load or call this code.  The CUDA library
 * shares no code, header, table or helper with it.
 *
 * Plain, slow, obviously-correct restatement of what the path computes:
 *   1. fp16 -> value from the IEEE-754 binary16 definition (sign, 5-bit
 *      exponent with bias 15, 10-bit fraction, subnormals, inf/NaN).
 *   2. Q8_0 block decode -- "GGUF: The File Format...", "How a Q8_0 block is
 *      stored": 32 weights share one fp16 scale d, each weight is a signed
 *      byte q, w = d * q.  Block = 2 bytes of d then 32 bytes of q; a row of
 *      `cols` weights is cols/32 consecutive blocks ("GGUF Inferencer in R",
 *      section 2.1, Q8_0 tensor blueprint).
 *   3. Q4_K super-block decode -- "GGUF: The File Format...", "How a Q8_0 block
 *      is stored" (k-quant paragraph): 256 weights in 8 sub-blocks of 32, each
 *      sub-block with a 6-bit scale and a 6-bit min, one fp16 super-scale for
 *      each (d, dmin), 144 bytes in all.  The byte order inside the 144 bytes is
 *      not printed on the pages; the reading used here (the layout of real
 *      Q4_K files) is: bytes 0-1 d, 2-3 dmin, 4-15 packed scales s[0..11],
 *      16-143 nibbles qs[0..127];
 *        j < 4 : sc_j = s[j] & 63,                      m_j = s[j+4] & 63
 *        j >= 4: sc_j = (s[j+4] & 15) | (s[j-4] >> 6) << 4,
 *                m_j  = (s[j+4] >> 4) | (s[j]   >> 6) << 4
 *      weight 64c+l (c = 0..3, l = 0..31) is the low nibble of qs[32c+l]
 *      (sub-block 2c), weight 64c+32+l its high nibble (sub-block 2c+1), and
 *      w = d*sc_j*q - dmin*m_j.
 *   4. Q4_0 block decode -- "GGUF: The File Format...", "How a Q8_0 block is
 *      stored": the Q8_0 layout with 4-bit integers, 2 + 16 = 18 bytes per 32
 *      weights.  Which nibble holds which weight and how a 4-bit code becomes
 *      a signed integer are not printed on the pages; the reading used here
 *      (the layout of real Q4_0 files) is: bytes 0-1 d, 2-17 qs[0..15];
 *      weight l (l < 16) is the low nibble of qs[l], weight 16+l its high
 *      nibble, and a code u in 0..15 stands for the integer u - 8, so
 *      w = d * (u - 8).
 *   5. Q6_K super-block decode -- "GGUF: The File Format...", "How a Q8_0
 *      block is stored" (k-quant paragraph: 256-weight super-blocks split into
 *      sub-blocks with their own scales under one 16-bit scale; the bits/weight
 *      loop: 210 bytes per 256 weights) and "Understanding quantization names
 *      like Q4_K_M" (Q4_K_M files hold some tensors as Q6_K).  The byte layout
 *      is not printed on the pages; the reading used here (the layout of real
 *      Q6_K files) is: bytes 0-127 ql (low 4 bits), 128-191 qh (high 2 bits),
 *      192-207 sixteen signed 8-bit sub-block scales sc[0..15] (one per 16
 *      weights), 208-209 d (fp16).  Weight k = 128h + 32g + l (h = 0..1,
 *      g = 0..3, l = 0..31) has the 6-bit code
 *        u = ((ql[64h + 32(g & 1) + l] >> 4(g >> 1)) & 15)
 *            | (((qh[32h + l] >> 2g) & 3) << 4)
 *      and w = d * sc[8h + 2g + l/16] * (u - 32).
 *   6. F32 rows -- "GGUF: The File Format...", the practice script's tensor
 *      payload: little-endian fp32 values, row after row.
 *   7. matvec -- culpeo.ws C++ engine blog, kernel list:
 *      the matrix-vector kernel (an r x c weight and a c-vector give an
 *      r-vector); "GGUF Inferencer in R" section 5.2.1 (the normalized input
 *      times the transposed weight): y[r] = sum_c w[r,c] * x[c].  For M activation
 *      rows, y[m][r] = sum_c w[r,c] * x[m][c].  Every product and sum is taken
 *      in double, columns in order.
 *
 * Decode produces fp32 exactly as the format defines it: the Q8_0 and Q4_0
 * products d*q, the Q6_K product d*sc*(u-32) (11 + 7 + 6 significant bits) and
 * the Q4_K products d*sc*q and dmin*m are exact in fp32, so the only rounding
 * is the final Q4_K subtraction (done here in double and rounded once more to
 * float, which gives the correctly rounded fp32 difference of two fp32 values
 * because 53 >= 2*24+2).
 *
 * Pins (tests/test_oracle_pins.py, tests/pin_checks.py): closed-form values of
 * hand-built blocks, IEEE binary16 special values, one-hot x (exact columns),
 * integer-valued inputs (exact sums), brute force against a library matmul on
 * tiny shapes, the pages' printed byte counts / offsets for the GGUF reader,
 * the practice script's printed mean errors (Q8_0 and its 4-bit block, through
 * the synth encoders), and Q4_0 / Q6_K blocks decoding like the Q8_0 blocks
 * of the same scale and integers.  tests/test_oracle_mutants.py plants slips
 * in copies of this file and checks that a pin fails for each.
 */
#include <stdint.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_Q4_0 = 2, ORC_Q8_0 = 8, ORC_Q4_K = 12, ORC_Q6_K = 14 };

/* IEEE-754 binary16 value, from the definition */
double orc_fp16_value(uint16_t h) {
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);               /* 2^(1-15) * frac/2^10 */
    } else if (expo == 31) {
        v = frac == 0 ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + frac), expo - 25); /* 2^(e-15) * (1 + frac/2^10) */
    }
    return sign ? -v : v;
}

/* bf16 is the top half of an fp32: widen exactly */
double orc_bf16_value(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

static uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* one Q8_0 block (34 bytes) -> 32 floats */
void orc_decode_q8_0_block(const uint8_t* blk, float* out) {
    double d = orc_fp16_value(rd16(blk));
    for (int i = 0; i < 32; ++i) {
        int q = (int8_t)blk[2 + i];
        out[i] = (float)(d * (double)q);
    }
}

/* one Q4_0 block (18 bytes) -> 32 floats */
void orc_decode_q4_0_block(const uint8_t* blk, float* out) {
    double d = orc_fp16_value(rd16(blk));
    const uint8_t* qs = blk + 2;
    for (int l = 0; l < 16; ++l) {
        int u_lo = qs[l] & 15;
        int u_hi = qs[l] >> 4;
        out[l] = (float)(d * (double)(u_lo - 8));
        out[16 + l] = (float)(d * (double)(u_hi - 8));
    }
}

/* the 6-bit scale and min of sub-block j of a Q4_K super-block */
void orc_q4_k_scale_min(const uint8_t* s, int j, int* sc, int* m) {
    if (j < 4) {
        *sc = s[j] & 63;
        *m = s[j + 4] & 63;
    } else {
        *sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
        *m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

/* one Q4_K super-block (144 bytes) -> 256 floats */
void orc_decode_q4_k_block(const uint8_t* blk, float* out) {
    double d = orc_fp16_value(rd16(blk));
    double dmin = orc_fp16_value(rd16(blk + 2));
    const uint8_t* s = blk + 4;
    const uint8_t* qs = blk + 16;
    for (int c = 0; c < 4; ++c) {
        int sc_lo, m_lo, sc_hi, m_hi;
        orc_q4_k_scale_min(s, 2 * c, &sc_lo, &m_lo);
        orc_q4_k_scale_min(s, 2 * c + 1, &sc_hi, &m_hi);
        for (int l = 0; l < 32; ++l) {
            int q_lo = qs[32 * c + l] & 15;
            int q_hi = qs[32 * c + l] >> 4;
            out[64 * c + l] = (float)(d * sc_lo * q_lo - dmin * m_lo);
            out[64 * c + 32 + l] = (float)(d * sc_hi * q_hi - dmin * m_hi);
        }
    }
}

/* one Q6_K super-block (210 bytes) -> 256 floats */
void orc_decode_q6_k_block(const uint8_t* blk, float* out) {
    const uint8_t* ql = blk;
    const uint8_t* qh = blk + 128;
    const int8_t* sc = (const int8_t*)(blk + 192);
    double d = orc_fp16_value(rd16(blk + 208));
    for (int h = 0; h < 2; ++h) {
        for (int g = 0; g < 4; ++g) {
            for (int l = 0; l < 32; ++l) {
                int lo = (ql[64 * h + 32 * (g & 1) + l] >> (4 * (g >> 1))) & 15;
                int hi = (qh[32 * h + l] >> (2 * g)) & 3;
                int u = lo | (hi << 4);
                int scale = sc[8 * h + 2 * g + l / 16];
                out[128 * h + 32 * g + l] = (float)(d * (double)scale * (double)(u - 32));
            }
        }
    }
}

/* bytes of one row of `cols` weights; 0 if the type or shape is not supported */
int64_t orc_row_bytes(int type, int64_t cols) {
    switch (type) {
    case ORC_F32: return 4 * cols;
    case ORC_F16: return 2 * cols;
    case ORC_Q8_0: return cols % 32 ? 0 : cols / 32 * 34;
    case ORC_Q4_0: return cols % 32 ? 0 : cols / 32 * 18;
    case ORC_Q4_K: return cols % 256 ? 0 : cols / 256 * 144;
    case ORC_Q6_K: return cols % 256 ? 0 : cols / 256 * 210;
    default: return 0;
    }
}

/* one row of weights -> floats */
static int decode_row(int type, const uint8_t* row, int64_t cols, float* out) {
    switch (type) {
    case ORC_F32:
        memcpy(out, row, (size_t)cols * 4);
        return 0;
    case ORC_F16:
        for (int64_t c = 0; c < cols; ++c) out[c] = (float)orc_fp16_value(rd16(row + 2 * c));
        return 0;
    case ORC_Q8_0:
        for (int64_t b = 0; b < cols / 32; ++b) orc_decode_q8_0_block(row + 34 * b, out + 32 * b);
        return 0;
    case ORC_Q4_K:
        for (int64_t b = 0; b < cols / 256; ++b) orc_decode_q4_k_block(row + 144 * b, out + 256 * b);
        return 0;
    case ORC_Q4_0:
        for (int64_t b = 0; b < cols / 32; ++b) orc_decode_q4_0_block(row + 18 * b, out + 32 * b);
        return 0;
    case ORC_Q6_K:
        for (int64_t b = 0; b < cols / 256; ++b) orc_decode_q6_k_block(row + 210 * b, out + 256 * b);
        return 0;
    default:
        return -1;
    }
}

int orc_dequantize(int type, const uint8_t* W, int64_t rows, int64_t cols, float* out) {
    int64_t rb = orc_row_bytes(type, cols);
    if (rb == 0 || rows < 0) return -1;
    for (int64_t r = 0; r < rows; ++r)
        if (decode_row(type, W + r * rb, cols, out + r * cols)) return -1;
    return 0;
}

/*
 * y[m*rows + r] = sum_c w[r,c] * x[m*cols + c]     (double, c in order)
 * absy[...]     = sum_c |w[r,c] * x[m*cols + c]|   (for the tolerance)
 * x is fp32 [M, cols]; `absy` may be NULL.
 */
int orc_gemv(int type, const uint8_t* W, int64_t rows, int64_t cols,
             const float* x, int64_t M, double* y, double* absy) {
    int64_t rb = orc_row_bytes(type, cols);
    if (rb == 0 || rows < 0 || M < 1) return -1;
    float* w = (float*)malloc((size_t)(cols > 0 ? cols : 1) * sizeof(float));
    if (!w) return -2;
    for (int64_t r = 0; r < rows; ++r) {
        decode_row(type, W + r * rb, cols, w);
        for (int64_t m = 0; m < M; ++m) {
            const float* xm = x + m * cols;
            double acc = 0.0, aacc = 0.0;
            for (int64_t c = 0; c < cols; ++c) {
                double p = (double)w[c] * (double)xm[c];
                acc += p;
                aacc += fabs(p);
            }
            y[m * rows + r] = acc;
            if (absy) absy[m * rows + r] = aacc;
        }
    }
    free(w);
    return 0;
}

/* Same with a bf16 activation matrix X [M, cols] (bit patterns), widened exactly. */
int orc_gemm_bf16(int type, const uint8_t* W, int64_t rows, int64_t cols,
                  const uint16_t* X, int64_t M, double* Y, double* absY) {
    int64_t rb = orc_row_bytes(type, cols);
    if (rb == 0 || rows < 0 || M < 1) return -1;
    float* w = (float*)malloc((size_t)(cols > 0 ? cols : 1) * sizeof(float));
    double* xd = (double*)malloc((size_t)(cols > 0 ? cols : 1) * sizeof(double) * (size_t)M);
    if (!w || !xd) { free(w); free(xd); return -2; }
    for (int64_t i = 0; i < M * cols; ++i) xd[i] = orc_bf16_value(X[i]);
    for (int64_t r = 0; r < rows; ++r) {
        decode_row(type, W + r * rb, cols, w);
        for (int64_t m = 0; m < M; ++m) {
            const double* xm = xd + m * cols;
            double acc = 0.0, aacc = 0.0;
            for (int64_t c = 0; c < cols; ++c) {
                double p = (double)w[c] * xm[c];
                acc += p;
                aacc += fabs(p);
            }
            Y[m * rows + r] = acc;
            if (absY) absY[m * rows + r] = aacc;
        }
    }
    free(w);
    free(xd);
    return 0;
}

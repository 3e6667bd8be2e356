// Per-lane decode + multiply of one weight tile row (one Q4_K super-block or one
// 8-block Q8_0 period), shared by the GEMV kernels.
//
// Decode trick (one AND per weight): a nibble (Q4_K) or an offset byte (Q8_0)
// masked in place inside its 32-bit word is the float bit pattern
// q * 2^(p - 149) for bit position p <= 20 -- a subnormal, or the first normal
// binade, which continues the subnormals linearly.  The activations are stored
// pre-scaled, x' = x * 2^(53 - p), so pattern * x' = q * x * 2^-96 exactly, and
// the per-sub-block sums P carry a factor 2^-96 that the scale removes.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace ggq {

constexpr float kTwo96 = pow2f(96);

// Pre-scale factor of the weight at position k of a Q4_K super-block (natural
// order): low nibbles sit at bits 0/8/16 (byte 3 shifted down to 16), high
// nibbles 4 higher.
__device__ __forceinline__ float q4k_xscale(int k) {
    const int hi = (k >> 5) & 1, b = k & 3;
    return hi ? (b == 0 ? pow2f(49) : b == 1 ? pow2f(41) : pow2f(33))
              : (b == 0 ? pow2f(53) : b == 1 ? pow2f(45) : pow2f(37));
}

// Pre-scale factor of the weight whose byte sits at position B of a 272-byte
// Q8_0 period (bytes 0..2 of a word in place, byte 3 shifted down to 2).
__device__ __forceinline__ float q8_xscale(int B) {
    const int pos = B & 3;
    return pos == 0 ? pow2f(53) : pos == 1 ? pow2f(45) : pow2f(37);
}

// acc(2) += a(2) * b(2), one packed instruction
__device__ __forceinline__ void ffma2(float& acc0, float& acc1, float a0, float a1, float b0, float b1) {
    uint64_t acc, a, b;
    asm("mov.b64 %0, {%1, %2};" : "=l"(acc) : "f"(acc0), "f"(acc1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(b) : "f"(b0), "f"(b1));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(acc0), "=f"(acc1) : "l"(acc));
}

// Packed accumulator pair kept in one 64-bit register across a loop.
struct F2 {
    uint64_t v;
};

__device__ __forceinline__ F2 f2_zero() { return F2{0ull}; }

__device__ __forceinline__ void f2_fma(F2& acc, float a0, float a1, float b0, float b1) {
    uint64_t a, b;
    asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(b) : "f"(b0), "f"(b1));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc.v) : "l"(a), "l"(b));
}

// sum of the four floats of two pairs: one packed add, one scalar add
__device__ __forceinline__ float f2_sum(F2 a, F2 b) {
    uint64_t s;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(s) : "l"(a.v), "l"(b.v));
    float s0, s1;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(s0), "=f"(s1) : "l"(s));
    return s0 + s1;
}

// Position of the x' value of weight k (natural order within a Q4_K
// super-block) in the layout the tile code reads: [c][lo/hi][byte b][word w],
// k = 64c + 32*hi + 4w + b.  x' values of words w and w+1 sit side by side, the
// operand pair of one packed FMA over two qs words.
__device__ __forceinline__ int q4k_xslot(int k) {
    return (k & ~31) | ((k & 3) << 3) | ((k >> 2) & 7);
}

__device__ __forceinline__ uint64_t and64(uint64_t a, uint64_t m) { return a & m; }

__device__ __forceinline__ void f2_fma64(F2& acc, uint64_t a, float b0, float b1) {
    uint64_t b;
    asm("mov.b64 %0, {%1, %2};" : "=l"(b) : "f"(b0), "f"(b1));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc.v) : "l"(a), "l"(b));
}

// Chunk c (weights 64c .. 64c+63, sub-blocks 2c and 2c+1) of R rows of Q4_K
// super-blocks per lane (rp: the lane's first row, `rstride` bytes to the next
// of its rows) against x' of that super-block and the per-sub-block sums of x.
// x' is read as float4 groups: slots 64c + 4q' .. +3 of the q4k_xslot layout
// (group q' of chunk c) of activation row m at xu + m*xs + c*cs + q'*gs.
// gs = 4, cs = 64: the 256 values contiguous; cs = 68: each chunk padded by 4
// floats, so lanes reading different chunks of one super-block hit different
// banks.  The sum of sub-block j of activation row m is su[m*ss + j*sj].
// acc[r][m] += sum_{k in chunk c} w_r[k] * x[m][k].
//
// Two consecutive qs words are handled as one 64-bit value: AND-ing it with a
// mask repeated in both halves gives the bit patterns of the same nibble of
// both words in one aligned register pair, the first operand of fma.f32x2.
template <int MMAX, int R>
__device__ __forceinline__ void q4k_chunk_rows(const uint8_t* rp, int rstride, int c, const float* xu, int xs,
                                               const float* su, int ss, float (&acc)[R][MMAX], int gs = 4,
                                               int sj = 1, int cs = 64) {
    // nibble masks (both halves): low nibble of bytes 0,1,2 in place, byte 3 after >> 8
    constexpr uint64_t kLo0 = 0x0000000F0000000Full, kLo1 = 0x00000F0000000F00ull, kLo2 = 0x000F0000000F0000ull;
    constexpr uint64_t kHi0 = 0x000000F0000000F0ull, kHi1 = 0x0000F0000000F000ull, kHi2 = 0x00F0000000F00000ull;
    float a_lo[R], a_hi[R], b_lo[R], b_hi[R];
    uint64_t wp[R][4];   // word pairs (0,1) (2,3) (4,5) (6,7) of the chunk
    // 6-bit scales and mins of sub-blocks 2c, 2c+1 (bytes jl, jh of the words
    // below).  Sub-blocks 0-3: the low 6 bits of scale bytes 0-3 / 4-7; 4-7: a
    // low nibble of bytes 8-11 plus the top 2 bits of bytes 0-3 / 4-7.  The
    // masks depend on c only, so they are worked out once per lane.
    const int jl = (2 * c) & 3, jh = (2 * c + 1) & 3;
    const bool upper = c >= 2;
    const uint32_t m1 = upper ? 0x0F0F0F0Fu : 0x3F3F3F3Fu, m2 = upper ? 0x30303030u : 0u;
    const uint32_t sel_lo = 0x7650u | (uint32_t)jl, sel_hi = 0x7650u | (uint32_t)jh;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const uint8_t* row = rp + r * rstride;
        const uint4 h = *reinterpret_cast<const uint4*>(row);
        const float d96 = half_bits_to_float(h.x) * kTwo96;
        const float dmin = half_bits_to_float(h.x >> 16);
        const uint32_t scw = ((upper ? h.w : h.y) & m1) | ((h.y >> 2) & m2);
        const uint32_t mw = ((upper ? (h.w >> 4) : h.z) & m1) | ((h.z >> 2) & m2);
        // 0x4B0000 | byte is the float 2^23 + byte
        const float2 sc = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(scw, 0x4B000000u, sel_lo)),
                                                 __uint_as_float(__byte_perm(scw, 0x4B000000u, sel_hi))),
                                     make_float2(-8388608.0f, -8388608.0f));
        const float2 mn = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(mw, 0x4B000000u, sel_lo)),
                                                 __uint_as_float(__byte_perm(mw, 0x4B000000u, sel_hi))),
                                     make_float2(-8388608.0f, -8388608.0f));
        const float2 a = __fmul2_rn(sc, make_float2(d96, d96));
        const float2 bb = __fmul2_rn(mn, make_float2(dmin, dmin));
        a_lo[r] = a.x;
        a_hi[r] = a.y;
        b_lo[r] = bb.x;
        b_hi[r] = bb.y;
        const ulonglong2 q0 = *reinterpret_cast<const ulonglong2*>(row + 16 + 32 * c);
        const ulonglong2 q1 = *reinterpret_cast<const ulonglong2*>(row + 32 + 32 * c);
        wp[r][0] = q0.x; wp[r][1] = q0.y; wp[r][2] = q1.x; wp[r][3] = q1.y;
    }
    // accumulator pairs per (low/high nibbles, byte position parity)
    F2 lo[R][MMAX][2], hi[R][MMAX][2];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MMAX; ++m)
#pragma unroll
            for (int b = 0; b < 2; ++b) lo[r][m][b] = hi[r][m][b] = f2_zero();
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        // x' of byte position b for the 8 words: low nibbles, high nibbles
        float4 xl[MMAX][2], xh[MMAX][2];
#pragma unroll
        for (int m = 0; m < MMAX; ++m) {
            const float* xm = xu + m * xs + c * cs + 2 * b * gs;
            xl[m][0] = *reinterpret_cast<const float4*>(xm);
            xl[m][1] = *reinterpret_cast<const float4*>(xm + gs);
            xh[m][0] = *reinterpret_cast<const float4*>(xm + 8 * gs);
            xh[m][1] = *reinterpret_cast<const float4*>(xm + 9 * gs);
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
#pragma unroll
            for (int pp = 0; pp < 4; ++pp) {
                const uint64_t v = b < 3 ? wp[r][pp] : (wp[r][pp] >> 8);
                const uint64_t ml = b == 0 ? kLo0 : b == 1 ? kLo1 : kLo2;
                const uint64_t mh = b == 0 ? kHi0 : b == 1 ? kHi1 : kHi2;
                const uint64_t pl = and64(v, ml), ph = and64(v, mh);
#pragma unroll
                for (int m = 0; m < MMAX; ++m) {
                    const float4 a = xl[m][pp >> 1], e = xh[m][pp >> 1];
                    if (pp & 1) {
                        f2_fma64(lo[r][m][b & 1], pl, a.z, a.w);
                        f2_fma64(hi[r][m][b & 1], ph, e.z, e.w);
                    } else {
                        f2_fma64(lo[r][m][b & 1], pl, a.x, a.y);
                        f2_fma64(hi[r][m][b & 1], ph, e.x, e.y);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
        for (int m = 0; m < MMAX; ++m) {
            const float* sm = su + m * ss;
            float a = acc[r][m];
            a = fmaf(a_lo[r], f2_sum(lo[r][m][0], lo[r][m][1]), a);
            a = fmaf(-b_lo[r], sm[2 * c * sj], a);
            a = fmaf(a_hi[r], f2_sum(hi[r][m][0], hi[r][m][1]), a);
            a = fmaf(-b_hi[r], sm[(2 * c + 1) * sj], a);
            acc[r][m] = a;
        }
    }
}

// All four chunks of R rows.
template <int MMAX, int R>
__device__ __forceinline__ void q4k_tile_rows(const uint8_t* rp, int rstride, const float* xu, int xs,
                                              const float* su, int ss, float (&acc)[R][MMAX], int gs = 4,
                                              int sj = 1, int cs = 64) {
#pragma unroll
    for (int c = 0; c < 4; ++c) q4k_chunk_rows<MMAX, R>(rp, rstride, c, xu, xs, su, ss, acc, gs, sj, cs);
}

// One row (R = 1) of the above.
template <int MMAX>
__device__ __forceinline__ void q4k_tile_row(const uint8_t* rp, const float* xu, int xs, const float* su, int ss,
                                             float (&acc)[MMAX]) {
    float a[1][MMAX];
#pragma unroll
    for (int m = 0; m < MMAX; ++m) a[0][m] = acc[m];
    q4k_tile_rows<MMAX, 1>(rp, 0, xu, xs, su, ss, a);
#pragma unroll
    for (int m = 0; m < MMAX; ++m) acc[m] = a[0][m];
}

// One 8-block Q8_0 period of one row (rp: 272 bytes) against x' indexed by
// byte position (272 values per activation row, read as float4 groups: group
// q of row m at xu + m*xs + q*gs) and 128 * sum(x) per block (block b of row m
// at su[m*ss + b*sj]).
template <int MMAX>
__device__ __forceinline__ void q8_tile_row(const uint8_t* rp, const float* xu, int xs, const float* su, int ss,
                                            float (&acc)[MMAX], int gs = 4, int sj = 1) {
    float pa[MMAX], pb[MMAX];
    float dcur = 0.0f;
#pragma unroll
    for (int m = 0; m < MMAX; ++m) pa[m] = pb[m] = 0.0f;
#pragma unroll
    for (int ch = 0; ch < 17; ++ch) {
        const uint4 q = *reinterpret_cast<const uint4*>(rp + 16 * ch);
        const uint32_t wq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int wi = ch * 4 + t;
            const uint32_t w = wq[t];
            float4 xv[MMAX];
#pragma unroll
            for (int m = 0; m < MMAX; ++m) xv[m] = *reinterpret_cast<const float4*>(xu + m * xs + wi * gs);
#pragma unroll
            for (int pos = 0; pos < 4; ++pos) {
                const int B = 4 * wi + pos;
                const int b = B / 34, o = B % 34;
                if (o == 0) {
                    dcur = half_bits_to_float(w >> (8 * pos));
                } else if (o >= 2) {
                    const uint32_t pat = pos < 3 ? ((w ^ 0x80808080u) & (0xFFu << (8 * pos)))
                                                 : (((w >> 8) ^ 0x00800000u) & 0x00FF0000u);
                    const float fw = __uint_as_float(pat);
#pragma unroll
                    for (int m = 0; m < MMAX; ++m) {
                        const float xsv = pos == 0 ? xv[m].x : pos == 1 ? xv[m].y : pos == 2 ? xv[m].z : xv[m].w;
                        if (pos & 1) pb[m] = fmaf(fw, xsv, pb[m]);
                        else pa[m] = fmaf(fw, xsv, pa[m]);
                    }
                    if (o == 33) {
#pragma unroll
                        for (int m = 0; m < MMAX; ++m) {
                            acc[m] = fmaf(dcur, fmaf(pa[m] + pb[m], kTwo96, -su[m * ss + b * sj]), acc[m]);
                            pa[m] = pb[m] = 0.0f;
                        }
                    }
                }
            }
        }
    }
}

// One quarter of a Q8_0 period: blocks 2c and 2c+1 (rp: their 68 bytes, 4-byte
// aligned) against x' of those byte positions (xu: 68 floats per activation
// row, 16-byte aligned, rows `xs` apart) and 128 * sum(x) of the two blocks
// (su[m*ss + 0 / 1]).  acc[m] += the 64 products.
template <int MMAX>
__device__ __forceinline__ void q8_chunk(const uint8_t* rp, const float* xu, int xs, const float* su, int ss,
                                         float (&acc)[MMAX]) {
    float pa[MMAX], pb[MMAX];
    float dcur = 0.0f;
#pragma unroll
    for (int m = 0; m < MMAX; ++m) pa[m] = pb[m] = 0.0f;
    const uint32_t* wp = reinterpret_cast<const uint32_t*>(rp);
#pragma unroll
    for (int wi = 0; wi < 17; ++wi) {
        const uint32_t w = wp[wi];
        float4 xv[MMAX];
#pragma unroll
        for (int m = 0; m < MMAX; ++m) xv[m] = *reinterpret_cast<const float4*>(xu + m * xs + 4 * wi);
#pragma unroll
        for (int pos = 0; pos < 4; ++pos) {
            const int B = 4 * wi + pos;
            const int b = B / 34, o = B % 34;
            if (o == 0) {
                dcur = half_bits_to_float(w >> (8 * pos));
            } else if (o >= 2) {
                const uint32_t pat = pos < 3 ? ((w ^ 0x80808080u) & (0xFFu << (8 * pos)))
                                             : (((w >> 8) ^ 0x00800000u) & 0x00FF0000u);
                const float fw = __uint_as_float(pat);
#pragma unroll
                for (int m = 0; m < MMAX; ++m) {
                    const float xsv = pos == 0 ? xv[m].x : pos == 1 ? xv[m].y : pos == 2 ? xv[m].z : xv[m].w;
                    if (pos & 1) pb[m] = fmaf(fw, xsv, pb[m]);
                    else pa[m] = fmaf(fw, xsv, pa[m]);
                }
                if (o == 33) {
#pragma unroll
                    for (int m = 0; m < MMAX; ++m) {
                        acc[m] = fmaf(dcur, fmaf(pa[m] + pb[m], kTwo96, -su[m * ss + b]), acc[m]);
                        pa[m] = pb[m] = 0.0f;
                    }
                }
            }
        }
    }
}

}  // namespace ggq

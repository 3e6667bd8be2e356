// Per-lane decode + multiply of one weight tile row (one Q4_K super-block, one
// 8-block Q8_0 period or a chunk of an 8-block Q4_0 period), shared by the
// GEMV kernels.
//
// Decode trick (one AND per weight): a nibble (Q4_K, Q4_0) or an offset byte
// (Q8_0) masked in place inside its 32-bit word is the float bit pattern
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
// order): low nibbles sit at bits 0/8/16 for bytes 0-2; byte 3 of an even word
// w = (k/4) % 8 is moved to bits 0-7 and that of the odd word w + 1 to bits
// 16-23 (one byte_perm for the pair); high nibbles 4 bits higher.
__device__ __forceinline__ float q4k_xscale(int k) {
    const int hi = (k >> 5) & 1, b = (k & 3) == 3 ? (((k >> 2) & 1) ? 2 : 0) : (k & 3);
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
// super-block) in the layout the tile code reads: [c][byte b][word w][lo/hi],
// k = 64c + 32*hi + 4w + b.  The x' values of the low and the high nibble of
// one byte sit side by side, the operand pair of one packed FMA over one qs
// word; a float4 holds those of words w and w+1.
__device__ __forceinline__ int q4k_xslot(int k) {
    return (k & ~63) | ((k & 3) << 4) | (((k >> 2) & 7) << 1) | ((k >> 5) & 1);
}

__device__ __forceinline__ uint64_t and64(uint64_t a, uint64_t m) { return a & m; }

__device__ __forceinline__ void f2_fma64(F2& acc, uint64_t a, float b0, float b1) {
    uint64_t b;
    asm("mov.b64 %0, {%1, %2};" : "=l"(b) : "f"(b0), "f"(b1));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc.v) : "l"(a), "l"(b));
}

// (w & m0, w & m1) as one register pair
__device__ __forceinline__ uint64_t and_pair(uint32_t w, uint32_t m0, uint32_t m1) {
    uint64_t r;
    asm("{\n\t.reg .b32 l, h;\n\tand.b32 l, %1, %2;\n\tand.b32 h, %1, %3;\n\tmov.b64 %0, {l, h};\n\t}"
        : "=l"(r) : "r"(w), "r"(m0), "r"(m1));
    return r;
}

// (w0 & m, w1 & m) as one register pair
__device__ __forceinline__ uint64_t and_two(uint32_t w0, uint32_t w1, uint32_t m) {
    uint64_t r;
    asm("{\n\t.reg .b32 l, h;\n\tand.b32 l, %1, %3;\n\tand.b32 h, %2, %3;\n\tmov.b64 %0, {l, h};\n\t}"
        : "=l"(r) : "r"(w0), "r"(w1), "r"(m));
    return r;
}

// acc(2) += a(2) * b(2) on float2 values
__device__ __forceinline__ void f2_fma(float2& acc, float2 a, float2 b) { acc = __ffma2_rn(a, b, acc); }

// Chunk c (weights 64c .. 64c+63, sub-blocks 2c and 2c+1) of R rows of Q4_K
// super-blocks per lane (rp: the lane's first row, `rstride` bytes to the next
// of its rows) against x' of that super-block and the per-sub-block sums of x.
// x' of chunk c of activation row m starts at xu + m*xs + c*cs in the
// q4k_xslot order (cs = 64: the 256 values contiguous; cs = 68: each chunk
// padded by 4 floats, so lanes reading different chunks of one super-block
// hit different banks).  The sums of sub-blocks 2c, 2c+1 of activation row m
// are the float pair at su + m*ss + 2c.
// acc[r][m].x + acc[r][m].y += sum_{k in chunk c} w_r[k] * x[m][k].
//
// Each qs word gives the bit patterns of its low and its high nibble at one
// byte position in one aligned register pair (two ANDs), the first operand of
// fma.f32x2; the accumulator pairs hold (low-nibble part, high-nibble part),
// so the sub-block scales and mins apply as one packed FMA each.
template <int MMAX, int R>
__device__ __forceinline__ void q4k_chunk_rows(const uint8_t* rp, int rstride, int c, const float* xu, int xs,
                                               const float* su, int ss, float2 (&acc)[R][MMAX], int cs = 64) {
    float2 a2[R], nb2[R];   // (d*sc, dmin*m) of sub-blocks 2c, 2c+1; the mins negated
    uint32_t wd[R][8];      // the chunk's 8 qs words
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
        const float ndmin = -half_bits_to_float(h.x >> 16);
        const uint32_t scw = ((upper ? h.w : h.y) & m1) | ((h.y >> 2) & m2);
        const uint32_t mw = ((upper ? (h.w >> 4) : h.z) & m1) | ((h.z >> 2) & m2);
        // 0x4B0000 | byte is the float 2^23 + byte
        const float2 sc = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(scw, 0x4B000000u, sel_lo)),
                                                 __uint_as_float(__byte_perm(scw, 0x4B000000u, sel_hi))),
                                     make_float2(-8388608.0f, -8388608.0f));
        const float2 mn = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(mw, 0x4B000000u, sel_lo)),
                                                 __uint_as_float(__byte_perm(mw, 0x4B000000u, sel_hi))),
                                     make_float2(-8388608.0f, -8388608.0f));
        a2[r] = __fmul2_rn(sc, make_float2(d96, d96));
        nb2[r] = __fmul2_rn(mn, make_float2(ndmin, ndmin));
        const uint4 q0 = *reinterpret_cast<const uint4*>(row + 16 + 32 * c);
        const uint4 q1 = *reinterpret_cast<const uint4*>(row + 32 + 32 * c);
        wd[r][0] = q0.x; wd[r][1] = q0.y; wd[r][2] = q0.z; wd[r][3] = q0.w;
        wd[r][4] = q1.x; wd[r][5] = q1.y; wd[r][6] = q1.z; wd[r][7] = q1.w;
    }
    // two accumulator chains per (row, activation row): even and odd words
    F2 t[R][MMAX][2];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MMAX; ++m) t[r][m][0] = t[r][m][1] = f2_zero();
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        // nibble masks at byte position b < 3 (byte 3: see below)
        const uint32_t ml = b == 0 ? 0x0000000Fu : b == 1 ? 0x00000F00u : 0x000F0000u;
        const uint32_t mh = ml << 4;
        // x' of byte position b: (w lo, w hi, w+1 lo, w+1 hi) for w = 0, 2, 4, 6
        float4 xv[MMAX][4];
#pragma unroll
        for (int m = 0; m < MMAX; ++m)
#pragma unroll
            for (int q = 0; q < 4; ++q)
                xv[m][q] = *reinterpret_cast<const float4*>(xu + m * xs + c * cs + 16 * b + 4 * q);
#pragma unroll
        for (int r = 0; r < R; ++r) {
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                // byte 3 of words w, w + 1 (w even) in one register: bits 0-7, 16-23
                const uint32_t v = b < 3 ? wd[r][w] : __byte_perm(wd[r][w & ~1], wd[r][w | 1], 0x7733u);
                const uint64_t pr = b < 3 ? and_pair(v, ml, mh)
                                          : ((w & 1) ? and_pair(v, 0x000F0000u, 0x00F00000u) : and_pair(v, 0x0Fu, 0xF0u));
#pragma unroll
                for (int m = 0; m < MMAX; ++m) {
                    const float4 x4 = xv[m][w >> 1];
                    if (w & 1) f2_fma64(t[r][m][1], pr, x4.z, x4.w);
                    else f2_fma64(t[r][m][0], pr, x4.x, x4.y);
                }
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MMAX; ++m) {
        const float2 s2 = *reinterpret_cast<const float2*>(su + m * ss + 2 * c);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            uint64_t sv;
            asm("add.rn.f32x2 %0, %1, %2;" : "=l"(sv) : "l"(t[r][m][0].v), "l"(t[r][m][1].v));
            float2 pv;
            asm("mov.b64 {%0, %1}, %2;" : "=f"(pv.x), "=f"(pv.y) : "l"(sv));
            f2_fma(acc[r][m], a2[r], pv);
            f2_fma(acc[r][m], nb2[r], s2);
        }
    }
}

// All four chunks of R rows.
template <int MMAX, int R>
__device__ __forceinline__ void q4k_tile_rows(const uint8_t* rp, int rstride, const float* xu, int xs,
                                              const float* su, int ss, float2 (&acc)[R][MMAX], int cs = 64) {
#pragma unroll
    for (int c = 0; c < 4; ++c) q4k_chunk_rows<MMAX, R>(rp, rstride, c, xu, xs, su, ss, acc, cs);
}

// One row (R = 1) of the above into plain float accumulators.
template <int MMAX>
__device__ __forceinline__ void q4k_tile_row(const uint8_t* rp, const float* xu, int xs, const float* su, int ss,
                                             float (&acc)[MMAX]) {
    float2 a[1][MMAX];
#pragma unroll
    for (int m = 0; m < MMAX; ++m) a[0][m] = make_float2(acc[m], 0.0f);
    q4k_tile_rows<MMAX, 1>(rp, 0, xu, xs, su, ss, a);
#pragma unroll
    for (int m = 0; m < MMAX; ++m) acc[m] = a[0][m].x + a[0][m].y;
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

// Pre-scale factor of the x' value at slot e = 2B + hi of a Q4_0 chunk (B: the
// byte position in the chunk, mod 36; hi: 1 for the high nibble).  Chunks start
// on 4-byte boundaries, so B mod 4 is the byte's position in its word.  Byte 3
// of the code words is gathered pairwise, words (0, 1), (2, 3), (5, 6), (7, 8),
// by one byte_perm: the first word's at bits 0-7, the second's at 16-23.
__device__ __forceinline__ float q40_xscale(int e) {
    const int B = (e >> 1) % 36, pos = B & 3, hi = e & 1, wi = B >> 2;
    const bool first = wi == 0 || wi == 2 || wi == 5 || wi == 7;
    const int p = (pos < 3 ? 8 * pos : first ? 0 : 16) + 4 * hi;   // bit position of the nibble
    return p == 0 ? pow2f(53) : p == 4 ? pow2f(49) : p == 8 ? pow2f(45) : p == 12 ? pow2f(41)
                              : p == 16 ? pow2f(37) : pow2f(33);
}

// Chunk c of a 144-byte Q4_0 period (blocks 2c and 2c+1: bytes 36c .. 36c+35,
// nine 32-bit words; block 2c has d in bytes 0-1 and its codes in 2-17, block
// 2c+1 has d in 18-19 and its codes in 20-35) for R rows per lane (rp: the
// chunk in the lane's first row, 4-byte aligned; `rstride` bytes to the next).
// The code of weight l (l < 16) of a block is the low nibble of its byte l,
// that of weight 16 + l the high nibble; the weight is d * (code - 8).
// x' of byte position B of the chunk sits at xu[2B] (low-nibble weight) and
// xu[2B + 1] (high-nibble weight), 72 floats per chunk, activation row m at
// xu + m*xs; 8 * sum(x) of blocks 2c, 2c+1 at su[m*ss + 0 / 1].
// acc[r][m] += the chunk's 64 products.
//
// A qs word gives the patterns of the low and the high nibble of one byte as
// one register pair (two ANDs), the first operand of fma.f32x2 against the
// pair (x'_lo, x'_hi); both belong to the same block, so one accumulator pair
// per block and the block's scale apply at the end.
template <int MMAX, int R>
__device__ __forceinline__ void q40_chunk_rows(const uint8_t* rp, int rstride, const float* xu, int xs,
                                               const float* su, int ss, float (&acc)[R][MMAX]) {
    uint32_t wd[R][9];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const uint32_t* wp = reinterpret_cast<const uint32_t*>(rp + r * rstride);
#pragma unroll
        for (int i = 0; i < 9; ++i) wd[r][i] = wp[i];
    }
    F2 t[R][MMAX][2];   // [block of the chunk]
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MMAX; ++m) t[r][m][0] = t[r][m][1] = f2_zero();
#pragma unroll
    for (int wi = 0; wi < 9; ++wi) {
        // byte positions of this word that hold codes, and their block
        const int p0 = wi == 0 ? 2 : 0, p1 = wi == 4 ? 2 : 4;
        const int blk = wi <= 4 ? 0 : 1;
#pragma unroll
        for (int q = 0; q < 2; ++q) {   // byte positions 2q, 2q + 1: one float4 of x' per activation row
            if (2 * q + 1 < p0 || 2 * q >= p1) continue;
            float4 xv[MMAX];
#pragma unroll
            for (int m = 0; m < MMAX; ++m) xv[m] = *reinterpret_cast<const float4*>(xu + m * xs + 8 * wi + 4 * q);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int pos = 2 * q + k;
                if (pos < p0 || pos >= p1) continue;
                // byte 3: words (0, 1), (2, 3), (5, 6), (7, 8) in one register each
                const bool first = wi == 0 || wi == 2 || wi == 5 || wi == 7;
                const uint32_t ml = pos == 0 ? 0x0000000Fu : pos == 1 ? 0x00000F00u
                                  : (pos == 2 || !first) ? 0x000F0000u : 0x0000000Fu;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const uint32_t v = pos < 3 ? wd[r][wi]
                                     : first ? __byte_perm(wd[r][wi], wd[r][wi < 8 ? wi + 1 : wi], 0x7733u)
                                             : __byte_perm(wd[r][wi > 0 ? wi - 1 : wi], wd[r][wi], 0x7733u);
                    const uint64_t pr = and_pair(v, ml, ml << 4);
#pragma unroll
                    for (int m = 0; m < MMAX; ++m) {
                        if (k) f2_fma64(t[r][m][blk], pr, xv[m].z, xv[m].w);
                        else f2_fma64(t[r][m][blk], pr, xv[m].x, xv[m].y);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const float d0 = half_bits_to_float(wd[r][0]);
        const float d1 = half_bits_to_float(wd[r][4] >> 16);
#pragma unroll
        for (int m = 0; m < MMAX; ++m) {
            float p0x, p0y, p1x, p1y;
            asm("mov.b64 {%0, %1}, %2;" : "=f"(p0x), "=f"(p0y) : "l"(t[r][m][0].v));
            asm("mov.b64 {%0, %1}, %2;" : "=f"(p1x), "=f"(p1y) : "l"(t[r][m][1].v));
            const float2 s2 = *reinterpret_cast<const float2*>(su + m * ss);
            acc[r][m] = fmaf(d0, fmaf(p0x + p0y, kTwo96, -s2.x), acc[r][m]);
            acc[r][m] = fmaf(d1, fmaf(p1x + p1y, kTwo96, -s2.y), acc[r][m]);
        }
    }
}

// Chunk c = (half h, quarter pair gp) of a Q6_K super-block for R rows per lane.
// rp: the lane's first row of the copy in shared memory, whose super-block bytes
// start at rp + r0 (r0 even: the copy starts at the 16-byte boundary below the
// super-block); `rstride` bytes to the next of its rows.  The chunk holds the
// weights 128h + 32g + l for g = gp, gp + 2 and l = 0..31: ql bytes 64h + 32gp
// + l (low nibble g = gp, high g = gp + 2) and qh bytes 32h + l (2 bits per g).
// Words are read aligned; when r0 is 2 mod 4 (every odd super-block) they are
// realigned with a 16-bit funnel shift (ALIGNED: r0 is 0 mod 4, none needed).
// Each byte of a code word holds one 6-bit code u, masked in place like a
// Q8_0 byte (x' scaled by its byte position); the pair (g = gp, g = gp + 2) at
// one (w, b) is one packed FMA.  A code word takes the low 4 bits of each byte
// from the ql word and bits 4-7 from the shifted qh word in one select; bits 6
// and 7 then hold other fields' bits, which the per-byte 6-bit mask drops.
// x' of chunk c: [b][w][pair] at xu + 16b + 2w, activation row m at xu + m*xs;
// byte 3's pair is masked at bits 0-7 (low word) and 16-23 (high word).
// 32 * sum(x) of the four 16-column groups of the chunk ((g, l < 16) for g =
// gp, gp + 2, then l >= 16) at su + m*ss.  acc[r][m] += the chunk's 64 products.
template <int MMAX, int R, bool ALIGNED>
__device__ __forceinline__ void q6k_chunk_rows_t(const uint8_t* rp, int r0, int rstride, int c, const float* xu,
                                                 int xs, const float* su, int ss, float (&acc)[R][MMAX]) {
    const int h = c >> 1, gp = c & 1;
    const int base = r0 & ~3;
    const uint32_t shl = 4u - 2u * (uint32_t)gp, shr = 2u * (uint32_t)gp;
    float ds[R][4];   // d * sc of the four groups
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const uint8_t* sb = rp + r * rstride + r0;
        const float d = half_bits_to_float(*reinterpret_cast<const unsigned short*>(sb + 208));
        // scales 8h + 2gp + {0, 1} and + {4, 5} (signed bytes) as bytes 0-3 of one
        // word, offset by 128; 0x4B0000 | byte is the float 2^23 + byte
        const unsigned short* sc16 = reinterpret_cast<const unsigned short*>(sb + 192 + 8 * h + 2 * gp);
        const uint32_t sw = ((uint32_t)sc16[0] | ((uint32_t)sc16[2] << 16)) ^ 0x80808080u;
        const float2 s01 = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(sw, 0x4B000000u, 0x7650)),
                                                  __uint_as_float(__byte_perm(sw, 0x4B000000u, 0x7652))),
                                      make_float2(-8388736.0f, -8388736.0f));   // (sc0, sc4)
        const float2 s23 = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(sw, 0x4B000000u, 0x7651)),
                                                  __uint_as_float(__byte_perm(sw, 0x4B000000u, 0x7653))),
                                      make_float2(-8388736.0f, -8388736.0f));   // (sc1, sc5)
        const float2 d01 = __fmul2_rn(s01, make_float2(d, d)), d23 = __fmul2_rn(s23, make_float2(d, d));
        ds[r][0] = d01.x;   // (gp, l < 16)
        ds[r][1] = d01.y;   // (gp + 2, l < 16)
        ds[r][2] = d23.x;   // (gp, l >= 16)
        ds[r][3] = d23.y;   // (gp + 2, l >= 16)
    }
    F2 t[R][MMAX][2];   // [half of the chunk: l < 16, l >= 16]
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MMAX; ++m) t[r][m][0] = t[r][m][1] = f2_zero();
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        uint32_t lo[R][4], hi[R][4];   // code words of quarters gp, gp + 2 for words 4*half .. +3
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t* wl = reinterpret_cast<const uint32_t*>(rp + r * rstride + base + 64 * h + 32 * gp + 16 * half);
            const uint32_t* wh = reinterpret_cast<const uint32_t*>(rp + r * rstride + base + 128 + 32 * h + 16 * half);
            constexpr int kWords = ALIGNED ? 4 : 5;
            uint32_t a[kWords], q[kWords];
#pragma unroll
            for (int i = 0; i < kWords; ++i) {
                a[i] = wl[i];
                q[i] = wh[i];
            }
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const uint32_t qlw = ALIGNED ? a[w] : __byte_perm(a[w], a[w + 1], 0x5432);
                const uint32_t qhw = ALIGNED ? q[w] : __byte_perm(q[w], q[w + 1], 0x5432);
                lo[r][w] = (qlw & 0x0F0F0F0Fu) | ((qhw << shl) & 0xF0F0F0F0u);
                hi[r][w] = ((qlw >> 4) & 0x0F0F0F0Fu) | ((qhw >> shr) & 0xF0F0F0F0u);
            }
        }
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const uint32_t mk = b == 0 ? 0x3Fu : b == 1 ? 0x3F00u : 0x3F0000u;
            float4 xv[MMAX][2];   // pairs of words 4*half .. +3 at byte position b
#pragma unroll
            for (int m = 0; m < MMAX; ++m)
#pragma unroll
                for (int qq = 0; qq < 2; ++qq)
                    xv[m][qq] = *reinterpret_cast<const float4*>(xu + m * xs + 16 * b + 8 * half + 4 * qq);
#pragma unroll
            for (int r = 0; r < R; ++r) {
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    // byte 3: the low word's at bits 0-7, the high word's at 16-23 (one byte_perm)
                    const uint64_t pr = b < 3 ? and_two(lo[r][w], hi[r][w], mk)
                                              : and_pair(__byte_perm(lo[r][w], hi[r][w], 0x7733u), 0x3Fu, 0x3F0000u);
#pragma unroll
                    for (int m = 0; m < MMAX; ++m) {
                        const float4 x4 = xv[m][w >> 1];
                        if (w & 1) f2_fma64(t[r][m][half], pr, x4.z, x4.w);
                        else f2_fma64(t[r][m][half], pr, x4.x, x4.y);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MMAX; ++m) {
        const float4 s4 = *reinterpret_cast<const float4*>(su + m * ss);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float a0, a1, b0, b1;
            asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(t[r][m][0].v));
            asm("mov.b64 {%0, %1}, %2;" : "=f"(b0), "=f"(b1) : "l"(t[r][m][1].v));
            float v = acc[r][m];
            v = fmaf(ds[r][0], fmaf(a0, kTwo96, -s4.x), v);
            v = fmaf(ds[r][1], fmaf(a1, kTwo96, -s4.y), v);
            v = fmaf(ds[r][2], fmaf(b0, kTwo96, -s4.z), v);
            v = fmaf(ds[r][3], fmaf(b1, kTwo96, -s4.w), v);
            acc[r][m] = v;
        }
    }
}

// The chunk for any r0: the copy of an even super-block starts 0 mod 4 bytes
// below it, that of an odd one 2 mod 4 (210 = 2 mod 4); warp-uniform.
template <int MMAX, int R>
__device__ __forceinline__ void q6k_chunk_rows(const uint8_t* rp, int r0, int rstride, int c, const float* xu, int xs,
                                               const float* su, int ss, float (&acc)[R][MMAX]) {
    if ((r0 & 2) == 0) q6k_chunk_rows_t<MMAX, R, true>(rp, r0, rstride, c, xu, xs, su, ss, acc);
    else q6k_chunk_rows_t<MMAX, R, false>(rp, r0, rstride, c, xu, xs, su, ss, acc);
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

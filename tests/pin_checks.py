"""Checks that pin the CPU oracle to facts outside itself.

Each ``check_*`` takes an ``oracle.Oracle`` (the real build, or a deliberately
broken copy in test_oracle_mutants.py) and raises AssertionError on a mismatch.
Expected values come from the pages (golden fixtures), from closed forms worked
out by hand for hand-built blocks, from IEEE-754 special values, from integer
arithmetic (exact), or from numpy library routines on tiny inputs.
"""
from __future__ import annotations

import struct

import numpy as np

F32, F16, Q4_0, Q8_0, Q4_K, Q6_K = 0, 1, 2, 8, 12, 14


# ------------------------------------------------------------ fp16 / bf16 ----

def check_fp16(orc):
    # IEEE-754 binary16 special values, written out by hand
    literal = {
        0x3C00: 1.0, 0xC000: -2.0, 0x3800: 0.5, 0x7BFF: 65504.0,
        0x0400: 2.0 ** -14, 0x0001: 2.0 ** -24, 0x03FF: 1023 * 2.0 ** -24,
        0x3555: 1365 / 4096, 0x0000: 0.0, 0x4B00: 14.0, 0x5BD0: 250.0,
    }
    for h, v in literal.items():
        assert orc.fp16_value(h) == v, hex(h)
    assert str(orc.fp16_value(0x8000)) == "-0.0"
    assert orc.fp16_value(0x7C00) == float("inf")
    assert orc.fp16_value(0xFC00) == float("-inf")
    assert np.isnan(orc.fp16_value(0x7E00)) and np.isnan(orc.fp16_value(0xFC01))
    # every pattern against numpy's binary16 (a library routine)
    pats = np.arange(65536, dtype=np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    got = np.array([orc.fp16_value(int(h)) for h in pats])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.all((ref == got) | both_nan)
    assert np.array_equal(np.signbit(ref[~both_nan]), np.signbit(got[~both_nan]))


def check_bf16(orc):
    assert orc.bf16_value(0x3F80) == 1.0
    assert orc.bf16_value(0xC040) == -3.0
    assert orc.bf16_value(0x0001) == 2.0 ** -133
    rng = np.random.default_rng(1)
    for b in rng.integers(0, 65536, 500):
        v = np.array([int(b) << 16], dtype=np.uint32).view(np.float32)[0]
        g = orc.bf16_value(int(b))
        assert (np.isnan(v) and np.isnan(g)) or g == float(v)


# ------------------------------------------------------------------- Q8_0 ----

def q8_block(d_bits: int, qs) -> bytes:
    assert len(qs) == 32
    return struct.pack("<H", d_bits) + bytes((q & 0xFF) for q in qs)


Q8_PATTERN = [-128, -127, 0, 1, 127, 2, -2, 64, -64, 3, 5, 7, 11, 13, 17, 19,
              23, 29, 31, 37, -41, -43, -47, 53, 59, 61, -67, 71, 73, -79, 83, 89]


def check_q8_0_blocks(orc):
    # d = 1 (0x3C00): weights are the signed bytes themselves
    got = orc.decode_q8_0_block(q8_block(0x3C00, Q8_PATTERN))
    assert got.tolist() == [float(q) for q in Q8_PATTERN]
    # d = 0.5 (0x3800)
    got = orc.decode_q8_0_block(q8_block(0x3800, Q8_PATTERN))
    assert got.tolist() == [q / 2 for q in Q8_PATTERN]
    # d = -2 (0xC000): sign of d applies
    got = orc.decode_q8_0_block(q8_block(0xC000, Q8_PATTERN))
    assert got.tolist() == [-2.0 * q for q in Q8_PATTERN]
    # d = smallest subnormal 2^-24
    got = orc.decode_q8_0_block(q8_block(0x0001, Q8_PATTERN))
    assert got.tolist() == [q * 2.0 ** -24 for q in Q8_PATTERN]
    # d = 65504 (largest finite half); 65504 * -128 = -8384512 is exact in fp32
    got = orc.decode_q8_0_block(q8_block(0x7BFF, [-128] + [0] * 30 + [127]))
    assert got[0] == -8384512.0 and got[31] == 65504.0 * 127 and not got[1:31].any()
    # block byte size from bits/weight: 8.5 bits * 32 = 34 bytes
    assert orc.row_bytes(Q8_0, 32) == 34 and orc.row_bytes(Q8_0, 2048) == 64 * 34
    assert orc.row_bytes(Q8_0, 48) == 0  # not a whole number of blocks


# ------------------------------------------------------------------- Q4_0 ----

def check_q4_0_blocks(orc):
    # Literal bytes, expected values worked out by hand for the reading (weight
    # l: low nibble of byte l; weight 16 + l: its high nibble; code u -> u - 8).
    # A: d = 1, byte l = l | (15 - l) << 4 -> weights -8..7, then 7..-8
    blk = bytes([0x00, 0x3C]) + bytes([0xF0, 0xE1, 0xD2, 0xC3, 0xB4, 0xA5, 0x96, 0x87,
                                       0x78, 0x69, 0x5A, 0x4B, 0x3C, 0x2D, 0x1E, 0x0F])
    got = orc.decode_q4_0_block(blk)
    assert got.tolist() == [float(v) for v in list(range(-8, 8)) + list(range(7, -9, -1))]
    # B: d = 0.5, every byte 0x08: low code 8 -> 0, high code 0 -> -8 * 0.5
    got = orc.decode_q4_0_block(bytes([0x00, 0x38]) + bytes([0x08] * 16))
    assert got.tolist() == [0.0] * 16 + [-4.0] * 16
    # C: d = -2, every byte 0xF0: low code 0 -> -8 * -2 = 16, high code 15 -> 7 * -2
    got = orc.decode_q4_0_block(bytes([0x00, 0xC0]) + bytes([0xF0] * 16))
    assert got.tolist() == [16.0] * 16 + [-14.0] * 16
    # D: the Q8_0 layout with 4-bit integers: a Q4_0 block and a Q8_0 block with
    # the same scale and the same integers decode alike (Q8_0 decode is pinned
    # to the pages' own values)
    rng = np.random.default_rng(3)
    for d_bits in (0x3C00, 0x2E66, 0x8123, 0x0001, 0x7BFF):
        codes = rng.integers(0, 16, 32)
        qs = bytes(int(codes[l]) | (int(codes[16 + l]) << 4) for l in range(16))
        q4 = orc.decode_q4_0_block(struct.pack("<H", d_bits) + qs)
        q8 = orc.decode_q8_0_block(q8_block(d_bits, [int(u) - 8 for u in codes]))
        assert np.array_equal(q4, q8), hex(d_bits)
    # block byte size from bits/weight: 2 + 16 = 18 bytes, 4.5 bits per weight
    assert orc.row_bytes(Q4_0, 32) == 18 and orc.row_bytes(Q4_0, 4096) == 128 * 18
    assert orc.row_bytes(Q4_0, 48) == 0


def q4_0_block(d_bits: int, codes) -> bytes:
    """32 codes in weight order -> 18 bytes (reading: weight l low nibble of byte l)."""
    assert len(codes) == 32
    return struct.pack("<H", d_bits) + bytes(int(codes[l]) | (int(codes[16 + l]) << 4) for l in range(16))


# ------------------------------------------------------------------- Q6_K ----

def q6k_raw(ql, qh, sc, d_bits) -> bytes:
    assert len(ql) == 128 and len(qh) == 64 and len(sc) == 16
    return bytes(ql) + bytes(qh) + bytes(v & 0xFF for v in sc) + struct.pack("<H", d_bits)


def q6k_block(d_bits: int, sc, codes) -> bytes:
    """256 six-bit codes in weight order + 16 signed scales -> 210 bytes, for the
    reading's bit placement: weight 128h + 32g + l keeps its low 4 bits in ql byte
    64h + 32(g % 2) + l (low nibble for g < 2, high nibble for g >= 2) and its high
    2 bits in qh byte 32h + l at bit 2g."""
    ql, qh = [0] * 128, [0] * 64
    for k, u in enumerate(codes):
        h, g, l = k // 128, (k % 128) // 32, k % 32
        ql[64 * h + 32 * (g % 2) + l] |= (int(u) & 15) << (4 * (g // 2))
        qh[32 * h + l] |= (int(u) >> 4) << (2 * g)
    return q6k_raw(ql, qh, sc, d_bits)


def check_q6_k_blocks(orc):
    ones = [1] * 16
    # all codes 0: every weight is (0 - 32) * d * 1
    got = orc.decode_q6_k_block(q6k_raw([0] * 128, [0] * 64, ones, 0x3C00))
    assert got.tolist() == [-32.0] * 256
    # every 2-bit high field 1 (qh bytes 0x55), low bits 0: codes 16 -> -16 * sc;
    # sub-block scales in natural order: weight k uses scale k // 16, signed
    sc = [1, -1, 2, -2, 3, -3, 4, -4, 5, -5, 6, -6, 7, -7, 127, -128]
    got = orc.decode_q6_k_block(q6k_raw([0] * 128, [0x55] * 64, sc, 0x3C00))
    assert got.tolist() == [-16.0 * sc[k // 16] for k in range(256)]
    # d = 0.5 (0x3800), all bits set: codes 63 -> 31 * 0.5 * sc
    got = orc.decode_q6_k_block(q6k_raw([0xFF] * 128, [0xFF] * 64, sc, 0x3800))
    assert got.tolist() == [15.5 * sc[k // 16] for k in range(256)]
    # one set nibble of ql byte b: its low nibble is weight 128(b // 64) + b % 64,
    # its high nibble the weight 64 after it; every other weight stays -32
    for b in (0, 1, 31, 32, 63, 64, 100, 127):
        ql = [0] * 128
        ql[b] = 0x0F
        got = orc.decode_q6_k_block(q6k_raw(ql, [0] * 64, ones, 0x3C00))
        want = [-32.0] * 256
        want[128 * (b // 64) + b % 64] = -17.0
        assert got.tolist() == want, b
        ql[b] = 0xF0
        got = orc.decode_q6_k_block(q6k_raw(ql, [0] * 64, ones, 0x3C00))
        want = [-32.0] * 256
        want[128 * (b // 64) + b % 64 + 64] = -17.0
        assert got.tolist() == want, b
    # one 2-bit field g of qh byte b is weight 128(b // 32) + 32g + b % 32
    for b in (0, 5, 31, 32, 63):
        for g in range(4):
            qh = [0] * 64
            qh[b] = 3 << (2 * g)
            got = orc.decode_q6_k_block(q6k_raw([0] * 128, qh, ones, 0x3C00))
            want = [-32.0] * 256
            want[128 * (b // 32) + 32 * g + b % 32] = 16.0
            assert got.tolist() == want, (b, g)
    # unit scales: a Q6_K super-block equals eight Q8_0 blocks with the same d
    # and the integers u - 32 (Q8_0 decode is pinned to the pages' own values)
    rng = np.random.default_rng(6)
    for d_bits in (0x3C00, 0x2E66, 0x8123, 0x0001):
        codes = rng.integers(0, 64, 256)
        q6 = orc.decode_q6_k_block(q6k_block(d_bits, ones, codes))
        q8 = np.concatenate([orc.decode_q8_0_block(q8_block(d_bits, [int(u) - 32 for u in codes[32 * i:32 * i + 32]]))
                             for i in range(8)])
        assert np.array_equal(q6, q8), hex(d_bits)
    # block byte size from bits/weight: 6.5625 bits * 256 = 210 bytes
    assert orc.row_bytes(Q6_K, 256) == 210 and orc.row_bytes(Q6_K, 4096) == 16 * 210
    assert orc.row_bytes(Q6_K, 288) == 0


# ------------------------------------------------------------------- Q4_K ----

def q4k_block(d_bits: int, dmin_bits: int, scales12, qs128) -> bytes:
    assert len(scales12) == 12 and len(qs128) == 128
    return struct.pack("<HH", d_bits, dmin_bits) + bytes(scales12) + bytes(qs128)


def check_q4_k_blocks(orc):
    # A: d = 1, dmin = 0, sc_j = j+1, m_j = 0, every nibble 1 -> w[k] = k//32 + 1
    #    scales bytes worked out by hand: s[0..3] = sc0..3, s[4..7] = m0..3 = 0,
    #    s[8..11] = low nibbles of sc4..7 (5,6,7,8) | m4..7 << 4 (0)
    blk = q4k_block(0x3C00, 0x0000, [1, 2, 3, 4, 0, 0, 0, 0, 5, 6, 7, 8], [0x11] * 128)
    got = orc.decode_q4_k_block(blk)
    assert got.tolist() == [float(k // 32 + 1) for k in range(256)]

    # B: the 2-bit high parts of sub-blocks 4..7.  sc = (0,0,0,0,63,32,16,48),
    #    m = (0,0,0,0,33,17,63,2), d = dmin = 1, every q = 2  ->  w = 2 sc - m
    #    bytes by hand: s[0..3] = (sc4..7 >> 4) << 6 = C0 80 40 C0,
    #    s[4..7] = (m4..7 >> 4) << 6 = 80 40 C0 00,
    #    s[8..11] = (sc & 15) | (m & 15) << 4 = 1F 10 F0 20
    blk = q4k_block(0x3C00, 0x3C00,
                    [0xC0, 0x80, 0x40, 0xC0, 0x80, 0x40, 0xC0, 0x00, 0x1F, 0x10, 0xF0, 0x20],
                    [0x22] * 128)
    got = orc.decode_q4_k_block(blk)
    expect = [0.0] * 128 + [93.0] * 32 + [47.0] * 32 + [-31.0] * 32 + [94.0] * 32
    assert got.tolist() == expect

    # C: mins and sign. d = 0.5, dmin = 0.25, sc = 1..8, m = 8..1, q = 3:
    #    w_j = 1.5 sc_j - 0.25 m_j = -0.5, 1.25, 3, 4.75, 6.5, 8.25, 10, 11.75
    blk = q4k_block(0x3800, 0x3400,
                    [1, 2, 3, 4, 8, 7, 6, 5, 0x45, 0x36, 0x27, 0x18], [0x33] * 128)
    got = orc.decode_q4_k_block(blk)
    vals = [-0.5, 1.25, 3.0, 4.75, 6.5, 8.25, 10.0, 11.75]
    assert got.tolist() == [vals[k // 32] for k in range(256)]

    # D: nibble positions.  d = 1, all sc = 1, m = 0; one nibble = 15.
    #    qs[i] low nibble -> weight 64*(i//32) + i%32, high nibble -> +32
    ones = [1, 1, 1, 1, 0, 0, 0, 0, 0x01, 0x01, 0x01, 0x01]
    cases = {(0, 0): 0, (0, 1): 32, (31, 0): 31, (31, 1): 63, (32, 0): 64, (32, 1): 96,
             (70, 0): 134, (70, 1): 166, (127, 0): 223, (127, 1): 255, (100, 0): 196,
             (100, 1): 228}
    for (i, hi), k in cases.items():
        qs = [0] * 128
        qs[i] = 0xF0 if hi else 0x0F
        got = orc.decode_q4_k_block(q4k_block(0x3C00, 0x0000, ones, qs))
        assert got[k] == 15.0 and np.count_nonzero(got) == 1, (i, hi, k)
    # every (byte, nibble) lands on a distinct weight
    seen = set()
    for i in range(128):
        for hi in (0, 1):
            qs = [0] * 128
            qs[i] = 0xF0 if hi else 0x0F
            got = orc.decode_q4_k_block(q4k_block(0x3C00, 0x0000, ones, qs))
            nz = np.flatnonzero(got)
            assert nz.size == 1
            seen.add(int(nz[0]))
    assert seen == set(range(256))

    # E: subnormal d = 2^-24 and dmin = 2^-23, sc = 1 everywhere, m_0 = 1, q = 1:
    #    sub-block 0 -> 2^-24 - 2^-23 = -2^-24, the others -> 2^-24
    blk = q4k_block(0x0001, 0x0002, [1, 1, 1, 1, 1, 0, 0, 0, 0x01, 0x01, 0x01, 0x01],
                    [0x11] * 128)
    got = orc.decode_q4_k_block(blk)
    assert got.tolist() == [-(2.0 ** -24)] * 32 + [2.0 ** -24] * 224
    # F: one rounding only: d*sc*q - dmin*m with d = 1 + 2^-10, sc = 63, q = 15,
    #    dmin = 2^-14 (0x0400), m = 1 -> exact 945.9228515625 - 2^-14, rounded to fp32
    blk = q4k_block(0x3C01, 0x0400, [63, 0, 0, 0, 1, 0, 0, 0, 0, 0, 0, 0], [0x0F] + [0] * 127)
    got = orc.decode_q4_k_block(blk)
    exact = (1 + 2.0 ** -10) * 63 * 15 - 2.0 ** -14
    assert got[0] == np.float32(exact)
    assert orc.row_bytes(Q4_K, 256) == 144 and orc.row_bytes(Q4_K, 4096) == 16 * 144
    assert orc.row_bytes(Q4_K, 128) == 0


# --------------------------------------------------------------- helpers ----

def pack_q4_k(d_bits, dmin_bits, sc, m, q):
    """Test-side packer for hand-chosen 6-bit scales/mins and 4-bit values."""
    s = [0] * 12
    for j in range(4):
        s[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        s[j + 4] = (m[j] & 63) | ((m[j + 4] >> 4) << 6)
        s[j + 8] = (sc[j + 4] & 15) | ((m[j + 4] & 15) << 4)
    qs = [0] * 128
    for c in range(4):
        for l in range(32):
            qs[32 * c + l] = q[64 * c + l] | (q[64 * c + 32 + l] << 4)
    return q4k_block(d_bits, dmin_bits, s, qs)


# ------------------------------------------------------------------- GEMV ----

def check_one_hot(orc):
    """x = e_c extracts column c exactly (every other product is an exact 0)."""
    rows = 3
    # Q8_0, cols 64: row r block b has d = 1 and q[i] = Q8_PATTERN[(i + 5r + 7b) % 32]
    W = b"".join(q8_block(0x3C00, [Q8_PATTERN[(i + 5 * r + 7 * b) % 32] for i in range(32)])
                 for r in range(rows) for b in range(2))
    for c in (0, 1, 31, 32, 45, 63):
        x = np.zeros(64, dtype=np.float32)
        x[c] = 1.0
        y, _ = orc.gemv(Q8_0, np.frombuffer(W, np.uint8), rows, 64, x)
        b, i = divmod(c, 32)
        assert y[0].tolist() == [float(Q8_PATTERN[(i + 5 * r + 7 * b) % 32]) for r in range(rows)]
    # Q4_K, cols 512: super-block (r, b): d = 1, dmin = 1, sc_j = j + 1 + r, m_j = 2b + j,
    # q = (k + r) % 16 -> w[k] = (j+1+r) * ((k+r)%16) - (2b + j), j = (k % 256) // 32
    blocks = []
    for r in range(rows):
        for b in range(2):
            sc = [j + 1 + r for j in range(8)]
            m = [2 * b + j for j in range(8)]
            q = [(k + r) % 16 for k in range(256)]
            blocks.append(pack_q4_k(0x3C00, 0x3C00, sc, m, q))
    W = b"".join(blocks)
    for c in (0, 31, 32, 100, 255, 256, 300, 511):
        x = np.zeros(512, dtype=np.float32)
        x[c] = 1.0
        y, _ = orc.gemv(Q4_K, np.frombuffer(W, np.uint8), rows, 512, x)
        b, k = divmod(c, 256)
        j = k // 32
        assert y[0].tolist() == [float((j + 1 + r) * ((k + r) % 16) - (2 * b + j))
                                 for r in range(rows)], c
    # Q4_0, cols 64: block (r, b) has d = 1 and code (i + 3r + 5b) % 16 for weight i
    W = b"".join(q4_0_block(0x3C00, [(i + 3 * r + 5 * b) % 16 for i in range(32)])
                 for r in range(rows) for b in range(2))
    for c in (0, 15, 16, 31, 32, 47, 63):
        x = np.zeros(64, dtype=np.float32)
        x[c] = 1.0
        y, _ = orc.gemv(Q4_0, np.frombuffer(W, np.uint8), rows, 64, x)
        b, i = divmod(c, 32)
        assert y[0].tolist() == [float((i + 3 * r + 5 * b) % 16 - 8) for r in range(rows)], c
    # Q6_K, cols 512: super-block (r, b) has d = 1, sc_j = j - 8 + r, code (k + 3r + b) % 64
    W = b"".join(q6k_block(0x3C00, [j - 8 + r for j in range(16)], [(k + 3 * r + b) % 64 for k in range(256)])
                 for r in range(rows) for b in range(2))
    for c in (0, 15, 16, 100, 255, 256, 300, 511):
        x = np.zeros(512, dtype=np.float32)
        x[c] = 1.0
        y, _ = orc.gemv(Q6_K, np.frombuffer(W, np.uint8), rows, 512, x)
        b, k = divmod(c, 256)
        assert y[0].tolist() == [float((k // 16 - 8 + r) * ((k + 3 * r + b) % 64 - 32)) for r in range(rows)], c
    # F32, cols 5 (no blocks): element (r, c) = 10r + c
    Wf = np.array([[10.0 * r + c for c in range(5)] for r in range(rows)], dtype=np.float32)
    for c in range(5):
        x = np.zeros(5, dtype=np.float32)
        x[c] = 1.0
        y, _ = orc.gemv(F32, Wf.reshape(-1).view(np.uint8), rows, 5, x)
        assert y[0].tolist() == [10.0 * r + c for r in range(rows)], c


def check_integer_exact(orc):
    """Integer-valued weights and x: every partial sum is an exact integer."""
    rng = np.random.default_rng(7)
    rows, cols, M = 17, 512, 3
    q = rng.integers(-128, 128, size=(rows, cols))
    W = b"".join(q8_block(0x3C00, list(q[r, 32 * b: 32 * b + 32]))
                 for r in range(rows) for b in range(cols // 32))
    x = rng.integers(-8, 9, size=(M, cols))
    y, ay = orc.gemv(Q8_0, np.frombuffer(W, np.uint8), rows, cols, x.astype(np.float32))
    ref = x @ q.T
    assert np.array_equal(y, ref.astype(np.float64))
    assert np.array_equal(ay, (np.abs(x) @ np.abs(q).T).astype(np.float64))
    # Q4_K with d = dmin = 1: w = sc*q - m
    sc = rng.integers(0, 64, size=(rows, cols // 256, 8))
    mm = rng.integers(0, 64, size=(rows, cols // 256, 8))
    qq = rng.integers(0, 16, size=(rows, cols))
    W = b"".join(pack_q4_k(0x3C00, 0x3C00, list(sc[r, b]), list(mm[r, b]),
                           list(qq[r, 256 * b: 256 * b + 256]))
                 for r in range(rows) for b in range(cols // 256))
    j = (np.arange(cols) % 256) // 32
    bidx = np.arange(cols) // 256
    w = sc[:, bidx, j] * qq - mm[:, bidx, j]
    y, _ = orc.gemv(Q4_K, np.frombuffer(W, np.uint8), rows, cols, x.astype(np.float32))
    assert np.array_equal(y, (x @ w.T).astype(np.float64))
    # Q4_0 with d = 1: w = code - 8
    u = rng.integers(0, 16, size=(rows, cols))
    W = b"".join(q4_0_block(0x3C00, list(u[r, 32 * b: 32 * b + 32]))
                 for r in range(rows) for b in range(cols // 32))
    y, ay = orc.gemv(Q4_0, np.frombuffer(W, np.uint8), rows, cols, x.astype(np.float32))
    assert np.array_equal(y, (x @ (u - 8).T).astype(np.float64))
    assert np.array_equal(ay, (np.abs(x) @ np.abs(u - 8).T).astype(np.float64))
    # Q6_K with d = 1: w = sc[k // 16] * (code - 32)
    sc = rng.integers(-128, 128, size=(rows, cols // 256, 16))
    u = rng.integers(0, 64, size=(rows, cols))
    W = b"".join(q6k_block(0x3C00, list(sc[r, b]), list(u[r, 256 * b:256 * b + 256]))
                 for r in range(rows) for b in range(cols // 256))
    w = sc[:, np.arange(cols) // 256, (np.arange(cols) % 256) // 16] * (u - 32)
    y, ay = orc.gemv(Q6_K, np.frombuffer(W, np.uint8), rows, cols, x.astype(np.float32))
    assert np.array_equal(y, (x @ w.T).astype(np.float64))
    assert np.array_equal(ay, (np.abs(x) @ np.abs(w).T).astype(np.float64))
    # F32 integer matrix
    wi = rng.integers(-1000, 1001, size=(rows, cols))
    y, _ = orc.gemv(F32, wi.astype(np.float32).reshape(-1).view(np.uint8), rows, cols, x.astype(np.float32))
    assert np.array_equal(y, (x @ wi.T).astype(np.float64))


def check_brute_force(orc):
    """Tiny shapes: oracle GEMV vs numpy float64 matmul of independently built weights."""
    rng = np.random.default_rng(11)
    for rows in (1, 3, 17):
        for cols in (256, 512, 2048):
            for M in (1, 2, 3, 16):
                # Q8_0 with random fp16 scales
                d = rng.uniform(0.001, 0.01, size=(rows, cols // 32)).astype(np.float16)
                q = rng.integers(-127, 128, size=(rows, cols))
                W = b"".join(struct.pack("<e", d[r, b]) +
                             bytes((int(v) & 0xFF) for v in q[r, 32 * b:32 * b + 32])
                             for r in range(rows) for b in range(cols // 32))
                w = np.repeat(d.astype(np.float64), 32, axis=1) * q
                x = rng.standard_normal((M, cols)).astype(np.float32)
                y, ay = orc.gemv(Q8_0, np.frombuffer(W, np.uint8), rows, cols, x)
                ref = x.astype(np.float64) @ w.T
                assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
                assert np.allclose(ay, np.abs(x.astype(np.float64)) @ np.abs(w).T, rtol=1e-12)
        # Q4_K with random fp16 d / dmin and 6-bit scales
        cols = 512
        d = rng.uniform(1e-4, 1e-3, size=(rows, 2)).astype(np.float16)
        dm = rng.uniform(1e-4, 1e-3, size=(rows, 2)).astype(np.float16)
        sc = rng.integers(0, 64, size=(rows, 2, 8))
        mm = rng.integers(0, 64, size=(rows, 2, 8))
        qq = rng.integers(0, 16, size=(rows, cols))
        W = b"".join(pack_q4_k(int(d[r, b].view(np.uint16)), int(dm[r, b].view(np.uint16)),
                               list(sc[r, b]), list(mm[r, b]), list(qq[r, 256 * b:256 * b + 256]))
                     for r in range(rows) for b in range(2))
        j = (np.arange(cols) % 256) // 32
        bi = np.arange(cols) // 256
        w = (d.astype(np.float64)[:, bi] * sc[:, bi, j] * qq
             - dm.astype(np.float64)[:, bi] * mm[:, bi, j]).astype(np.float32)
        x = rng.standard_normal((2, cols)).astype(np.float32)
        y, _ = orc.gemv(Q4_K, np.frombuffer(W, np.uint8), rows, cols, x)
        assert np.allclose(y, x.astype(np.float64) @ w.astype(np.float64).T, rtol=1e-12, atol=1e-15)
        Wd = orc.dequantize(Q4_K, np.frombuffer(W, np.uint8), rows, cols)
        assert np.array_equal(Wd, w)
        # Q4_0 with random fp16 d, cols 96 (three blocks)
        cols = 96
        d = rng.uniform(1e-3, 1e-2, size=(rows, 3)).astype(np.float16)
        u = rng.integers(0, 16, size=(rows, cols))
        W = b"".join(q4_0_block(int(d[r, b].view(np.uint16)), list(u[r, 32 * b:32 * b + 32]))
                     for r in range(rows) for b in range(3))
        w = np.repeat(d.astype(np.float64), 32, axis=1) * (u - 8)
        x = rng.standard_normal((3, cols)).astype(np.float32)
        y, ay = orc.gemv(Q4_0, np.frombuffer(W, np.uint8), rows, cols, x)
        assert np.allclose(y, x.astype(np.float64) @ w.T, rtol=1e-12, atol=1e-15)
        assert np.allclose(ay, np.abs(x.astype(np.float64)) @ np.abs(w).T, rtol=1e-12)
        assert np.array_equal(orc.dequantize(Q4_0, np.frombuffer(W, np.uint8), rows, cols),
                              w.astype(np.float32))
        # Q6_K with random fp16 d and signed scales, cols 512
        cols = 512
        d = rng.uniform(1e-5, 1e-4, size=(rows, 2)).astype(np.float16)
        sc = rng.integers(-128, 128, size=(rows, 2, 16))
        u = rng.integers(0, 64, size=(rows, cols))
        W = b"".join(q6k_block(int(d[r, b].view(np.uint16)), list(sc[r, b]), list(u[r, 256 * b:256 * b + 256]))
                     for r in range(rows) for b in range(2))
        bi, j = np.arange(cols) // 256, (np.arange(cols) % 256) // 16
        w = d.astype(np.float64)[:, bi] * sc[:, bi, j] * (u - 32)
        x = rng.standard_normal((2, cols)).astype(np.float32)
        y, _ = orc.gemv(Q6_K, np.frombuffer(W, np.uint8), rows, cols, x)
        assert np.allclose(y, x.astype(np.float64) @ w.T, rtol=1e-12, atol=1e-15)
        assert np.array_equal(orc.dequantize(Q6_K, np.frombuffer(W, np.uint8), rows, cols), w.astype(np.float32))
        # F32, cols 7
        wf = rng.standard_normal((rows, 7)).astype(np.float32)
        x = rng.standard_normal((2, 7)).astype(np.float32)
        y, _ = orc.gemv(F32, wf.reshape(-1).view(np.uint8), rows, 7, x)
        assert np.allclose(y, x.astype(np.float64) @ wf.astype(np.float64).T, rtol=1e-12, atol=1e-15)


def check_gemm_bf16(orc):
    """bf16 X is widened exactly: Y = X W^T with X taken as the bf16 values."""
    rng = np.random.default_rng(13)
    rows, cols, M = 5, 256, 4
    q = rng.integers(-127, 128, size=(rows, cols))
    W = b"".join(q8_block(0x3800, list(q[r, 32 * b:32 * b + 32]))
                 for r in range(rows) for b in range(cols // 32))
    xf = rng.standard_normal((M, cols)).astype(np.float32)
    bits = (xf.view(np.uint32) >> 16).astype(np.uint16)      # truncation: any bf16 pattern
    xv = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    Y, _ = orc.gemm_bf16(Q8_0, np.frombuffer(W, np.uint8), rows, cols, bits)
    assert np.allclose(Y, xv @ (0.5 * q).T, rtol=1e-12, atol=1e-12)
    y2, _ = orc.gemv(Q8_0, np.frombuffer(W, np.uint8), rows, cols, xv.astype(np.float32))
    assert np.array_equal(Y, y2)


ALL_CHECKS = [check_fp16, check_bf16, check_q8_0_blocks, check_q4_0_blocks, check_q6_k_blocks, check_q4_k_blocks,
              check_one_hot, check_integer_exact, check_brute_force, check_gemm_bf16]

"""Pins for two oracle parts every parity test leans on (no GPU):

* ``oracle.tolerance_ok`` -- the parity bar |y - y_ref| <= 1e-3 * sum|w x| + 1e-6,
  checked on hand-made cases just inside and just outside the bound, with the
  bound driven by sum|w x| and not by |y_ref| (a cancelling row), NaN and inf
  in the device result, a zero sum|w x| (only the absolute term left) and one
  bad element among good ones;
* ``oracle.read_gguf``'s metadata walk for every value type of the GGUF v3
  table ("GGUF: The File Format...", "What is stored inside a GGUF file": the
  type code tells the reader how many bytes follow), scalars, strings and
  nested arrays, on bytes assembled here field by field.

Each pin is then shown to catch plausible slips planted in a copy of the
oracle's own source (any for all, the bound from |y_ref|, NaN hidden by a
nan-aware max, the array count read as 32 bits, signed/unsigned or width
swaps in the type table)."""
import inspect
import math
import struct
import types

import numpy as np
import pytest

import oracle
from oracle import gguf_reader


# ------------------------------------------------------------ tolerance ----

def check_tolerance(tol_ok):
    # inside: |err| = 1.0 against 1e-3 * 1000 + 1e-6
    ok, worst = tol_ok(np.array([2.0]), np.array([1.0]), np.array([1000.0]))
    assert ok and 0.99 < worst < 1.0
    # outside by 2e-6
    ok, worst = tol_ok(np.array([2.0 + 2e-6]), np.array([1.0]), np.array([1000.0]))
    assert not ok and worst > 1.0
    # the same distance below y_ref
    ok, worst = tol_ok(np.array([-1.0 - 2e-6]), np.array([1.0]), np.array([1000.0]))
    assert not ok and worst > 1.0
    # 1e-2 would let this through; 1e-3 does not
    ok, _ = tol_ok(np.array([3.0]), np.array([1.0]), np.array([1000.0]))
    assert not ok
    # a row whose terms cancel: y_ref = 0, sum|w x| = 1000 -> error 0.5 allowed
    ok, worst = tol_ok(np.array([0.5]), np.array([0.0]), np.array([1000.0]))
    assert ok and abs(worst - 0.5 / (1.0 + 1e-6)) < 1e-9
    # sum|w x| = 0: only the absolute term, 1e-6
    assert tol_ok(np.array([5e-7]), np.array([0.0]), np.array([0.0]))[0]
    assert not tol_ok(np.array([2e-6]), np.array([0.0]), np.array([0.0]))[0]
    # NaN or inf in the device result never passes, and shows in the ratio
    ok, worst = tol_ok(np.array([1.0, np.nan]), np.array([1.0, 1.0]), np.array([10.0, 10.0]))
    assert not ok and not (worst <= 1.0)
    ok, _ = tol_ok(np.array([np.inf]), np.array([1.0]), np.array([10.0]))
    assert not ok
    # one bad element among good ones
    y_ref = np.linspace(-1.0, 1.0, 64)
    a_ref = np.full(64, 10.0)
    y_dev = y_ref.copy()
    assert tol_ok(y_dev, y_ref, a_ref)[0]
    y_dev[37] += 0.02
    ok, worst = tol_ok(y_dev, y_ref, a_ref)
    assert not ok and 1.9 < worst < 2.1
    # exact agreement: ratio 0; empty input passes
    assert tol_ok(y_ref, y_ref, a_ref) == (True, 0.0)
    assert tol_ok(np.zeros(0), np.zeros(0), np.zeros(0))[0]


def test_tolerance_pins():
    check_tolerance(oracle.tolerance_ok)


TOL_MUTANTS = {
    "any_for_all": ("bool(np.all(err <= bound))", "bool(np.any(err <= bound))"),
    "bound_from_y_ref": ("bound = rel * abs_ref + abs_", "bound = rel * np.abs(y_ref) + abs_"),
    "nan_hidden_in_ratio": ("worst = float(np.max(ratio))", "worst = float(np.nanmax(ratio))"),
    "ok_from_nan_aware_max": ("worst = float(np.max(ratio)) if ratio.size else 0.0\n    return bool(np.all(err <= bound)), worst",
                              "worst = float(np.nanmax(ratio)) if ratio.size else 0.0\n    return bool(worst <= 1.0), worst"),
    "rel_1e2": ("rel: float = 1e-3", "rel: float = 1e-2"),
    "abs_term_dropped": ("bound = rel * abs_ref + abs_", "bound = rel * abs_ref"),
    "signed_error": ("err = np.abs(np.asarray(y_dev, dtype=np.float64) - y_ref)",
                     "err = np.asarray(y_dev, dtype=np.float64) - y_ref"),
}


@pytest.mark.parametrize("name", sorted(TOL_MUTANTS))
def test_tolerance_mutant_is_caught(name):
    before, after = TOL_MUTANTS[name]
    src = inspect.getsource(oracle.tolerance_ok)
    assert src.count(before) == 1, name
    ns = {"np": np}
    exec(src.replace(before, after), ns)
    with pytest.raises(AssertionError):
        check_tolerance(ns["tolerance_ok"])


# ------------------------------------------------------- metadata values ----

def _s(text: str) -> bytes:
    b = text.encode()
    return struct.pack("<Q", len(b)) + b


# (key, type code, encoded value bytes, expected value as read)
_KVS = [
    ("t.u8", 0, bytes([0xF3]), 243),
    ("t.i8", 1, bytes([0xF3]), -13),
    ("t.u16", 2, bytes([0x34, 0xF2]), 0xF234),
    ("t.i16", 3, bytes([0x34, 0xF2]), 0xF234 - 0x10000),
    ("t.u32", 4, bytes([0x78, 0x56, 0x34, 0xF2]), 0xF2345678),
    ("t.i32", 5, bytes([0xFE, 0xFF, 0xFF, 0xFF]), -2),
    ("t.f32", 6, bytes([0x00, 0x00, 0xC0, 0x3F]), 1.5),
    ("t.bool", 7, bytes([1]), True),
    ("t.str", 8, struct.pack("<Q", 5) + b"hello", "hello"),
    ("t.u64", 10, bytes([0xEF, 0xCD, 0xAB, 0x89, 0x67, 0x45, 0x23, 0xF1]), 0xF123456789ABCDEF),
    ("t.i64", 11, bytes([0xFD] + [0xFF] * 7), -3),
    ("t.f64", 12, bytes([0, 0, 0, 0, 0, 0, 0x04, 0xC0]), -2.5),
    # array of 3 u16: element type 2, count 3 (8 bytes), elements
    ("t.arr_u16", 9, struct.pack("<IQ", 2, 3) + bytes([1, 0, 0, 1, 0xFF, 0xFF]), (2, [1, 256, 65535])),
    # array of 2 strings
    ("t.arr_str", 9, struct.pack("<IQ", 8, 2) + struct.pack("<Q", 2) + b"en" + struct.pack("<Q", 1) + b"x",
     (8, ["en", "x"])),
    # array of arrays: [[-1 (i8), 2 (i8)], []] then an f32 array [0.25]
    ("t.nested", 9, struct.pack("<IQ", 9, 3) + struct.pack("<IQ", 1, 2) + bytes([0xFF, 0x02])
     + struct.pack("<IQ", 1, 0) + struct.pack("<IQ", 6, 1) + bytes([0, 0, 0x80, 0x3E]),
     (9, [(1, [-1, 2]), (1, []), (6, [0.25])])),
    # empty array of u64
    ("t.empty", 9, struct.pack("<IQ", 10, 0), (10, [])),
]


def _typed_file() -> bytes:
    out = b"GGUF" + struct.pack("<IQQ", 3, 1, len(_KVS))
    for key, code, enc, _ in _KVS:
        out += _s(key) + struct.pack("<I", code) + enc
    out += _s("w") + struct.pack("<I", 1) + struct.pack("<Q", 8) + struct.pack("<IQ", 0, 0)
    out += b"\0" * (-len(out) % 32)
    return out + struct.pack("<8f", *range(8))


def check_reader(read):
    buf = _typed_file()
    r = read(buf)
    assert r["n_kv"] == len(_KVS)
    got = r["kvs"]
    assert [k for k, _, _ in got] == [k for k, _, _, _ in _KVS]
    for (key, code, _, want), (k, t, v) in zip(_KVS, got):
        assert t == code, key
        assert v == want and type(v) is type(want), (key, v, want)
    # the walk ends exactly where the tensor info starts: the tensor reads back
    t = r["tensors"][0]
    assert t["name"] == "w" and t["ne"] == [8] and t["type"] == 0
    assert r["data_start"] % 32 == 0 and r["data_start"] == len(buf) - 32
    assert struct.unpack("<8f", t["data"]) == tuple(float(i) for i in range(8))
    # an unknown type code is an error, not a skip of unknown size
    bad = b"GGUF" + struct.pack("<IQQ", 3, 0, 1) + _s("k") + struct.pack("<I", 13) + b"\0" * 16
    with pytest.raises(ValueError) as e:
        read(bad)
    assert type(e.value).__name__ == "GGUFError"


def test_reader_every_value_type():
    check_reader(oracle.read_gguf)


def _ieee(enc: bytes, ebits: int) -> float:
    """A normal IEEE-754 binary32/64 value from its little-endian bytes:
    sign, biased exponent, implicit leading 1."""
    n = int.from_bytes(enc, "little")
    mbits = len(enc) * 8 - 1 - ebits
    sign = -1.0 if n >> (len(enc) * 8 - 1) else 1.0
    e = (n >> mbits) & ((1 << ebits) - 1)
    m = n & ((1 << mbits) - 1)
    return sign * math.ldexp(1.0 + m / (1 << mbits), e - ((1 << (ebits - 1)) - 1))


def test_typed_values_are_what_the_bytes_say():
    """The expected values above, cross-checked from the same bytes by
    fixed-width integer decoding and the IEEE-754 field layout."""
    for key, code, enc, want in _KVS:
        if code in (0, 2, 4, 10):
            assert want == int.from_bytes(enc, "little"), key
        elif code in (1, 3, 5, 11):
            assert want == int.from_bytes(enc, "little", signed=True), key
        elif code == 6:
            assert want == _ieee(enc, 8), key
        elif code == 12:
            assert want == _ieee(enc, 11), key


READER_MUTANTS = {
    "array_count_u32": ('etype, count = self.take("<I"), self.take("<Q")',
                        'etype, count = self.take("<I"), self.take("<I")'),
    "array_etype_u64": ('etype, count = self.take("<I"), self.take("<Q")',
                        'etype, count = self.take("<Q"), self.take("<Q")'),
    "i8_unsigned": ('1: "<b"', '1: "<B"'),
    "u16_signed": ('2: "<H"', '2: "<h"'),
    "i32_unsigned": ('5: "<i"', '5: "<I"'),
    "f32_as_i32": ('6: "<f"', '6: "<i"'),
    "bool_wide": ('7: "<?"', '7: "<I"'),
    "u64_signed": ('10: "<Q"', '10: "<q"'),
    "f64_as_f32x2": ('12: "<d"', '12: "<ff"'),
    "string_len_u32": ('n = self.take("<Q")\n        if self.pos + n', 'n = self.take("<I")\n        if self.pos + n'),
    "nested_elem_type_ignored": ("[self.value(etype, depth + 1) for _ in range(count)]",
                                 "[self.value(4, depth + 1) for _ in range(count)]"),
}


@pytest.mark.parametrize("name", sorted(READER_MUTANTS))
def test_reader_mutant_is_caught(name):
    before, after = READER_MUTANTS[name]
    src = inspect.getsource(gguf_reader)
    assert src.count(before) == 1, name
    mod = types.ModuleType(f"mutant_{name}")
    exec(src.replace(before, after), mod.__dict__)
    with pytest.raises((AssertionError, struct.error, ValueError, UnicodeDecodeError, OverflowError)):
        check_reader(mod.read_gguf)

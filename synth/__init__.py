"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

Holds input generation only (no decode, no dot products):

* ``normal_f32`` / ``normal_bf16`` -- counter-based N(0, sigma) draws;
* ``weight_rows`` -- rows of a seeded weight tensor, encoded to Q8_0 (34 B /
  32 weights), Q4_K (144 B / 256 weights), Q4_0 (18 B / 32 weights) or Q6_K
  (210 B / 256 weights) bytes, or stored as F32;
* ``quantize_q8_0`` / ``quantize_q4_k`` / ``quantize_q4_0`` /
  ``quantize_q6_k`` -- the same encoders on given floats;
* ``write_gguf`` -- a GGUF v3 writer (header, typed KVs, tensor-info table,
  32-byte padding, 32-byte-aligned payloads), laid out as in "GGUF: The File
  Format..." (section "What is stored inside a GGUF file") and the byte
  blueprint of "GGUF Inferencer in R" section 2.1;
* ``workloads`` -- the shapes of the benchmark configurations.

The C part is built in-tree on first use (gcc, OpenMP, -ffp-contract=off).
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import struct
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ggq_synth.c")
_LIB = os.path.join(_HERE, "libggq_synth.so")
_lock = threading.Lock()
_lib = None

BASE_SEED = 20261202


def build(force: bool = False) -> str:
    """Compile libggq_synth.so next to its source (idempotent)."""
    with _lock:
        if (not force and os.path.exists(_LIB)
                and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
            return _LIB
        tmp = _LIB + ".tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
        return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        u64, i64, f32, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
        lib.synth_normal_f32.argtypes = [u64, u64, u64, i64, f32, vp]
        lib.synth_normal_bf16.argtypes = [u64, u64, u64, i64, f32, vp]
        lib.synth_quantize_q8_0.argtypes = [vp, i64, vp]
        lib.synth_quantize_q4_k.argtypes = [vp, i64, vp]
        lib.synth_quantize_q4_0.argtypes = [vp, i64, vp]
        lib.synth_quantize_q6_k.argtypes = [vp, i64, vp]
        lib.synth_q6_k_rows.argtypes = [u64, u64, i64, i64, i64, f32, vp]
        lib.synth_q8_0_rows.argtypes = [u64, u64, i64, i64, i64, f32, vp]
        lib.synth_q4_k_rows.argtypes = [u64, u64, i64, i64, i64, f32, vp]
        lib.synth_q4_0_rows.argtypes = [u64, u64, i64, i64, i64, f32, vp]
        lib.synth_f32_rows.argtypes = [u64, u64, i64, i64, i64, f32, vp]
        lib.synth_f32_to_f16_array.argtypes = [vp, i64, vp]
        lib.synth_f32_to_bf16_array.argtypes = [vp, i64, vp]
        lib.synth_set_threads.argtypes = [ctypes.c_int]
        lib.synth_mix64.argtypes = [u64]
        lib.synth_mix64.restype = u64
        _lib = lib
    return _lib


def set_threads(n: int) -> None:
    _load().synth_set_threads(int(n))


def stream_id(*parts) -> int:
    """Stable 64-bit stream id for a tensor name / config tuple."""
    h = hashlib.sha256("/".join(str(p) for p in parts).encode()).digest()
    return int.from_bytes(h[:8], "little")


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


QK8_0, Q8_0_BYTES = 32, 34
QK_K, Q4_K_BYTES = 256, 144
QK4_0, Q4_0_BYTES = 32, 18
Q6_K_BYTES = 210
TYPE_F32, TYPE_F16, TYPE_Q4_0, TYPE_Q8_0, TYPE_Q4_K, TYPE_Q6_K = 0, 1, 2, 8, 12, 14


def row_bytes(qtype: int, cols: int) -> int:
    if qtype == TYPE_Q8_0:
        return cols // QK8_0 * Q8_0_BYTES
    if qtype == TYPE_Q4_K:
        return cols // QK_K * Q4_K_BYTES
    if qtype == TYPE_Q4_0:
        return cols // QK4_0 * Q4_0_BYTES
    if qtype == TYPE_Q6_K:
        return cols // QK_K * Q6_K_BYTES
    if qtype == TYPE_F32:
        return cols * 4
    raise ValueError(f"unsupported type {qtype}")


def normal_f32(n: int, stream: int, sigma: float = 1.0, seed: int = BASE_SEED,
               first: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    _load().synth_normal_f32(seed, stream, first, n, sigma, _ptr(out))
    return out


def normal_bf16(n: int, stream: int, sigma: float = 1.0, seed: int = BASE_SEED,
                first: int = 0) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(0, sigma) draws."""
    out = np.empty(n, dtype=np.uint16)
    _load().synth_normal_bf16(seed, stream, first, n, sigma, _ptr(out))
    return out


def quantize_q8_0(w: np.ndarray) -> np.ndarray:
    w = np.ascontiguousarray(w, dtype=np.float32).reshape(-1)
    assert w.size % QK8_0 == 0
    out = np.empty(w.size // QK8_0 * Q8_0_BYTES, dtype=np.uint8)
    _load().synth_quantize_q8_0(_ptr(w), w.size, _ptr(out))
    return out


def quantize_q4_k(w: np.ndarray) -> np.ndarray:
    w = np.ascontiguousarray(w, dtype=np.float32).reshape(-1)
    assert w.size % QK_K == 0
    out = np.empty(w.size // QK_K * Q4_K_BYTES, dtype=np.uint8)
    _load().synth_quantize_q4_k(_ptr(w), w.size, _ptr(out))
    return out


def quantize_q4_0(w: np.ndarray) -> np.ndarray:
    w = np.ascontiguousarray(w, dtype=np.float32).reshape(-1)
    assert w.size % QK4_0 == 0
    out = np.empty(w.size // QK4_0 * Q4_0_BYTES, dtype=np.uint8)
    _load().synth_quantize_q4_0(_ptr(w), w.size, _ptr(out))
    return out


def quantize_q6_k(w: np.ndarray) -> np.ndarray:
    w = np.ascontiguousarray(w, dtype=np.float32).reshape(-1)
    assert w.size % QK_K == 0
    out = np.empty(w.size // QK_K * Q6_K_BYTES, dtype=np.uint8)
    _load().synth_quantize_q6_k(_ptr(w), w.size, _ptr(out))
    return out


def weight_rows(qtype: int, stream: int, rows: int, cols: int, row0: int = 0,
                sigma: float = 0.02, seed: int = BASE_SEED,
                out: np.ndarray | None = None) -> np.ndarray:
    """Encoded bytes of rows [row0, row0+rows) of a seeded rows x cols tensor."""
    nb = rows * row_bytes(qtype, cols)
    if out is None:
        out = np.empty(nb, dtype=np.uint8)
    assert out.dtype == np.uint8 and out.size >= nb and out.flags["C_CONTIGUOUS"]
    lib = _load()
    if qtype == TYPE_Q8_0:
        lib.synth_q8_0_rows(seed, stream, row0, rows, cols, sigma, _ptr(out))
    elif qtype == TYPE_Q4_K:
        lib.synth_q4_k_rows(seed, stream, row0, rows, cols, sigma, _ptr(out))
    elif qtype == TYPE_Q4_0:
        lib.synth_q4_0_rows(seed, stream, row0, rows, cols, sigma, _ptr(out))
    elif qtype == TYPE_Q6_K:
        lib.synth_q6_k_rows(seed, stream, row0, rows, cols, sigma, _ptr(out))
    elif qtype == TYPE_F32:
        lib.synth_f32_rows(seed, stream, row0, rows, cols, sigma, _ptr(out))
    else:
        raise ValueError(f"unsupported type {qtype}")
    return out[:nb]


def f32_to_f16_bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32).reshape(-1)
    out = np.empty(a.size, dtype=np.uint16)
    _load().synth_f32_to_f16_array(_ptr(a), a.size, _ptr(out))
    return out


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32).reshape(-1)
    out = np.empty(a.size, dtype=np.uint16)
    _load().synth_f32_to_bf16_array(_ptr(a), a.size, _ptr(out))
    return out


# ------------------------------------------------------------------ GGUF ----

# metadata value types (GGUF v3): fixed-size scalars by code
KV_SCALAR = {0: "<B", 1: "<b", 2: "<H", 3: "<h", 4: "<I", 5: "<i", 6: "<f",
             7: "<?", 10: "<Q", 11: "<q", 12: "<d"}
KV_STRING, KV_ARRAY = 8, 9


def gguf_string(s: str | bytes) -> bytes:
    b = s.encode() if isinstance(s, str) else s
    return struct.pack("<Q", len(b)) + b


def _kv_value(vtype: int, value) -> bytes:
    if vtype in KV_SCALAR:
        return struct.pack(KV_SCALAR[vtype], value)
    if vtype == KV_STRING:
        return gguf_string(value)
    if vtype == KV_ARRAY:
        etype, items = value
        out = struct.pack("<IQ", etype, len(items))
        for it in items:
            out += _kv_value(etype, it)
        return out
    raise ValueError(f"bad kv type {vtype}")


def tensor_nbytes(qtype: int, ne) -> int:
    n = 1
    for e in ne:
        n *= int(e)
    if qtype == TYPE_F32:
        return 4 * n
    if qtype == TYPE_F16:
        return 2 * n
    if qtype == TYPE_Q8_0:
        return n // QK8_0 * Q8_0_BYTES
    if qtype == TYPE_Q4_K:
        return n // QK_K * Q4_K_BYTES
    if qtype == TYPE_Q4_0:
        return n // 32 * 18
    if qtype == TYPE_Q6_K:
        return n // 256 * 210
    raise ValueError(f"unsupported type {qtype}")


def gguf_header(kvs, tensors, alignment: int = 32):
    """Header bytes (up to and including the padding) and the payload offsets.

    kvs: [(key, vtype, value)]; tensors: [(name, ne (fastest first), qtype)].
    Offsets are relative to the start of the data blob; each is the previous
    tensor's end rounded up to `alignment`.
    """
    out = b"GGUF" + struct.pack("<IQQ", 3, len(tensors), len(kvs))
    for key, vtype, value in kvs:
        out += gguf_string(key) + struct.pack("<I", vtype) + _kv_value(vtype, value)
    offsets, off = [], 0
    for name, ne, qtype in tensors:
        off = (off + alignment - 1) // alignment * alignment
        offsets.append(off)
        out += gguf_string(name) + struct.pack("<I", len(ne))
        out += struct.pack(f"<{len(ne)}Q", *[int(e) for e in ne])
        out += struct.pack("<IQ", qtype, off)
        off += tensor_nbytes(qtype, ne)
    out += b"\0" * (-len(out) % alignment)
    return out, offsets, off


def write_gguf(path, kvs, tensors, payloads, alignment: int = 32) -> int:
    """Write a GGUF v3 file; payloads[i] is a bytes-like of tensor i. Returns size."""
    head, offsets, end = gguf_header(kvs, tensors, alignment)
    with open(path, "wb") as f:
        f.write(head)
        pos = 0
        for off, p in zip(offsets, payloads):
            if off > pos:
                f.write(b"\0" * (off - pos))
                pos = off
            mv = memoryview(p).cast("B")
            f.write(mv)
            pos += mv.nbytes
        if end > pos:
            f.write(b"\0" * (end - pos))
    return len(head) + end

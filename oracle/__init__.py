"""CPU oracle for the block-quantized dequantize + GEMV path.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / ``--impl reference`` leg may import this package.
The CUDA library (``gguf_block_quantized_q8_gb300``) never imports it and
shares no code with it; the two meet only on input bytes from ``synth``.

* ``ggq_oracle.c`` -- fp16 decode from IEEE-754, Q8_0 / Q4_K / Q4_0 / Q6_K block decode to
  fp32, GEMV / GEMM with every product and sum in double (see its header for
  the passages followed);
* ``gguf_reader.py`` -- a plain byte walk of GGUF v3;
* ``layer_ops.py`` -- RMSNorm, SiLU(gate) * up and the residual add in float64,
  the element-wise steps the chain fuses into its GEMV stages.

Parity status: fp16 decode, Q8_0 decode, GEMV/GEMM and the GGUF reader are
pinned by the tests in tests/test_oracle_pins.py.  Q4_K decode is pinned by
closed-form hand-built super-blocks for the byte layout read here; no page
prints a Q4_K block, so agreement with Q4_K files made by other tools is
unpinned (the path and the oracle decode the same bytes either way).  Q4_0
decode is pinned the same way and, beyond that, against the Q8_0 decode: a
Q4_0 block and a Q8_0 block holding the same scale and the same integers
decode to the same 32 values.  Which nibble holds which weight, and the offset
of 8, are a reading of the format (real Q4_0 files), not on the pages.  Q6_K:
only the size (210 bytes per 256 weights) and the k-quant idea are on the pages;
its byte layout is a reading (real Q6_K files), pinned by hand-built
super-blocks and against the Q8_0 decode (a Q6_K super-block with unit
sub-block scales equals eight Q8_0 blocks of the same scale and integers).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .gguf_reader import GGUFError, read_gguf, tensor_nbytes  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ggq_oracle.c")
_LIB = os.path.join(_HERE, "libggq_oracle.so")
_lock = threading.Lock()
_lib = None

F32, F16, Q4_0, Q8_0, Q4_K, Q6_K = 0, 1, 2, 8, 12, 14


def compile_oracle(src: str, out: str) -> str:
    """gcc the oracle source `src` into shared library `out`."""
    tmp = out + ".tmp"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-fno-fast-math", src, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile libggq_oracle.so next to its source (idempotent)."""
    with _lock:
        if (not force and os.path.exists(_LIB)
                and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
            return _LIB
        return compile_oracle(_SRC, _LIB)


SOURCE = _SRC


class Oracle:
    """Bound to one compiled oracle library (the default one, or a test build)."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        i64, vp = ctypes.c_int64, ctypes.c_void_p
        lib.orc_fp16_value.argtypes = [ctypes.c_uint16]
        lib.orc_fp16_value.restype = ctypes.c_double
        lib.orc_bf16_value.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_value.restype = ctypes.c_double
        lib.orc_decode_q8_0_block.argtypes = [vp, vp]
        lib.orc_decode_q4_k_block.argtypes = [vp, vp]
        lib.orc_decode_q4_0_block.argtypes = [vp, vp]
        lib.orc_decode_q6_k_block.argtypes = [vp, vp]
        lib.orc_row_bytes.argtypes = [ctypes.c_int, i64]
        lib.orc_row_bytes.restype = i64
        lib.orc_dequantize.argtypes = [ctypes.c_int, vp, i64, i64, vp]
        lib.orc_gemv.argtypes = [ctypes.c_int, vp, i64, i64, vp, i64, vp, vp]
        lib.orc_gemm_bf16.argtypes = [ctypes.c_int, vp, i64, i64, vp, i64, vp, vp]
        self.lib = lib

    def fp16_value(self, h: int) -> float:
        return self.lib.orc_fp16_value(int(h) & 0xFFFF)

    def bf16_value(self, b: int) -> float:
        return self.lib.orc_bf16_value(int(b) & 0xFFFF)

    def row_bytes(self, qtype: int, cols: int) -> int:
        return int(self.lib.orc_row_bytes(qtype, cols))

    def dequantize(self, qtype: int, W: np.ndarray, rows: int, cols: int) -> np.ndarray:
        """fp32 [rows, cols] decoded weights."""
        W = _c(W, np.uint8).reshape(-1)
        rb = self.row_bytes(qtype, cols)
        if rb == 0 or W.size < rows * rb:
            raise ValueError("bad shape for type")
        out = np.empty((rows, cols), dtype=np.float32)
        if self.lib.orc_dequantize(qtype, W.ctypes.data, rows, cols, out.ctypes.data):
            raise ValueError("oracle dequantize failed")
        return out

    def gemv(self, qtype: int, W: np.ndarray, rows: int, cols: int, x: np.ndarray):
        """(y, abs_y): float64 [M, rows] each; x is fp32 [M, cols] (or [cols])."""
        W = _c(W, np.uint8).reshape(-1)
        x = _c(x, np.float32).reshape(-1, cols)
        M = x.shape[0]
        rb = self.row_bytes(qtype, cols)
        if rb == 0 or W.size < rows * rb:
            raise ValueError("bad shape for type")
        y = np.empty((M, rows), dtype=np.float64)
        ay = np.empty((M, rows), dtype=np.float64)
        if self.lib.orc_gemv(qtype, W.ctypes.data, rows, cols, x.ctypes.data, M,
                             y.ctypes.data, ay.ctypes.data):
            raise ValueError("oracle gemv failed")
        return y, ay

    def gemm_bf16(self, qtype: int, W: np.ndarray, rows: int, cols: int, X_bits: np.ndarray):
        """(Y, abs_Y): float64 [M, rows]; X_bits is uint16 bf16 patterns [M, cols]."""
        W = _c(W, np.uint8).reshape(-1)
        X_bits = _c(X_bits, np.uint16).reshape(-1, cols)
        M = X_bits.shape[0]
        rb = self.row_bytes(qtype, cols)
        if rb == 0 or W.size < rows * rb:
            raise ValueError("bad shape for type")
        Y = np.empty((M, rows), dtype=np.float64)
        aY = np.empty((M, rows), dtype=np.float64)
        if self.lib.orc_gemm_bf16(qtype, W.ctypes.data, rows, cols, X_bits.ctypes.data, M,
                                  Y.ctypes.data, aY.ctypes.data):
            raise ValueError("oracle gemm failed")
        return Y, aY

    def decode_q8_0_block(self, blk: bytes) -> np.ndarray:
        b = np.frombuffer(bytes(blk), dtype=np.uint8)
        assert b.size == 34
        out = np.empty(32, dtype=np.float32)
        self.lib.orc_decode_q8_0_block(b.ctypes.data, out.ctypes.data)
        return out

    def decode_q4_k_block(self, blk: bytes) -> np.ndarray:
        b = np.frombuffer(bytes(blk), dtype=np.uint8)
        assert b.size == 144
        out = np.empty(256, dtype=np.float32)
        self.lib.orc_decode_q4_k_block(b.ctypes.data, out.ctypes.data)
        return out

    def decode_q6_k_block(self, blk: bytes) -> np.ndarray:
        b = np.frombuffer(bytes(blk), dtype=np.uint8)
        assert b.size == 210
        out = np.empty(256, dtype=np.float32)
        self.lib.orc_decode_q6_k_block(b.ctypes.data, out.ctypes.data)
        return out

    def decode_q4_0_block(self, blk: bytes) -> np.ndarray:
        b = np.frombuffer(bytes(blk), dtype=np.uint8)
        assert b.size == 18
        out = np.empty(32, dtype=np.float32)
        self.lib.orc_decode_q4_0_block(b.ctypes.data, out.ctypes.data)
        return out


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def default() -> Oracle:
    """The oracle compiled from ggq_oracle.c (built on first use)."""
    global _lib
    if _lib is None:
        build()
        _lib = Oracle(_LIB)
    return _lib


def fp16_value(h):
    return default().fp16_value(h)


def bf16_value(b):
    return default().bf16_value(b)


def row_bytes(qtype, cols):
    return default().row_bytes(qtype, cols)


def dequantize(qtype, W, rows, cols):
    return default().dequantize(qtype, W, rows, cols)


def gemv(qtype, W, rows, cols, x):
    return default().gemv(qtype, W, rows, cols, x)


def gemm_bf16(qtype, W, rows, cols, X_bits):
    return default().gemm_bf16(qtype, W, rows, cols, X_bits)


def decode_q8_0_block(blk):
    return default().decode_q8_0_block(blk)


def decode_q4_k_block(blk):
    return default().decode_q4_k_block(blk)


def decode_q4_0_block(blk):
    return default().decode_q4_0_block(blk)


def decode_q6_k_block(blk):
    return default().decode_q6_k_block(blk)


def _widen_bf16(X_bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64, exactly (the pattern is the top half of an
    IEEE binary32)."""
    b = np.ascontiguousarray(X_bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def gemv_dense(qtype, W, rows, cols, x, chunk=16384):
    """The same quantities as gemv -- y[m, r] = sum_c w[r, c] x[m, c] and
    sum_c |w[r, c] x[m, c]| in float64 -- for full-size matrices: the weights
    decoded exactly by the oracle (dequantize), widened to float64, then one
    float64 matrix product per block of rows (the plain definition y = W x,
    in another summation order than gemv's column loop)."""
    W = _c(W, np.uint8).reshape(-1)
    x64 = _c(x, np.float32).reshape(-1, cols).astype(np.float64)
    M = x64.shape[0]
    rb = row_bytes(qtype, cols)
    y = np.empty((M, rows), dtype=np.float64)
    ay = np.empty((M, rows), dtype=np.float64)
    ax = np.abs(x64)
    for r0 in range(0, rows, chunk):
        n = min(chunk, rows - r0)
        w = dequantize(qtype, W[r0 * rb:(r0 + n) * rb], n, cols).astype(np.float64)
        y[:, r0:r0 + n] = x64 @ w.T
        ay[:, r0:r0 + n] = ax @ np.abs(w).T
    return y, ay


def gemm_bf16_dense(qtype, W, rows, cols, X_bits, chunk=8192):
    """gemm_bf16 for full-size matrices, as gemv_dense: decoded weights times
    the exactly widened bf16 activations, in float64."""
    W = _c(W, np.uint8).reshape(-1)
    X64 = _widen_bf16(np.asarray(X_bits).reshape(-1, cols))
    M = X64.shape[0]
    rb = row_bytes(qtype, cols)
    Y = np.empty((M, rows), dtype=np.float64)
    aY = np.empty((M, rows), dtype=np.float64)
    aX = np.abs(X64)
    for r0 in range(0, rows, chunk):
        n = min(chunk, rows - r0)
        w = dequantize(qtype, W[r0 * rb:(r0 + n) * rb], n, cols).astype(np.float64)
        Y[:, r0:r0 + n] = X64 @ w.T
        aY[:, r0:r0 + n] = aX @ np.abs(w).T
    return Y, aY


def tolerance_ok(y_dev: np.ndarray, y_ref: np.ndarray, abs_ref: np.ndarray,
                 rel: float = 1e-3, abs_: float = 1e-6):
    """|y - y_ref| <= rel * sum|w x| + abs_, elementwise. Returns (ok, worst ratio).

    Every element must be within its bound; a NaN or inf anywhere in y_dev
    fails, and the worst ratio is then NaN or inf too (never hidden)."""
    err = np.abs(np.asarray(y_dev, dtype=np.float64) - y_ref)
    bound = rel * abs_ref + abs_
    ratio = err / bound
    worst = float(np.max(ratio)) if ratio.size else 0.0
    return bool(np.all(err <= bound)), worst

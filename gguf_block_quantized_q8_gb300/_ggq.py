"""ctypes binding of libggq.so (include/ggq.h): argument marshalling only.

Every entry point of the C ABI is exposed under its own name.  The torch
helpers below accept CUDA tensors and pass their data pointers and the current
stream; torch is used for device memory and streams only.  If the shared
library is missing or cannot be loaded, importing this module raises: there is
no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

OK, EINVAL, ETYPE, EIO, EFORMAT, ENOMEM, ECUDA, ETIMEOUT, ENOTFOUND = 0, -1, -2, -3, -4, -5, -6, -7, -8
F32, F16, Q4_0, Q8_0, Q4_K, Q6_K = 0, 1, 2, 8, 12, 14
LOAD_METADATA_ONLY = 1


class GGQError(RuntimeError):
    def __init__(self, code: int, where: str, message: str):
        super().__init__(f"{where}: {message} (code {code})")
        self.code = code


class Tensor(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("type", ctypes.c_int32), ("n_dims", ctypes.c_int32),
                ("ne", ctypes.c_int64 * 4), ("offset", ctypes.c_uint64), ("nbytes", ctypes.c_uint64),
                ("data", ctypes.c_void_p)]


class ChainStage(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int), ("W", ctypes.c_void_p * 4), ("rows", ctypes.c_int64 * 4),
                ("cols", ctypes.c_int64), ("x", ctypes.c_void_p), ("y", ctypes.c_void_p * 4)]


X_PLAIN, X_RMSNORM, X_SILU_MUL = 0, 1, 2


class ChainOps(ctypes.Structure):
    _fields_ = [("x_op", ctypes.c_int), ("eps", ctypes.c_float), ("norm_w", ctypes.c_void_p),
                ("up", ctypes.c_void_p), ("res", ctypes.c_void_p * 4)]


def _bind(lib):
    vp, i64, u64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int32
    sig = {
        "ggq_load": ([ctypes.c_char_p, ctypes.POINTER(vp)], ctypes.c_int),
        "ggq_load_ex": ([ctypes.c_char_p, ctypes.c_uint, ctypes.POINTER(vp)], ctypes.c_int),
        "ggq_load_memory": ([vp, ctypes.c_size_t, ctypes.c_uint, ctypes.POINTER(vp)], ctypes.c_int),
        "ggq_free": ([vp], None),
        "ggq_version_of": ([vp, ctypes.POINTER(ctypes.c_uint32)], ctypes.c_int),
        "ggq_data_start": ([vp, ctypes.POINTER(u64)], ctypes.c_int),
        "ggq_num_tensors": ([vp, ctypes.POINTER(i64)], ctypes.c_int),
        "ggq_tensor_info": ([vp, i64, ctypes.POINTER(Tensor)], ctypes.c_int),
        "ggq_find_tensor": ([vp, ctypes.c_char_p, ctypes.POINTER(i64)], ctypes.c_int),
        "ggq_num_kv": ([vp, ctypes.POINTER(i64)], ctypes.c_int),
        "ggq_kv_info": ([vp, i64, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(i32),
                         ctypes.POINTER(vp), ctypes.POINTER(u64)], ctypes.c_int),
        "ggq_kv_find": ([vp, ctypes.c_char_p, ctypes.POINTER(i64)], ctypes.c_int),
        "ggq_gemv": ([ctypes.c_int, vp, i64, i64, vp, vp, ctypes.c_int, vp], ctypes.c_int),
        "ggq_gemv_multi": ([ctypes.c_int, ctypes.c_int, ctypes.POINTER(vp), ctypes.POINTER(i64), i64, vp,
                            ctypes.POINTER(vp), ctypes.c_int, vp], ctypes.c_int),
        "ggq_gemv_noalloc": ([ctypes.c_int, vp, i64, i64, vp, vp, ctypes.c_int, vp], ctypes.c_int),
        "ggq_chain_create": ([ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ChainStage),
                              ctypes.POINTER(vp)], ctypes.c_int),
        "ggq_chain_create_ops": ([ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ChainStage),
                                  ctypes.POINTER(ChainOps), ctypes.POINTER(vp)], ctypes.c_int),
        "ggq_chain_create_typed": ([ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ChainStage),
                                    ctypes.POINTER(ChainOps), ctypes.POINTER(vp)], ctypes.c_int),
        "ggq_chain_run": ([vp, vp], ctypes.c_int),
        "ggq_embed": ([ctypes.c_int, vp, i64, i64, vp, ctypes.c_int, vp, vp], ctypes.c_int),
        "ggq_chain_reset": ([vp], ctypes.c_int),
        "ggq_chain_free": ([vp], None),
        "ggq_gemm_prefill": ([ctypes.c_int, vp, i64, i64, vp, vp, ctypes.c_int, vp], ctypes.c_int),
        "ggq_dequantize": ([ctypes.c_int, vp, i64, i64, vp, vp], ctypes.c_int),
        "ggq_device_status": ([], ctypes.c_int),
        "ggq_strerror": ([ctypes.c_int], ctypes.c_char_p),
        "ggq_last_error": ([], ctypes.c_char_p),
        "ggq_abi_version": ([], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


def _load():
    path = _build.LIB
    if _build.is_stale():
        if os.environ.get("GGQ_NO_AUTOBUILD"):
            raise ImportError(f"{path} is missing or stale; run __graft_entry__.build()")
        _build.build()
    return _bind(ctypes.CDLL(path))


lib = _load()
LIB_PATH = _build.LIB


def check(rc: int, where: str) -> None:
    if rc != OK:
        msg = lib.ggq_last_error().decode(errors="replace") or lib.ggq_strerror(rc).decode()
        raise GGQError(rc, where, msg)


def strerror(code: int) -> str:
    return lib.ggq_strerror(code).decode()


# ------------------------------------------------------------------ raw calls

def ggq_gemv(qtype: int, W: int, rows: int, cols: int, x: int, y: int, M: int, stream: int) -> int:
    return lib.ggq_gemv(qtype, W, rows, cols, x, y, M, stream)


def ggq_gemv_noalloc(qtype: int, W: int, rows: int, cols: int, x: int, y: int, M: int, stream: int) -> int:
    return lib.ggq_gemv_noalloc(qtype, W, rows, cols, x, y, M, stream)


def ggq_gemv_multi(qtype: int, Ws, rows, cols: int, x: int, ys, M: int, stream: int) -> int:
    n = len(Ws)
    Wa = (ctypes.c_void_p * n)(*Ws)
    ra = (ctypes.c_int64 * n)(*rows)
    ya = (ctypes.c_void_p * n)(*ys)
    return lib.ggq_gemv_multi(qtype, n, Wa, ra, cols, x, ya, M, stream)


def _chain_arrays(stages, ops):
    arr = (ChainStage * len(stages))()
    for i, (Ws, rows, cols, x, ys) in enumerate(stages):
        st = arr[i]
        st.n = len(Ws)                     # n > 4 is passed through for the library to reject
        for j in range(min(len(Ws), 4)):
            st.W[j] = Ws[j]
            st.rows[j] = rows[j]
            st.y[j] = ys[j]
        st.cols = cols
        st.x = x
    if ops is None:
        return arr, None
    oa = (ChainOps * len(stages))()
    for i, o in enumerate(ops):
        if not o:
            continue
        oa[i].x_op = o.get("x_op", X_PLAIN)
        oa[i].eps = o.get("eps", 0.0)
        oa[i].norm_w = o.get("norm_w") or None
        oa[i].up = o.get("up") or None
        for j, r in enumerate((o.get("res") or [])[:4]):
            oa[i].res[j] = r or None
    return arr, oa


def ggq_chain_create(qtype: int, M: int, stages, ops=None) -> tuple[int, int]:
    """stages: sequence of (Ws, rows, cols, x, ys) with device pointers; ops: None, or
    per stage None or a dict with keys x_op, eps, norm_w, up, res (a list of up to 4
    pointers or None), pointers as ints; returns (rc, handle)."""
    arr, oa = _chain_arrays(stages, ops)
    h = ctypes.c_void_p()
    if oa is None:
        rc = lib.ggq_chain_create(qtype, M, len(stages), arr, ctypes.byref(h))
    else:
        rc = lib.ggq_chain_create_ops(qtype, M, len(stages), arr, oa, ctypes.byref(h))
    return rc, (h.value or 0)


def ggq_chain_create_typed(M: int, types, stages, ops=None) -> tuple[int, int]:
    """ggq_chain_create with one weight type per stage (types[s] for stages[s])."""
    arr, oa = _chain_arrays(stages, ops)
    ta = (ctypes.c_int * len(stages))(*[int(t) for t in types][:len(stages)])
    h = ctypes.c_void_p()
    rc = lib.ggq_chain_create_typed(M, len(stages), ta, arr, oa, ctypes.byref(h))
    return rc, (h.value or 0)


def ggq_chain_run(chain: int, stream: int) -> int:
    return lib.ggq_chain_run(chain, stream)


def ggq_chain_reset(chain: int) -> int:
    return lib.ggq_chain_reset(chain)


def ggq_chain_free(chain: int) -> None:
    lib.ggq_chain_free(chain)


def ggq_gemm_prefill(qtype: int, W: int, rows: int, cols: int, X: int, Y: int, M: int, stream: int) -> int:
    return lib.ggq_gemm_prefill(qtype, W, rows, cols, X, Y, M, stream)


def ggq_dequantize(qtype: int, W: int, rows: int, cols: int, out: int, stream: int) -> int:
    return lib.ggq_dequantize(qtype, W, rows, cols, out, stream)


def ggq_device_status() -> int:
    return lib.ggq_device_status()


# --------------------------------------------------------------- model handle

class Model:
    """A loaded GGUF file (ggq_load / ggq_load_memory); payloads live on the device."""

    def __init__(self, handle: int):
        self._h = ctypes.c_void_p(handle)

    @classmethod
    def load(cls, path: str, metadata_only: bool = False) -> "Model":
        h = ctypes.c_void_p()
        check(lib.ggq_load_ex(path.encode(), LOAD_METADATA_ONLY if metadata_only else 0, ctypes.byref(h)),
              "ggq_load")
        return cls(h.value)

    @classmethod
    def from_bytes(cls, buf: bytes, metadata_only: bool = False) -> "Model":
        h = ctypes.c_void_p()
        b = ctypes.create_string_buffer(bytes(buf), len(buf)) if buf else None
        check(lib.ggq_load_memory(b, len(buf), LOAD_METADATA_ONLY if metadata_only else 0, ctypes.byref(h)),
              "ggq_load_memory")
        return cls(h.value)

    def close(self):
        if self._h:
            lib.ggq_free(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    @property
    def version(self) -> int:
        v = ctypes.c_uint32()
        check(lib.ggq_version_of(self._h, ctypes.byref(v)), "ggq_version_of")
        return v.value

    @property
    def data_start(self) -> int:
        v = ctypes.c_uint64()
        check(lib.ggq_data_start(self._h, ctypes.byref(v)), "ggq_data_start")
        return v.value

    def __len__(self) -> int:
        n = ctypes.c_int64()
        check(lib.ggq_num_tensors(self._h, ctypes.byref(n)), "ggq_num_tensors")
        return n.value

    def tensor(self, i: int) -> dict:
        t = Tensor()
        check(lib.ggq_tensor_info(self._h, i, ctypes.byref(t)), "ggq_tensor_info")
        return dict(name=t.name.decode(), type=t.type, n_dims=t.n_dims, ne=list(t.ne)[:t.n_dims],
                    offset=t.offset, nbytes=t.nbytes, data=t.data or 0)

    def tensors(self):
        return [self.tensor(i) for i in range(len(self))]

    def find(self, name: str) -> dict:
        i = ctypes.c_int64()
        check(lib.ggq_find_tensor(self._h, name.encode(), ctypes.byref(i)), "ggq_find_tensor")
        return self.tensor(i.value)

    def kvs(self):
        n = ctypes.c_int64()
        check(lib.ggq_num_kv(self._h, ctypes.byref(n)), "ggq_num_kv")
        out = []
        for i in range(n.value):
            key, vt, val, nb = ctypes.c_char_p(), ctypes.c_int32(), ctypes.c_void_p(), ctypes.c_uint64()
            check(lib.ggq_kv_info(self._h, i, ctypes.byref(key), ctypes.byref(vt), ctypes.byref(val),
                                  ctypes.byref(nb)), "ggq_kv_info")
            raw = ctypes.string_at(val.value, nb.value) if nb.value else b""
            out.append((key.value.decode(), vt.value, raw))
        return out


# -------------------------------------------------------------- torch helpers

def _stream_ptr(stream) -> int:
    """A torch stream, a raw cudaStream_t value (int), or None (the current stream)."""
    if isinstance(stream, int):
        return stream
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def gemv(qtype: int, W, rows: int, cols: int, x, y=None, stream=None):
    """y[M, rows] = x[M, cols] @ W^T with W a uint8 CUDA tensor of encoded blocks."""
    import torch
    x2 = x.reshape(-1, cols)
    M = x2.shape[0]
    if y is None:
        y = torch.empty((M, rows), dtype=torch.float32, device=x.device)
    check(ggq_gemv(qtype, W.data_ptr(), rows, cols, x2.data_ptr(), y.data_ptr(), M, _stream_ptr(stream)),
          "ggq_gemv")
    return y


def gemv_multi(qtype: int, Ws, rows, cols: int, x, ys=None, stream=None):
    """ys[i][M, rows[i]] = x[M, cols] @ W_i^T for matrices sharing x, one launch."""
    import torch
    x2 = x.reshape(-1, cols)
    M = x2.shape[0]
    if ys is None:
        ys = [torch.empty((M, r), dtype=torch.float32, device=x.device) for r in rows]
    check(ggq_gemv_multi(qtype, [w.data_ptr() for w in Ws], list(rows), cols, x2.data_ptr(),
                         [y.data_ptr() for y in ys], M, _stream_ptr(stream)), "ggq_gemv_multi")
    return ys


def ggq_embed(qtype: int, table: int, rows: int, cols: int, ids: int, n: int, out: int, stream: int) -> int:
    return lib.ggq_embed(qtype, table, rows, cols, ids, n, out, stream)


def embed(qtype: int, table, rows: int, cols: int, ids, out=None, stream=None):
    """out[i] = row ids[i] of the block-quantized table, decoded to fp32 (CUDA tensors)."""
    import torch
    ids = ids.to(device=table.device, dtype=torch.int32).contiguous()
    if out is None:
        out = torch.empty((ids.numel(), cols), dtype=torch.float32, device=table.device)
    check(ggq_embed(qtype, table.data_ptr(), rows, cols, ids.data_ptr(), ids.numel(), out.data_ptr(),
                    _stream_ptr(stream)), "ggq_embed")
    return out


class Chain:
    """A sequence of GEMV stages run as one launch (ggq_chain_create / ggq_chain_run).

    qtype: the weight type of every stage, or a list with one per stage
    (ggq_chain_create_typed).  stages: sequence of (Ws, rows, cols, x, ys) with
    CUDA tensors; the chain keeps references to them (their memory is bound at
    creation).  ops: None, or per stage None or a dict {x_op: X_RMSNORM /
    X_SILU_MUL, eps, norm_w, up, res: [..]} with CUDA tensors
    (ggq_chain_create_ops).
    """

    def __init__(self, qtype: int, M: int, stages, ops=None):
        raw = [([w.data_ptr() for w in Ws], list(rows), cols, x.data_ptr(), [y.data_ptr() for y in ys])
               for (Ws, rows, cols, x, ys) in stages]
        rops = None
        if ops is not None:
            def ptr(t):
                return t.data_ptr() if t is not None else None
            rops = [None if o is None else
                    {"x_op": o.get("x_op", X_PLAIN), "eps": o.get("eps", 0.0), "norm_w": ptr(o.get("norm_w")),
                     "up": ptr(o.get("up")), "res": [ptr(t) for t in (o.get("res") or [])]}
                    for o in ops]
        if isinstance(qtype, (list, tuple)):
            if len(qtype) != len(raw):
                raise ValueError("one weight type per stage")
            rc, h = ggq_chain_create_typed(M, qtype, raw, rops)
        else:
            rc, h = ggq_chain_create(qtype, M, raw, rops)
        check(rc, "ggq_chain_create")
        self._h = h
        self._keep = list(stages) + ([ops] if ops is not None else [])

    def run(self, stream=None) -> None:
        check(ggq_chain_run(self._h, _stream_ptr(stream)), "ggq_chain_run")

    def close(self) -> None:
        if self._h:
            ggq_chain_free(self._h)
            self._h = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def gemm_prefill(qtype: int, W, rows: int, cols: int, X_bf16, Y=None, stream=None):
    """Y[M, rows] = X[M, cols] @ W^T, X a bf16 CUDA tensor (or uint16 bit patterns)."""
    import torch
    M = X_bf16.shape[0]
    if Y is None:
        Y = torch.empty((M, rows), dtype=torch.float32, device=X_bf16.device)
    check(ggq_gemm_prefill(qtype, W.data_ptr(), rows, cols, X_bf16.data_ptr(), Y.data_ptr(), M,
                           _stream_ptr(stream)), "ggq_gemm_prefill")
    return Y


def dequantize(qtype: int, W, rows: int, cols: int, out=None, stream=None):
    import torch
    if out is None:
        out = torch.empty((rows, cols), dtype=torch.float32, device=W.device)
    check(ggq_dequantize(qtype, W.data_ptr(), rows, cols, out.data_ptr(), _stream_ptr(stream)),
          "ggq_dequantize")
    return out


def device_status() -> int:
    return ggq_device_status()

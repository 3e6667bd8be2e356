"""Oracle GGUF v3 reader: a plain byte walk.  TEST INFRASTRUCTURE (see oracle/__init__.py).

Follows the layout the pages give:

* header -- "GGUF Inferencer in R" section 2.1 (byte blueprint): magic
  ``47 47 55 46``, uint32 version, uint64 tensor count, uint64 metadata count;
  "GGUF: The File Format...", gguf_demo.py: ``struct.pack("<IQQ", 3, ...)``;
* strings -- uint64 length + UTF-8 bytes.  The R page's blueprint says uint32;
  the lesson's writer uses uint64 and its "Worked example, step by step" only
  reaches data start 224 with 8-byte lengths, so uint64 is the reading taken;
* metadata -- key string, uint32 value type, value.  Codes 4 (uint32), 8
  (string) and 9 (array: uint32 element type, uint64 count, elements) are on
  the pages; the rest of the v3 code table (0 u8, 1 i8, 2 u16, 3 i16, 5 i32,
  6 f32, 7 bool, 10 u64, 11 i64, 12 f64) is the reading used to step over
  unknown keys ("Pause and think": the type tells the reader the size);
* tensor infos -- name, uint32 n_dims, n_dims x uint64 extents (fastest
  first: a 2x4 tensor is stored as dims (4, 2)), uint32 type, uint64 offset
  relative to the blob;
* the blob starts at the next multiple of 32 (padding after the tensor infos).

Payload sizes by type: F32 4 B, F16 2 B per value; Q8_0 34 B per 32 values;
Q4_K 144 B per 256; Q4_0 18 B per 32; Q6_K 210 B per 256 (the lesson's bits/weight
table).
"""
from __future__ import annotations

import struct

ALIGN = 32
_SCALAR = {0: "<B", 1: "<b", 2: "<H", 3: "<h", 4: "<I", 5: "<i", 6: "<f", 7: "<?",
           10: "<Q", 11: "<q", 12: "<d"}
# (values per block, bytes per block)
_BLOCK = {0: (1, 4), 1: (1, 2), 8: (32, 34), 12: (256, 144), 2: (32, 18), 14: (256, 210)}


class GGUFError(ValueError):
    pass


class _Cursor:
    def __init__(self, buf: bytes):
        self.buf = buf
        self.pos = 0

    def take(self, fmt: str):
        size = struct.calcsize(fmt)
        if self.pos + size > len(self.buf):
            raise GGUFError("truncated file")
        v = struct.unpack_from(fmt, self.buf, self.pos)
        self.pos += size
        return v if len(v) > 1 else v[0]

    def string(self) -> str:
        n = self.take("<Q")
        if self.pos + n > len(self.buf):
            raise GGUFError("string runs past end of file")
        s = self.buf[self.pos:self.pos + n]
        self.pos += n
        return s.decode("utf-8", errors="replace")

    def value(self, vtype: int, depth: int = 0):
        if vtype in _SCALAR:
            return self.take(_SCALAR[vtype])
        if vtype == 8:
            return self.string()
        if vtype == 9:
            if depth > 8:
                raise GGUFError("array nesting too deep")
            etype, count = self.take("<I"), self.take("<Q")
            return (etype, [self.value(etype, depth + 1) for _ in range(count)])
        raise GGUFError(f"unknown metadata value type {vtype}")


def tensor_nbytes(qtype: int, ne) -> int:
    if qtype not in _BLOCK:
        raise GGUFError(f"unsupported tensor type {qtype}")
    per, nb = _BLOCK[qtype]
    n = 1
    for e in ne:
        n *= int(e)
    if n % per:
        raise GGUFError("element count not a multiple of the block size")
    return n // per * nb


def read_gguf(buf: bytes, need_payload: bool = True) -> dict:
    """Parse a GGUF v3 byte string.  Returns a dict with version, kvs (ordered
    list of (key, vtype, value)), tensors (list of dicts: name, n_dims, ne,
    type, offset, nbytes, data) and data_start."""
    cur = _Cursor(buf)
    if len(buf) < 4 or buf[:4] != b"GGUF":
        raise GGUFError("bad magic")
    cur.pos = 4
    version = cur.take("<I")
    if version != 3:
        raise GGUFError(f"unsupported version {version}")
    n_tensors, n_kv = cur.take("<Q"), cur.take("<Q")
    kvs = []
    for _ in range(n_kv):
        key = cur.string()
        vtype = cur.take("<I")
        kvs.append((key, vtype, cur.value(vtype)))
    tensors = []
    for _ in range(n_tensors):
        name = cur.string()
        nd = cur.take("<I")
        if not 1 <= nd <= 4:
            raise GGUFError(f"bad n_dims {nd}")
        ne = [cur.take("<Q") for _ in range(nd)]
        qtype = cur.take("<I")
        off = cur.take("<Q")
        tensors.append(dict(name=name, n_dims=nd, ne=ne, type=qtype, offset=off,
                            nbytes=tensor_nbytes(qtype, ne)))
    data_start = (cur.pos + ALIGN - 1) // ALIGN * ALIGN
    for t in tensors:
        if t["offset"] % ALIGN:
            raise GGUFError("tensor offset not 32-byte aligned")
        if need_payload:
            a = data_start + t["offset"]
            if a + t["nbytes"] > len(buf):
                raise GGUFError("tensor data runs past end of file")
            t["data"] = buf[a:a + t["nbytes"]]
    return dict(version=version, n_tensors=n_tensors, n_kv=n_kv, kvs=kvs,
                tensors=tensors, data_start=data_start)

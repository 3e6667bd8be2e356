"""C-ABI library: loads, exports every declared symbol, and its host logic
(GGUF parsing/validation, argument checks) behaves -- no GPU needed."""
import ctypes
import os
import random
import re
import struct

import numpy as np
import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ggq.h")


@pytest.fixture(scope="module")
def ggq():
    import gguf_block_quantized_q8_gb300 as g
    return g


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ggq_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(ggq):
    names = _declared_functions()
    assert len(names) >= 18
    lib = ctypes.CDLL(ggq.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert ggq.lib.ggq_abi_version() == 1
    assert ggq.strerror(-4) == "malformed GGUF file"


def _tiny():
    """tiny.gguf of the lesson, via the synthetic writer."""
    head, offsets, end = synth.gguf_header(
        [("general.architecture", 8, "llama"), ("general.name", 8, "tiny-demo"),
         ("llama.context_length", 4, 4096)], [("blk.0.ffn_up.weight", [4, 2], 0)])
    return head + np.arange(8, dtype=np.float32).tobytes()


def test_metadata_only_load_of_tiny_gguf(ggq):
    with ggq.Model.from_bytes(_tiny(), metadata_only=True) as m:
        assert m.version == 3 and m.data_start == 224 and len(m) == 1
        t = m.tensor(0)
        assert t["name"] == "blk.0.ffn_up.weight" and t["ne"] == [4, 2] and t["type"] == 0
        assert t["nbytes"] == 32 and t["offset"] == 0 and t["data"] == 0
        kv = m.kvs()
        assert kv[0] == ("general.architecture", 8, b"llama")
        assert kv[2] == ("llama.context_length", 4, struct.pack("<I", 4096))
        assert m.find("blk.0.ffn_up.weight")["ne"] == [4, 2]
        with pytest.raises(ggq.GGQError) as e:
            m.find("nope")
        assert e.value.code == -8


def _mixed_file():
    kvs = [("general.architecture", 8, "llama"),
           ("general.languages", 9, (8, ["en", "fr"])),
           ("x.nested", 9, (9, [(4, [1, 2]), (6, [1.5])])),
           ("x.f64", 12, 2.5), ("x.bool", 7, True), ("x.i64", 11, -3), ("x.u8", 0, 7)]
    q8 = synth.weight_rows(synth.TYPE_Q8_0, 1, 3, 64)
    q4 = synth.weight_rows(synth.TYPE_Q4_K, 2, 2, 512)
    tensors = [("a.weight", [64, 3], 8), ("norm", [64], 0), ("b.weight", [512, 2], 12)]
    head, offs, end = synth.gguf_header(kvs, tensors)
    payloads = [q8.tobytes(), np.ones(64, np.float32).tobytes(), q4.tobytes()]
    blob = bytearray(end)
    for o, p in zip(offs, payloads):
        blob[o:o + len(p)] = p
    return head + bytes(blob), head, offs


def test_metadata_only_load_of_mixed_file(ggq):
    buf, head, offs = _mixed_file()
    with ggq.Model.from_bytes(buf, metadata_only=True) as m:
        ts = m.tensors()
        assert [t["offset"] for t in ts] == offs
        assert [t["nbytes"] for t in ts] == [3 * 68, 256, 2 * 288]
        assert m.data_start == len(head)
        keys = [k for k, _, _ in m.kvs()]
        assert keys[-1] == "x.u8" and len(keys) == 7


def test_loader_rejects_malformed(ggq):
    good, head, _ = _mixed_file()
    cases = {
        "magic": b"GGUX" + good[4:],
        "version": good[:4] + struct.pack("<I", 2) + good[8:],
        "truncated_header": good[:20],
        "truncated_payload": good[:-10],
        "huge_tensor_count": good[:8] + struct.pack("<Q", 1 << 60) + good[16:],
        "huge_kv_count": good[:16] + struct.pack("<Q", 1 << 60) + good[24:],
    }
    for name, buf in cases.items():
        with pytest.raises(ggq.GGQError) as e:
            ggq.Model.from_bytes(buf, metadata_only=True)
        assert e.value.code == -4, name
    with pytest.raises(ggq.GGQError) as e:
        ggq.Model.load("/nonexistent/file.gguf", metadata_only=True)
    assert e.value.code == -3


def test_loader_rejects_bad_tensor_fields(ggq):
    def one(ne, qtype, off):
        out = b"GGUF" + struct.pack("<IQQ", 3, 1, 0)
        out += synth.gguf_string("t") + struct.pack("<I", len(ne)) + struct.pack(f"<{len(ne)}Q", *ne)
        out += struct.pack("<IQ", qtype, off)
        out += b"\0" * (-len(out) % 32)
        return out + b"\0" * 4096
    assert ggq.Model.from_bytes(one([64, 2], 8, 0), metadata_only=True).tensor(0)["nbytes"] == 136
    bad = {
        "unaligned_offset": (one([64, 2], 8, 16), -4),
        "past_end": (one([64, 2], 8, 4096), -4),
        "ragged_q8_row": (one([48, 2], 8, 0), -4),
        "ragged_q4k_row": (one([128, 2], 12, 0), -4),
        "unknown_type": (one([64], 99, 0), -2),
        "zero_dims": (one([], 0, 0), -4),
        "overflowing_dims": (one([1 << 40, 1 << 40], 0, 0), -4),
    }
    for name, (buf, code) in bad.items():
        with pytest.raises(ggq.GGQError) as e:
            ggq.Model.from_bytes(buf, metadata_only=True)
        assert e.value.code == code, name


def test_loader_fuzz_never_crashes(ggq):
    """Every truncation and random byte flips of a valid file: an error code or a
    consistent model, never a crash."""
    buf, _, _ = _mixed_file()
    for n in range(0, len(buf), 7):
        try:
            ggq.Model.from_bytes(buf[:n], metadata_only=True).close()
        except ggq.GGQError as e:
            assert e.code in (-4, -2)
    rnd = random.Random(3)
    for _ in range(400):
        b = bytearray(buf)
        for _ in range(rnd.randint(1, 6)):
            b[rnd.randrange(0, 200)] = rnd.randrange(256)
        try:
            with ggq.Model.from_bytes(bytes(b), metadata_only=True) as m:
                for t in m.tensors():
                    assert t["offset"] % 32 == 0
                    assert m.data_start + t["offset"] + t["nbytes"] <= len(b)
        except ggq.GGQError as e:
            assert e.code in (-4, -2, -5)


def test_compute_entry_points_validate_arguments(ggq):
    """Argument errors are reported before any device work."""
    g = ggq.ggq_gemv
    assert g(ggq.Q8_0, 0, 4, 64, 16, 16, 1, 0) == -1                 # NULL W
    assert g(ggq.Q8_0, 16, 4, 48, 16, 16, 1, 0) == -1                # ragged cols
    assert g(ggq.Q4_K, 16, 4, 128, 16, 16, 1, 0) == -1
    assert g(ggq.Q8_0, 16, 4, 64, 16, 16, 0, 0) == -1                # M = 0
    assert g(ggq.Q8_0, 16, 4, 64, 16, 16, 17, 0) == -1               # M = 17
    assert g(ggq.Q8_0, 8, 4, 64, 16, 16, 1, 0) == -1                 # W misaligned
    assert g(ggq.Q8_0, 16, 0, 64, 16, 16, 1, 0) == -1                # rows = 0
    assert g(ggq.Q8_0, 16, 4, 64, 8, 16, 1, 0) == -1                 # x misaligned
    assert g(ggq.F16, 16, 4, 64, 16, 16, 1, 0) == -2                 # type
    assert g(ggq.Q6_K, 16, 4, 288, 16, 16, 1, 0) == -1                # Q6_K: cols % 256
    assert g(ggq.Q6_K, 16, 4, 256, 16, 16, 17, 0) == -1
    assert g(ggq.Q4_0, 16, 4, 48, 16, 16, 1, 0) == -1                # Q4_0: cols % 32
    assert g(ggq.Q4_0, 16, 4, 64, 16, 16, 17, 0) == -1
    assert g(ggq.F32, 16, 4, 0, 16, 16, 1, 0) == -1                  # F32: cols >= 1
    assert g(ggq.F32, 8, 4, 5, 16, 16, 1, 0) == -1                   # F32: W misaligned
    n = ggq.ggq_gemv_noalloc
    assert n(ggq.Q4_0, 16, 4, 512, 16, 16, 1, 0) == -1               # Q4_0 stream kernel: cols >= 768
    assert n(ggq.F32, 16, 4, 1024, 16, 16, 1, 0) == -2               # F32 has no allocation-free kernel
    p = ggq.ggq_gemm_prefill
    assert p(ggq.F16, 16, 128, 256, 16, 16, 128, 0) == -2
    assert p(ggq.Q8_0, 16, 100, 256, 16, 16, 128, 0) == -1           # Q8_0 too: rows % 128
    assert p(ggq.Q8_0, 16, 128, 224, 16, 16, 128, 0) == -1           # cols % 256
    assert p(ggq.Q4_K, 16, 100, 256, 16, 16, 128, 0) == -1           # rows % 128
    assert p(ggq.Q4_K, 16, 128, 256, 16, 16, 100, 0) == -1           # M % 128
    assert p(ggq.Q4_K, 16, 128, 256, 8, 16, 128, 0) == -1            # X misaligned
    d = ggq.ggq_dequantize
    assert d(ggq.Q4_K, 16, 2, 100, 16, 0) == -1
    assert d(ggq.F16, 16, 2, 256, 16, 0) == -2
    assert d(ggq.Q4_0, 16, 2, 40, 16, 0) == -1                       # cols % 32
    assert d(ggq.Q6_K, 16, 2, 100, 16, 0) == -1                      # cols % 256
    # Q6_K rows start on 16 bytes only when cols % 2048 == 0: other widths are refused
    assert ggq.ggq_chain_create(ggq.Q6_K, 1, [([16], [64], 1024, 16, [16])])[0] == -1
    assert "stage 0 shape unsupported" in ggq.lib.ggq_last_error().decode()
    assert ggq.ggq_gemv_noalloc(ggq.Q6_K, 16, 4, 1024, 16, 16, 1, 0) == -1
    rc, h = ggq.ggq_chain_create(ggq.Q6_K, 1, [([16], [64], 2048, 16, [16])])
    assert rc not in (-1, -2)                     # past validation (no device here: fails later)
    if rc == 0:
        ggq.ggq_chain_free(h)
    assert g(ggq.Q8_0, 16, 4, 64, 16, 16, 17, 0) == -1
    assert "M 17 outside 1..16" in ggq.lib.ggq_last_error().decode()


def test_chain_create_validates_stages(ggq):
    """ggq_chain_create rejects malformed stages before touching the device."""
    ok = ([16], [64], 2048, 16, [16])
    assert ggq.ggq_chain_create(ggq.F32, 1, [ok])[0] == -2                          # type
    assert ggq.ggq_chain_create(ggq.Q4_K, 0, [ok])[0] == -1                         # M = 0
    assert ggq.ggq_chain_create(ggq.Q4_K, 5, [ok])[0] == -1                         # M = 5
    assert ggq.ggq_chain_create(ggq.Q4_K, 1, [])[0] == -1                           # no stages
    assert ggq.ggq_chain_create(ggq.Q4_K, 1, [ok, ([0], [64], 256, 16, [16])])[0] == -1      # NULL W
    assert "stage 1" in ggq.lib.ggq_last_error().decode()
    assert ggq.ggq_chain_create(ggq.Q4_K, 1, [([16], [64], 256, 8, [16])])[0] == -1          # x misaligned
    assert ggq.ggq_chain_create(ggq.Q4_K, 1, [([8], [64], 256, 16, [16])])[0] == -1          # W misaligned
    assert ggq.ggq_chain_create(ggq.Q4_K, 1, [([16], [0], 256, 16, [16])])[0] == -1          # rows = 0
    assert ggq.ggq_chain_create(ggq.Q4_K, 1, [([16], [64], 320, 16, [16])])[0] == -1         # cols % 256
    assert ggq.ggq_chain_create(ggq.Q4_K, 1, [([16] * 5, [64] * 5, 256, 16, [16] * 5)])[0] == -1   # n = 5
    assert ggq.ggq_chain_create(ggq.Q4_0, 1, [([16], [64], 512, 16, [16])])[0] == -1         # Q4_0: cols >= 768
    assert ggq.ggq_chain_create(ggq.Q4_0, 1, [([16], [64], 800, 16, [16])])[0] == -1         # Q4_0: cols % 256
    assert ggq.ggq_chain_run(0, 0) == -1
    ggq.ggq_chain_free(0)


def test_chain_create_typed_validates_each_stage(ggq):
    """ggq_chain_create_typed: one type per stage, each checked with its own
    shape limits; the error names the stage."""
    ok = ([16], [64], 2048, 16, [16])
    t = ggq.ggq_chain_create_typed
    assert t(1, [ggq.Q4_K, ggq.F32], [ok, ok])[0] == -2
    assert "stage 1 type 0" in ggq.lib.ggq_last_error().decode()
    assert t(1, [ggq.Q4_K, ggq.F16], [ok, ok])[0] == -2
    assert t(5, [ggq.Q4_K, ggq.Q6_K], [ok, ok])[0] == -1                               # M = 5
    assert t(1, [], [])[0] == -1                                                       # no stages
    q6_narrow = ([16], [64], 1024, 16, [16])                                           # Q6_K needs cols % 2048
    assert t(1, [ggq.Q4_K, ggq.Q6_K], [q6_narrow, q6_narrow])[0] == -1
    assert "stage 1 shape unsupported" in ggq.lib.ggq_last_error().decode()
    q40_narrow = ([16], [64], 512, 16, [16])                                           # Q4_0 needs cols >= 768
    assert t(1, [ggq.Q6_K, ggq.Q4_0], [ok, q40_narrow])[0] == -1
    assert "stage 1" in ggq.lib.ggq_last_error().decode()
    assert t(1, [ggq.Q4_K, ggq.Q6_K, ggq.Q4_0], [ok] * 3)[0] == -2                  # two types besides Q6_K
    assert "stage 2 type 2" in ggq.lib.ggq_last_error().decode()
    assert t(1, [ggq.Q8_0, ggq.Q6_K], [ok] * 2)[0] == -2                             # Q8_0 is not mixed
    for types in ([ggq.Q4_K, ggq.Q6_K, ggq.Q4_K], [ggq.Q6_K, ggq.Q4_0], [ggq.Q8_0, ggq.Q8_0]):
        rc, h = t(1, types, [ok] * len(types))
        assert rc not in (-1, -2), types          # past validation (no device here: fails later)
        if rc == 0:
            ggq.ggq_chain_free(h)
    with pytest.raises(ValueError):
        ggq.Chain([ggq.Q4_K], 1, [])              # one type per stage


def test_chain_create_ops_validates_fused_steps(ggq):
    """ggq_chain_create_ops rejects malformed fused steps before touching the device."""
    ok = ([16], [64], 2048, 16, [16])

    def rc(op, stages=None):
        stages = stages or [ok, ok]
        return ggq.ggq_chain_create(ggq.Q4_K, 1, stages, [None, op])[0]

    assert rc({"x_op": ggq.X_RMSNORM, "eps": 1e-6, "norm_w": 0}) == -1             # norm_w missing
    assert "stage 1" in ggq.lib.ggq_last_error().decode()
    assert rc({"x_op": ggq.X_RMSNORM, "eps": 1e-6, "norm_w": 24}) == -1            # norm_w misaligned
    assert rc({"x_op": ggq.X_RMSNORM, "eps": -1.0, "norm_w": 32}) == -1            # eps < 0
    assert rc({"x_op": ggq.X_RMSNORM, "eps": float("nan"), "norm_w": 32}) == -1    # eps NaN
    assert rc({"x_op": ggq.X_RMSNORM, "eps": float("inf"), "norm_w": 32}) == -1    # eps infinite
    assert rc({"x_op": ggq.X_SILU_MUL, "up": 0}) == -1                             # up missing
    assert rc({"x_op": ggq.X_SILU_MUL, "up": 8}) == -1                             # up misaligned
    assert rc({"x_op": 7}) == -1                                                   # unknown step
    assert "x_op 7" in ggq.lib.ggq_last_error().decode()
    assert rc({"res": [6]}) == -1                                                  # residual misaligned
    assert "res[0]" in ggq.lib.ggq_last_error().decode()


def test_embed_validates_arguments(ggq):
    """ggq_embed rejects bad arguments before any launch."""
    assert ggq.ggq_embed(ggq.F16, 16, 4, 64, 16, 1, 16, 0) == -2          # type
    assert ggq.ggq_embed(ggq.Q4_0, 16, 4, 40, 16, 1, 16, 0) == -1         # Q4_0: cols % 32
    assert ggq.ggq_embed(ggq.Q6_K, 16, 4, 320, 16, 1, 16, 0) == -1        # Q6_K: cols % 256
    assert ggq.ggq_embed(ggq.F32, 18, 4, 5, 16, 1, 16, 0) == -1           # F32 table: 4-byte aligned
    assert ggq.ggq_embed(ggq.Q8_0, 0, 4, 64, 16, 1, 16, 0) == -1          # NULL table
    assert ggq.ggq_embed(ggq.Q8_0, 16, 4, 64, 0, 1, 16, 0) == -1          # NULL ids
    assert ggq.ggq_embed(ggq.Q8_0, 16, 4, 63, 16, 1, 16, 0) == -1         # cols % 32
    assert ggq.ggq_embed(ggq.Q4_K, 16, 4, 288, 16, 1, 16, 0) == -1        # cols % 256
    assert ggq.ggq_embed(ggq.Q8_0, 16, 0, 64, 16, 1, 16, 0) == -1         # rows = 0
    assert ggq.ggq_embed(ggq.Q8_0, 16, 4, 64, 16, 0, 16, 0) == -1         # n = 0
    assert ggq.ggq_embed(ggq.Q8_0, 16, 4, 64, 16, 65536, 16, 0) == -1     # n too large
    assert ggq.ggq_embed(ggq.Q8_0, 17, 4, 64, 16, 1, 16, 0) == -1         # table misaligned
    assert ggq.ggq_embed(ggq.Q8_0, 16, 4, 64, 18, 1, 16, 0) == -1         # ids misaligned
    assert "misaligned" in ggq.lib.ggq_last_error().decode()

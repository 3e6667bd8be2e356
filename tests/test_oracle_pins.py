"""The CPU oracle pinned to the pages, closed forms and library routines (no GPU)."""
import json
import os
import struct

import numpy as np
import pytest

import oracle
import synth
from tests import pin_checks

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("check", pin_checks.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(orc, check):
    check(orc)


# ------------------------------------------------------------ GGUF reader ----

def _lesson():
    with open(os.path.join(GOLDEN, "gguf_lesson_values.json")) as f:
        return json.load(f)


def _s(text: str) -> bytes:
    b = text.encode()
    return struct.pack("<Q", len(b)) + b


def _tiny_gguf_bytes(extra_kv: bytes = b"", n_kv: int = 3) -> bytes:
    """tiny.gguf built from the lesson's description of the layout."""
    out = b"GGUF" + struct.pack("<IQQ", 3, 1, n_kv)
    out += _s("general.architecture") + struct.pack("<I", 8) + _s("llama")
    out += _s("general.name") + struct.pack("<I", 8) + _s("tiny-demo")
    out += _s("llama.context_length") + struct.pack("<I", 4) + struct.pack("<I", 4096)
    out += extra_kv
    out += _s("blk.0.ffn_up.weight") + struct.pack("<I", 2)
    out += struct.pack("<QQIQ", 4, 2, 0, 0)
    out += b"\0" * (-len(out) % 32)
    return out + np.arange(8, dtype=np.float32).tobytes()


def test_tiny_gguf_layout():
    g = _lesson()["tiny_gguf"]
    buf = _tiny_gguf_bytes()
    parts = g["part_bytes"]
    assert len(buf) == g["file_size"]
    assert parts["header"] + parts["kv_architecture"] + parts["kv_name"] + \
        parts["kv_context_length"] + parts["tensor_info"] == parts["before_padding"]
    r = oracle.read_gguf(buf)
    assert r["version"] == g["version"] and r["n_tensors"] == g["tensors"]
    assert r["n_kv"] == g["metadata_keys"]
    assert [[k, t, v] for k, t, v in r["kvs"]] == g["kvs"]
    assert r["data_start"] == g["data_start"]
    t = r["tensors"][0]
    assert t["name"] == g["tensor_name"] and t["ne"] == g["dims"] and t["type"] == g["tensor_type"]
    vals = np.frombuffer(t["data"], dtype="<f4").reshape(t["ne"][1], t["ne"][0])
    assert vals.tolist() == g["values"]


def test_tiny_gguf_extra_key_moves_data_to_256():
    e = _lesson()["extra_kv"]
    # a uint32 entry with a 14-character key: (8 + 14) + 4 + 4 = 30 bytes
    key = _s("extra.key.abcd") + struct.pack("<I", 4) + struct.pack("<I", 7)
    assert len(key) == e["entry_bytes"]
    buf = _tiny_gguf_bytes(key, n_kv=4)
    r = oracle.read_gguf(buf)
    assert r["data_start"] == e["data_start"]
    assert r["kvs"][3] == ("extra.key.abcd", 4, 7)


def test_synth_writer_matches_lesson_bytes(tmp_path):
    g = _lesson()["tiny_gguf"]
    kvs = [tuple(kv) for kv in g["kvs"]]
    path = tmp_path / "tiny.gguf"
    size = synth.write_gguf(str(path), kvs, [(g["tensor_name"], g["dims"], 0)],
                            [np.arange(8, dtype=np.float32).tobytes()])
    assert size == g["file_size"]
    assert path.read_bytes() == _tiny_gguf_bytes()


def test_block_sizes_from_bits_per_weight():
    lesson = _lesson()
    for name, (nbytes, nweights) in lesson["block_bytes"].items():
        assert f"{nbytes * 8 / nweights:.4g}" == lesson["bits_per_weight"][name]
    assert oracle.tensor_nbytes(8, [32]) == 34
    assert oracle.tensor_nbytes(12, [256]) == 144
    assert oracle.tensor_nbytes(2, [32]) == 18
    assert oracle.tensor_nbytes(14, [256]) == 210


def _smollm3_table():
    rows = []
    with open(os.path.join(GOLDEN, "smollm3_q8_0_tensor_table.txt")) as f:
        for line in f:
            if line.startswith("#") or line.startswith("cols") or not line.strip():
                continue
            name, cols, nrows, typ, off = line.split()
            rows.append((name, int(cols), int(nrows), {"F32": 0, "Q8_0": 8}[typ], int(off)))
    return rows


def test_smollm3_table_offsets_follow_block_sizes():
    """Every printed offset = previous offset + that tensor's payload size."""
    with open(os.path.join(GOLDEN, "smollm3_header.json")) as f:
        hdr = json.load(f)
    table = _smollm3_table()
    assert len(table) == hdr["tensor_count"]
    ex = hdr["example_tensor"]
    assert (ex["name"], ex["cols"], ex["rows"], ex["type"], ex["offset"]) in table
    for (n0, c0, r0, t0, o0), (_, _, _, _, o1) in zip(table, table[1:]):
        ne = [c0] if r0 == 1 else [c0, r0]
        assert o0 % 32 == 0
        assert o0 + oracle.tensor_nbytes(t0, ne) == o1, n0
    # 64 Q8_0 chunks per 2048-wide row
    assert oracle.tensor_nbytes(8, [2048]) == hdr["q8_0_chunks_per_row_2048"] * 34
    n, c, r, t, o = table[-1]
    assert o + oracle.tensor_nbytes(t, [c, r]) == 3267731456   # blob end: a "3GB GGUF"


def test_smollm3_table_roundtrip_through_writer_and_reader():
    table = _smollm3_table()
    tensors = [(n, [c] if r == 1 else [c, r], t) for n, c, r, t, _ in table]
    kvs = [("general.architecture", 8, "smollm3"), ("smollm3.block_count", 4, 36)]
    head, offsets, end = synth.gguf_header(kvs, tensors)
    assert offsets == [o for *_, o in table]
    parsed = oracle.read_gguf(head, need_payload=False)
    assert [t["offset"] for t in parsed["tensors"]] == offsets
    assert [t["name"] for t in parsed["tensors"]] == [n for n, *_ in table]
    assert parsed["data_start"] == len(head)


def test_reader_rejects_malformed():
    good = _tiny_gguf_bytes()
    with pytest.raises(oracle.GGUFError):
        oracle.read_gguf(b"GGUX" + good[4:])
    with pytest.raises(oracle.GGUFError):
        oracle.read_gguf(good[:4] + struct.pack("<I", 2) + good[8:])
    with pytest.raises(oracle.GGUFError):
        oracle.read_gguf(good[:-4])           # payload truncated
    with pytest.raises(oracle.GGUFError):
        oracle.read_gguf(good[:40])           # header truncated


# ------------------------------------------------- encoder round trip (P2) ----

def test_practice_script_mean_error():
    """The lesson's practice script: two blocks of N(0, 0.05) with numpy seed 5
    round-trip through the Q8_0 block with mean error 0.00020."""
    p = _lesson()["practice"]
    rng = np.random.default_rng(p["seed"])
    w = rng.normal(0, p["sigma"], size=p["n"]).astype(np.float32)
    packed = synth.quantize_q8_0(w)
    assert packed.size // (p["n"] // p["block"]) == p["q8_bytes_per_block"]
    assert packed.size * 8 / p["n"] == p["q8_bits_per_weight"]
    back = oracle.dequantize(8, packed, 1, p["n"]).reshape(-1)
    assert f"{np.abs(back - w).mean():.5f}" == p["q8_mean_error"]


def test_practice_script_mean_error_4bit():
    """The same two blocks through a Q4_0 block (fp16 scale absmax/7, 4-bit codes
    q + 8): 18 bytes per block, 4.5 bits per weight, mean error 0.00324 as the
    practice script prints for its 4-bit block (same value mapping; only the
    pairing of weights in a byte differs, which the mean error cannot see)."""
    p = _lesson()["practice"]
    rng = np.random.default_rng(p["seed"])
    w = rng.normal(0, p["sigma"], size=p["n"]).astype(np.float32)
    packed = synth.quantize_q4_0(w)
    assert packed.size // (p["n"] // p["block"]) == p["q4_bytes_per_block"]
    assert packed.size * 8 / p["n"] == p["q4_bits_per_weight"]
    back = oracle.dequantize(2, packed, 1, p["n"]).reshape(-1)
    assert f"{np.abs(back - w).mean():.5f}" == p["q4_mean_error"]


def test_synth_rows_are_counter_based():
    """Any row range regenerates the same bytes (used for full-size spot checks)."""
    full = synth.weight_rows(12, 99, 8, 512)
    part = synth.weight_rows(12, 99, 3, 512, row0=4)
    rb = 2 * 144
    assert np.array_equal(full[4 * rb:7 * rb], part)
    full8 = synth.weight_rows(8, 5, 6, 256)
    assert np.array_equal(full8[2 * 272:], synth.weight_rows(8, 5, 4, 256, row0=2))


def test_synth_q4_0_roundtrip_error():
    """Q4_0 of N(0, 0.02): every decoded weight within half a step (d / 2) of its
    source, and the scale is absmax / 7 rounded to fp16."""
    w = synth.normal_f32(32 * 64, 4, sigma=0.02)
    packed = synth.quantize_q4_0(w)
    back = oracle.dequantize(2, packed, 64, 32).reshape(64, 32)
    d = packed.reshape(64, 18)[:, :2].copy().view(np.float16).astype(np.float64).reshape(64)
    amax = np.abs(w.reshape(64, 32)).max(axis=1)
    assert np.allclose(d, amax / 7, rtol=2 ** -10)
    assert np.all(np.abs(back - w.reshape(64, 32)) <= d[:, None] / 2 * (1 + 2 ** -10))


def test_synth_q6_k_roundtrip_error():
    """Q6_K of N(0, 0.02): every decoded weight within half a step (d * sc / 2)
    of its source; scales are non-negative and d = fp16(max scale / 127)."""
    w = synth.normal_f32(256 * 32, 5, sigma=0.02)
    packed = synth.quantize_q6_k(w).reshape(32, 210)
    back = oracle.dequantize(14, packed.reshape(-1), 32, 256)
    d = packed[:, 208:210].copy().view(np.float16).astype(np.float64).reshape(32)
    sc = packed[:, 192:208].view(np.int8).astype(np.float64)
    assert (sc >= 0).all() and (sc.max(axis=1) >= 126).all()
    step = d[:, None] * np.repeat(sc, 16, axis=1)
    assert np.all(np.abs(back - w.reshape(32, 256)) <= step / 2 * (1 + 2 ** -10) + 1e-12)


def test_synth_q4_k_roundtrip_error():
    """RTN Q4_K of N(0, 0.02): decoded weights stay within one step of the grid."""
    w = synth.normal_f32(256 * 64, 3, sigma=0.02)
    packed = synth.quantize_q4_k(w)
    back = oracle.dequantize(12, packed, 64, 256).reshape(-1)
    err = np.abs(back - w)
    assert err.mean() < 0.0025 and err.max() < 0.01


def test_synth_encoders_edge_blocks():
    """Encoder edge cases (the inputs both sides read): an all-zero block has
    scale 0 and decodes to zeros; the largest magnitude of a block lands on the
    end of its grid (Q4_0: code 8 + 7 or 8 - 7; Q6_K: 32 + 31 or 32 - 31)."""
    z = np.zeros(256, np.float32)
    assert not oracle.dequantize(2, synth.quantize_q4_0(z), 1, 256).any()
    assert not oracle.dequantize(14, synth.quantize_q6_k(z), 1, 256).any()
    w = synth.normal_f32(256, 9, sigma=0.02)
    w[37] = 0.5                       # the largest magnitude, positive
    w[200] = -0.5
    q4 = synth.quantize_q4_0(w).reshape(8, 18)
    assert (q4[1, 2 + 5] & 15) == 15          # weight 37 = block 1, weight 5: low nibble, code 15
    assert (q4[6, 2 + 8] & 15) == 1           # weight 200 = block 6, weight 8: low nibble, code 1
    q6 = synth.quantize_q6_k(w)
    back = oracle.dequantize(14, q6, 1, 256).reshape(-1)
    assert abs(back[37] - 0.5) <= 0.5 / 31 / 2 * 1.01 and abs(back[200] + 0.5) <= 0.5 / 31 / 2 * 1.01

"""The library's pass planner (gguf_block_quantized_q8_gb300.plan) on the CPU:
the stages a file's tensor table gives (split by type in order), the layer
count from the metadata, and the launches they make (runs of chain-kernel
types as one chain launch, every other stage on its own)."""
import pytest

import synth
from synth import workloads as WL


def _bench():
    from gguf_block_quantized_q8_gb300 import plan
    return plan


class FakeModel:
    """Tensor table of a Q4_K_M-style file, as Model.find returns it."""

    def __init__(self, layers, vocab):
        self.t = {g.name: dict(name=g.name, type=g.qtype, ne=[g.cols] if g.rows == 1 else [g.cols, g.rows],
                               nbytes=0, data=0) for g in WL.llama8b_q4km_tensors(layers, vocab)}

    def find(self, name):
        return self.t[name]

    def tensors(self):
        return list(self.t.values())

    def kvs(self):
        return [("general.architecture", 8, b"llama")]


def test_plan_splits_stages_by_type_in_order():
    b = _bench()
    plan = b.plan_from_table(FakeModel(2, 1000), 2)
    got = [(qt, [t["name"].split(".")[2] if t["name"].startswith("blk") else t["name"] for t in ts]) for qt, ts in plan]
    assert got == [
        (12, ["attn_q", "attn_k", "attn_v"]), (12, ["attn_output"]), (12, ["ffn_gate", "ffn_up"]), (12, ["ffn_down"]),
        (12, ["attn_q", "attn_k"]), (14, ["attn_v"]), (12, ["attn_output"]), (12, ["ffn_gate", "ffn_up"]),
        (14, ["ffn_down"]), (14, ["output.weight"]),
    ]


def test_segments():
    b = _bench()
    assert b.segments([12, 12, 12, 12, 12, 14, 12, 12, 14, 14]) == [
        (0, 5, True), (5, 6, False), (6, 8, True), (8, 9, False), (9, 10, False)]
    assert b.segments([]) == []
    assert b.segments([8, 12, 12, 2, 0]) == [(0, 1, True), (1, 3, True), (3, 4, True), (4, 5, False)]


def test_q4km_file_size_matches_the_pages():
    """An 8B model in Q4_K_M is roughly 4.9 GB ("GGUF: The File Format...",
    "Understanding quantization names like Q4_K_M")."""
    import synth
    ts = WL.llama8b_q4km_tensors(32, 128256)
    total = sum(g.rows * synth.row_bytes(g.qtype, g.cols) for g in ts)
    assert 4.85e9 < total < 4.95e9
    plan_types = [g.qtype for g in ts if g.rows > 1 and g.name != "token_embd.weight"]
    assert plan_types.count(14) == 16 * 2 + 1


def test_block_count_from_metadata_and_table(tmp_path):
    import gguf_block_quantized_q8_gb300 as ggq
    from gguf_block_quantized_q8_gb300 import plan
    # from the table alone
    assert plan.block_count(FakeModel(3, 100)) == 3
    # from the <arch>.block_count key of a real file (metadata-only load)
    q4 = synth.weight_rows(12, 5, 2, 256)
    head, offs, end = synth.gguf_header([("general.architecture", 8, "llama"), ("llama.block_count", 4, 7)],
                                        [("blk.0.attn_q.weight", [256, 2], 12)])
    blob = bytearray(end)
    blob[offs[0]:offs[0] + q4.nbytes] = q4.tobytes()
    with ggq.Model.from_bytes(head + bytes(blob), metadata_only=True) as m:
        assert plan.block_count(m) == 7


def test_decode_pass_checks_its_arguments():
    from gguf_block_quantized_q8_gb300 import plan
    with pytest.raises(ValueError):
        plan.DecodePass([], [], [], M=5)
    with pytest.raises(ValueError):
        plan.DecodePass([(12, [dict(ne=[256, 2], data=0, nbytes=0)])], [], [])

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
    """Runs of chainable stages of any types are one chain; a stage outside
    the chain kernel's limits (F32, Q6_K at cols % 2048, Q4_K/Q4_0 below 768
    columns, cols % 256 for Q8_0) is a launch of its own."""
    b = _bench()
    q4km = [12, 12, 12, 12, 12, 14, 12, 12, 14, 14]
    assert b.segments(q4km, [4096] * 10) == [(0, 10, True)]
    assert b.segments(q4km, [4096] * 5 + [11008] + [4096] * 4) == [(0, 5, True), (5, 6, False), (6, 10, True)]
    assert b.segments([], []) == []
    # a chain holds one type, or Q6_K with Q4_K or with Q4_0
    assert b.segments([8, 12, 12, 2, 0], [4096] * 5) == [(0, 1, True), (1, 3, True), (3, 4, True), (4, 5, False)]
    assert b.segments([2, 14, 2, 14, 12, 14], [4096] * 6) == [(0, 4, True), (4, 6, True)]
    assert b.segments([8, 14], [4096] * 2) == [(0, 1, True), (1, 2, True)]
    assert b.segments([14, 8, 8], [4096] * 3) == [(0, 1, True), (1, 3, True)]
    assert b.segments([8, 12, 8, 2, 8], [4096, 512, 4096, 512, 4000]) == [
        (0, 1, True), (1, 2, False), (2, 3, True), (3, 4, False), (4, 5, False)]
    assert b.segments([14, 14], [2048, 6144]) == [(0, 2, True)]
    with pytest.raises(ValueError):
        b.segments([12], [])


def test_mixable():
    b = _bench()
    assert b.mixable([12, 14, 12]) and b.mixable([2, 14]) and b.mixable([14]) and b.mixable([8, 8])
    assert not b.mixable([12, 2]) and not b.mixable([8, 14]) and not b.mixable([12, 14, 2])


def test_chainable_limits():
    b = _bench()
    assert b.chainable(8, 256) and not b.chainable(8, 288)
    assert b.chainable(12, 768) and not b.chainable(12, 512)
    assert b.chainable(2, 1024) and not b.chainable(2, 512)
    assert b.chainable(14, 2048) and not b.chainable(14, 1024) and not b.chainable(14, 2304)
    assert not b.chainable(0, 4096) and not b.chainable(1, 4096)
    assert not b.chainable(8, (1 << 20) + 256)


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


class _Buf:
    """Stands in for a device tensor: only its address is used."""

    def __init__(self, addr):
        self.addr = addr

    def data_ptr(self):
        return self.addr


def _fake_chains(monkeypatch, plan, max_cols):
    """ggq_chain_create_typed that refuses (EINVAL) a run holding a stage wider
    than max_cols, as the library does for a stage whose pre-scaled x for M rows
    would not fit in shared memory; records every run it was asked for."""
    asked, live = [], set()

    def create(M, types, raw):
        asked.append([r[2] for r in raw])
        if any(r[2] > max_cols for r in raw):
            return plan._ggq.EINVAL, 0
        h = 1000 + len(asked)
        live.add(h)
        return 0, h

    monkeypatch.setattr(plan._ggq, "ggq_chain_create_typed", create)
    monkeypatch.setattr(plan._ggq, "ggq_chain_free", lambda h: live.discard(h))
    return asked, live


def _stages(cols_list, qtype=12):
    stages, xs, ys = [], [], []
    for i, cols in enumerate(cols_list):
        stages.append((qtype, [dict(ne=[cols, 64], data=16 * (i + 1), nbytes=0)]))
        xs.append(_Buf(4096 * (i + 1)))
        ys.append([_Buf(8192 * (i + 1))])
    return stages, xs, ys


def test_decode_pass_takes_too_wide_stages_out_of_the_chain(monkeypatch):
    """Runs of chainable stages become chains; a stage the chain kernel refuses
    at this M (too wide) becomes a launch of its own between them, and stages
    that fit keep sharing one chain on each side of it."""
    from gguf_block_quantized_q8_gb300 import plan
    asked, live = _fake_chains(monkeypatch, plan, max_cols=8192)
    cols = [4096, 4096, 14336, 4096, 4096, 4096, 14336, 14336, 4096]
    stages, xs, ys = _stages(cols)
    dp = plan.DecodePass(stages, xs, ys, M=4)
    kinds = [(k, c["cols"] if k == "stage" else c) for k, c in dp.calls]
    assert [k for k, _ in kinds] == ["chain", "stage", "chain", "stage", "stage", "chain"]
    assert [c for k, c in kinds if k == "stage"] == [14336, 14336, 14336]
    # the whole run first, each stage alone once the run was refused, then the
    # runs between the too-wide stages
    assert asked[0] == cols
    assert asked[1:1 + len(cols)] == [[c] for c in cols]
    assert asked[1 + len(cols):] == [[4096, 4096], [4096, 4096, 4096], [4096]]
    assert len(dp.chains) == 3 and live == set(dp.chains)
    dp.close()
    assert not live


def test_decode_pass_one_chain_when_every_stage_fits(monkeypatch):
    from gguf_block_quantized_q8_gb300 import plan
    asked, live = _fake_chains(monkeypatch, plan, max_cols=1 << 20)
    stages, xs, ys = _stages([4096, 14336, 4096])
    dp = plan.DecodePass(stages, xs, ys, M=2)
    assert dp.launches == 1 and asked == [[4096, 14336, 4096]]
    dp.close()
    assert not live


def test_decode_pass_other_errors_propagate(monkeypatch):
    """A refusal for another reason than EINVAL is an error, not a split."""
    from gguf_block_quantized_q8_gb300 import plan
    live = set()

    def create(M, types, raw):
        return plan._ggq.ECUDA, 0

    monkeypatch.setattr(plan._ggq, "ggq_chain_create_typed", create)
    monkeypatch.setattr(plan._ggq, "ggq_chain_free", lambda h: live.discard(h))
    stages, xs, ys = _stages([4096, 4096])
    with pytest.raises(Exception):
        plan.DecodePass(stages, xs, ys, M=1)

"""GPU parity for a mixed-type decode pass planned from a file's tensor table:
a 2-layer Q4_K_M-style GGUF (Q4_K matrices, Q6_K attn_v / ffn_down in layer 1,
F32 norms, a Q6_K head of 32000 rows) written, loaded with ggq_load, planned by
the library's planner (gguf_block_quantized_q8_gb300.plan: the whole pass,
Q4_K and Q6_K stages and the head, as one chain of mixed types) and run twice;
every output row of every stage checked against the oracle."""
import numpy as np
import pytest

import oracle
import synth
from synth import workloads as WL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("-m gpu tests need a CUDA device")
    import gguf_block_quantized_q8_gb300 as ggq
    return torch, ggq


def test_q4km_file_pass(env, tmp_path):
    torch, ggq = env
    from gguf_block_quantized_q8_gb300 import plan as P
    layers, vocab = 2, 32000
    path = str(tmp_path / "q4km.gguf")
    ts = WL.write_q4km_file(path, layers, vocab)
    byname = {g.name: g for g in ts}
    with ggq.Model.load(path) as model:
        assert P.block_count(model) == layers
        stages = P.plan_from_table(model)
        xs, ys = [], []
        for si, (qtype, tl) in enumerate(stages):
            xs.append(torch.from_numpy(synth.normal_f32(tl[0]["ne"][0], 9000 + si)).cuda())
            ys.append([torch.full((t["ne"][1],), float("nan"), device="cuda") for t in tl])
        dp = P.DecodePass(stages, xs, ys)
        assert len(dp.chains) == 1 and dp.launches == 1   # one chain: Q4_K, Q6_K and the head
        for _ in range(2):                                  # twice: chains reset their counters
            dp.run()
            torch.cuda.synchronize()
            assert ggq.device_status() == 0
        for si, (qtype, tl) in enumerate(stages):
            x = xs[si].cpu().numpy().reshape(1, -1)
            for t, y in zip(tl, ys[si]):
                g = byname[t["name"]]
                assert g.qtype == qtype and g.rows == t["ne"][1] and g.cols == t["ne"][0]
                W = synth.weight_rows(g.qtype, g.stream, g.rows, g.cols)
                y_ref, a_ref = oracle.gemv_dense(g.qtype, W, g.rows, g.cols, x)
                ok, worst = oracle.tolerance_ok(y.cpu().numpy().reshape(1, -1), y_ref, a_ref)
                assert ok, f"{t['name']}: worst error / bound {worst:.3g}"
        dp.close()

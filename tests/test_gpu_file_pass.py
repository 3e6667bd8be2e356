"""GPU parity for a mixed-type decode pass planned from a file's tensor table:
a 2-layer Q4_K_M-style GGUF (Q4_K matrices, Q6_K attn_v / ffn_down in layer 1,
F32 norms, a Q6_K head of 32000 rows) written, loaded with ggq_load, planned by
bench.py's FilePass (Q4_K runs as chain launches, Q6_K stages on their own) and
run once; every stage's outputs checked on sampled rows against the oracle."""
import importlib.util
import os

import numpy as np
import pytest

import oracle
import synth
from synth import workloads as WL

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("-m gpu tests need a CUDA device")
    import gguf_block_quantized_q8_gb300 as ggq
    return torch, ggq


def test_q4km_file_pass(env, tmp_path):
    torch, ggq = env
    spec = importlib.util.spec_from_file_location("bench_fp", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    layers, vocab = 2, 32000
    path = str(tmp_path / "q4km.gguf")
    ts = WL.write_q4km_file(path, layers, vocab)
    byname = {g.name: g for g in ts}
    with ggq.Model.load(path) as model:
        fp = bench.FilePass(model, layers, torch, ggq, synth)
        assert len(fp.chains) == 2 and len(fp.calls) == 5   # chain, v, chain, down, head
        for _ in range(2):                                    # twice: chains reset their counters
            fp.run(torch.cuda.current_stream().cuda_stream)
            torch.cuda.synchronize()
            assert ggq.device_status() == 0
        rng = np.random.default_rng(3)
        for p in fp.plan:
            x = synth.normal_f32(p["cols"], p["x_stream"]).reshape(1, -1)
            for name, rows, y in zip(p["names"], p["rows"], p["ys"]):
                g = byname[name]
                assert g.qtype == p["qtype"] and g.rows == rows and g.cols == p["cols"]
                rs = np.unique(np.r_[0, rows - 1, rng.integers(0, rows, 40)])
                W = np.concatenate([synth.weight_rows(g.qtype, g.stream, 1, g.cols, row0=int(r)) for r in rs])
                y_ref, a_ref = oracle.gemv(g.qtype, W, len(rs), g.cols, x)
                got = y.cpu().numpy()[rs].reshape(1, -1)
                ok, worst = oracle.tolerance_ok(got, y_ref, a_ref)
                assert ok, f"{name}: worst error / bound {worst:.3g}"
        fp.close()

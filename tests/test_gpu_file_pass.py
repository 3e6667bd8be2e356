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


@pytest.mark.parametrize("M", [1, 3])
def test_decode_pass_splits_at_stages_the_chain_kernel_does_not_take(env, M):
    """A plan whose stages alternate between what the chain kernel streams and
    what it does not (Q6_K at 2304 columns, F32): chains for the runs, one
    ggq_gemv / ggq_gemv_multi launch for each other stage, every output
    against the oracle."""
    torch, ggq = env
    from gguf_block_quantized_q8_gb300 import plan as P
    spec = [(ggq.Q4_K, [(512, 2048)]), (ggq.Q6_K, [(384, 2304)]), (ggq.Q4_K, [(256, 1024), (128, 1024)]),
            (ggq.F32, [(100, 515)]), (ggq.Q6_K, [(64, 2048)]), (ggq.Q4_K, [(96, 2048)])]
    keep, stages, xs, ys, host = [], [], [], [], []
    for si, (qtype, mats) in enumerate(spec):
        infos, ylist, hw = [], [], []
        for mi, (rows, cols) in enumerate(mats):
            W = synth.weight_rows(qtype, 700 + 10 * si + mi, rows, cols)
            Wd = torch.from_numpy(W).cuda()
            keep.append(Wd)
            infos.append({"name": f"s{si}.{mi}", "type": qtype, "ne": [cols, rows], "nbytes": W.nbytes,
                          "data": Wd.data_ptr()})
            ylist.append(torch.full((M, rows), float("nan"), device="cuda"))
            hw.append(W)
        cols = mats[0][1]
        x = synth.normal_f32(M * cols, 800 + si).reshape(M, cols)
        xs.append(torch.from_numpy(x).cuda())
        ys.append(ylist)
        stages.append((qtype, infos))
        host.append((qtype, mats, hw, x))
    dp = P.DecodePass(stages, xs, ys, M=M)
    assert P.segments([q for q, _ in stages], [t[0]["ne"][0] for _, t in stages]) == [
        (0, 1, True), (1, 2, False), (2, 3, True), (3, 4, False), (4, 6, True)]
    assert len(dp.chains) == 3 and dp.launches == 5
    dp.run()
    torch.cuda.synchronize()
    assert ggq.device_status() == 0
    for (qtype, mats, hw, x), ylist in zip(host, ys):
        for (rows, cols), W, y in zip(mats, hw, ylist):
            y_ref, a_ref = oracle.gemv(qtype, W, rows, cols, x)
            ok, worst = oracle.tolerance_ok(y.cpu().numpy(), y_ref, a_ref)
            assert ok, f"type {qtype} {rows}x{cols}: worst error / bound {worst:.3g}"
    dp.close()


def test_decode_pass_takes_stages_too_wide_for_the_chain_out_of_it(env):
    """At M = 4 the pre-scaled x of a 14336-column stage does not fit in shared
    memory: that stage (and a Q6_K one of the same width) runs as ggq_gemv
    between two chains; at M = 2 the same plan is one chain."""
    torch, ggq = env
    from gguf_block_quantized_q8_gb300 import plan as P
    spec = [(ggq.Q4_K, [(128, 4096), (64, 4096)]), (ggq.Q4_K, [(72, 14336)]), (ggq.Q6_K, [(40, 14336)]),
            (ggq.Q4_K, [(96, 4096)]), (ggq.Q6_K, [(48, 4096)])]
    for M, n_chains, n_launches in ((4, 2, 4), (2, 1, 1)):
        keep, stages, xs, ys, host = [], [], [], [], []
        for si, (qtype, mats) in enumerate(spec):
            infos, ylist, hw = [], [], []
            for mi, (rows, cols) in enumerate(mats):
                W = synth.weight_rows(qtype, 900 + 10 * si + mi, rows, cols)
                Wd = torch.from_numpy(W).cuda()
                keep.append(Wd)
                infos.append({"name": f"s{si}.{mi}", "type": qtype, "ne": [cols, rows], "nbytes": W.nbytes,
                              "data": Wd.data_ptr()})
                ylist.append(torch.full((M, rows), float("nan"), device="cuda"))
                hw.append(W)
            cols = mats[0][1]
            x = synth.normal_f32(M * cols, 950 + si).reshape(M, cols)
            xs.append(torch.from_numpy(x).cuda())
            ys.append(ylist)
            stages.append((qtype, infos))
            host.append((qtype, mats, hw, x))
        dp = P.DecodePass(stages, xs, ys, M=M)
        assert (len(dp.chains), dp.launches) == (n_chains, n_launches), M
        dp.run()
        torch.cuda.synchronize()
        assert ggq.device_status() == 0
        for (qtype, mats, hw, x), ylist in zip(host, ys):
            for (rows, cols), W, y in zip(mats, hw, ylist):
                y_ref, a_ref = oracle.gemv(qtype, W, rows, cols, x)
                ok, worst = oracle.tolerance_ok(y.cpu().numpy(), y_ref, a_ref)
                assert ok, f"M={M} type {qtype} {rows}x{cols}: worst error / bound {worst:.3g}"
        dp.close()

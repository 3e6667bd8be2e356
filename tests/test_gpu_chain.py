"""GPU parity: ggq_chain (a sequence of dependent GEMV stages in one launch)
against the CPU oracle, through the C ABI.

Each stage is checked against the oracle fed with the x that stage actually
read on the GPU (the y the chain wrote for the stage before it), so a stage
that started before its input was complete shows up as a mismatch: outputs
start as NaN and the input of the second run differs from the first.
"""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

REL, ABS = 1e-3, 1e-6


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("-m gpu tests need a CUDA device")
    import gguf_block_quantized_q8_gb300 as ggq
    return torch, ggq


def _dev(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


class Net:
    """Stages given as lists of (name, rows, cols, source); source is 'x0' or
    the name of an earlier output whose rows equal this stage's cols.  qtype:
    one weight type for every stage, or a list with one per stage (a chain of
    mixed types)."""

    def __init__(self, env, qtype, M, stages, seed=0):
        torch, ggq = env
        self.torch, self.ggq, self.M = torch, ggq, M
        self.types = list(qtype) if isinstance(qtype, (list, tuple)) else [qtype] * len(stages)
        self.qtype = {}
        self.W, self.Wd, self.y, self.shape = {}, {}, {}, {}
        cols0 = stages[0][0][2]
        self.x0 = torch.empty((M, cols0), dtype=torch.float32, device="cuda")
        self.plan = []
        for si, stage in enumerate(stages):
            src = stage[0][3]
            cols = stage[0][2]
            assert all(s[2] == cols and s[3] == src for s in stage)
            for (name, rows, _, _) in stage:
                self.qtype[name] = self.types[si]
                self.W[name] = synth.weight_rows(self.types[si], 100 + 17 * seed + len(self.W), rows, cols)
                self.Wd[name] = _dev(torch, self.W[name])
                self.y[name] = torch.full((M, rows), float("nan"), dtype=torch.float32, device="cuda")
                self.shape[name] = (rows, cols)
            x = self.x0 if src == "x0" else self.y[src]
            self.plan.append(([self.Wd[n] for (n, _, _, _) in stage], [r for (_, r, _, _) in stage], cols, x,
                              [self.y[n] for (n, _, _, _) in stage]))
        self.names = [[n for (n, _, _, _) in stage] for stage in stages]
        self.srcs = [stage[0][3] for stage in stages]
        self.chain = ggq.Chain(qtype if isinstance(qtype, int) else self.types, M, self.plan)

    def run(self, x0):
        self.x0.copy_(self.torch.from_numpy(x0))
        for y in self.y.values():
            y.fill_(float("nan"))
        self.chain.run()
        self.torch.cuda.synchronize()
        assert self.ggq.device_status() == 0
        return {n: y.cpu().numpy() for n, y in self.y.items()}

    def check(self, x0, out):
        worst = 0.0
        for names, src in zip(self.names, self.srcs):
            x = x0 if src == "x0" else out[src]
            assert np.isfinite(x).all()
            for n in names:
                rows, cols = self.shape[n]
                y_ref, a_ref = oracle.gemv(self.qtype[n], self.W[n], rows, cols, x)
                ok, w = oracle.tolerance_ok(out[n], y_ref, a_ref, REL, ABS)
                assert ok, f"{n}: worst error / bound = {w:.3g}"
                worst = max(worst, w)
        return worst


def _layer(prefix, hidden, kv, ffn, src):
    return [
        [(f"{prefix}q", hidden, hidden, src), (f"{prefix}k", kv, hidden, src), (f"{prefix}v", kv, hidden, src)],
        [(f"{prefix}o", hidden, hidden, f"{prefix}q")],
        [(f"{prefix}gate", ffn, hidden, f"{prefix}o"), (f"{prefix}up", ffn, hidden, f"{prefix}o")],
        [(f"{prefix}down", hidden, ffn, f"{prefix}gate")],
    ]


@pytest.mark.parametrize("qtype,M", [(12, 1), (12, 2), (12, 3), (8, 1), (8, 4), (2, 1), (2, 3)])
def test_chain_two_layers(env, qtype, M):
    """Two small layers: every stage after the first reads the previous stage's y."""
    stages = _layer("a.", 1280, 256, 2816, "x0") + _layer("b.", 1280, 256, 2816, "a.down")
    net = Net(env, qtype, M, stages)
    for run in range(2):
        x0 = synth.normal_f32(M * 1280, 40 + run).reshape(M, 1280)
        net.check(x0, net.run(x0))


def test_chain_repeat_is_bit_identical(env):
    stages = _layer("a.", 2048, 512, 5632, "x0")
    net = Net(env, 12, 1, stages, seed=1)
    x0 = synth.normal_f32(2048, 50).reshape(1, 2048)
    a = net.run(x0)
    b = net.run(x0)
    for n in a:
        assert np.array_equal(a[n].view(np.uint32), b[n].view(np.uint32)), n
    net.check(x0, a)


@pytest.mark.parametrize("qtype", [12, 8, 2, 14])
@pytest.mark.parametrize("rows", [3000, 151 * 16, 152 * 16, 152 * 16 + 5, 40000])
def test_chain_single_stage_matches_oracle_and_gemv(env, qtype, rows):
    """A one-stage chain against the oracle and against ggq_gemv, for each
    streamed weight type.  Row counts below, at and above one 16-row group per
    SM, and ragged: each CTA takes whole 16-row groups, whose tiles its
    consumer warps share in equal runs (a group cut between warps is added in
    warp order); both within the bound, and repeated chain runs bit-identical."""
    torch, ggq = env
    cols = 4096
    W = synth.weight_rows(qtype, 60, rows, cols)
    x = synth.normal_f32(cols, 61).reshape(1, cols)
    y_ref, a_ref = oracle.gemv(qtype, W, rows, cols, x)
    Wd, xd = _dev(torch, W), _dev(torch, x)
    y1 = ggq.gemv(qtype, Wd, rows, cols, xd)
    y2 = torch.full_like(y1, float("nan"))
    ch = ggq.Chain(qtype, 1, [([Wd], [rows], cols, xd, [y2])])
    outs = []
    for _ in range(3):
        y2.fill_(float("nan"))
        ch.run()
        torch.cuda.synchronize()
        outs.append(y2.cpu().numpy().copy())
    assert ggq.device_status() == 0
    for y in (y1.cpu().numpy(), outs[0]):
        ok, w = oracle.tolerance_ok(y, y_ref, a_ref, REL, ABS)
        assert ok, f"worst error / bound = {w:.3g}"
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32))


def test_chain_uneven_stages(env):
    """Stages far smaller than the grid (a few tiles) next to large ones, and
    ragged row counts that end inside a row block."""
    stages = [
        [("s0", 1280, 1280, "x0"), ("t0", 33, 1280, "x0")],
        [("s1", 4099, 1280, "s0"), ("s2", 1, 1280, "s0"), ("s3", 65, 1280, "s0")],
        [("s4", 1536, 1280, "s0")],                 # reads the output of two stages back
        [("s5", 70000, 1536, "s4")],
    ]
    net = Net(env, 12, 1, stages, seed=2)
    x0 = synth.normal_f32(1280, 70).reshape(1, 1280)
    net.check(x0, net.run(x0))


def test_chain_llama8b_layers(env):
    """Two Llama-8B-shaped Q4_K layers (hidden 4096, kv 1024, ffn 14336)."""
    stages = _layer("a.", 4096, 1024, 14336, "x0") + _layer("b.", 4096, 1024, 14336, "a.down")
    net = Net(env, 12, 1, stages, seed=3)
    x0 = synth.normal_f32(4096, 80).reshape(1, 4096)
    net.check(x0, net.run(x0))


# ---- chains of mixed weight types (Q4_K_M-style files) ------------------------

Q8_0, Q4_K, Q4_0, Q6_K = 8, 12, 2, 14


def _mixed_stages(other=Q4_K):
    """Two layers (hidden 2048, kv 512, ffn 4096) as in a Q4_K_M file: q/k,
    o and gate/up in `other` (Q4_K, or Q4_0), v and down in Q6_K in the first
    layer, only down in the second."""
    stages = [
        [("a.q", 2048, 2048, "x0"), ("a.k", 512, 2048, "x0")],
        [("a.v", 512, 2048, "x0")],
        [("a.o", 2048, 2048, "a.q")],
        [("a.gate", 4096, 2048, "a.o"), ("a.up", 4096, 2048, "a.o")],
        [("a.down", 2048, 4096, "a.gate")],
        [("b.q", 2048, 2048, "a.down"), ("b.k", 512, 2048, "a.down"), ("b.v", 512, 2048, "a.down")],
        [("b.o", 2048, 2048, "b.q")],
        [("b.gate", 4096, 2048, "b.o"), ("b.up", 4096, 2048, "b.o")],
        [("b.down", 2048, 4096, "b.gate")],
    ]
    types = [other, Q6_K, other, other, Q6_K, other, other, other, Q6_K]
    return stages, types


@pytest.mark.parametrize("other,M", [(Q4_K, 1), (Q4_K, 2), (Q4_K, 3), (Q4_0, 1), (Q4_0, 4)])
def test_chain_mixed_types(env, other, M):
    """One launch over stages of two weight types, each stage decoded by its
    own type; every stage against the oracle fed with what it read."""
    stages, types = _mixed_stages(other)
    net = Net(env, types, M, stages, seed=7)
    for run in range(2):
        x0 = synth.normal_f32(M * 2048, 150 + run).reshape(M, 2048)
        net.check(x0, net.run(x0))


def test_chain_mixed_stage_equals_uniform_chain(env):
    """A stage of a mixed chain is computed exactly as in a chain of its own
    type (same tiles, same order of sums): its outputs are bit-identical."""
    torch, ggq = env
    stages, types = _mixed_stages()
    net = Net(env, types, 1, stages, seed=8)
    x0 = synth.normal_f32(2048, 160).reshape(1, 2048)
    out = net.run(x0)
    for names, qt in ((["a.q", "a.k"], Q4_K), (["a.v"], Q6_K)):
        ys = [torch.full((1, net.shape[n][0]), float("nan"), dtype=torch.float32, device="cuda") for n in names]
        ch = ggq.Chain(qt, 1, [([net.Wd[n] for n in names], [net.shape[n][0] for n in names], 2048, net.x0, ys)])
        ch.run()
        torch.cuda.synchronize()
        for n, y in zip(names, ys):
            assert np.array_equal(y.cpu().numpy().view(np.uint32), out[n].view(np.uint32)), n


def test_chain_typed_with_one_type_is_the_uniform_chain(env):
    """ggq_chain_create_typed with every stage of one type runs the same kernel
    as ggq_chain_create: bit-identical outputs."""
    stages = _layer("a.", 2048, 512, 4096, "x0")
    a = Net(env, Q4_K, 1, stages, seed=9)
    b = Net(env, [Q4_K] * len(stages), 1, stages, seed=9)
    x0 = synth.normal_f32(2048, 170).reshape(1, 2048)
    ya, yb = a.run(x0), b.run(x0)
    for n in ya:
        assert np.array_equal(ya[n].view(np.uint32), yb[n].view(np.uint32)), n


def test_chain_in_cuda_graph(env):
    torch, ggq = env
    stages = _layer("a.", 1280, 256, 2816, "x0")
    net = Net(env, 12, 1, stages, seed=4)
    x0 = synth.normal_f32(1280, 90).reshape(1, 1280)
    net.run(x0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    net.chain.run(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            net.chain.run(s)
    torch.cuda.synchronize()
    x1 = synth.normal_f32(1280, 91).reshape(1, 1280)
    net.x0.copy_(torch.from_numpy(x1))
    for y in net.y.values():
        y.fill_(float("nan"))
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert ggq.device_status() == 0
    out = {n: y.cpu().numpy() for n, y in net.y.items()}
    net.check(x1, out)


# ---- fused steps: RMSNorm / SiLU(gate)*up on x, residual add on y -----------

from oracle import layer_ops  # noqa: E402


def _fused_layers(torch, ggq, qtype, M, H, KV, F, layers, seed, types=None):
    """A residual stream through `layers` Llama-style layers as one fused chain:
    [q,k,v](rmsnorm(h)), [o](q) + h, [gate,up](rmsnorm(h2)), [down](silu(gate)*up) + h2.
    types: None (every matrix qtype) or {(layer, name): type} for the matrices
    that differ; a stage whose matrices differ in type is split by type (same
    x and fused step).  Returns the chain, the buffers and, per stage, what the
    oracle needs."""
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()   # noqa: E731
    h0 = torch.empty((M, H), dtype=torch.float32, device="cuda")
    stages, ops, plan, stypes = [], [], [], []
    h = h0
    for l in range(layers):
        W, T = {}, {}
        for j, (name, r, c) in enumerate([("q", H, H), ("k", KV, H), ("v", KV, H), ("o", H, H),
                                          ("gate", F, H), ("up", F, H), ("down", H, F)]):
            T[name] = (types or {}).get((l, name), qtype)
            W[name] = (synth.weight_rows(T[name], 300 + 31 * seed + 10 * l + j, r, c), r, c, T[name])
        Wd = {n: dev(w[0]) for n, w in W.items()}
        y = {n: torch.full((M, w[1]), float("nan"), dtype=torch.float32, device="cuda") for n, w in W.items()}
        g_attn = (1.0 + 0.1 * synth.normal_f32(H, 400 + 7 * seed + 2 * l)).astype(np.float32)
        g_ffn = (1.0 + 0.1 * synth.normal_f32(H, 401 + 7 * seed + 2 * l)).astype(np.float32)
        ga, gf = dev(g_attn), dev(g_ffn)
        eps = 1e-6
        layer = [(["q", "k", "v"], H, h, {"x_op": ggq.X_RMSNORM, "eps": eps, "norm_w": ga}, ("rms", h, g_attn, eps), None),
                 (["o"], H, y["q"], {"res": [h]}, ("plain", y["q"]), h),
                 (["gate", "up"], H, y["o"], {"x_op": ggq.X_RMSNORM, "eps": eps, "norm_w": gf},
                  ("rms", y["o"], g_ffn, eps), None),
                 (["down"], F, y["gate"], {"x_op": ggq.X_SILU_MUL, "up": y["up"]}, ("silu", y["gate"], y["up"]), y["o"])]
        for names, cols, x, op, xin, res in layer:
            for t in dict.fromkeys(T[n] for n in names):     # split by type, in order of first use
                part = [n for n in names if T[n] == t]
                stages.append(([Wd[n] for n in part], [W[n][1] for n in part], cols, x, [y[n] for n in part]))
                o = dict(op)
                if res is not None:
                    o["res"] = [res] * len(part)
                ops.append(o)
                stypes.append(t)
                plan.append((part, W, y, xin, res))
        h = y["down"]
    chain = ggq.Chain(qtype if types is None else stypes, M, stages, ops)
    return chain, h0, plan, (stages, ops)


def _check_fused(qtype, plan):
    worst = 0.0
    for names, W, y, xin, res in plan:
        xa = xin[1].cpu().numpy().astype(np.float64)          # what the stage read
        if xin[0] == "rms":
            xr = layer_ops.rmsnorm(xa, xin[2], xin[3])
        elif xin[0] == "silu":
            xr = layer_ops.silu_mul(xa, xin[2].cpu().numpy().astype(np.float64))
        else:
            xr = xa
        assert np.isfinite(xr).all()
        for n in names:
            w, rows, cols, wt = W[n]
            wd = oracle.dequantize(wt, w, rows, cols).astype(np.float64)   # exact decoded weights
            y_ref = xr @ wd.T
            a_ref = np.abs(xr) @ np.abs(wd).T
            if res is not None:
                r = res.cpu().numpy().astype(np.float64)
                y_ref = layer_ops.add(y_ref, r)
                a_ref = a_ref + np.abs(r)
            ok, wr = oracle.tolerance_ok(y[n].cpu().numpy(), y_ref, a_ref, REL, ABS)
            assert ok, f"{n}: worst error / bound = {wr:.3g}"
            worst = max(worst, wr)
    return worst


@pytest.mark.parametrize("qtype,M", [(12, 1), (12, 2), (12, 3), (8, 1), (8, 4), (2, 1), (2, 2), (2, 4)])
def test_chain_fused_layers(env, qtype, M):
    """Two fused layers (RMSNorm before q/k/v and gate/up, SiLU(gate)*up into down,
    residual adds after o and down) against the oracle's layer steps + GEMV,
    each stage fed with what it actually read on the GPU."""
    torch, ggq = env
    chain, h0, plan, _ = _fused_layers(torch, ggq, qtype, M, 1280, 256, 2816, 2, seed=qtype + M)
    for run in range(2):
        h0.copy_(torch.from_numpy((3.0 * synth.normal_f32(M * 1280, 500 + run)).reshape(M, 1280)))
        chain.run()
        torch.cuda.synchronize()
        assert ggq.device_status() == 0
        _check_fused(qtype, plan)


@pytest.mark.parametrize("M", [1, 3])
def test_chain_fused_layers_mixed_types(env, M):
    """Fused layers of a Q4_K_M-style file: v (first layer) and down in Q6_K
    (v's stage split from q/k, with the same fused step), the rest Q4_K."""
    torch, ggq = env
    types = {(0, "v"): Q6_K, (0, "down"): Q6_K, (1, "down"): Q6_K}
    chain, h0, plan, _ = _fused_layers(torch, ggq, Q4_K, M, 2048, 512, 4096, 2, seed=60 + M, types=types)
    for run in range(2):
        h0.copy_(torch.from_numpy((3.0 * synth.normal_f32(M * 2048, 530 + run)).reshape(M, 2048)))
        chain.run()
        torch.cuda.synchronize()
        assert ggq.device_status() == 0
        _check_fused(Q4_K, plan)


def test_chain_fused_residual_into_own_output(env):
    """res may be the stage's own y: y = W x + y_before."""
    torch, ggq = env
    rows, cols = 3000, 2048
    W = synth.weight_rows(12, 610, rows, cols)
    x = synth.normal_f32(cols, 611).reshape(1, cols)
    y0 = synth.normal_f32(rows, 612).reshape(1, rows)
    Wd, xd = _dev(torch, W), _dev(torch, x)
    yd = _dev(torch, y0)
    ch = ggq.Chain(12, 1, [([Wd], [rows], cols, xd, [yd])], [{"res": [yd]}])
    ch.run()
    torch.cuda.synchronize()
    assert ggq.device_status() == 0
    wd = oracle.dequantize(12, W, rows, cols).astype(np.float64)
    y_ref = x.astype(np.float64) @ wd.T + y0
    a_ref = np.abs(x.astype(np.float64)) @ np.abs(wd).T + np.abs(y0)
    ok, wr = oracle.tolerance_ok(yd.cpu().numpy(), y_ref, a_ref, REL, ABS)
    assert ok, wr


@pytest.mark.parametrize("M,cols", [(3, 4096), (2, 2048), (1, 12288)])
def test_chain_fused_rmsnorm_spiky_and_zero_rows(env, M, cols):
    """RMSNorm on activation rows of very different scale, one of them all zero
    (eps keeps it finite: its normalized x is 0); x held in one load batch a
    thread (cols 2048) or read twice (sum of squares first: cols 12288, M = 3)."""
    torch, ggq = env
    rows = 1500
    W = synth.weight_rows(12, 620, rows, cols)
    x = synth.normal_f32(M * cols, 621).reshape(M, cols).astype(np.float64)
    x[0] *= 1e-4
    if M > 1:
        x[1] = 0.0
    x[0 if M == 2 else M - 1, 17] = 5e4    # one spike, never in the zero row
    x = x.astype(np.float32)
    g = (1.0 + 0.1 * synth.normal_f32(cols, 622)).astype(np.float32)
    Wd, xd, gd = _dev(torch, W), _dev(torch, x), _dev(torch, g)
    yd = torch.full((M, rows), float("nan"), dtype=torch.float32, device="cuda")
    ch = ggq.Chain(12, M, [([Wd], [rows], cols, xd, [yd])], [{"x_op": ggq.X_RMSNORM, "eps": 1e-5, "norm_w": gd}])
    ch.run()
    torch.cuda.synchronize()
    assert ggq.device_status() == 0
    xr = layer_ops.rmsnorm(x.astype(np.float64), g, 1e-5)
    wd = oracle.dequantize(12, W, rows, cols).astype(np.float64)
    ok, wr = oracle.tolerance_ok(yd.cpu().numpy(), xr @ wd.T, np.abs(xr) @ np.abs(wd).T, REL, ABS)
    assert ok, wr
    if M > 1:
        assert np.array_equal(yd.cpu().numpy()[1], np.zeros(rows, dtype=np.float32))

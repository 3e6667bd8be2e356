"""GPU parity for Q6_K weights: decode and row gather bit-exact, GEMV within
the tolerance, one-hot and integer-valued cases exact, against the CPU oracle.
GEMVs with cols % 2048 == 0 run on the streaming kernel at M 1..4 and on the
tensor-core small-M kernel at M 5..16, the others on the warp-per-row kernel;
all are covered, and so are Q6_K chains of dependent stages.

Bar as for the other types: |y - y_ref| <= 1e-3 * sum_c |w[r,c] x[c]| + 1e-6
(y_ref in double).
"""
import numpy as np
import pytest

import oracle
import synth
from tests.pin_checks import q6k_block, q6k_raw
from tests.test_gpu_gemv import REL, ABS, _dev, assert_close, env, gpu_gemv  # noqa: F401

pytestmark = pytest.mark.gpu

Q6_K = 14


def weights(rows, cols, stream=7):
    return synth.weight_rows(Q6_K, stream, rows, cols)


def xs(M, cols, stream=8):
    return synth.normal_f32(M * cols, stream).reshape(M, cols)


@pytest.mark.parametrize("rows,cols", [(1, 256), (3, 512), (17, 2304), (40, 4096)])
def test_dequantize_bit_exact(env, rows, cols):
    torch, ggq = env
    W = weights(rows, cols)
    out = ggq.dequantize(Q6_K, _dev(torch, W), rows, cols)
    torch.cuda.synchronize()
    ref = oracle.dequantize(Q6_K, W, rows, cols)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_dequantize_every_code_extreme_scales_and_special_d(env):
    """Every code 0..63 in every quarter, scales -128 .. 127, and d = 1,
    subnormal, largest finite, -0, inf, NaN."""
    torch, ggq = env
    codes = [(k * 7) % 64 for k in range(256)]
    sc = [-128, 127, -1, 1, 0, 64, -64, 2, 3, -3, 100, -100, 5, -7, 11, -13]
    blocks = [q6k_block(d, sc, codes) for d in (0x3C00, 0x0001, 0x7BFF, 0x8000, 0x7C00, 0x7E00)]
    blocks.append(q6k_raw([0xFF] * 128, [0xFF] * 64, sc, 0x3800))
    W = np.frombuffer(b"".join(blocks), np.uint8).copy()
    rows = len(blocks)
    out = ggq.dequantize(Q6_K, _dev(torch, W), rows, 256)
    torch.cuda.synchronize()
    ref = oracle.dequantize(Q6_K, W, rows, 256)
    got = out.cpu().numpy()
    both_nan = np.isnan(got) & np.isnan(ref)
    assert np.array_equal(got.view(np.uint32)[~both_nan], ref.view(np.uint32)[~both_nan])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


# warp-per-row: cols % 2048 != 0; streaming: (33, 2048) a ragged row group,
# (100, 4096) fewer groups than SMs, (2056, 6144) 24 SBs a row, (4096, 14336)
SHAPES = [(1, 256), (31, 512), (33, 2304), (257, 11008), (4099, 1280),
          (33, 2048), (100, 4096), (2056, 6144), (4096, 14336)]


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("M", [1, 2, 3, 5, 8, 16])
def test_gemv_q6_k(env, rows, cols, M):
    W = weights(rows, cols, stream=17)
    x = xs(M, cols, stream=18)
    y_ref, a_ref = oracle.gemv(Q6_K, W, rows, cols, x)
    assert_close(gpu_gemv(env, Q6_K, W, rows, cols, x), y_ref, a_ref, f"q6_k {rows}x{cols} M={M}")


@pytest.mark.parametrize("cols", [256, 2304, 2048, 4096])
def test_gemv_one_hot_extracts_exact_columns(env, cols):
    rows = 37
    W = weights(rows, cols, stream=3)
    Wf = oracle.dequantize(Q6_K, W, rows, cols)
    for c in sorted({0, 1, 15, 16, 31, 32, 127, 128, 200, cols // 2 + 3, cols - 1}):
        x = np.zeros((1, cols), np.float32)
        x[0, c] = 1.0
        y = gpu_gemv(env, Q6_K, W, rows, cols, x)
        assert np.array_equal(y[0].view(np.uint32), Wf[:, c].view(np.uint32)), c


@pytest.mark.parametrize("M", [1, 4, 9])
def test_gemv_integer_inputs_are_exact(env, M):
    """d = 1, scales in -4..4, codes 0..63, x in -4..4: every partial sum is an
    integer below 2^24 in magnitude, so any summation order is exact."""
    rng = np.random.default_rng(M)
    rows, cols = 45, 2048
    sc = rng.integers(-4, 5, size=(rows, cols // 256, 16))
    u = rng.integers(0, 64, size=(rows, cols))
    W = np.frombuffer(b"".join(q6k_block(0x3C00, list(sc[r, b]), list(u[r, 256 * b:256 * b + 256]))
                               for r in range(rows) for b in range(cols // 256)), np.uint8).copy()
    w = sc[:, np.arange(cols) // 256, (np.arange(cols) % 256) // 16] * (u - 32)
    x = rng.integers(-4, 5, size=(M, cols)).astype(np.float32)
    y = gpu_gemv(env, Q6_K, W, rows, cols, x)
    assert np.array_equal(y.astype(np.int64), x.astype(np.int64) @ w.T)
    # the same weights at cols 2304 (warp-per-row kernel): the first 9 SBs of each row
    W9 = W.reshape(rows, cols // 256, 210)[:, :1].repeat(9, axis=1).reshape(-1).copy()
    w9 = np.tile(w[:, :256], 9)
    y9 = gpu_gemv(env, Q6_K, W9, rows, 2304, np.tile(x[:, :256], 9))
    assert np.array_equal(y9.astype(np.int64), np.tile(x[:, :256], 9).astype(np.int64) @ w9.T)


def test_gemv_multi_q6_k(env):
    torch, ggq = env
    cols, rows = 2048, [512, 2048]
    Ws = [weights(r, cols, stream=60 + i) for i, r in enumerate(rows)]
    x = xs(2, cols, stream=63)
    ys = ggq.gemv_multi(Q6_K, [_dev(torch, W) for W in Ws], rows, cols, _dev(torch, x))
    torch.cuda.synchronize()
    for W, r, y in zip(Ws, rows, ys):
        y_ref, a_ref = oracle.gemv(Q6_K, W, r, cols, x)
        assert_close(y.cpu().numpy(), y_ref, a_ref, f"multi {r}")


@pytest.mark.parametrize("rows,cols", [(14336, 4096), (4096, 14336)])
def test_full_size_sampled(env, rows, cols):
    """Full-size matrices in the bench's launch configuration (M = 1); rows
    sampled for the oracle (regenerated alone from their counters)."""
    W = synth.weight_rows(Q6_K, 70, rows, cols)
    x = synth.normal_f32(cols, 71).reshape(1, -1)
    y = gpu_gemv(env, Q6_K, W, rows, cols, x)
    rng = np.random.default_rng(2)
    rows_s = np.unique(np.r_[0, 15, 16, rows - 1, rng.integers(0, rows, 96)])
    rb = oracle.row_bytes(Q6_K, cols)
    Ws = np.concatenate([synth.weight_rows(Q6_K, 70, 1, cols, row0=int(r)) for r in rows_s])
    assert np.array_equal(Ws[:rb], W[:rb])
    y_ref, a_ref = oracle.gemv(Q6_K, Ws, len(rows_s), cols, x)
    assert_close(y[:, rows_s], y_ref, a_ref, f"q6_k {rows}x{cols}")


def test_repeated_calls_are_bit_identical(env):
    torch, ggq = env
    rows, cols = 3000, 4096
    W = weights(rows, cols, stream=64)
    x = xs(3, cols, stream=65)
    Wd, xd = _dev(torch, W), _dev(torch, x)
    outs = [ggq.gemv(Q6_K, Wd, rows, cols, xd).cpu().numpy() for _ in range(3)]
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32))


@pytest.mark.parametrize("cols", [256, 4096])
def test_embed_rows_bit_exact(env, cols):
    torch, ggq = env
    rows = 300
    W = weights(rows, cols, stream=80)
    ids = np.array([0, 299, 17, 17, 150, 1], dtype=np.int32)
    out = ggq.embed(Q6_K, _dev(torch, W), rows, cols, _dev(torch, ids))
    torch.cuda.synchronize()
    assert ggq.device_status() == 0
    ref = oracle.dequantize(Q6_K, W, rows, cols)[ids]
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


# ---- Q6_K chains (the streaming kernel's stage boundaries) ---------------------

from tests.test_gpu_chain import Net, _layer, _fused_layers, _check_fused  # noqa: E402


@pytest.mark.parametrize("M", [1, 2, 4])
def test_chain_q6_k_two_layers(env, M):
    """Two layers (hidden 2048, kv 512, ffn 4096): each stage reads the
    previous stage's y, checked against the oracle fed with what it read."""
    stages = _layer("a.", 2048, 512, 4096, "x0") + _layer("b.", 2048, 512, 4096, "a.down")
    net = Net(env, Q6_K, M, stages, seed=5)
    for run in range(2):
        x0 = synth.normal_f32(M * 2048, 140 + run).reshape(M, 2048)
        net.check(x0, net.run(x0))


@pytest.mark.parametrize("M", [1, 3])
def test_chain_q6_k_fused_layers(env, M):
    torch, ggq = env
    chain, h0, plan, _ = _fused_layers(torch, ggq, Q6_K, M, 2048, 512, 4096, 2, seed=40 + M)
    for run in range(2):
        h0.copy_(torch.from_numpy((3.0 * synth.normal_f32(M * 2048, 520 + run)).reshape(M, 2048)))
        chain.run()
        torch.cuda.synchronize()
        assert ggq.device_status() == 0
        _check_fused(Q6_K, plan)

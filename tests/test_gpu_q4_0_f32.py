"""GPU parity for Q4_0 and F32 weights: decode bit-exact, GEMV (the streaming
kernel for Q4_0 at cols % 256 == 0, cols >= 768, M <= 4; the warp-per-row
kernel for F32 and the other Q4_0 shapes), row gather, against the CPU oracle.

Bar as for the other types: decode and row gather bit-exact; GEMV within
|y - y_ref| <= 1e-3 * sum_c |w[r,c] x[c]| + 1e-6 (y_ref in double);
one-hot and integer-valued cases exact.
"""
import numpy as np
import pytest

import oracle
import synth
from tests.pin_checks import q4_0_block
from tests.test_gpu_gemv import REL, ABS, _dev, assert_close, env, gpu_gemv  # noqa: F401

pytestmark = pytest.mark.gpu

Q4_0, F32 = 2, 0


def weights(qtype, rows, cols, stream=7):
    return synth.weight_rows(qtype, stream, rows, cols)


def xs(M, cols, stream=8):
    return synth.normal_f32(M * cols, stream).reshape(M, cols)


# streaming-kernel shapes (one and several 256-column periods, ragged row
# groups) and warp-per-row shapes (cols % 256 != 0 or cols < 768)
Q40_STREAM = [(1, 768), (31, 1024), (33, 2304), (100, 4096), (257, 11008), (4099, 1280)]
Q40_ROWS = [(1, 32), (3, 96), (31, 256), (33, 512), (9, 4096 + 32)]
F32_SHAPES = [(1, 1), (3, 5), (31, 7), (33, 512), (100, 2048), (257, 4096 + 4), (64, 4099)]


@pytest.mark.parametrize("qtype,rows,cols", [(Q4_0, 1, 32), (Q4_0, 3, 96), (Q4_0, 17, 512), (Q4_0, 65, 2304),
                                             (F32, 3, 5), (F32, 17, 512)])
def test_dequantize_bit_exact(env, qtype, rows, cols):
    torch, ggq = env
    W = weights(qtype, rows, cols)
    out = ggq.dequantize(qtype, _dev(torch, W), rows, cols)
    torch.cuda.synchronize()
    ref = oracle.dequantize(qtype, W, rows, cols)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_dequantize_q4_0_every_code_and_special_scales(env):
    """Every code 0..15 in both nibbles, with scales 1, subnormal, largest
    finite, -0, inf and NaN."""
    torch, ggq = env
    codes = [(i % 16) for i in range(32)]
    codes2 = [15 - c for c in codes]
    blocks = [q4_0_block(d, c) for d in (0x3C00, 0x0001, 0x7BFF, 0x8000, 0x7C00, 0x7E00) for c in (codes, codes2)]
    W = np.frombuffer(b"".join(blocks), np.uint8).copy()
    rows = len(blocks)
    out = ggq.dequantize(Q4_0, _dev(torch, W), rows, 32)
    torch.cuda.synchronize()
    ref = oracle.dequantize(Q4_0, W, rows, 32)
    got = out.cpu().numpy()
    both_nan = np.isnan(got) & np.isnan(ref)
    assert np.array_equal(got.view(np.uint32)[~both_nan], ref.view(np.uint32)[~both_nan])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


@pytest.mark.parametrize("rows,cols", Q40_STREAM + Q40_ROWS)
def test_gemv_q4_0_m1(env, rows, cols):
    W = weights(Q4_0, rows, cols)
    x = xs(1, cols)
    y_ref, a_ref = oracle.gemv(Q4_0, W, rows, cols, x)
    assert_close(gpu_gemv(env, Q4_0, W, rows, cols, x), y_ref, a_ref, f"q4_0 {rows}x{cols}")


@pytest.mark.parametrize("rows,cols", [(33, 2304), (70, 4096), (9, 96), (40, 512)])
@pytest.mark.parametrize("M", [2, 3, 4, 5, 8, 16])
def test_gemv_q4_0_small_m(env, rows, cols, M):
    W = weights(Q4_0, rows, cols, stream=13)
    x = xs(M, cols, stream=14)
    y_ref, a_ref = oracle.gemv(Q4_0, W, rows, cols, x)
    assert_close(gpu_gemv(env, Q4_0, W, rows, cols, x), y_ref, a_ref, f"q4_0 {rows}x{cols} M={M}")


@pytest.mark.parametrize("rows,cols", F32_SHAPES)
@pytest.mark.parametrize("M", [1, 2, 3, 8, 16])
def test_gemv_f32(env, rows, cols, M):
    W = weights(F32, rows, cols, stream=15)
    x = xs(M, cols, stream=16)
    y_ref, a_ref = oracle.gemv(F32, W, rows, cols, x)
    assert_close(gpu_gemv(env, F32, W, rows, cols, x), y_ref, a_ref, f"f32 {rows}x{cols} M={M}")


@pytest.mark.parametrize("qtype,cols", [(Q4_0, 2304), (Q4_0, 96), (F32, 7), (F32, 2048)])
def test_gemv_one_hot_extracts_exact_columns(env, qtype, cols):
    rows = 37
    W = weights(qtype, rows, cols, stream=3)
    Wf = oracle.dequantize(qtype, W, rows, cols)
    for c in sorted(c for c in {0, 1, 17, cols // 2 + 3, cols - 1} if c < cols):
        x = np.zeros((1, cols), np.float32)
        x[0, c] = 1.0
        y = gpu_gemv(env, qtype, W, rows, cols, x)
        assert np.array_equal(y[0].view(np.uint32), Wf[:, c].view(np.uint32)), c


@pytest.mark.parametrize("cols,M", [(2048, 1), (2048, 3), (4096, 4), (512, 2), (2048, 7)])
def test_gemv_q4_0_integer_inputs_are_exact(env, cols, M):
    """d = 1 and small integer x: every partial sum is an exact integer."""
    rng = np.random.default_rng(cols + M)
    rows = 45
    u = rng.integers(0, 16, size=(rows, cols))
    W = np.frombuffer(b"".join(q4_0_block(0x3C00, list(u[r, 32 * b:32 * b + 32]))
                               for r in range(rows) for b in range(cols // 32)), np.uint8).copy()
    x = rng.integers(-8, 9, size=(M, cols)).astype(np.float32)
    y = gpu_gemv(env, Q4_0, W, rows, cols, x)
    assert np.array_equal(y.astype(np.int64), x.astype(np.int64) @ (u - 8).T)


def test_gemv_f32_integer_inputs_are_exact(env):
    rng = np.random.default_rng(4)
    rows, cols, M = 50, 1031, 3
    w = rng.integers(-64, 65, size=(rows, cols)).astype(np.float32)
    x = rng.integers(-8, 9, size=(M, cols)).astype(np.float32)
    y = gpu_gemv(env, F32, w.reshape(-1).view(np.uint8), rows, cols, x)
    assert np.array_equal(y.astype(np.int64), x.astype(np.int64) @ w.astype(np.int64).T)


def test_gemv_multi_q4_0(env):
    """q, k, v of one layer sharing x in one launch."""
    torch, ggq = env
    cols, rows = 2048, [2048, 512, 512]
    Ws = [weights(Q4_0, r, cols, stream=60 + i) for i, r in enumerate(rows)]
    x = xs(2, cols, stream=63)
    ys = ggq.gemv_multi(Q4_0, [_dev(torch, W) for W in Ws], rows, cols, _dev(torch, x))
    torch.cuda.synchronize()
    for W, r, y in zip(Ws, rows, ys):
        y_ref, a_ref = oracle.gemv(Q4_0, W, r, cols, x)
        assert_close(y.cpu().numpy(), y_ref, a_ref, f"multi {r}")


def test_gemv_q4_0_repeated_calls_are_bit_identical(env):
    torch, ggq = env
    rows, cols = 3000, 4096
    W = weights(Q4_0, rows, cols, stream=64)
    x = xs(1, cols, stream=65)
    Wd, xd = _dev(torch, W), _dev(torch, x)
    outs = [ggq.gemv(Q4_0, Wd, rows, cols, xd).cpu().numpy() for _ in range(3)]
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32))
    y_ref, a_ref = oracle.gemv(Q4_0, W, rows, cols, x)
    assert_close(outs[0], y_ref, a_ref, "repeat")


@pytest.mark.parametrize("qtype,rows,cols", [(Q4_0, 14336, 4096), (Q4_0, 4096, 14336), (F32, 14336, 4096)])
def test_full_size_sampled(env, qtype, rows, cols):
    """Full-size matrices in the bench's launch configuration (M = 1); rows
    sampled for the oracle (regenerated alone from their counters)."""
    W = synth.weight_rows(qtype, 70, rows, cols)
    x = synth.normal_f32(cols, 71).reshape(1, -1)
    y = gpu_gemv(env, qtype, W, rows, cols, x)
    rng = np.random.default_rng(2)
    rows_s = np.unique(np.r_[0, 15, 16, rows - 1, rng.integers(0, rows, 96)])
    rb = oracle.row_bytes(qtype, cols)
    Ws = np.concatenate([synth.weight_rows(qtype, 70, 1, cols, row0=int(r)) for r in rows_s])
    assert np.array_equal(Ws[:rb], W[:rb])
    y_ref, a_ref = oracle.gemv(qtype, Ws, len(rows_s), cols, x)
    assert_close(y[:, rows_s], y_ref, a_ref, f"type {qtype} {rows}x{cols}")


@pytest.mark.parametrize("qtype,cols", [(Q4_0, 64), (Q4_0, 2048), (F32, 7), (F32, 4096)])
def test_embed_rows_bit_exact(env, qtype, cols):
    torch, ggq = env
    rows = 300
    W = weights(qtype, rows, cols, stream=80)
    ids = np.array([0, 299, 17, 17, 150, 1], dtype=np.int32)
    out = ggq.embed(qtype, _dev(torch, W), rows, cols, _dev(torch, ids))
    torch.cuda.synchronize()
    assert ggq.device_status() == 0
    ref = oracle.dequantize(qtype, W, rows, cols)[ids]
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))

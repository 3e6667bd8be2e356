"""The oracle's full-size GEMV / GEMM (decoded weights times x in one float64
matrix product per row block) against its column-loop GEMV and GEMM on the
same inputs: the same definition in another summation order, so they agree to
float64 rounding on random data and exactly on integer data (no GPU)."""
import numpy as np
import pytest

import oracle
import synth


@pytest.mark.parametrize("qtype,rows,cols,M", [(8, 37, 512, 1), (12, 70, 768, 3), (2, 19, 160, 2), (14, 33, 512, 4),
                                               (0, 9, 40, 2), (12, 300, 256, 1)])
def test_dense_gemv_matches_loop(qtype, rows, cols, M):
    W = synth.weight_rows(qtype, 300 + qtype, rows, cols)
    x = synth.normal_f32(M * cols, 301).reshape(M, cols)
    y1, a1 = oracle.gemv(qtype, W, rows, cols, x)
    y2, a2 = oracle.gemv_dense(qtype, W, rows, cols, x, chunk=16)   # several row blocks, one ragged
    assert y2.shape == (M, rows)
    np.testing.assert_allclose(y2, y1, rtol=0, atol=1e-12 * np.max(a1))
    np.testing.assert_allclose(a2, a1, rtol=1e-13)


def test_dense_gemv_integer_exact():
    # Q8_0 blocks with d = 1 and integer codes, integer x: every sum exact
    rows, cols = 24, 256
    rng = np.random.default_rng(5)
    q = rng.integers(-127, 128, size=(rows, cols // 32, 32))
    blk = np.zeros((rows, cols // 32, 34), np.uint8)
    blk[:, :, 0:2] = np.frombuffer(np.float16(1.0).tobytes(), np.uint8)
    blk[:, :, 2:] = q.astype(np.int8).view(np.uint8)
    x = rng.integers(-8, 9, size=(2, cols)).astype(np.float32)
    y, a = oracle.gemv_dense(8, blk.reshape(-1), rows, cols, x, chunk=7)
    want = x.astype(np.int64) @ q.reshape(rows, cols).T
    assert np.array_equal(y, want.astype(np.float64))
    assert np.array_equal(a, (np.abs(x).astype(np.int64) @ np.abs(q.reshape(rows, cols)).T).astype(np.float64))


@pytest.mark.parametrize("qtype", [12, 8])
def test_dense_gemm_matches_loop(qtype):
    rows, cols, M = 40, 512, 5
    W = synth.weight_rows(qtype, 310, rows, cols)
    X = synth.normal_bf16(M * cols, 311).reshape(M, cols)
    Y1, A1 = oracle.gemm_bf16(qtype, W, rows, cols, X)
    Y2, A2 = oracle.gemm_bf16_dense(qtype, W, rows, cols, X, chunk=16)
    np.testing.assert_allclose(Y2, Y1, rtol=0, atol=1e-12 * np.max(A1))
    np.testing.assert_allclose(A2, A1, rtol=1e-13)


def test_dense_gemm_widens_bf16_exactly():
    # one-hot bf16 X: Y[m] is a decoded column exactly; a bf16 of 1.5 widened is 1.5
    rows, cols = 16, 256
    W = synth.weight_rows(12, 312, rows, cols)
    X = np.zeros((2, cols), np.uint16)
    X[0, 7] = 0x3FC0          # 1.5
    X[1, 200] = 0xBF80        # -1.0
    w = oracle.dequantize(12, W, rows, cols).astype(np.float64)
    Y, _ = oracle.gemm_bf16_dense(12, W, rows, cols, X)
    assert np.array_equal(Y[0], 1.5 * w[:, 7]) and np.array_equal(Y[1], -w[:, 200])

"""GPU parity of the tcgen05 prefill dequant-GEMM (ggq_gemm_prefill) against the oracle.

Y[M, rows] = X[M, cols] W^T with W Q4_K or Q8_0 and X bf16.  The GPU decodes W to bf16
in shared memory; the oracle uses the exact fp32 weights.  Bar:
|Y - Y_ref| <= 1e-3 * sum_c |w x| + 1e-6.  Integer-valued cases whose weights
are exact in bf16 must match exactly; one-hot rows of X return bf16(w) exactly.
"""
import numpy as np
import pytest

import oracle
import synth
from synth import workloads as WL
from tests.pin_checks import pack_q4_k

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("-m gpu tests need a CUDA device")
    import gguf_block_quantized_q8_gb300 as ggq
    return torch, ggq


def gpu_prefill(env, W, rows, cols, X_bits, qtype=12):
    torch, ggq = env
    M = X_bits.shape[0]
    Wd = torch.from_numpy(np.ascontiguousarray(W)).cuda()
    Xd = torch.from_numpy(np.ascontiguousarray(X_bits).view(np.int16)).cuda()
    guard = 256
    buf = torch.full((M * rows + 2 * guard,), float("nan"), dtype=torch.float32, device="cuda")
    Y = buf[guard:guard + M * rows]
    ggq.check(ggq.ggq_gemm_prefill(qtype, Wd.data_ptr(), rows, cols, Xd.data_ptr(), Y.data_ptr(), M,
                                   torch.cuda.current_stream().cuda_stream), "ggq_gemm_prefill")
    torch.cuda.synchronize()
    assert ggq.device_status() == 0, "a bounded wait timed out"
    out = buf.cpu().numpy()
    assert np.isnan(out[:guard]).all() and np.isnan(out[guard + M * rows:]).all(), "write outside Y"
    return out[guard:guard + M * rows].reshape(M, rows)


def bf16_round(a: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def int_q4k(rng, rows, cols, sc_max=16, m_max=63):
    sc = rng.integers(0, sc_max + 1, size=(rows, cols // 256, 8))
    mm = rng.integers(0, m_max + 1, size=(rows, cols // 256, 8))
    qq = rng.integers(0, 16, size=(rows, cols))
    W = np.frombuffer(b"".join(pack_q4_k(0x3C00, 0x3C00, list(sc[r, b]), list(mm[r, b]),
                                         list(qq[r, 256 * b:256 * b + 256]))
                               for r in range(rows) for b in range(cols // 256)), np.uint8).copy()
    j = (np.arange(cols) % 256) // 32
    bi = np.arange(cols) // 256
    return W, sc[:, bi, j] * qq - mm[:, bi, j]


@pytest.mark.parametrize("rows,cols,M", [(128, 256, 128), (256, 512, 256), (128, 2048, 512), (384, 1024, 384),
                                         (256, 768, 1024), (1280, 512, 512)])
def test_prefill_integer_exact(env, rows, cols, M):
    """Weights |w| <= 240 and X in [-8, 8] are exact in bf16; every sum is exact."""
    rng = np.random.default_rng(rows + cols + M)
    W, w = int_q4k(rng, rows, cols)
    X = rng.integers(-8, 9, size=(M, cols)).astype(np.float32)
    bits = (X.view(np.uint32) >> 16).astype(np.uint16)
    Y = gpu_prefill(env, W, rows, cols, bits)
    assert np.array_equal(Y.astype(np.int64), X.astype(np.int64) @ w.T)


def int_q8_0(rng, rows, cols):
    """Q8_0 blocks with d = 1 and q in [-127, 127]: every weight an integer, exact in bf16."""
    q = rng.integers(-127, 128, size=(rows, cols))
    blocks = q.reshape(rows, cols // 32, 32).astype(np.int8)
    W = np.empty((rows, cols // 32, 34), np.uint8)
    W[:, :, 0:2] = np.frombuffer(np.uint16(0x3C00).tobytes(), np.uint8)   # fp16 1.0
    W[:, :, 2:] = blocks.view(np.uint8)
    return W.reshape(-1).copy(), q


@pytest.mark.parametrize("rows,cols,M", [(128, 256, 128), (256, 1024, 256), (128, 2304, 384)])
def test_prefill_q8_0_integer_exact(env, rows, cols, M):
    """Q8_0 with d = 1: |w| <= 127 and X in [-8, 8] are exact in bf16; every sum is exact."""
    rng = np.random.default_rng(rows + cols + M + 1)
    W, w = int_q8_0(rng, rows, cols)
    X = rng.integers(-8, 9, size=(M, cols)).astype(np.float32)
    bits = (X.view(np.uint32) >> 16).astype(np.uint16)
    Y = gpu_prefill(env, W, rows, cols, bits, qtype=8)
    assert np.array_equal(Y.astype(np.int64), X.astype(np.int64) @ w.T)


@pytest.mark.parametrize("qtype,M", [(12, 256), (8, 256), (12, 512)])
def test_prefill_one_hot_rows(env, qtype, M):
    rows, cols = 256, 1024
    W = synth.weight_rows(qtype, 61, rows, cols)
    wb = bf16_round(oracle.dequantize(qtype, W, rows, cols))
    X = np.zeros((M, cols), np.float32)
    cs = (np.arange(M) * 37) % cols
    X[np.arange(M), cs] = 1.0
    bits = (X.view(np.uint32) >> 16).astype(np.uint16)
    Y = gpu_prefill(env, W, rows, cols, bits, qtype=qtype)
    assert np.array_equal(Y, wb[:, cs].T)


@pytest.mark.parametrize("qtype", [12, 8])
@pytest.mark.parametrize("rows,cols,M", [(128, 256, 128), (256, 4096, 256), (512, 2304, 512), (384, 1536, 1024),
                                         (128, 1024, 1536), (20352, 512, 512)])
def test_prefill_random(env, qtype, rows, cols, M):
    W = synth.weight_rows(qtype, 62, rows, cols)
    X = synth.normal_bf16(M * cols, 63).reshape(M, cols)
    Y = gpu_prefill(env, W, rows, cols, X, qtype=qtype)
    Y_ref, A_ref = oracle.gemm_bf16(qtype, W, rows, cols, X)
    ok, worst = oracle.tolerance_ok(Y, Y_ref, A_ref)
    assert ok, f"worst error / bound = {worst:.3g}"


def test_prefill_cfg5_full(env):
    """The full prefill shape (Q4_K 14336 x 4096, X 512 x 4096 bf16): all
    512 x 14336 outputs against the oracle (decoded weights times the exactly
    widened X, float64)."""
    g = WL.CFG5
    W = synth.weight_rows(g.qtype, g.stream, g.rows, g.cols)
    X = synth.normal_bf16(WL.CFG5_M * g.cols, g.x_stream).reshape(WL.CFG5_M, g.cols)
    Y = gpu_prefill(env, W, g.rows, g.cols, X)
    assert np.isfinite(Y).all()
    Y_ref, A_ref = oracle.gemm_bf16_dense(g.qtype, W, g.rows, g.cols, X)
    ok, worst = oracle.tolerance_ok(Y, Y_ref, A_ref)
    assert ok, f"worst error / bound = {worst:.3g}"


def test_prefill_cfg5_q8_0_full(env):
    """The same shape with Q8_0 weights: every output against the oracle."""
    g = WL.CFG5
    W = synth.weight_rows(8, g.stream, g.rows, g.cols)
    X = synth.normal_bf16(WL.CFG5_M * g.cols, g.x_stream).reshape(WL.CFG5_M, g.cols)
    Y = gpu_prefill(env, W, g.rows, g.cols, X, qtype=8)
    Y_ref, A_ref = oracle.gemm_bf16_dense(8, W, g.rows, g.cols, X)
    ok, worst = oracle.tolerance_ok(Y, Y_ref, A_ref)
    assert ok, f"worst error / bound = {worst:.3g}"

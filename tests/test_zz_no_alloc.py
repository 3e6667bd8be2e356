"""ggq_gemv_noalloc: the GEMV for callers that may not allocate device memory
(a server whose device memory all belongs to its own pool, or a loop where a
cudaMalloc/cudaFree and the device-wide synchronisation it may bring are not
allowed).  Through the C ABI, on two calls in a row, it must agree with the
oracle and with ggq_gemv within the parity bound, and allocate nothing.

Kept in a file pytest collects last, so that a run stopping at the first
failure has already run every other test; it also passes alone in a fresh
process.
"""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("-m gpu tests need a CUDA device")
    import gguf_block_quantized_q8_gb300 as ggq
    return torch, ggq


@pytest.mark.parametrize("qtype,rows,cols,M", [(12, 4096, 4096, 1), (12, 1000, 11008, 2), (8, 2048, 2048, 1),
                                               (8, 777, 4096, 3), (2, 3000, 4096, 1), (2, 500, 1024, 4),
                                               (14, 3000, 4096, 1), (14, 1000, 14336, 2)])
def test_noalloc_matches_oracle_and_gemv_twice(env, qtype, rows, cols, M):
    """Two calls in a row: each result within the parity bound of the
    oracle's float64 GEMV, and of ggq_gemv's result; free device memory is
    the same before and after (nothing allocated, nothing left behind)."""
    torch, ggq = env
    W = synth.weight_rows(qtype, 70 + qtype, rows, cols)
    x = synth.normal_f32(M * cols, 71).reshape(M, cols)
    y_ref, a_ref = oracle.gemv(qtype, W, rows, cols, x)
    Wd = torch.from_numpy(W).cuda()
    xd = torch.from_numpy(x).cuda()
    stream = torch.cuda.current_stream().cuda_stream
    y_gemv = torch.empty((M, rows), dtype=torch.float32, device="cuda")
    ggq.check(ggq.ggq_gemv(qtype, Wd.data_ptr(), rows, cols, xd.data_ptr(), y_gemv.data_ptr(), M, stream),
              "ggq_gemv")
    ys = [torch.full((M, rows), float("nan"), dtype=torch.float32, device="cuda") for _ in range(2)]
    torch.cuda.synchronize()
    ok, worst = oracle.tolerance_ok(y_gemv.cpu().numpy(), y_ref, a_ref)
    assert ok, f"ggq_gemv: worst {worst}"
    free_before = torch.cuda.mem_get_info()[0]
    for call in range(2):
        rc = ggq.ggq_gemv_noalloc(qtype, Wd.data_ptr(), rows, cols, xd.data_ptr(), ys[call].data_ptr(), M, stream)
        ggq.check(rc, "ggq_gemv_noalloc")
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    assert ggq.device_status() == 0
    for call in range(2):
        y = ys[call].cpu().numpy()
        ok, worst = oracle.tolerance_ok(y, y_ref, a_ref)
        assert ok, f"call {call} vs oracle: worst {worst}"
        ok, worst = oracle.tolerance_ok(y, y_gemv.cpu().numpy().astype(np.float64), a_ref)
        assert ok, f"call {call} vs ggq_gemv: worst {worst}"


def test_noalloc_refuses_shapes_it_cannot_run_without_allocating(env):
    torch, ggq = env
    buf = torch.empty(64, dtype=torch.float32, device="cuda")
    p = buf.data_ptr()
    assert ggq.ggq_gemv_noalloc(12, p, 64, 256, p, p, 5, 0) == -1                  # M > 4
    assert ggq.ggq_gemv_noalloc(8, p, 64, 96, p, p, 1, 0) == -1                    # cols % 256
    assert ggq.ggq_gemv_noalloc(12, p, 64, 1 << 20, p, p, 1, 0) == -1              # x' beyond shared memory
    assert "allocation-free kernel" in ggq.lib.ggq_last_error().decode()

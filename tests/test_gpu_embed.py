"""GPU parity: ggq_embed (token embedding rows of a block-quantized table,
"GGUF Inferencer in R" section 4 "Input Embedding") against the oracle's
decode, bit for bit (the decode is exact)."""
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


@pytest.mark.parametrize("qtype,rows,cols", [(8, 1000, 2048), (8, 3, 32), (12, 777, 4096), (12, 5, 256)])
def test_embed_rows_bit_exact(env, qtype, rows, cols):
    torch, ggq = env
    W = synth.weight_rows(qtype, 700 + qtype, rows, cols)
    ref = oracle.dequantize(qtype, W, rows, cols)          # [rows, cols] fp32, exact
    rng = np.random.default_rng(rows)
    ids = np.concatenate([[0, rows - 1, 0], rng.integers(0, rows, size=34)]).astype(np.int32)
    Wd = torch.from_numpy(W).cuda()
    out = ggq.embed(qtype, Wd, rows, cols, torch.from_numpy(ids))
    torch.cuda.synchronize()
    assert ggq.device_status() == 0
    got = out.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref[ids].astype(np.float32).view(np.uint32))
    one = ggq.embed(qtype, Wd, rows, cols, torch.tensor([rows - 1]))
    torch.cuda.synchronize()
    assert np.array_equal(one.cpu().numpy()[0].view(np.uint32), ref[rows - 1].astype(np.float32).view(np.uint32))


def test_embed_out_of_range_id_is_reported(env):
    """An id outside the table gives a zero row and GGQ_EINVAL from the next
    ggq_device_status (the kernel's own bounds check); other rows are intact."""
    torch, ggq = env
    rows, cols = 64, 256
    W = synth.weight_rows(8, 710, rows, cols)
    ref = oracle.dequantize(8, W, rows, cols)
    Wd = torch.from_numpy(W).cuda()
    out = ggq.embed(8, Wd, rows, cols, torch.tensor([3, rows, -1, 5], dtype=torch.int32))
    assert ggq.device_status() == -1
    assert "embedding" in ggq.lib.ggq_last_error().decode()
    got = out.cpu().numpy()
    assert np.array_equal(got[1], np.zeros(cols, np.float32)) and np.array_equal(got[2], np.zeros(cols, np.float32))
    assert np.array_equal(got[0], ref[3]) and np.array_equal(got[3], ref[5])
    assert ggq.device_status() == 0                        # the record was cleared

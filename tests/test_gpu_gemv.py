"""GPU parity: ggq_dequantize / ggq_gemv (through the C ABI) against the CPU oracle.

Bar: decoded weights bit-exact; GEMV outputs within
|y - y_ref| <= 1e-3 * sum_c |w[r,c] x[c]| + 1e-6  (y_ref in double);
integer-valued and one-hot cases exact.
"""
import numpy as np
import pytest

import oracle
import synth
from synth import workloads as WL

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


def gpu_gemv(env, qtype, W, rows, cols, x, guard=64):
    """Run ggq_gemv with guard cells around y; check they survive."""
    torch, ggq = env
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, cols)
    M = x.shape[0]
    Wd, xd = _dev(torch, W), _dev(torch, x)
    buf = torch.full((M * rows + 2 * guard,), float("nan"), dtype=torch.float32, device="cuda")
    y = buf[guard:guard + M * rows]
    rc = ggq.ggq_gemv(qtype, Wd.data_ptr(), rows, cols, xd.data_ptr(), y.data_ptr(), M,
                      torch.cuda.current_stream().cuda_stream)
    ggq.check(rc, "ggq_gemv")
    torch.cuda.synchronize()
    assert ggq.device_status() == 0
    out = buf.cpu().numpy()
    assert np.isnan(out[:guard]).all() and np.isnan(out[guard + M * rows:]).all(), "write outside y"
    return out[guard:guard + M * rows].reshape(M, rows)


def assert_close(y, y_ref, a_ref, what=""):
    ok, worst = oracle.tolerance_ok(y, y_ref, a_ref, REL, ABS)
    assert ok, f"{what}: worst error / bound = {worst:.3g}"
    return worst


def weights(qtype, rows, cols, stream=7):
    return synth.weight_rows(qtype, stream, rows, cols)


def xs(M, cols, stream=8):
    return synth.normal_f32(M * cols, stream).reshape(M, cols)


# ----------------------------------------------------------------- dequant ----

@pytest.mark.parametrize("qtype,rows,cols", [(8, 1, 32), (8, 3, 96), (8, 17, 512), (8, 65, 2304),
                                             (12, 1, 256), (12, 3, 512), (12, 40, 2304)])
def test_dequantize_bit_exact(env, qtype, rows, cols):
    torch, ggq = env
    W = weights(qtype, rows, cols)
    out = ggq.dequantize(qtype, _dev(torch, W), rows, cols)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    ref = oracle.dequantize(qtype, W, rows, cols)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_dequantize_special_scales(env):
    """fp16 scales that are subnormal, the largest finite, inf and NaN."""
    torch, ggq = env
    from tests.pin_checks import Q8_PATTERN, q8_block, pack_q4_k
    d_bits = [0x0001, 0x03FF, 0x7BFF, 0xFBFF, 0x7C00, 0xFC00, 0x7E00, 0x8000]
    W8 = b"".join(q8_block(d, Q8_PATTERN) for d in d_bits)
    rng = np.random.default_rng(0)
    W4 = b"".join(pack_q4_k(d, dm, list(rng.integers(0, 64, 8)), list(rng.integers(0, 64, 8)),
                            list(rng.integers(0, 16, 256)))
                  for d, dm in [(0x0001, 0x0002), (0x7BFF, 0x03FF), (0x7C00, 0x3C00), (0x3C00, 0x7E00)])
    for qtype, W, cols in [(8, W8, 32), (12, W4, 256)]:
        Wn = np.frombuffer(W, np.uint8).copy()
        rows = Wn.size // oracle.row_bytes(qtype, cols)
        got = ggq.dequantize(qtype, _dev(torch, Wn), rows, cols).cpu().numpy()
        ref = oracle.dequantize(qtype, Wn, rows, cols)
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(got), nan)
        assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


# -------------------------------------------------------------------- GEMV ----

SHAPES_Q8 = [(1, 32), (3, 96), (31, 256), (33, 512), (100, 2048), (257, 2304), (64, 4096 + 32)]
SHAPES_Q4 = [(1, 256), (31, 512), (33, 2304), (100, 4096), (257, 11008)]


@pytest.mark.parametrize("rows,cols", SHAPES_Q8)
def test_gemv_q8_0_m1(env, rows, cols):
    W = weights(8, rows, cols)
    x = xs(1, cols)
    y_ref, a_ref = oracle.gemv(8, W, rows, cols, x)
    assert_close(gpu_gemv(env, 8, W, rows, cols, x), y_ref, a_ref, f"q8_0 {rows}x{cols}")


@pytest.mark.parametrize("rows,cols", SHAPES_Q4)
def test_gemv_q4_k_m1(env, rows, cols):
    W = weights(12, rows, cols)
    x = xs(1, cols)
    y_ref, a_ref = oracle.gemv(12, W, rows, cols, x)
    assert_close(gpu_gemv(env, 12, W, rows, cols, x), y_ref, a_ref, f"q4_k {rows}x{cols}")


@pytest.mark.parametrize("qtype,rows,cols", [(8, 33, 512), (8, 70, 2304), (8, 9, 96), (12, 33, 512),
                                             (12, 70, 2304)])
@pytest.mark.parametrize("M", [2, 3, 4, 5, 8, 9, 16])
def test_gemv_small_m(env, qtype, rows, cols, M):
    W = weights(qtype, rows, cols)
    x = xs(M, cols)
    y_ref, a_ref = oracle.gemv(qtype, W, rows, cols, x)
    y = gpu_gemv(env, qtype, W, rows, cols, x)
    assert_close(y, y_ref, a_ref, f"type {qtype} M={M}")
    # the last activation row alone (M = 1 kernel) meets the same bar
    y1 = gpu_gemv(env, qtype, W, rows, cols, x[M - 1:M])
    assert_close(y1, y_ref[M - 1:M], a_ref[M - 1:M], f"type {qtype} row {M - 1} alone")


@pytest.mark.parametrize("qtype,rows,cols,M", [(8, 1, 256, 5), (8, 129, 2304, 8), (8, 300, 4096, 16),
                                             (12, 127, 256, 6), (12, 257, 11008, 13), (12, 1000, 4096, 16)])
def test_gemv_tensor_core_small_batch(env, qtype, rows, cols, M):
    """M >= 5 runs on the tcgen05 path: ragged 128-row tiles, one and many
    256-column periods, padded activation rows."""
    W = weights(qtype, rows, cols, stream=11)
    x = xs(M, cols, stream=12)
    y_ref, a_ref = oracle.gemv(qtype, W, rows, cols, x)
    y = gpu_gemv(env, qtype, W, rows, cols, x)
    assert_close(y, y_ref, a_ref, f"type {qtype} {rows}x{cols} M={M}")


# 2-4 activation rows whose pre-scaled x does not fit in shared memory at
# once (4 x 14336 fp32 = 229 KB): the streaming kernel runs on groups of rows
# (2 + 1, 2 + 2; one row at a time at 32768 columns), y rows of each group at
# their own offset.
@pytest.mark.parametrize("qtype,rows,cols,M", [(12, 97, 14336, 3), (12, 70, 14336, 4), (8, 33, 14336, 4),
                                             (8, 40, 16384, 3), (14, 65, 14336, 4), (2, 50, 14336, 3),
                                             (12, 40, 32768, 3), (8, 24, 32768, 2)])
def test_gemv_wide_rows_in_groups(env, qtype, rows, cols, M):
    W = weights(qtype, rows, cols, stream=31)
    x = xs(M, cols, stream=32)
    y_ref, a_ref = oracle.gemv(qtype, W, rows, cols, x)
    y = gpu_gemv(env, qtype, W, rows, cols, x)
    assert_close(y, y_ref, a_ref, f"type {qtype} {rows}x{cols} M={M}")


# Tiles split along K (the y zeroed, both parts added): big/small parts when
# the 128-row tiles fill more than half of the 152 SMs in one wave (14336 rows:
# 112 tiles), halves of the last wave's tiles otherwise (20480 rows: 160
# tiles, 8 of them split; 12800 x 2048: 100 tiles, 8 blocks a row).
@pytest.mark.parametrize("qtype,rows,cols,M", [(2, 14336, 4096, 16), (12, 14336, 4096, 8), (8, 20480, 1024, 16),
                                             (2, 12800, 2048, 5), (12, 300, 4096, 9)])
def test_gemv_tensor_core_split_layouts(env, qtype, rows, cols, M):
    W = weights(qtype, rows, cols, stream=21)
    x = xs(M, cols, stream=22)
    y = gpu_gemv(env, qtype, W, rows, cols, x)
    y_ref, a_ref = oracle.gemv_dense(qtype, W, rows, cols, x)
    assert_close(y, y_ref, a_ref, f"type {qtype} {rows}x{cols} M={M}")


def test_gemv_tensor_core_split_repeat_and_graph(env):
    """The two parts of a split tile add in whichever order they finish: the
    same fp32 sum, so repeated calls agree bit for bit; captured in a CUDA
    graph (the zeroing of y and the kernel), replays with new x are right."""
    torch, ggq = env
    rows, cols, M = 14336, 4096, 16
    W = weights(8, rows, cols, stream=23)
    x = xs(M, cols, stream=24)
    Wd, xd = _dev(torch, W), _dev(torch, x)
    outs = [ggq.gemv(8, Wd, rows, cols, xd).cpu().numpy() for _ in range(3)]
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32))
    s = torch.cuda.Stream()
    y = torch.full((M, rows), float("nan"), dtype=torch.float32, device="cuda")
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            ggq.check(ggq.ggq_gemv(8, Wd.data_ptr(), rows, cols, xd.data_ptr(), y.data_ptr(), M, s.cuda_stream),
                      "ggq_gemv")
    x2 = xs(M, cols, stream=25)
    xd.copy_(torch.from_numpy(x2))
    y.fill_(float("nan"))
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert ggq.device_status() == 0
    y_ref, a_ref = oracle.gemv_dense(8, W, rows, cols, x2)
    assert_close(y.cpu().numpy(), y_ref, a_ref, "graph replay")


def test_gemv_tensor_core_integer_inputs_are_exact(env):
    """Q8_0 with d = 1 and small integer x at M = 8: every product and sum is an
    exact integer in fp32, so the bf16 hi/lo parts and the tensor-core sums give
    the exact result."""
    from tests.pin_checks import q8_block
    rng = np.random.default_rng(9)
    rows, cols, M = 200, 1024, 8
    q = rng.integers(-128, 128, size=(rows, cols))
    W = np.frombuffer(b"".join(q8_block(0x3C00, list(q[r, 32 * b:32 * b + 32]))
                               for r in range(rows) for b in range(cols // 32)), np.uint8).copy()
    x = rng.integers(-8, 9, size=(M, cols)).astype(np.float32)
    y = gpu_gemv(env, 8, W, rows, cols, x)
    assert np.array_equal(y.astype(np.int64), x.astype(np.int64) @ q.T)


def test_gemv_many_rounds(env):
    """Columns wide enough that a CTA streams its slice in several rounds."""
    for qtype, cols, M in [(12, 65536, 16), (8, 65536, 16), (12, 65536, 1)]:
        rows = 40
        W = weights(qtype, rows, cols, stream=21)
        x = xs(M, cols, stream=22)
        y_ref, a_ref = oracle.gemv(qtype, W, rows, cols, x)
        assert_close(gpu_gemv(env, qtype, W, rows, cols, x), y_ref, a_ref, f"wide {qtype} M={M}")


@pytest.mark.parametrize("qtype,cols", [(8, 512), (8, 96), (12, 512), (12, 2304)])
def test_gemv_one_hot_extracts_exact_columns(env, qtype, cols):
    rows = 37
    W = weights(qtype, rows, cols, stream=3)
    Wf = oracle.dequantize(qtype, W, rows, cols)
    for c in [0, 1, cols // 2 + 3, cols - 1]:
        x = np.zeros((1, cols), np.float32)
        x[0, c] = 1.0
        y = gpu_gemv(env, qtype, W, rows, cols, x)
        assert np.array_equal(y[0].view(np.uint32), Wf[:, c].view(np.uint32)), c


def test_gemv_integer_inputs_are_exact(env):
    from tests.pin_checks import q8_block, pack_q4_k
    rng = np.random.default_rng(5)
    rows, cols = 45, 2048
    q = rng.integers(-128, 128, size=(rows, cols))
    W = np.frombuffer(b"".join(q8_block(0x3C00, list(q[r, 32 * b:32 * b + 32]))
                               for r in range(rows) for b in range(cols // 32)), np.uint8).copy()
    x = rng.integers(-8, 9, size=(3, cols)).astype(np.float32)
    y = gpu_gemv(env, 8, W, rows, cols, x)
    assert np.array_equal(y.astype(np.int64), x.astype(np.int64) @ q.T)
    sc = rng.integers(0, 8, size=(rows, cols // 256, 8))
    mm = rng.integers(0, 8, size=(rows, cols // 256, 8))
    qq = rng.integers(0, 16, size=(rows, cols))
    W = np.frombuffer(b"".join(pack_q4_k(0x3C00, 0x3C00, list(sc[r, b]), list(mm[r, b]),
                                         list(qq[r, 256 * b:256 * b + 256]))
                               for r in range(rows) for b in range(cols // 256)), np.uint8).copy()
    j = (np.arange(cols) % 256) // 32
    bi = np.arange(cols) // 256
    w = sc[:, bi, j] * qq - mm[:, bi, j]
    x = rng.integers(-4, 5, size=(2, cols)).astype(np.float32)
    y = gpu_gemv(env, 12, W, rows, cols, x)
    assert np.array_equal(y.astype(np.int64), x.astype(np.int64) @ w.T)


def test_gemv_zero_weights_and_zero_x(env):
    rows, cols = 33, 512
    x = xs(2, cols)
    for qtype in (8, 12):
        W = np.zeros(rows * oracle.row_bytes(qtype, cols), np.uint8)
        assert not gpu_gemv(env, qtype, W, rows, cols, x).any()
        W = weights(qtype, rows, cols)
        assert not gpu_gemv(env, qtype, W, rows, cols, np.zeros((1, cols), np.float32)).any()


def test_gemv_on_a_side_stream(env):
    torch, ggq = env
    rows, cols = 300, 4096
    W = weights(12, rows, cols, stream=30)
    x = xs(1, cols, stream=31)
    y_ref, a_ref = oracle.gemv(12, W, rows, cols, x)
    s = torch.cuda.Stream()
    Wd, xd = _dev(torch, W), _dev(torch, x)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        y = ggq.gemv(12, Wd, rows, cols, xd)
    s.synchronize()
    assert_close(y.cpu().numpy(), y_ref, a_ref, "side stream")


# ----------------------------------------------------- the benchmark shapes ----

def test_cfg1_q8_0_2048(env):
    g = WL.CFG1[0]
    W = synth.weight_rows(g.qtype, g.stream, g.rows, g.cols)
    x = synth.normal_f32(g.cols, g.x_stream).reshape(1, -1)
    y_ref, a_ref = oracle.gemv(g.qtype, W, g.rows, g.cols, x)
    assert_close(gpu_gemv(env, g.qtype, W, g.rows, g.cols, x), y_ref, a_ref, "cfg1")


@pytest.mark.parametrize("g", WL.CFG2, ids=lambda g: g.name.split(".")[-2])
def test_cfg2_smollm3_layer(env, g):
    W = synth.weight_rows(g.qtype, g.stream, g.rows, g.cols)
    x = synth.normal_f32(g.cols, g.x_stream).reshape(1, -1)
    y_ref, a_ref = oracle.gemv(g.qtype, W, g.rows, g.cols, x)
    assert_close(gpu_gemv(env, g.qtype, W, g.rows, g.cols, x), y_ref, a_ref, g.name)


@pytest.mark.parametrize("M", WL.CFG4_M)
def test_cfg4_q8_0_small_batch(env, M):
    """Q8_0 14336 x 4096 at every M of the sweep: every output row against the
    oracle (decoded weights, float64 product)."""
    g = WL.CFG4
    W = synth.weight_rows(g.qtype, g.stream, g.rows, g.cols)
    x = synth.normal_f32(M * g.cols, g.x_stream).reshape(M, -1)
    y = gpu_gemv(env, g.qtype, W, g.rows, g.cols, x)
    y_ref, a_ref = oracle.gemv_dense(g.qtype, W, g.rows, g.cols, x)
    assert_close(y, y_ref, a_ref, f"cfg4 M={M}")


def _distinct_shapes():
    seen, out = set(), []
    for g in WL.llama8b_pass(1):
        key = (g.qtype, g.rows, g.cols)
        if key not in seen:
            seen.add(key)
            out.append(g)
    return out


@pytest.mark.parametrize("g", _distinct_shapes(), ids=lambda g: g.name)
def test_cfg3_llama8b_shapes_full(env, g):
    """Every distinct tensor shape of the Llama-8B-shaped decode pass (the Q8_0
    head included) at full size, in the bench's launch configuration: every
    output row against the oracle.  A few rows are also regenerated alone from
    their counters (the generator is row-addressable)."""
    W = synth.weight_rows(g.qtype, g.stream, g.rows, g.cols)
    x = synth.normal_f32(g.cols, g.x_stream).reshape(1, -1)
    y = gpu_gemv(env, g.qtype, W, g.rows, g.cols, x)
    rb = oracle.row_bytes(g.qtype, g.cols)
    for r in (0, 31, g.rows - 1):
        assert np.array_equal(synth.weight_rows(g.qtype, g.stream, 1, g.cols, row0=int(r)), W[r * rb:(r + 1) * rb])
    y_ref, a_ref = oracle.gemv_dense(g.qtype, W, g.rows, g.cols, x)
    assert_close(y, y_ref, a_ref, g.name)


# ---------------------------------------------------------------- loading ----

def test_load_file_to_device_and_multiply(env, tmp_path):
    torch, ggq = env
    q8 = synth.weight_rows(8, 41, 70, 512)
    q4 = synth.weight_rows(12, 42, 50, 2304)
    norm = synth.normal_f32(512, 43)
    kvs = [("general.architecture", 8, "llama"), ("llama.block_count", 4, 1)]
    tensors = [("blk.0.attn_q.weight", [512, 70], 8), ("blk.0.attn_norm.weight", [512], 0),
               ("blk.0.ffn_up.weight", [2304, 50], 12)]
    path = str(tmp_path / "m.gguf")
    synth.write_gguf(path, kvs, tensors, [q8.tobytes(), norm.tobytes(), q4.tobytes()])
    with ggq.Model.load(path) as m:
        t8, t4 = m.find("blk.0.attn_q.weight"), m.find("blk.0.ffn_up.weight")
        assert t8["data"] % 256 == 0 and t4["data"] % 256 == 0
        for t, W, rows, cols, qt in [(t8, q8, 70, 512, 8), (t4, q4, 50, 2304, 12)]:
            out = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
            ggq.check(ggq.ggq_dequantize(qt, t["data"], rows, cols, out.data_ptr(),
                                         torch.cuda.current_stream().cuda_stream), "dequantize")
            got = out.cpu().numpy()
            assert np.array_equal(got.view(np.uint32), oracle.dequantize(qt, W, rows, cols).view(np.uint32))
            x = xs(1, cols, stream=44)
            xd = _dev(torch, x)
            y = torch.empty((1, rows), dtype=torch.float32, device="cuda")
            ggq.check(ggq.ggq_gemv(qt, t["data"], rows, cols, xd.data_ptr(), y.data_ptr(), 1,
                                   torch.cuda.current_stream().cuda_stream), "gemv")
            y_ref, a_ref = oracle.gemv(qt, W, rows, cols, x)
            assert_close(y.cpu().numpy(), y_ref, a_ref, t["name"])


@pytest.mark.parametrize("qtype,rows,cols,M", [(12, 33, 4096, 1), (8, 100, 2048, 1), (12, 1000, 11008, 2),
                                               (8, 4000, 4096, 4)])
def test_gemv_repeated_calls_are_bit_identical(env, qtype, rows, cols, M):
    """Groups of rows cut between warps are added in a fixed warp order, so
    repeated calls agree bit for bit (and with the oracle within the bound)."""
    torch, ggq = env
    W = weights(qtype, rows, cols, stream=50)
    x = xs(M, cols, stream=51)
    y_ref, a_ref = oracle.gemv(qtype, W, rows, cols, x)
    Wd, xd = _dev(torch, W), _dev(torch, x)
    outs = [ggq.gemv(qtype, Wd, rows, cols, xd).cpu().numpy() for _ in range(4)]
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32))
    assert_close(outs[0], y_ref, a_ref, "repeat")
    assert ggq.device_status() == 0


def test_gemv_in_cuda_graph(env):
    torch, ggq = env
    rows, cols = 2000, 4096
    W = weights(12, rows, cols, stream=52)
    x = xs(1, cols, stream=53)
    y_ref, a_ref = oracle.gemv(12, W, rows, cols, x)
    Wd, xd = _dev(torch, W), _dev(torch, x)
    y = torch.empty((1, rows), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ggq.gemv(12, Wd, rows, cols, xd, y)       # outside capture first: kernel attributes are set once
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ggq.gemv(12, Wd, rows, cols, xd, y)
    for _ in range(3):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert_close(y.cpu().numpy(), y_ref, a_ref, "graph replay")


@pytest.mark.parametrize("qtype,rows,cols,M", [(12, 4096, 4096, 1), (8, 2048, 4096, 3), (12, 300, 512, 2),
                                               (8, 1024, 4096, 8), (12, 1024, 4096, 16)])
def test_gemv_reads_weights_written_by_the_previous_kernel(env, qtype, rows, cols, M):
    """A device kernel (an element-wise OR, not a copy) rewrites W on the same
    stream right before the GEMV: the GEMV must read the new weights.  The
    shapes reach the streaming kernel (M <= 4), the narrow-shape cluster
    kernel and the tensor-core small-batch kernel (M 8, 16)."""
    torch, ggq = env
    W_old = weights(qtype, rows, cols, stream=60)
    W_new = weights(qtype, rows, cols, stream=61)
    x = xs(M, cols, stream=62)
    y_ref, a_ref = oracle.gemv(qtype, W_new, rows, cols, x)
    Wd = _dev(torch, W_old)
    W_src = _dev(torch, W_new)
    zero = torch.zeros((), dtype=torch.uint8, device="cuda")
    xd = _dev(torch, x)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        Wd.copy_(_dev(torch, W_old))
        y = torch.full((M, rows), float("nan"), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        torch.bitwise_or(W_src, zero, out=Wd)      # a kernel writes W
        if call == 0:
            rc = ggq.ggq_gemv(qtype, Wd.data_ptr(), rows, cols, xd.data_ptr(), y.data_ptr(), M, stream)
        elif M <= 4 and cols % 256 == 0 and cols >= 768:
            rc = ggq.ggq_gemv_noalloc(qtype, Wd.data_ptr(), rows, cols, xd.data_ptr(), y.data_ptr(), M, stream)
        else:
            continue
        ggq.check(rc, "gemv after a kernel wrote W")
        torch.cuda.synchronize()
        assert ggq.device_status() == 0
        assert_close(y.cpu().numpy(), y_ref, a_ref, f"call {call}")

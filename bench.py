#!/usr/bin/env python3
"""Benchmark of the block-quantized decode weight pass on GB300.

Default workload: one batch-1 decode weight pass over a Llama-8B-shaped stack
(32 layers of Q4_K projections, hidden 4096, 32/8 heads of 128, ffn 14336, and a
4096 -> 128256 Q8_0 output head): 4,484,038,656 weight bytes per pass.  The
weights are seeded synthetic N(0, 0.02) values encoded to Q4_K / Q8_0, written
to a GGUF file and loaded with ggq_load; activations are N(0, 1).

A step is one pass in dependency order: per layer the stages [q,k,v], [o],
[gate,up], [down] (128 Q4_K stages, each reading its own x only after the
previous stage's outputs are complete) run as ONE ggq_chain launch, then the
Q8_0 head (ggq_gemv) -- 2 launches, replayed as a CUDA graph.  The same pass
as one launch per stage (129 launches) is reported beside it.  The weights
(4.48 GB) exceed the L2 cache, so successive steps read them from HBM.

Prints ONE JSON line (rank 0).  --impl reference times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "dequant-GEMV achieved HBM GB/s (fraction of ~8 TB/s); decode weight-pass tok/s"
WORKLOAD = "llama8b_decode_weight_pass_q4k_q8head"


def args_parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ggq", choices=["ggq", "reference"])
    ap.add_argument("--layers", type=int, default=32, help="layers in the stack (32 = the benchmark)")
    ap.add_argument("--no-extras", action="store_true", help="skip the per-config kernel timings")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle sample budget")
    ap.add_argument("--kernel", choices=sorted(KERNEL_SHAPES),
                    help="run one configuration's GEMV a few times and exit (a small command to profile)")
    ap.add_argument("--M", type=int, default=1, help="activation rows for --kernel")
    ap.add_argument("--file-pass-layers", type=int, default=0,
                    help="run only the Q4_K_M-style file pass with this many layers and exit "
                         "(a small command to profile its mixed-type chain)")
    return ap.parse_args()


# one GEMV configuration each: (workload attribute, description)
KERNEL_SHAPES = {
    "q8_0_head": ("HEAD", "Q8_0 4096 -> 128256 output head of the Llama-8B-shaped pass"),
    "q6_k_14336x4096": ("Q6K_GEMV", "Q6_K 14336 x 4096"),
    "q6_k_4096x14336": ("Q6K_DOWN_GEMV", "Q6_K 4096 x 14336 (ffn_down shape)"),
    "q8_0_14336x4096": ("CFG4", "Q8_0 14336 x 4096"),
    "q4_0_14336x4096": ("Q40_GEMV", "Q4_0 14336 x 4096"),
    "prefill_q4_k_512x14336x4096": ("CFG5", "prefill: Q4_K 14336 x 4096 times bf16 X 512 x 4096"),
    "prefill_q8_0_512x14336x4096": ("CFG4", "prefill: Q8_0 14336 x 4096 times bf16 X 512 x 4096"),
}


def run_kernel(a):
    """Five launches of one configuration's ggq_gemv (seeded weights, random x)
    after one warm-up; prints the per-launch time of the last five."""
    import torch
    import gguf_block_quantized_q8_gb300 as ggq
    import synth
    from synth import workloads as WL
    attr, desc = KERNEL_SHAPES[a.kernel]
    g = WL.llama8b_pass(1)[-1] if attr == "HEAD" else getattr(WL, attr)
    torch.cuda.set_device(0)
    W = torch.from_numpy(synth.weight_rows(g.qtype, g.stream, g.rows, g.cols)).cuda()
    s = torch.cuda.current_stream().cuda_stream
    if a.kernel.startswith("prefill"):
        import numpy as np
        a.M = WL.CFG5_M
        x = torch.from_numpy(synth.normal_bf16(a.M * g.cols, WL.CFG5.x_stream).view(np.int16)).cuda()
    else:
        x = torch.randn(a.M, g.cols, device="cuda")
    y = torch.empty(a.M, g.rows, device="cuda")

    def once():
        if a.kernel.startswith("prefill"):
            ggq.check(ggq.ggq_gemm_prefill(g.qtype, W.data_ptr(), g.rows, g.cols, x.data_ptr(), y.data_ptr(), a.M,
                                           s), "prefill")
        else:
            ggq.check(ggq.ggq_gemv(g.qtype, W.data_ptr(), g.rows, g.cols, x.data_ptr(), y.data_ptr(), a.M, s),
                      "gemv")
    once()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(5):
        once()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / 5
    nb = g.rows * synth.row_bytes(g.qtype, g.cols)
    print(json.dumps({"kernel": a.kernel, "desc": desc, "M": a.M, "us": round(us, 2),
                      "GB_s": round(nb / us / 1e3, 1), "TFLOP_s": round(2 * a.M * g.rows * g.cols / us / 1e6, 1),
                      "status": ggq.device_status()}))
    return 0


# ------------------------------------------------------------ distributed ----

def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_max(value: float, ws: int, device=None) -> float:
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ clocks ----

class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.dev)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, mx, pw, reasons = [], None, [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            try:
                pw.append(float(f[3].split()[0]))
            except (ValueError, IndexError):
                pass
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "power_w": statistics.median(pw) if pw else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------- workload ----

def build_pass_file(path: str, layers: int):
    """Write the seeded synthetic stack as a GGUF v3 file; returns the tensor list."""
    import synth
    from synth import workloads as WL
    gem = WL.llama8b_pass(layers)
    kvs = [("general.architecture", 8, "llama"), ("general.name", 8, "synthetic-llama8b-shape"),
           ("llama.block_count", 4, layers), ("llama.embedding_length", 4, 4096),
           ("llama.feed_forward_length", 4, 14336), ("llama.attention.head_count", 4, 32),
           ("llama.attention.head_count_kv", 4, 8)]
    tensors = [(g.name, [g.cols, g.rows], g.qtype) for g in gem]
    payloads = (synth.weight_rows(g.qtype, g.stream, g.rows, g.cols) for g in gem)
    synth.write_gguf(path, kvs, tensors, payloads)
    return gem


def stage_plan(layers: int):
    from synth import workloads as WL
    return WL.llama8b_stages(layers)


class DecodePass:
    """Device state for one pass: loaded weights, per-stage x and y, launch list.

    run(): the Q4_K stages (128 for 32 layers) as ONE ggq_chain launch, then
    the Q8_0 head with ggq_gemv -- 2 launches.  run_launches(): every stage as
    its own ggq_gemv / ggq_gemv_multi launch (129), for comparison."""

    def __init__(self, model, stages, torch, ggq, synth):
        self.torch, self.ggq = torch, ggq
        self.stages = []
        self.weight_bytes = 0
        # every stage's x and every output y are slices of one pinned host buffer
        # and one device buffer each (x slices start on 1 KB boundaries: cols is a
        # multiple of 256), so a step's inputs and outputs move in one copy each way
        nx = sum(st[0].cols for st in stages)
        ny = sum(g.rows for st in stages for g in st)
        self.x_host = torch.empty(nx, dtype=torch.float32).pin_memory()
        self.y_host = torch.empty(ny, dtype=torch.float32).pin_memory()
        self.x_dev = torch.empty(nx, dtype=torch.float32, device="cuda")
        self.y_dev = torch.empty(ny, dtype=torch.float32, device="cuda")
        xo = yo = 0
        for st in stages:
            tinfo = [model.find(g.name) for g in st]
            cols = st[0].cols
            self.x_host[xo:xo + cols].copy_(torch.from_numpy(synth.normal_f32(cols, st[0].x_stream)))
            xd = self.x_dev[xo:xo + cols]
            xo += cols
            ys = []
            for g in st:
                ys.append(self.y_dev[yo:yo + g.rows])
                yo += g.rows
            nbytes = sum(t["nbytes"] for t in tinfo)
            self.weight_bytes += nbytes
            self.stages.append(dict(qtype=st[0].qtype, W=[t["data"] for t in tinfo], rows=[g.rows for g in st],
                                    cols=cols, x=xd.data_ptr(), y=[y.data_ptr() for y in ys], nbytes=nbytes,
                                    io_bytes=4 * cols + 4 * sum(g.rows for g in st)))
        self.x_dev.copy_(self.x_host)
        self.io_bytes = sum(s["io_bytes"] for s in self.stages)
        self.x_bytes = sum(4 * s["cols"] for s in self.stages)
        self.y_bytes = sum(4 * sum(s["rows"]) for s in self.stages)
        self.q4 = [s for s in self.stages if s["qtype"] == 12]
        self.rest = [s for s in self.stages if s["qtype"] != 12]
        rc, self.chain = ggq.ggq_chain_create(12, 1, [(s["W"], s["rows"], s["cols"], s["x"], s["y"]) for s in self.q4])
        ggq.check(rc, "ggq_chain_create")
        self.q4_bytes = sum(s["nbytes"] + s["io_bytes"] for s in self.q4)
        # the pass's result: the output head's logits (the last stage's y)
        self.head_rows = self.stages[-1]["rows"][0]
        self.head_y = self.y_dev[ny - self.head_rows:]

    def launch_stage(self, st, stream_ptr):
        ggq = self.ggq
        if len(st["W"]) == 1:
            rc = ggq.ggq_gemv(st["qtype"], st["W"][0], st["rows"][0], st["cols"], st["x"], st["y"][0], 1, stream_ptr)
        else:
            rc = ggq.ggq_gemv_multi(st["qtype"], st["W"], st["rows"], st["cols"], st["x"], st["y"], 1, stream_ptr)
        ggq.check(rc, "gemv")

    def run_chain(self, stream_ptr):
        self.ggq.check(self.ggq.ggq_chain_run(self.chain, stream_ptr), "ggq_chain_run")

    def run(self, stream_ptr):
        self.run_chain(stream_ptr)
        for st in self.rest:
            self.launch_stage(st, stream_ptr)

    def run_launches(self, stream_ptr):
        for st in self.stages:
            self.launch_stage(st, stream_ptr)

    def run_per_tensor(self, stream_ptr):
        """Every weight matrix as its own ggq_gemv (225 launches for 32 layers)."""
        for st in self.stages:
            for W, rows, y in zip(st["W"], st["rows"], st["y"]):
                self.ggq.check(self.ggq.ggq_gemv(st["qtype"], W, rows, st["cols"], st["x"], y, 1, stream_ptr), "gemv")

    @property
    def launches(self):
        return 1 + len(self.rest)

    def fused_pass(self, synth):
        """The same weights as a real layer data flow, every element-wise step fused
        into the chain (ggq_chain_create_ops): h = the embedding row of one token
        (ggq_embed; the Q8_0 head matrix read as a tied embedding table), then per
        layer h -> [q,k,v](rmsnorm(h)), [o](q) + h = h2, [gate,up](rmsnorm(h2)),
        [down](silu(gate) * up) + h2; then the head on rmsnorm(h) as a one-stage
        Q8_0 chain.  Returns a callable running the pass (3 launches) and the
        objects it keeps."""
        torch, ggq = self.torch, self.ggq
        q4 = self.q4
        assert len(q4) % 4 == 0 and len(self.rest) == 1
        H = q4[0]["cols"]
        norms = []

        def norm_w(stream_id):
            g = torch.from_numpy((1.0 + 0.1 * synth.normal_f32(H, stream_id)).astype("float32")).cuda()
            norms.append(g)
            return g.data_ptr()

        h = q4[0]["x"]
        stages, ops = [], []
        for L in range(len(q4) // 4):
            qkv, o, gu, dn = q4[4 * L: 4 * L + 4]
            yq, yo, yg, yu = qkv["y"][0], o["y"][0], gu["y"][0], gu["y"][1]
            stages += [(qkv["W"], qkv["rows"], H, h, qkv["y"]), (o["W"], o["rows"], H, yq, o["y"]),
                       (gu["W"], gu["rows"], H, yo, gu["y"]), (dn["W"], dn["rows"], dn["cols"], yg, dn["y"])]
            ops += [{"x_op": ggq.X_RMSNORM, "eps": 1e-5, "norm_w": norm_w(7000 + 2 * L)},
                    {"res": [h]},
                    {"x_op": ggq.X_RMSNORM, "eps": 1e-5, "norm_w": norm_w(7001 + 2 * L)},
                    {"x_op": ggq.X_SILU_MUL, "up": yu, "res": [yo]}]
            h = dn["y"][0]
        rc, body = ggq.ggq_chain_create(12, 1, stages, ops)
        ggq.check(rc, "ggq_chain_create_ops")
        hd = self.rest[0]
        rc, head = ggq.ggq_chain_create(hd["qtype"], 1, [(hd["W"], hd["rows"], hd["cols"], h, hd["y"])],
                                        [{"x_op": ggq.X_RMSNORM, "eps": 1e-5, "norm_w": norm_w(7999)}])
        ggq.check(rc, "ggq_chain_create_ops")

        tok = torch.tensor([1234], dtype=torch.int32, device="cuda")
        norms.append(tok)
        h_in = q4[0]["x"]

        def run(sp):
            ggq.check(ggq.ggq_embed(hd["qtype"], hd["W"][0], hd["rows"][0], hd["cols"], tok.data_ptr(), 1, h_in, sp),
                      "ggq_embed")
            ggq.check(ggq.ggq_chain_run(body, sp), "ggq_chain_run")
            ggq.check(ggq.ggq_chain_run(head, sp), "ggq_chain_run")

        def free():
            ggq.ggq_chain_free(body)
            ggq.ggq_chain_free(head)

        return run, free, norms

    def close(self):
        if self.chain:
            self.ggq.ggq_chain_free(self.chain)
            self.chain = 0


# ----------------------------------------------- a pass planned from a file ----

class FilePass:
    """The library's planned pass (gguf_block_quantized_q8_gb300.plan) of a loaded
    file, every stage reading its own seeded x (as in DecodePass) and writing
    NaN-initialised outputs."""

    def __init__(self, model, layers, torch, ggq, synth, x_stream0=9000):
        from gguf_block_quantized_q8_gb300 import plan as P
        stages = P.plan_from_table(model, layers)
        self.plan, xs, ys = [], [], []
        self.type_bytes = {}   # weight bytes per tensor type
        for si, (qtype, ts) in enumerate(stages):
            cols = ts[0]["ne"][0]
            rows = [t["ne"][1] for t in ts]
            x = torch.from_numpy(synth.normal_f32(cols, x_stream0 + si)).cuda()
            y = [torch.full((r,), float("nan"), device="cuda") for r in rows]
            xs.append(x)
            ys.append(y)
            self.type_bytes[qtype] = self.type_bytes.get(qtype, 0) + sum(t["nbytes"] for t in ts)
            self.plan.append(dict(qtype=qtype, rows=rows, cols=cols, x=x, ys=y, names=[t["name"] for t in ts],
                                  x_stream=x_stream0 + si))
        self.dp = P.DecodePass(stages, xs, ys)
        self.weight_bytes = self.dp.weight_bytes
        self.calls, self.chains = self.dp.calls, self.dp.chains

    def run(self, sp):
        self.dp.run(sp)

    def close(self):
        self.dp.close()


def q4km_file_pass(torch, ggq, synth, stream, steps: int = 20, layers: int = 32):
    """The mixed-type pass of a Q4_K_M-style file: write it (synth.workloads.
    write_q4km_file, 4.9 GB), load it with ggq_load, plan the pass from the tensor
    table (FilePass) and time it as a CUDA graph.  The weights exceed L2."""
    from synth import workloads as WL
    shm = "/dev/shm" if os.path.isdir("/dev/shm") else tempfile.gettempdir()
    path = os.path.join(shm, f"ggq_q4km_{os.getpid()}.gguf")
    t0 = time.perf_counter()
    try:
        WL.write_q4km_file(path, layers)
        t_gen = time.perf_counter() - t0
        file_bytes = os.path.getsize(path)
        model = ggq.Model.load(path)
    finally:
        if os.path.exists(path):
            os.remove(path)
    fp = FilePass(model, layers, torch, ggq, synth)
    sp = stream.cuda_stream
    with torch.cuda.stream(stream):
        fp.run(sp)
    torch.cuda.synchronize()
    g = capture(torch, lambda: fp.run(sp), stream)
    time_graph(torch, g, stream, 3)
    ms = time_graph(torch, g, stream, steps)
    rc = ggq.device_status()
    out = {"ms": round(ms, 4), "GB_s": round(fp.weight_bytes / ms / 1e6, 1), "launches": len(fp.calls),
           "chain_launches": len(fp.chains), "weight_bytes_per_pass": fp.weight_bytes,
           "q6_k_bytes_per_pass": fp.type_bytes.get(14, 0), "file_bytes": file_bytes,
           "generate_s": round(t_gen, 2), "status": rc,
           "plan": "per layer [q,k,v] [o] [gate,up] [down], split by type; every stage (Q4_K, Q6_K, "
                   "the Q6_K head) in one chain launch of mixed types; attn_v and ffn_down Q6_K in odd layers"}
    del g
    fp.close()
    model.close()
    return out


def time_graph(torch, graph, stream, steps):
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps   # ms per step


def capture(torch, fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    g.replay()
    torch.cuda.synchronize()
    return g


def roofline_chain(torch, dp, stream, steps):
    """Average launch of the dominant kernel (the Q4_K chain kernel running the
    pass's Q4_K stages) in the bench's launch configuration: one launch per
    CUDA-graph replay, CUDA events on the launching stream around `steps`
    replays.  Returns (algorithmic bytes per launch, seconds per launch)."""
    g = capture(torch, lambda: dp.run_chain(stream.cuda_stream), stream)
    ms = time_graph(torch, g, stream, steps)
    return dp.q4_bytes, ms * 1e-3


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def _on_threads(calls, threads: int) -> float:
    """Run the oracle calls (callables) on `threads` Python threads -- the
    oracle's C functions release the interpreter lock -- and return the wall
    seconds."""
    import concurrent.futures as cf
    t0 = time.perf_counter()
    if threads <= 1:
        for c in calls:
            c()
    else:
        with cf.ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda c: c(), calls))
    return time.perf_counter() - t0


def _row_jobs(qtype, W, rows, cols, x, pieces, gemm=False):
    """The oracle over `rows` rows of W as `pieces` calls on contiguous row blocks."""
    import oracle
    rb = oracle.row_bytes(qtype, cols)
    jobs = []
    for k in range(pieces):
        r0, r1 = rows * k // pieces, rows * (k + 1) // pieces
        if r1 > r0:
            Wk = W[r0 * rb:r1 * rb]
            if gemm:
                jobs.append(lambda Wk=Wk, n=r1 - r0: oracle.gemm_bf16(qtype, Wk, n, cols, x))
            else:
                jobs.append(lambda Wk=Wk, n=r1 - r0: oracle.gemv(qtype, Wk, n, cols, x))
    return jobs


def cpu_oracle_jobs(budget_s: float, layers: int = 32):
    """A bounded sample of the decode pass for the oracle: whole rows drawn
    from every tensor of the stack in turn (regenerated from their counters),
    64 rows per tensor, about budget_s of single-thread oracle work.  Returns
    (oracle calls, weight bytes, description)."""
    import numpy as np
    import oracle
    import synth
    from synth import workloads as WL
    gem = WL.llama8b_pass(layers)
    rng = np.random.default_rng(0)
    budget_bytes = budget_s * 0.4e9   # the oracle's single-thread rate, about 0.4 GB/s of weights
    jobs, done_bytes, n_rows, i = [], 0, 0, 0
    while done_bytes < budget_bytes:
        g = gem[i % len(gem)]
        i += 1
        rows = 64
        r0 = int(rng.integers(0, g.rows - rows + 1))
        W = synth.weight_rows(g.qtype, g.stream, rows, g.cols, row0=r0)
        x = synth.normal_f32(g.cols, g.x_stream).reshape(1, -1)
        jobs.append(lambda W=W, g=g, x=x, rows=rows: oracle.gemv(g.qtype, W, rows, g.cols, x))
        done_bytes += W.nbytes
        n_rows += rows
    desc = (f"{n_rows} whole rows ({done_bytes / 1e6:.1f} MB of Q4_K/Q8_0 weights) sampled 64 at a time from "
            f"{i} tensors of the {layers}-layer pass, oracle decode + fp64 dot products (generation not timed)")
    return jobs, done_bytes, desc


def cpu_oracle_sample(budget_s: float, layers: int = 32, threads: int = 1):
    """The oracle on a bounded sample of the pass (cpu_oracle_jobs) on
    `threads` threads.  Returns (GB/s of weight bytes, description, seconds)."""
    jobs, nbytes, desc = cpu_oracle_jobs(budget_s, layers)
    used = _on_threads(jobs, threads)
    return nbytes / used / 1e9, f"{desc}, {threads} thread(s)", used


def cpu_oracle_configs(threads: int):
    """The oracle per configuration, single-threaded and on `threads` threads
    (row blocks of the same matrices): cfg1 and cfg2 whole, cfg4 on 1024 of its
    14336 rows at every M, cfg5 on 16 of its 14336 rows for all 512 tokens.
    GB/s of weight bytes (TFLOP/s for cfg5).  Generation is not timed."""
    import numpy as np
    import synth
    from synth import workloads as WL
    out = {}

    def both(name, qtype, W, rows, cols, x, work, unit, gemm=False):
        r = {}
        for n in (1, threads):
            t = _on_threads(_row_jobs(qtype, W, rows, cols, x, max(n, 1) * (4 if n > 1 else 1), gemm), n)
            r["threads_%d" % n] = round(work / t / (1e12 if unit == "TFLOP/s" else 1e9), 6 if unit == "TFLOP/s" else 4)
        r["unit"] = unit
        out[name] = r

    g = WL.CFG1[0]
    W = synth.weight_rows(g.qtype, g.stream, g.rows, g.cols)
    both("cfg1_q8_0_2048x2048", g.qtype, W, g.rows, g.cols, synth.normal_f32(g.cols, g.x_stream).reshape(1, -1),
         W.nbytes, "GB/s")
    # cfg2: the 7 projections one after another
    tot, t1, tn = 0, 0.0, 0.0
    for g in WL.CFG2:
        W = synth.weight_rows(g.qtype, g.stream, g.rows, g.cols)
        x = synth.normal_f32(g.cols, g.x_stream).reshape(1, -1)
        t1 += _on_threads(_row_jobs(g.qtype, W, g.rows, g.cols, x, 1), 1)
        tn += _on_threads(_row_jobs(g.qtype, W, g.rows, g.cols, x, 4 * threads), threads)
        tot += W.nbytes
    out["cfg2_smollm3_layer_q4_k"] = {"threads_1": round(tot / t1 / 1e9, 4),
                                      "threads_%d" % threads: round(tot / tn / 1e9, 4), "unit": "GB/s"}
    g = WL.CFG4
    rows = 1024
    W = synth.weight_rows(g.qtype, g.stream, rows, g.cols)
    res = {}
    for M in WL.CFG4_M:
        x = synth.normal_f32(M * g.cols, g.x_stream).reshape(M, -1)
        r = {}
        for n in (1, threads):
            t = _on_threads(_row_jobs(g.qtype, W, rows, g.cols, x, 4 * n if n > 1 else 1), n)
            r["threads_%d" % n] = round(W.nbytes / t / 1e9, 4)
        res[str(M)] = r
    out["cfg4_q8_0_14336x4096"] = {"rows_sampled": rows, "unit": "GB/s", **res}
    g = WL.CFG5
    rows = 16
    W = synth.weight_rows(g.qtype, g.stream, rows, g.cols)
    X = synth.normal_bf16(WL.CFG5_M * g.cols, g.x_stream).reshape(WL.CFG5_M, g.cols)
    both("cfg5_prefill_q4_k_512x14336x4096", g.qtype, W, rows, g.cols, X, 2.0 * WL.CFG5_M * rows * g.cols,
         "TFLOP/s", gemm=True)
    out["cfg5_prefill_q4_k_512x14336x4096"]["rows_sampled"] = rows
    del np
    return out


# -------------------------------------------------------------- extras ----

L2_BYTES = 129 * 1000 * 1000          # GB300 L2
ROTATE_BYTES = 4 * L2_BYTES           # distinct weight bytes cycled through between reuses
MIN_LAUNCHES = 200


def copies_for(nbytes: int, cap: int = 160) -> int:
    """Weight copies to cycle so that one pass over them moves at least
    4 x L2 of distinct bytes (each launch reads its weights cold)."""
    return max(1, min(cap, -(-ROTATE_BYTES // max(1, nbytes))))


def kernel_time(torch, fn, stream, per_graph, min_launches=MIN_LAUNCHES, min_replays=5):
    """Per-launch time of fn (a C-ABI call on `stream`): a CUDA graph of
    `per_graph` launches (fn cycles its weight copies), replayed until at
    least `min_launches` launches and `min_replays` replays; each replay timed
    with CUDA events on the stream.  Returns (median seconds per launch over
    the replays, launches timed)."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(per_graph):
            fn()
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    replays = max(min_replays, -(-min_launches // per_graph))
    e = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(replays)]
    with torch.cuda.stream(stream):
        for e0, e1 in e:
            e0.record(stream)
            g.replay()
            e1.record(stream)
    torch.cuda.synchronize()
    per = sorted(e0.elapsed_time(e1) * 1e-3 / per_graph for e0, e1 in e)
    return per[len(per) // 2], replays * per_graph


def extras(torch, ggq, synth, stream):
    """Kernel timings for the other configurations: weights cycled through
    copies totalling at least 4 x L2 (cold reads), the median over replays of
    a graph, at least 200 launches each."""
    import numpy as np
    from synth import workloads as WL
    out = {}
    sp = stream.cuda_stream

    def rotating(gs):
        base = [torch.from_numpy(synth.weight_rows(g.qtype, g.stream, g.rows, g.cols)).cuda() for g in gs]
        n = copies_for(sum(int(b.numel()) for b in base))
        return [base] + [[b.clone() for b in base] for _ in range(n - 1)]

    def timing(t, launches, copies, nbytes, **kw):
        return {"us": round(t * 1e6, 2), "GB_s": round(nbytes / t / 1e9, 1), **kw,
                "launches": launches, "weight_copies": copies,
                "rotated_MB": round(copies * nbytes / 1e6, 1)}

    # cfg1: Q8_0 2048x2048, M=1
    g = WL.CFG1[0]
    Ws = rotating([g])
    x = torch.randn(g.cols, device="cuda")
    y = torch.empty(g.rows, device="cuda")
    nb = g.rows * synth.row_bytes(g.qtype, g.cols)
    k = [0]

    def f1():
        W = Ws[k[0] % len(Ws)][0]
        k[0] += 1
        ggq.check(ggq.ggq_gemv(g.qtype, W.data_ptr(), g.rows, g.cols, x.data_ptr(), y.data_ptr(), 1, sp), "gemv")
    t, n = kernel_time(torch, f1, stream, len(Ws))
    out["cfg1_q8_0_2048x2048"] = timing(t, n, len(Ws), nb)
    del Ws

    # cfg2: one SmolLM3 layer, 7 Q4_K GEMVs in 4 launches ([q,k,v], [o], [gate,up], [down])
    gs = WL.CFG2
    Ws = rotating(gs)
    xs = {c: torch.randn(c, device="cuda") for c in (2048, 11008)}
    ys = [torch.empty(gg.rows, device="cuda") for gg in gs]
    groups = [[0, 1, 2], [3], [4, 5], [6]]
    nb = sum(gg.rows * synth.row_bytes(gg.qtype, gg.cols) for gg in gs)
    k = [0]

    def f2():
        Wc = Ws[k[0] % len(Ws)]
        k[0] += 1
        for grp in groups:
            ggq.check(ggq.ggq_gemv_multi(12, [Wc[i].data_ptr() for i in grp], [gs[i].rows for i in grp],
                                         gs[grp[0]].cols, xs[gs[grp[0]].cols].data_ptr(),
                                         [ys[i].data_ptr() for i in grp], 1, sp), "gemv")
    t, n = kernel_time(torch, f2, stream, len(Ws), min_launches=MIN_LAUNCHES // 4)
    out["cfg2_smollm3_layer_q4_k"] = timing(t, 4 * n, len(Ws), nb, launches_per_layer=4)
    # the same 4 stages as one chain launch (one chain per weight copy: a chain
    # binds its pointers at creation)
    chains = []
    try:
        for Wc in Ws:
            rc, h = ggq.ggq_chain_create(12, 1, [([Wc[i].data_ptr() for i in grp], [gs[i].rows for i in grp],
                                                  gs[grp[0]].cols, xs[gs[grp[0]].cols].data_ptr(),
                                                  [ys[i].data_ptr() for i in grp]) for grp in groups])
            ggq.check(rc, "ggq_chain_create")
            chains.append(h)
        k = [0]

        def f2c():
            h = chains[k[0] % len(chains)]
            k[0] += 1
            ggq.check(ggq.ggq_chain_run(h, sp), "ggq_chain_run")
        t, n = kernel_time(torch, f2c, stream, len(chains))
        out["cfg2_smollm3_layer_q4_k_one_chain"] = timing(t, n, len(Ws), nb, launches_per_layer=1)
    finally:
        for h in chains:
            ggq.ggq_chain_free(h)
    del Ws

    # cfg4: Q8_0 14336x4096, M in 1..16
    g = WL.CFG4
    Ws = rotating([g])
    nb = g.rows * synth.row_bytes(g.qtype, g.cols)
    res = {}
    for M in WL.CFG4_M:
        x = torch.randn(M, g.cols, device="cuda")
        y = torch.empty(M, g.rows, device="cuda")
        k = [0]

        def f4():
            W = Ws[k[0] % len(Ws)][0]
            k[0] += 1
            ggq.check(ggq.ggq_gemv(g.qtype, W.data_ptr(), g.rows, g.cols, x.data_ptr(), y.data_ptr(), M, sp),
                      "gemv")
        t, n = kernel_time(torch, f4, stream, len(Ws))
        res[str(M)] = timing(t, n, len(Ws), nb, TFLOP_s=round(2 * M * g.rows * g.cols / t / 1e12, 2))
    out["cfg4_q8_0_14336x4096"] = res
    del Ws

    # cfg5: prefill Q4_K 14336x4096 x bf16 X 512x4096 (compute-bound), and the
    # same with the Q8_0 14336x4096 matrix of cfg4
    g = WL.CFG5
    X = torch.from_numpy(synth.normal_bf16(WL.CFG5_M * g.cols, g.x_stream).view(np.int16)).cuda()
    Y = torch.empty(WL.CFG5_M, g.rows, device="cuda")
    flops = 2 * WL.CFG5_M * g.rows * g.cols
    for name, gq in (("cfg5_prefill_q4_k_512x14336x4096", g), ("prefill_q8_0_512x14336x4096", WL.CFG4)):
        Ws = rotating([gq])
        k = [0]

        def f5():
            W = Ws[k[0] % len(Ws)][0]
            k[0] += 1
            ggq.check(ggq.ggq_gemm_prefill(gq.qtype, W.data_ptr(), gq.rows, gq.cols, X.data_ptr(), Y.data_ptr(),
                                           WL.CFG5_M, sp), "prefill")
        t, n = kernel_time(torch, f5, stream, len(Ws))
        out[name] = {"us": round(t * 1e6, 2), "TFLOP_s": round(flops / t / 1e12, 1), "launches": n,
                     "weight_copies": len(Ws)}
        del Ws
    del X, Y

    # the cfg4 shape as Q4_0, as F32 and as Q6_K; Q4_0 14336x4128 (warp-per-row
    # kernel); the Q6_K ffn_down shape
    for name, g, Ms in [("q4_0_14336x4096", WL.Q40_GEMV, (1, 2, 4, 8, 16)),
                        ("q4_0_14336x4128_warp_per_row", WL.Q40_ODD_GEMV, (1, 8)),
                        ("f32_14336x4096", WL.F32_GEMV, (1,)),
                        ("q6_k_14336x4096", WL.Q6K_GEMV, (1, 2, 8)),
                        ("q6_k_4096x14336", WL.Q6K_DOWN_GEMV, (1,))]:
        Ws = rotating([g])
        nb = g.rows * synth.row_bytes(g.qtype, g.cols)
        res = {}
        for M in Ms:
            x = torch.randn(M, g.cols, device="cuda")
            y = torch.empty(M, g.rows, device="cuda")
            k = [0]

            def fx():
                W = Ws[k[0] % len(Ws)][0]
                k[0] += 1
                ggq.check(ggq.ggq_gemv(g.qtype, W.data_ptr(), g.rows, g.cols, x.data_ptr(), y.data_ptr(), M, sp),
                          "gemv")
            t, n = kernel_time(torch, fx, stream, len(Ws))
            res[str(M)] = timing(t, n, len(Ws), nb)
        out[name] = res
        del Ws
    return out


def roofline_traffic(bytes_per_launch: int):
    """DRAM traffic per launch of the dominant kernel from the committed ncu
    capture (profiles/roofline_traffic.json), scaled to the full launch by the
    bytes it streams; None if the kernel sources changed since the capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "roofline_traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        h = hashlib.sha256()
        for src in t["kernel_sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        if h.hexdigest()[:16] != t["kernel_sources_sha256_16"]:
            return None
        captured = t["dram_bytes_read"] + t["dram_bytes_write"]
        return int(captured * bytes_per_launch / t["captured_algorithmic_bytes"])
    except (OSError, KeyError, ValueError):
        return None


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs"), d.get("bf16_tflops"), "measured"
    except (OSError, ValueError):
        return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------------- main ----

def run_reference(a, ws, rank):
    """The reference arm: the CPU oracle as it stands, on the bench workload.
    K timed steps after W warm-up steps, each step a bounded sample of the
    pass (whole rows of every tensor in turn) sized so the whole run stays
    within about two minutes.  Under torchrun only rank 0 runs and prints."""
    if rank != 0:
        return 0
    import multiprocessing
    steps = max(1, a.steps)
    threads = host_threads()
    # one sample of about `per` seconds of single-thread oracle work, generated
    # once; each step runs the oracle over all of it on every host thread
    per = max(0.05, min(a.cpu_seconds / 6, 120.0 * threads / (steps + a.warmup)))
    jobs, nbytes, desc = cpu_oracle_jobs(per, a.layers)
    desc = f"{desc}, {threads} threads"
    for _ in range(a.warmup):
        _on_threads(jobs, threads)
    vals, walls = [], []
    for _ in range(steps):
        t = _on_threads(jobs, threads)
        walls.append(t)
        vals.append(nbytes / t / 1e9)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": a.gpus, "steps": steps, "warmup": a.warmup,
        "ms_per_step": round(1e3 * statistics.median(walls), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "layers": a.layers, "sampled": True},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"per step: {desc}", "host_cpus": multiprocessing.cpu_count()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    a = args_parse()
    if a.kernel:
        return run_kernel(a)
    if a.file_pass_layers:
        import torch
        import gguf_block_quantized_q8_gb300 as ggq
        import synth
        torch.cuda.set_device(0)
        stream = torch.cuda.Stream()
        out = q4km_file_pass(torch, ggq, synth, stream, steps=5, layers=a.file_pass_layers)
        print(json.dumps({"file_pass_layers": a.file_pass_layers, **out}))
        return 0 if out["status"] == 0 else 1
    ws, rank, local = dist_setup()
    if a.impl == "reference":
        return run_reference(a, ws, rank)

    import torch
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.cuda.current_device()
    import gguf_block_quantized_q8_gb300 as ggq
    import synth

    # ---- weights: seeded synthetic GGUF -> ggq_load (rows a1-a3 of the path)
    shm = "/dev/shm" if os.path.isdir("/dev/shm") else tempfile.gettempdir()
    path = os.path.join(shm, f"ggq_bench_{os.getpid()}_{rank}.gguf")
    t0 = time.perf_counter()
    gem = build_pass_file(path, a.layers)
    t_gen = time.perf_counter() - t0
    t0 = time.perf_counter()
    model = ggq.Model.load(path)
    t_load = time.perf_counter() - t0
    file_bytes = os.path.getsize(path)
    os.remove(path)

    stream = torch.cuda.Stream()
    sp = stream.cuda_stream
    dp = DecodePass(model, stage_plan(a.layers), torch, ggq, synth)
    weight_bytes = dp.weight_bytes
    assert weight_bytes == sum(g.rows * synth.row_bytes(g.qtype, g.cols) for g in gem)

    clocks = ClockSampler(dev)
    clocks.start()
    # ---- warm-up (kernel attributes are set on first launch), then capture one pass
    with torch.cuda.stream(stream):
        for _ in range(max(1, a.warmup)):
            dp.run(sp)
    torch.cuda.synchronize()
    rc = ggq.device_status()
    if rc:
        raise SystemExit(f"device status {rc} after warm-up")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        dp.run(sp)
    # keep the GPU busy >= 1.5 s before timing so the clock samples see load
    t_end = time.perf_counter() + 1.5
    while time.perf_counter() < t_end:
        time_graph(torch, graph, stream, 20)

    # ---- timed region: K passes (graph replays), barrier + sync on both sides
    dist_barrier(ws)
    ms = time_graph(torch, graph, stream, a.steps)
    dist_barrier(ws)
    ms = dist_max(ms, ws, device="cuda")

    # ---- end to end through the C ABI with host buffers: every step uploads
    # the x of all its stages from pinned memory (one copy: they are
    # contiguous) and reads back its result, the head's logits, all inside the
    # timed region.  Two device buffer sets (a second pass bound to them):
    # step k+1's upload runs on a copy stream while step k computes, and step
    # k's logits come back while step k+1 computes.
    dp2 = DecodePass(model, stage_plan(a.layers), torch, ggq, synth)
    with torch.cuda.stream(stream):
        dp2.run(sp)
    torch.cuda.synchronize()
    graph2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph2, stream=stream):
        dp2.run(sp)
    passes = [(dp, graph), (dp2, graph2)]
    head_host = torch.empty(dp.head_rows, dtype=torch.float32).pin_memory()
    cstream = torch.cuda.Stream()
    e2e_steps = max(3, min(a.steps, 50))
    ev_up = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_free = [torch.cuda.Event() for _ in range(2)]
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    cstream.wait_event(e0)
    with torch.cuda.stream(cstream):
        passes[0][0].x_dev.copy_(dp.x_host, non_blocking=True)
        ev_up[0].record(cstream)
    for k in range(e2e_steps):
        b = k % 2
        pk, gk = passes[b]
        stream.wait_event(ev_up[b])
        with torch.cuda.stream(stream):
            gk.replay()
        ev_done[b].record(stream)
        with torch.cuda.stream(cstream):
            if k + 1 < e2e_steps:
                nb_ = (k + 1) % 2
                if k >= 1:
                    cstream.wait_event(ev_free[nb_])   # step k-1 read its x and its logits are home
                passes[nb_][0].x_dev.copy_(dp.x_host, non_blocking=True)
                ev_up[nb_].record(cstream)
            cstream.wait_event(ev_done[b])
            head_host.copy_(pk.head_y, non_blocking=True)
            ev_free[b].record(cstream)
    stream.wait_stream(cstream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = dist_max(e0.elapsed_time(e1) / e2e_steps, ws, device="cuda")
    del graph2
    dp2.close()

    # ---- roofline of the dominant kernel (Q4_K GEMV launches)
    r_steps = max(3, min(a.steps, 20))
    per_launch_bytes, per_launch_s = roofline_chain(torch, dp, stream, r_steps)
    # the same pass as one launch per stage (129 launches), for comparison
    g_l = capture(torch, lambda: dp.run_launches(sp), stream)
    ms_launches = time_graph(torch, g_l, stream, r_steps)
    del g_l
    # and as one launch per weight matrix (225 launches)
    g_t = capture(torch, lambda: dp.run_per_tensor(sp), stream)
    ms_tensors = time_graph(torch, g_t, stream, r_steps)
    del g_t
    clk = clocks.stop()
    rc = ggq.device_status()
    if rc:
        raise SystemExit(f"device status {rc} after the timed region")

    extra = {} if a.no_extras else extras(torch, ggq, synth, stream)
    if not a.no_extras:
        extra["q4_k_m_file_pass_llama8b"] = q4km_file_pass(torch, ggq, synth, stream)
    if not a.no_extras and len(dp.rest) == 1:
        # the pass with the layer's element-wise steps fused in (real data flow)
        frun, ffree, _norms = dp.fused_pass(synth)
        frun(sp)
        torch.cuda.synchronize()
        g_f = capture(torch, lambda: frun(sp), stream)
        ms_f = time_graph(torch, g_f, stream, r_steps)
        del g_f
        if ggq.device_status():
            raise SystemExit("device status set by the fused pass")
        ffree()
        extra["cfg3_fused_layer_pass"] = {
            "ms": round(ms_f, 4), "GB_s": round(weight_bytes / (ms_f * 1e-3) / 1e9, 1), "launches": 3,
            "fused": "token embedding row (ggq_embed), rmsnorm into q/k/v and gate/up, silu(gate)*up into down, "
                     "residual adds after o and down, final rmsnorm into the head"}
    hbm_peak, bf16_peak, peak_kind = measured_peaks()

    step_bytes = weight_bytes + dp.io_bytes
    value = step_bytes * ws / (ms * 1e-3) / 1e9
    achieved = per_launch_bytes / per_launch_s / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": a.steps,
        "warmup": a.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp32 accumulate over Q4_K/Q8_0 blocks",
        "data": "synthetic (seeded N(0,0.02) weights encoded to Q4_K/Q8_0, N(0,1) activations)",
        "config": {"workload": WORKLOAD, "layers": a.layers, "hidden": 4096, "ffn": 14336,
                   "heads": 32, "kv_heads": 8, "vocab": 128256, "batch": 1,
                   "weight_bytes_per_pass": weight_bytes, "launches_per_pass": dp.launches,
                   "l2": "weights (4.48 GB) exceed the 129 MB L2 between passes",
                   "parallelism": "replicas" if ws > 1 else "single GPU"},
        "tok_s": round(1000.0 / ms * ws, 2),
        "frac_of_8tbs": round(value / 8000.0, 4),
        "frac_of_measured_hbm": round(value / hbm_peak, 4),
        "e2e": {"value": round(step_bytes * ws / (ms_e2e * 1e-3) / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": dp.x_bytes, "d2h_bytes_per_step": 4 * dp.head_rows,
                "ms_per_step": round(ms_e2e, 4),
                "how": "per step: every stage's x uploaded from pinned host memory (one copy), the pass, the "
                       "head's logits read back to pinned memory; two device buffer sets, step k+1's upload and "
                       "step k's read-back on a copy stream overlapping the passes"},
        "gpu_launches": dp.launches * a.steps,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "traffic": roofline_traffic(int(per_launch_bytes)),
                     "kernel": f"rows_kernel<Q4_K, M=1, 16 warps> (one ggq_chain_run over {len(dp.q4)} stages)",
                     "peak_kind": f"{peak_kind} (copy, burst)",
                     "bytes_per_launch": int(per_launch_bytes), "us_per_launch": round(per_launch_s * 1e6, 3),
                     "timing": "one chain launch per CUDA-graph replay, events on its stream"},
        "per_stage_launches": {"ms_per_step": round(ms_launches, 4), "launches_per_pass": len(dp.stages),
                               "value": round(step_bytes * ws / (ms_launches * 1e-3) / 1e9, 1), "unit": "GB/s"},
        "per_tensor_launches": {"ms_per_step": round(ms_tensors, 4),
                                "launches_per_pass": sum(len(st["W"]) for st in dp.stages),
                                "value": round(step_bytes * ws / (ms_tensors * 1e-3) / 1e9, 1), "unit": "GB/s"},
        "clocks": clk,
        "load": {"generate_s": round(t_gen, 2), "ggq_load_s": round(t_load, 3), "file_bytes": file_bytes},
        "configs": extra,
    }
    if not a.no_cpu_baseline and rank == 0 and ws == 1:
        import multiprocessing
        threads = host_threads()
        jobs, nbytes, desc = cpu_oracle_jobs(a.cpu_seconds / 6, a.layers)
        used1 = _on_threads(jobs, 1)
        used = _on_threads(jobs, threads)
        line["cpu_baseline"] = {"value": round(nbytes / used / 1e9, 4), "unit": "GB/s", "cores": threads,
                                "kind": "oracle", "sample": f"{desc}, {threads} threads", "seconds": round(used, 2),
                                "single_thread": {"value": round(nbytes / used1 / 1e9, 4), "seconds": round(used1, 2)},
                                "host_cpus": multiprocessing.cpu_count(),
                                "configs": cpu_oracle_configs(threads)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    dp.close()
    model.close()
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

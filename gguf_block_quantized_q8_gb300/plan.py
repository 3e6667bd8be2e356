"""The decode weight pass of a loaded GGUF model, planned from its tensor table.

A transformer layer's projections run in dependency order ("GGUF Inferencer in R"
section 4: the normalized input through the query/key/value weights, attention
through the output weight, then the feed-forward gate/up and down weights), so a
pass is, per layer, the stages [attn_q, attn_k, attn_v], [attn_output],
[ffn_gate, ffn_up], [ffn_down], then the output head.  Files mix weight types
("GGUF: The File Format Powering Local LLM Inference", "Understanding
quantization names like Q4_K_M": Q4_K_M keeps part of attn_v and ffn_down in
Q6_K), so a stage whose matrices differ in type is split by type, in order.

Launches: each run of consecutive stages the chain kernel streams (Q8_0;
Q4_K and Q4_0 with cols >= 768; Q6_K with cols % 2048 == 0), of one type or of
Q6_K and one other type, is one ``ggq_chain_run``; every other stage (F32, or
a shape outside those limits) is one ``ggq_gemv`` / ``ggq_gemv_multi``.  A
Q4_K_M file's whole pass, head included, is then one launch.  Everything here is host-side
planning: the arithmetic runs in the library's kernels.
"""
from __future__ import annotations

from . import _ggq

# the GEMV stages of a layer in dependency order, by GGUF tensor name
LAYER_STAGES = (("attn_q", "attn_k", "attn_v"), ("attn_output",), ("ffn_gate", "ffn_up"), ("ffn_down",))
# the types the chain kernel streams
CHAIN_TYPES = (_ggq.Q4_0, _ggq.Q8_0, _ggq.Q4_K, _ggq.Q6_K)


def chainable(qtype: int, cols: int) -> bool:
    """Whether a stage of this type and width can be a chain stage (the limits
    ggq_chain_create documents; the library checks them again)."""
    if qtype not in CHAIN_TYPES or cols % 256 or cols > (1 << 20):
        return False
    if qtype in (_ggq.Q4_K, _ggq.Q4_0) and cols < 768:
        return False
    return not (qtype == _ggq.Q6_K and cols % 2048)


def block_count(model) -> int:
    """Layers of the model: the ``<arch>.block_count`` key, else the number of
    distinct ``blk.N.`` tensor prefixes."""
    kv = {k: (t, v) for k, t, v in model.kvs()}
    arch = kv.get("general.architecture")
    if arch is not None and arch[0] == 8:
        key = arch[1].decode() + ".block_count"
        if key in kv and kv[key][0] in (4, 5, 10, 11):
            return int.from_bytes(kv[key][1], "little", signed=kv[key][0] in (5, 11))
    blocks = {t["name"].split(".")[1] for t in model.tensors() if t["name"].startswith("blk.")}
    return len(blocks)


def plan_from_table(model, layers: int | None = None, head: str = "output.weight"):
    """The stages of the pass from the tensor table alone: a list of
    ``(type, [tensor info])`` in dependency order, each stage's matrices of one
    type.  ``layers`` defaults to ``block_count(model)``; ``head`` is left out
    if None."""
    if layers is None:
        layers = block_count(model)
    stages = []
    for L in range(layers):
        for names in LAYER_STAGES:
            groups = {}
            for n in names:
                t = model.find(f"blk.{L}.{n}.weight")
                groups.setdefault(t["type"], []).append(t)
            stages += list(groups.items())
    if head is not None:
        t = model.find(head)
        stages.append((t["type"], [t]))
    return stages


def mixable(types) -> bool:
    """Whether one chain may hold stages of these types: one type, or Q6_K and
    one other (the mixes ggq_chain_create_typed runs)."""
    return len(set(types) - {_ggq.Q6_K}) <= 1 and (len(set(types)) == 1 or _ggq.Q8_0 not in types)


def segments(types, cols):
    """Launches for stages of the given types and widths, in order: each run of
    consecutive chainable stages whose types may share a chain is one chain
    launch, every other stage a launch of its own.  Returns
    ``[(start, end, is_chain)]``."""
    if len(types) != len(cols):
        raise ValueError("one width per stage")
    out, i = [], 0
    while i < len(types):
        if chainable(types[i], cols[i]):
            j = i
            while j < len(types) and chainable(types[j], cols[j]) and mixable(types[i:j + 1]):
                j += 1
            out.append((i, j, True))
            i = j
        else:
            out.append((i, i + 1, False))
            i += 1
    return out


class DecodePass:
    """A planned pass bound to activation and output buffers.

    stages: ``plan_from_table`` output.  xs[i]: CUDA fp32 tensor [M, cols] read
    by stage i; ys[i]: one CUDA fp32 tensor [M, rows] per matrix of stage i.
    Stage s+1 reads its x only after every output of stage s is written (the
    chain's stage boundaries, or stream order between launches), so an x may be
    an earlier stage's y.  M is 1..4 (the chain kernel's range); at M > 2 the
    widest stages of a large model (the 14336-column down projection) leave the
    chain and run as ggq_gemv calls of their own.
    """

    def __init__(self, stages, xs, ys, M: int = 1):
        if not (1 <= M <= 4):
            raise ValueError("M must be 1..4")
        if len(xs) != len(stages) or len(ys) != len(stages):
            raise ValueError("one x and one list of ys per stage")
        self.M = M
        self.stages = []
        for (qtype, ts), x, y in zip(stages, xs, ys):
            cols = int(ts[0]["ne"][0])
            rows = [int(t["ne"][1]) if len(t["ne"]) > 1 else 1 for t in ts]
            if any(int(t["ne"][0]) != cols for t in ts) or len(y) != len(ts):
                raise ValueError("a stage's matrices share cols and have one output each")
            self.stages.append(dict(qtype=qtype, W=[t["data"] for t in ts], rows=rows, cols=cols, x=x, ys=list(y),
                                    nbytes=sum(int(t["nbytes"]) for t in ts)))
        self.weight_bytes = sum(s["nbytes"] for s in self.stages)
        self.calls, self.chains = [], []
        try:
            for i, j, is_chain in segments([s["qtype"] for s in self.stages], [s["cols"] for s in self.stages]):
                if is_chain:
                    self._chain_run(self.stages[i:j])
                else:
                    self.calls.append(("stage", self.stages[i]))
        except Exception:
            self.close()
            raise

    def _create(self, run):
        raw = [(s["W"], s["rows"], s["cols"], s["x"].data_ptr(), [y.data_ptr() for y in s["ys"]]) for s in run]
        return _ggq.ggq_chain_create_typed(self.M, [s["qtype"] for s in run], raw)

    def _chain_run(self, run):
        """Calls for a run of chainable stages: one chain, unless a stage is too
        wide for the chain kernel at M rows (the pre-scaled x of all M rows must
        fit in shared memory: 4 rows of 14336 columns do not).  Such a stage is
        a ggq_gemv of its own, which runs the rows in groups that fit; the
        stages between them form chains."""
        rc, h = self._create(run)
        if rc == 0:
            self.chains.append(h)
            self.calls.append(("chain", h))
            return
        if len(run) == 1:
            if rc != _ggq.EINVAL:
                _ggq.check(rc, "ggq_chain_create")
            self.calls.append(("stage", run[0]))
            return
        fits = []
        for s in run:
            rc1, h1 = self._create([s])
            if rc1 == 0:
                _ggq.ggq_chain_free(h1)
            elif rc1 != _ggq.EINVAL:
                _ggq.check(rc1, "ggq_chain_create")
            fits.append(rc1 == 0)
        if all(fits):   # every stage fits alone, the run does not: not a width limit
            _ggq.check(rc, "ggq_chain_create")
        i = 0
        while i < len(run):
            j = i + 1
            while j < len(run) and fits[j] == fits[i]:
                j += 1
            if fits[i]:
                self._chain_run(run[i:j])
            else:
                self.calls += [("stage", s) for s in run[i:j]]
            i = j

    @property
    def launches(self) -> int:
        return len(self.calls)

    def run(self, stream=None) -> None:
        """Launch the pass on `stream` (a torch stream, a cudaStream_t value or
        None: the current stream); asynchronous."""
        sp = _ggq._stream_ptr(stream)
        for kind, c in self.calls:
            if kind == "chain":
                _ggq.check(_ggq.ggq_chain_run(c, sp), "ggq_chain_run")
            elif len(c["W"]) == 1:
                _ggq.check(_ggq.ggq_gemv(c["qtype"], c["W"][0], c["rows"][0], c["cols"], c["x"].data_ptr(),
                                         c["ys"][0].data_ptr(), self.M, sp), "ggq_gemv")
            else:
                _ggq.check(_ggq.ggq_gemv_multi(c["qtype"], c["W"], c["rows"], c["cols"], c["x"].data_ptr(),
                                               [y.data_ptr() for y in c["ys"]], self.M, sp), "ggq_gemv_multi")

    def close(self) -> None:
        for h in self.chains:
            _ggq.ggq_chain_free(h)
        self.chains = []
        self.calls = []

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

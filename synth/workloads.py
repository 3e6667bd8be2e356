"""Shapes of the benchmark workloads (synthetic, seeded; no model file is read).

Every weight is N(0, 0.02) before encoding, activations N(0, 1).  Tensor names
follow the GGUF naming of "GGUF Inferencer in R" section 2.1 (blk.N.attn_q.weight,
..., token_embd.weight).  rows = output features, cols = input features (ne0).
"""
from __future__ import annotations

from dataclasses import dataclass

from . import TYPE_F32, TYPE_Q4_0, TYPE_Q4_K, TYPE_Q6_K, TYPE_Q8_0, stream_id

W_SIGMA = 0.02
X_SIGMA = 1.0


@dataclass(frozen=True)
class Gemv:
    name: str
    qtype: int
    rows: int
    cols: int

    @property
    def stream(self) -> int:
        return stream_id("w", self.name, self.qtype, self.rows, self.cols)

    @property
    def x_stream(self) -> int:
        return stream_id("x", self.name, self.rows, self.cols)


def _layer(prefix: str, hidden: int, n_q: int, n_kv: int, head_dim: int, ffn: int,
           qtype: int):
    kv = n_kv * head_dim
    return [
        Gemv(f"{prefix}.attn_q.weight", qtype, n_q * head_dim, hidden),
        Gemv(f"{prefix}.attn_k.weight", qtype, kv, hidden),
        Gemv(f"{prefix}.attn_v.weight", qtype, kv, hidden),
        Gemv(f"{prefix}.attn_output.weight", qtype, hidden, n_q * head_dim),
        Gemv(f"{prefix}.ffn_gate.weight", qtype, ffn, hidden),
        Gemv(f"{prefix}.ffn_up.weight", qtype, ffn, hidden),
        Gemv(f"{prefix}.ffn_down.weight", qtype, hidden, ffn),
    ]


# single Q8_0 GEMV 2048 x 2048, M = 1
CFG1 = [Gemv("cfg1.q8_0.weight", TYPE_Q8_0, 2048, 2048)]

# one SmolLM3-shaped layer (hidden 2048, 16 q heads, 4 kv heads, head_dim 128,
# ffn 11008), all Q4_K, M = 1
CFG2 = _layer("smollm3.blk.0", 2048, 16, 4, 128, 11008, TYPE_Q4_K)


def llama8b_pass(n_layers: int = 32):
    """Batch-1 decode weight pass over a Llama-8B-shaped stack: 32 layers of Q4_K
    projections (hidden 4096, 32 q / 8 kv heads of 128, ffn 14336) and a Q8_0
    4096 -> 128256 output head."""
    out = []
    for L in range(n_layers):
        out += _layer(f"blk.{L}", 4096, 32, 8, 128, 14336, TYPE_Q4_K)
    out.append(Gemv("output.weight", TYPE_Q8_0, 128256, 4096))
    return out


def llama8b_stages(n_layers: int = 32):
    """The pass grouped into dependency stages: GEMVs within a stage share their
    input vector (q/k/v; gate/up) and can run in one launch."""
    gem = llama8b_pass(n_layers)
    stages = []
    for L in range(n_layers):
        g = gem[7 * L: 7 * L + 7]
        stages += [g[0:3], [g[3]], g[4:6], [g[6]]]
    stages.append([gem[-1]])
    return stages


CFG3 = llama8b_pass()

# small-batch Q8_0 GEMM on 14336 x 4096
CFG4 = Gemv("cfg4.q8_0.weight", TYPE_Q8_0, 14336, 4096)
CFG4_M = (1, 2, 4, 8, 16)

# prefill: Q4_K 14336 x 4096 times bf16 X [512, 4096]
CFG5 = Gemv("cfg5.q4_k.weight", TYPE_Q4_K, 14336, 4096)
CFG5_M = 512


# the cfg4 shape in the other weight types the GEMV takes, M = 1 (and 2..8 for Q4_0)
Q40_GEMV = Gemv("extra.q4_0.weight", TYPE_Q4_0, 14336, 4096)
F32_GEMV = Gemv("extra.f32.weight", TYPE_F32, 14336, 4096)
# a Q4_0 width that is not a multiple of 256 (the warp-per-row kernel)
Q40_ODD_GEMV = Gemv("extra.q4_0_odd.weight", TYPE_Q4_0, 14336, 4128)
# Q6_K in the shapes a Q4_K_M file gives it (ffn_down 4096 x 14336) and the cfg4 shape
Q6K_GEMV = Gemv("extra.q6_k.weight", TYPE_Q6_K, 14336, 4096)
Q6K_DOWN_GEMV = Gemv("extra.q6_k_down.weight", TYPE_Q6_K, 4096, 14336)


def q6k_layer(L: int) -> bool:
    """Layers whose attn_v and ffn_down are Q6_K in the Q4_K_M-style mixture:
    every other layer (the pages name only some of those tensors as Q6_K)."""
    return L % 2 == 1


def llama8b_q4km_tensors(n_layers: int = 32, vocab: int = 128256):
    """Every tensor of a Llama-8B-shaped file in a Q4_K_M-style mixture, in file
    order: token_embd (Q4_K), per layer attn_norm (F32), q, k, v, o, ffn_norm
    (F32), gate, up, down, then output_norm (F32) and the output head.  attn_v
    and ffn_down are Q6_K in the layers q6k_layer picks, the head is Q6_K (as in
    real Q4_K_M files), every other matrix Q4_K: 4.9 GB for 32 layers, the size
    the pages give for an 8B model in Q4_K_M.  Norms are rows = 1."""
    out = [Gemv("token_embd.weight", TYPE_Q4_K, vocab, 4096)]
    for L in range(n_layers):
        p = f"blk.{L}"
        six = TYPE_Q6_K if q6k_layer(L) else TYPE_Q4_K
        out += [Gemv(f"{p}.attn_norm.weight", TYPE_F32, 1, 4096),
                Gemv(f"{p}.attn_q.weight", TYPE_Q4_K, 4096, 4096),
                Gemv(f"{p}.attn_k.weight", TYPE_Q4_K, 1024, 4096),
                Gemv(f"{p}.attn_v.weight", six, 1024, 4096),
                Gemv(f"{p}.attn_output.weight", TYPE_Q4_K, 4096, 4096),
                Gemv(f"{p}.ffn_norm.weight", TYPE_F32, 1, 4096),
                Gemv(f"{p}.ffn_gate.weight", TYPE_Q4_K, 14336, 4096),
                Gemv(f"{p}.ffn_up.weight", TYPE_Q4_K, 14336, 4096),
                Gemv(f"{p}.ffn_down.weight", six, 4096, 14336)]
    out += [Gemv("output_norm.weight", TYPE_F32, 1, 4096), Gemv("output.weight", TYPE_Q6_K, vocab, 4096)]
    return out


def write_q4km_file(path: str, n_layers: int = 32, vocab: int = 128256):
    """Write llama8b_q4km_tensors as a GGUF v3 file (seeded payloads); returns
    the tensor list."""
    from . import weight_rows, write_gguf
    ts = llama8b_q4km_tensors(n_layers, vocab)
    kvs = [("general.architecture", 8, "llama"), ("general.name", 8, "synthetic-llama8b-q4_k_m-shape"),
           ("llama.block_count", 4, n_layers), ("llama.embedding_length", 4, 4096),
           ("llama.feed_forward_length", 4, 14336), ("llama.attention.head_count", 4, 32),
           ("llama.attention.head_count_kv", 4, 8)]
    tensors = [(g.name, [g.cols] if g.rows == 1 else [g.cols, g.rows], g.qtype) for g in ts]
    write_gguf(path, kvs, tensors, (weight_rows(g.qtype, g.stream, g.rows, g.cols) for g in ts))
    return ts


def weight_bytes(gemvs) -> int:
    from . import row_bytes
    return sum(g.rows * row_bytes(g.qtype, g.cols) for g in gemvs)

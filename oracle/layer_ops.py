"""Oracle for the element-wise steps that sit between the GEMVs of a decode
pass and that the chain fuses into its GEMV stages.

TEST INFRASTRUCTURE (see the package docstring): plain numpy, every value in
float64, one step per function in the order the pages give it.

* rmsnorm -- "GGUF Inferencer in R", section 4 ("Normalize Input", before the
  q/k/v projections and again before gate/up): the input vector is divided by
  the square root of the mean of its squares plus the model's epsilon, then
  multiplied element-wise by the layer's norm weights.  The C++ engine post
  (culpeo.ws, its list of kernels) names the same operation
  rmsnorm(x, w, eps).
* silu_mul -- "GGUF Inferencer in R", section 4 ("Activate Weights"): SiLU of
  the gate projection, SiLU(v) = v / (1 + e^-v), times the up projection,
  element by element; the engine post's silu_mul(gate, up).
* add -- "GGUF Inferencer in R", section 4 ("Add to Input", after the output
  projection and after the down projection); the engine post's add(a, b) and
  its residual stream, x_{i+1} = x_i + f(x_i).

Rows of a [M, n] array are independent activation vectors (one per token).
Parity status: pinned by closed forms and invariants in
tests/test_oracle_layer_ops.py (no page prints a numeric example of these steps).
"""
from __future__ import annotations

import numpy as np


def rmsnorm(x, w, eps):
    """x [M, n] (or [n]), w [n], eps >= 0 -> w * x / sqrt(mean(x^2) + eps), per row."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    x2 = np.atleast_2d(x)
    ms = np.mean(x2 * x2, axis=1, keepdims=True)   # mean of the squares of the row
    out = w[None, :] * x2 / np.sqrt(ms + float(eps))
    return out.reshape(x.shape)


def silu(v):
    """v / (1 + e^-v), element-wise."""
    v = np.asarray(v, dtype=np.float64)
    with np.errstate(over="ignore"):
        return v / (1.0 + np.exp(-v))


def silu_mul(gate, up):
    """SiLU(gate) * up, element-wise (gate and up of the same shape)."""
    return silu(gate) * np.asarray(up, dtype=np.float64)


def add(a, b):
    """a + b, element-wise."""
    return np.asarray(a, dtype=np.float64) + np.asarray(b, dtype=np.float64)

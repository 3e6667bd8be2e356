"""ggq -- GB300-native block-quantized (Q8_0 / Q4_K / Q4_0 / Q6_K, and F32) dequantize + GEMV.

The compute path is ``libggq.so`` (C ABI in ``include/ggq.h``), built in-tree for
sm_103a by ``build.build()``.  This package is its thin Python binding.
"""
from . import build, plan  # noqa: F401
from ._ggq import (F16, F32, Q4_0, Q4_K, Q6_K, Q8_0, X_PLAIN, X_RMSNORM, X_SILU_MUL, Chain, ChainOps, GGQError, Model, check, dequantize,  # noqa: F401
                   device_status, gemm_prefill, gemv, gemv_multi, ggq_chain_create, ggq_chain_create_typed, ggq_chain_free,
                   ggq_chain_reset, ggq_chain_run, ggq_dequantize, ggq_embed, embed, ggq_device_status, ggq_gemm_prefill, ggq_gemv, ggq_gemv_multi,
                   ggq_gemv_noalloc, lib, LIB_PATH, strerror)

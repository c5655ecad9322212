"""Oracle package: TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct CPU implementation of the batch-1 Qwen-style
decoder step and its causal prefill (numpy; float32 tensors, float64 inside each
operation). Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference legs of ``bench.py`` may import it. The CUDA product path never does.

Parity status per function (pins live in ``tests/test_oracle_pins.py``):
every function here is pinned; nothing is "parity unpinned" except agreement
with a real Hugging Face checkpoint, which needs weights this project does not have.
"""
from .qwen_ref import (  # noqa: F401
    Config, OracleModel, apply_rope, build_oracle, causal_gqa_attention, greedy_argmax,
    int4_dequantize, int4_quantize, kv_cache_bytes, linear, rmsnorm, rope_cos_sin, silu_mul,
    widen_bf16,
)

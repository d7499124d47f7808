"""CPU oracle for the Qwen3 decoder stack -- test infrastructure only.

Imported by the tests, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline
leg; never by the library.  See ``qwen3_oracle.py``.
"""
from .qwen3_oracle import (Qwen3Oracle, Qwen3OracleF32Acc, rnd, rms_norm, rope, rope_table, softmax,  # noqa: F401
                           attention_probs, silu, dequant_affine, router_topk, moe_layer,
                           embed_rows, head_logits, l2_pool_last)

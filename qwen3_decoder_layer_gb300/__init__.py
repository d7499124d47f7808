"""GB300-native Qwen3 decoder-stack forward (dense and MoE) over a static
per-sequence KV cache.

The compute lives in ``libqwen3_gb300.so`` (hand-written sm_103a CUDA kernels
behind the C ABI declared in ``include/qwen3.h``).  ``binding`` wraps that ABI
with the same function names; nothing here computes any part of the forward
pass in Python.
"""

__all__ = ["binding", "inputs"]


def __getattr__(name):
    if name in ("binding", "inputs", "build"):
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)

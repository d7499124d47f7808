"""Host-side checks of the C-ABI library that need no GPU: it builds for
sm_103a, loads, exports every symbol include/qwen3.h declares, and validates
configurations on the host."""
import os
import re

import pytest
import torch

from qwen3_decoder_layer_gb300 import build as B
from qwen3_decoder_layer_gb300 import binding as Q
from qwen3_decoder_layer_gb300 import inputs as I

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return Q.lib()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "qwen3.h")).read()
    return sorted(set(re.findall(r"QWEN3_API[^;(]*?\b(qwen3_\w+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    assert Q.qwen3_status_string(0) == "ok"
    assert "capacity" in Q.qwen3_status_string(3)


@pytest.mark.parametrize("name", list(I.CONFIGS))
def test_workload_configs_are_valid(lib, name):
    assert Q.qwen3_check_config(I.CONFIGS[name]) == Q.QWEN3_OK


@pytest.mark.parametrize("change,status", [
    (dict(dtype="fp16"), 2),                       # dtype gate: only fp32 or bf16
    (dict(head_dim=96), 8),
    (dict(n_heads=5), 1),                          # kv heads must divide q heads
    (dict(n_heads=64, n_kv_heads=2), 8),          # G > 16 not built
    (dict(hidden=100), 1),
    (dict(capacity=0), 1),
    (dict(max_seqs=0), 1),
    (dict(weight_format="int8", dtype="fp32"), 8),
    (dict(num_experts=8, top_k=9, moe_intermediate=64), 1),
    (dict(num_experts=512, top_k=8, moe_intermediate=64), 1),
])
def test_bad_configs_are_rejected(lib, change, status):
    cfg = I.with_sizes(I.TINY_FP32, **change)
    assert Q.qwen3_check_config(cfg) == status


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_create_without_a_device_fails_cleanly(lib):
    cfg = I.TINY_FP32
    w = I.make_weights(cfg, seed=1)   # CPU tensors: pointers are never dereferenced
    with pytest.raises(Q.Qwen3Error) as e:
        Q.qwen3_create(cfg, w)
    assert e.value.status == 9

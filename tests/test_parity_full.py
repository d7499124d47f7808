"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark uses (CUDA graphs + programmatic dependent launch for decode).

The oracle checks every output row it can afford: all rows of the dense and
MoE workloads, and two of the 32 sequences (shortest and longest context) of
the batched int8 decode -- each sequence's rows depend only on its own cache.
Bounds: gpu_helpers (fp32 1e-4; bf16 max(2e-2, 1.5 x the oracle-twin drift)).
fp32 runs of the same shapes are the strict gate (the Backbone's own strict
gates run in fp32)."""
import gc

import numpy as np
import pytest
import torch

from gpu_helpers import TOL, Parity, rel_err
from test_parity_small import moe_layer_check
from qwen3_decoder_layer_gb300 import binding as Q
from qwen3_decoder_layer_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _free():
    yield
    gc.collect()
    torch.cuda.empty_cache()


def _gpu_weights(cfg, seed):
    wd = I.make_weights(cfg, seed=seed, device="cuda")
    from gpu_helpers import to_device
    return wd, to_device(wd, "cpu")


@pytest.mark.parametrize("dtype,steps,fused", [("bf16", 4, 0), ("fp32", 2, 0), ("bf16", 2, 1)])
def test_dense_1p7b_decode(cuda_ok, dtype, steps, fused):
    """28 layers, cache prefilled to 4096 positions with N(0,1) K/V, decode steps
    (fused = 1: the whole step as one persistent cooperative kernel)."""
    cfg = I.with_sizes(I.DENSE_1P7B_DECODE, dtype=dtype)
    wd, w = _gpu_weights(cfg, I.SEEDS["dense_1p7b_decode"])
    p = Parity(cfg, weights=w, device_weights=wd)
    Q.qwen3_set_option(p.stack.h, Q.QWEN3_OPT_FUSED_DECODE, fused)
    p.fill_cache(0, 4096, seed=3000)
    for s in range(steps):
        p.step(I.make_rows(cfg, 1, seed=3001 + s, device="cuda"))
    p.close()
    p.check()


def test_dense_1p7b_prefill_bf16_and_chunked(cuda_ok):
    """T=2048 from an empty cache (causal), and 4 x 512 chunks equal to it."""
    cfg = I.DENSE_1P7B_PREFILL
    wd, w = _gpu_weights(cfg, I.SEEDS[cfg.name])
    p = Parity(cfg, weights=w, device_weights=wd)
    x = I.make_rows(cfg, 2048, seed=3100, device="cuda")
    one, _ = p.step(x)
    p.check()
    s2 = Q.Qwen3Stack(cfg, wd)
    chunks = torch.cat([s2.forward(x[i:i + 512]) for i in range(0, 2048, 512)])
    assert rel_err(chunks, one) <= TOL["bf16"]
    s2.close()
    p.close()


def test_dense_prefill_fp32_strict(cuda_ok):
    """The prefill shapes in fp32 (4 of the 28 layers): strict 1e-4."""
    cfg = I.with_sizes(I.DENSE_1P7B_PREFILL, dtype="fp32", num_layers=4)
    wd, w = _gpu_weights(cfg, 3200)
    p = Parity(cfg, weights=w, device_weights=wd)
    p.step(I.make_rows(cfg, 2048, seed=3201, device="cuda"))
    p.close()
    p.check()


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_moe_decode_at_context_2048(cuda_ok, dtype):
    cfg = I.with_sizes(I.MOE_A3B_4LAYER, dtype=dtype)
    wd, w = _gpu_weights(cfg, I.SEEDS["moe_a3b_4layer"])
    p = Parity(cfg, weights=w, device_weights=wd)
    p.fill_cache(0, 2048, seed=3300)
    for s in range(3):
        p.step(I.make_rows(cfg, 1, seed=3301 + s, device="cuda"))
    p.close()
    p.check()


def test_moe_prefill_1024(cuda_ok):
    cfg = I.MOE_A3B_4LAYER
    wd, w = _gpu_weights(cfg, I.SEEDS[cfg.name])
    p = Parity(cfg, weights=w, device_weights=wd)
    p.step(I.make_rows(cfg, 1024, seed=3400, device="cuda"))
    p.close()
    p.check()


@pytest.mark.parametrize("T", [1, 4, 1024])
def test_moe_layer_full_size_indices(cuda_ok, T):
    """qwen3_moe_layer at the MoE workload's sizes (128 experts, top-8): indices
    bit-exact by the margin protocol, output within the bf16 bound."""
    cfg = I.MOE_A3B_4LAYER
    wd, w = _gpu_weights(cfg, I.SEEDS[cfg.name])
    p = Parity(cfg, weights=w, device_weights=wd, twin=False)
    for layer in (0, 3):
        err, clear = moe_layer_check(cfg, p.stack, p.orc, layer,
                                     I.make_rows(cfg, T, seed=3500 + layer, device="cuda"))
        assert err <= TOL["bf16"]
        assert clear >= (0.99 if T > 100 else 1.0)
    p.close()


def test_int8_batched_decode_32_sequences(cuda_ok):
    """32 sequences with contexts uniform in [1024, 16384], int8 weights; the
    oracle follows the shortest and the longest sequence."""
    cfg = I.DENSE_1P7B_INT8_B32
    wd, w = _gpu_weights(cfg, I.SEEDS[cfg.name])
    ctx = I.batch_context_lengths(32, 1024, 16384, seed=3600)
    sampled = [int(np.argmin(ctx)), int(np.argmax(ctx))]
    p = Parity(cfg, weights=w, device_weights=wd)
    for s, n in enumerate(ctx):
        p.fill_cache(s, n, seed=3601 + s, to_oracle=s in sampled)
    for step in range(2):
        x = I.make_rows(cfg, 32, seed=3700 + step, device="cuda")
        p.step(x, seq_ids=list(range(32)), oracle_rows=sampled)
    p.close()
    p.check()

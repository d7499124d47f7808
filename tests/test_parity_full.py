"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark uses (CUDA graphs + programmatic dependent launch for decode).

Each bf16 workload is checked twice on the same oracle run:

* layer by layer (the primary bf16 claim): layers 0, 13 and 27 of the
  28-layer stacks and every layer of the 4-layer MoE stack, each run alone as a
  one-layer stack on the oracle's own input rows and cache, at 2e-2
  (gpu_helpers.LayerGate);
* end to end: the 28-layer output against the oracle within 2e-2 or twice the
  oracle-twin drift (gpu_helpers.Parity.bound).

The oracle follows every row of the dense and MoE workloads and 8 of the 32
sequences of the batched int8 decode (the shortest, the longest and six drawn
at random) -- each sequence's rows depend only on its own cache.  fp32 runs of
the same shapes are the strict gate (1e-4)."""
import gc

import numpy as np
import pytest
import torch

from gpu_helpers import TOL, Parity, rel_err, report, to_device
from test_parity_small import moe_layer_check
from qwen3_decoder_layer_gb300 import binding as Q
from qwen3_decoder_layer_gb300 import inputs as I

pytestmark = pytest.mark.gpu

GATED_28 = (0, 13, 27)


@pytest.fixture(autouse=True)
def _free():
    yield
    gc.collect()
    torch.cuda.empty_cache()


def _gpu_weights(cfg, seed):
    wd = I.make_weights(cfg, seed=seed, device="cuda")
    return wd, to_device(wd, "cpu")


@pytest.mark.parametrize("dtype,steps", [("bf16", 16), ("fp32", 2)])
def test_dense_1p7b_decode(cuda_ok, dtype, steps):
    """28 layers, cache prefilled to 4096 positions with N(0,1) K/V, decode steps
    at contexts 4096..; bf16: layers 0, 13, 27 gated one by one at every step."""
    cfg = I.with_sizes(I.DENSE_1P7B_DECODE, dtype=dtype)
    wd, w = _gpu_weights(cfg, I.SEEDS["dense_1p7b_decode"])
    p = Parity(cfg, weights=w, device_weights=wd)
    if dtype == "bf16":
        p.add_layer_gate(GATED_28)
    p.fill_cache(0, 4096, seed=3000)
    for s in range(steps):
        p.step(I.make_rows(cfg, 1, seed=3001 + s, device="cuda"))
    p.close()
    p.check()


def test_dense_1p7b_prefill_bf16_and_chunked(cuda_ok):
    """T=2048 from an empty cache (causal) with layers 0, 13, 27 gated; then the
    same rows as 4 x 512 chunks, against the oracle and against the one pass."""
    cfg = I.DENSE_1P7B_PREFILL
    wd, w = _gpu_weights(cfg, I.SEEDS[cfg.name])
    p = Parity(cfg, weights=w, device_weights=wd)
    p.add_layer_gate(GATED_28)
    x = I.make_rows(cfg, 2048, seed=3100, device="cuda")
    one, ref = p.step(x)
    p.close()
    p.check()
    s2 = Q.Qwen3Stack(cfg, wd)
    chunks = torch.cat([s2.forward(x[i:i + 512]) for i in range(0, 2048, 512)])
    s2.close()
    e_orc, e_one = rel_err(chunks, ref), rel_err(chunks, one)
    report("4 x 512 chunks vs oracle", e_orc, p.bound())
    report("4 x 512 chunks vs one pass", e_one, TOL["bf16"])
    assert e_orc <= p.bound()
    assert e_one <= TOL["bf16"]


def test_dense_prefill_fp32_strict(cuda_ok):
    """The prefill shapes in fp32 (4 of the 28 layers): strict 1e-4."""
    cfg = I.with_sizes(I.DENSE_1P7B_PREFILL, dtype="fp32", num_layers=4)
    wd, w = _gpu_weights(cfg, 3200)
    p = Parity(cfg, weights=w, device_weights=wd)
    p.step(I.make_rows(cfg, 2048, seed=3201, device="cuda"))
    p.close()
    p.check()


@pytest.mark.parametrize("dtype,steps", [("bf16", 16), ("fp32", 3)])
def test_moe_decode_at_context_2048(cuda_ok, dtype, steps):
    cfg = I.with_sizes(I.MOE_A3B_4LAYER, dtype=dtype)
    wd, w = _gpu_weights(cfg, I.SEEDS["moe_a3b_4layer"])
    p = Parity(cfg, weights=w, device_weights=wd)
    if dtype == "bf16":
        p.add_layer_gate(range(cfg.num_layers))
    p.fill_cache(0, 2048, seed=3300)
    for s in range(steps):
        p.step(I.make_rows(cfg, 1, seed=3301 + s, device="cuda"))
    p.close()
    p.check()


def test_moe_prefill_1024(cuda_ok):
    cfg = I.MOE_A3B_4LAYER
    wd, w = _gpu_weights(cfg, I.SEEDS[cfg.name])
    p = Parity(cfg, weights=w, device_weights=wd)
    p.add_layer_gate(range(cfg.num_layers))
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
        report(f"moe block layer {layer}, {T} rows", err, TOL["bf16"], f"{clear:.3f} of rows clear of a near-tie")
        assert err <= TOL["bf16"]
        assert clear >= (0.99 if T > 100 else 1.0)
    p.close()


def test_int8_batched_decode_32_sequences(cuda_ok):
    """32 sequences with contexts uniform in [1024, 16384], int8 weights, all 32
    rows per step; the oracle follows 8 sequences (shortest, longest, six at
    random), the twin the shortest and the longest; layers 0, 13, 27 gated."""
    cfg = I.DENSE_1P7B_INT8_B32
    wd, w = _gpu_weights(cfg, I.SEEDS[cfg.name])
    ctx = I.batch_context_lengths(32, 1024, 16384, seed=3600)
    ends = [int(np.argmin(ctx)), int(np.argmax(ctx))]
    others = [s for s in range(32) if s not in ends]
    sampled = sorted(ends + [int(s) for s in np.random.default_rng(3650).choice(others, 6, replace=False)])
    p = Parity(cfg, weights=w, device_weights=wd)
    p.add_layer_gate(GATED_28)
    for s, n in enumerate(ctx):
        p.fill_cache(s, n, seed=3601 + s, to_oracle=s in sampled, to_twin=s in ends)
    for step in range(2):
        x = I.make_rows(cfg, 32, seed=3700 + step, device="cuda")
        p.step(x, seq_ids=list(range(32)), oracle_rows=sampled, twin_rows=sorted(ends))
    p.close()
    p.check()

"""Seeded synthetic inputs for the Qwen3 decoder stack.

This module only draws random numbers and lays them out; it holds none of the
forward pass's arithmetic.  Both the CUDA library's callers (tests, bench.py,
smoke) and the CPU oracle take their inputs from here, so the two sides see
the same values.

Draws use ``torch.Generator`` seeded per call, on the device asked for (CPU for
small cases, CUDA for full-size ones so that generating a 60 GB cache takes
seconds).  Values are drawn in fp32 and cast to the model dtype (bf16 or fp32)
with torch's own round-to-nearest-even conversion; the oracle reads the cast
values back exactly.

Workloads (sizes from the Qwen3 pages: the MLX ``Backbone`` of
maya2_mlx/backbone.py for the dense stack, and @mlx-bun/inference qwen3-moe.ts
for the MoE block):

* ``tiny_fp32``        2 layers, hidden 256, 4 q / 2 kv heads, head_dim 64,
                       intermediate 768, fp32, capacity 64.
* ``dense_1p7b_decode`` 28 layers, hidden 2048, 16 q / 8 kv heads, head_dim 128,
                       intermediate 6144, bf16, capacity 8192 (batch-1 decode
                       at context 4096..4351).
* ``dense_1p7b_prefill`` the same stack, capacity 2048 (one 2048-token prefill).
* ``moe_a3b_4layer``   4 Qwen3-MoE layers: hidden 2048, 32 q / 4 kv heads,
                       128 experts, top-8, moe_intermediate 768, theta 1e7.
* ``dense_1p7b_int8_b32`` the 1.7B-shaped stack with int8 affine group-64
                       weights, 32 sequences, capacity 16512.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

DTYPES = {"fp32": torch.float32, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Qwen3Config:
    num_layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    capacity: int = 64
    max_seqs: int = 1
    dtype: str = "bf16"             # "fp32" (strict) or "bf16" (production)
    weight_format: str = "dense"    # "dense" or "int8" (affine, per-group scale/bias)
    group_size: int = 64
    num_experts: int = 0            # 0 = dense stack
    top_k: int = 0
    moe_intermediate: int = 0
    norm_topk_prob: bool = True
    decoder_sparse_step: int = 1
    mlp_only_layers: tuple = ()     # layers of a MoE stack that keep the dense MLP
    name: str = field(default="custom", compare=False)

    @property
    def qkv_rows(self) -> int:
        return (self.n_heads + 2 * self.n_kv_heads) * self.head_dim

    def has_experts(self, layer: int) -> bool:
        """Whether the generator draws expert weights (rather than a dense MLP)
        for this layer: the layer schedule the config describes (experts exist,
        the layer is not in mlp_only_layers, (layer + 1) % decoder_sparse_step
        == 0).  Only the weight layout depends on it; the oracle and the
        library each decide a layer's kind with their own code."""
        return (self.num_experts > 0 and layer not in tuple(self.mlp_only_layers)
                and (layer + 1) % self.decoder_sparse_step == 0)

    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]


TINY_FP32 = Qwen3Config(
    name="tiny_fp32", num_layers=2, hidden=256, n_heads=4, n_kv_heads=2, head_dim=64,
    intermediate=768, rms_eps=1e-6, rope_theta=1e6, capacity=64, dtype="fp32")
DENSE_1P7B_DECODE = Qwen3Config(
    name="dense_1p7b_decode", num_layers=28, hidden=2048, n_heads=16, n_kv_heads=8,
    head_dim=128, intermediate=6144, rms_eps=1e-6, rope_theta=1e6, capacity=8192,
    dtype="bf16")
DENSE_1P7B_PREFILL = replace(DENSE_1P7B_DECODE, name="dense_1p7b_prefill", capacity=2048)
MOE_A3B_4LAYER = Qwen3Config(
    name="moe_a3b_4layer", num_layers=4, hidden=2048, n_heads=32, n_kv_heads=4,
    head_dim=128, intermediate=6144, rms_eps=1e-6, rope_theta=1e7, capacity=2112,
    dtype="bf16", num_experts=128, top_k=8, moe_intermediate=768, norm_topk_prob=True,
    decoder_sparse_step=1)
DENSE_1P7B_INT8_B32 = replace(
    DENSE_1P7B_DECODE, name="dense_1p7b_int8_b32", capacity=16512, max_seqs=32,
    weight_format="int8", group_size=64)

CONFIGS = {c.name: c for c in
           (TINY_FP32, DENSE_1P7B_DECODE, DENSE_1P7B_PREFILL, MOE_A3B_4LAYER, DENSE_1P7B_INT8_B32)}

# One seed per workload, in the order the workloads are listed above.
SEEDS = {name: 20261202 + i for i, name in enumerate(CONFIGS)}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def _normal(shape, std, g, device, dt, mean=0.0):
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(dt)


def _int8_linear(out_f, in_f, group, g, device):
    """Affine int8 group quantised linear: codes uniform in 0..255, one bf16
    scale and bias per group of ``group`` consecutive inputs of each row.
    scale = bf16(0.02*sqrt(12)/256 * (1 + U(-0.1, 0.1))) and bias = bf16(-128*scale)
    give weights of mean ~0 and standard deviation ~0.02."""
    codes = torch.randint(0, 256, (out_f, in_f), generator=g, device=device,
                          dtype=torch.int32).to(torch.uint8)
    u = torch.rand((out_f, in_f // group), generator=g, device=device, dtype=torch.float32)
    scale = (0.02 * math.sqrt(12.0) / 256.0) * (1.0 + (u * 0.2 - 0.1))
    scale = scale.to(torch.bfloat16)
    bias = (scale.float() * -128.0).to(torch.bfloat16)
    return {"w": codes, "scale": scale, "bias": bias}


def _stack(parts):
    """Stack per-expert int8 linears into [E, ...] codes, scales and biases."""
    return {k: torch.stack([p[k] for p in parts]) for k in parts[0]}


def make_weights(cfg: Qwen3Config, seed: int | None = None, device="cpu") -> dict:
    """Random-init weights with the stack's architecture.

    Draw order (fixed): for each layer, in_norm, post_norm, q_norm, k_norm,
    qkv, o, gate_up, down (dense layers) or router, expert gate|up, expert down
    (MoE layers; int8 experts: every expert's gate|up codes, scales and biases,
    then every expert's down); then the final norm.  Linear weights are
    nn.Linear ``[out, in]`` row-major; q|k|v rows and gate|up rows are concatenated
    (the fused projections of the MLX Backbone).  Gains are 1 + N(0, 0.1),
    weights N(0, 0.02).
    """
    seed = SEEDS.get(cfg.name, 1234) if seed is None else seed
    g = _gen(seed, device)
    dt = cfg.torch_dtype()
    H, D = cfg.hidden, cfg.head_dim

    def lin(out_f, in_f):
        if cfg.weight_format == "int8":
            return _int8_linear(out_f, in_f, cfg.group_size, g, device)
        return {"w": _normal((out_f, in_f), 0.02, g, device, dt)}

    layers = []
    for i in range(cfg.num_layers):
        L = {
            "in_norm": _normal((H,), 0.1, g, device, dt, mean=1.0),
            "post_norm": _normal((H,), 0.1, g, device, dt, mean=1.0),
            "q_norm": _normal((D,), 0.1, g, device, dt, mean=1.0),
            "k_norm": _normal((D,), 0.1, g, device, dt, mean=1.0),
            "qkv": lin(cfg.qkv_rows, H),
            "o": lin(H, cfg.n_heads * D),
        }
        if cfg.has_experts(i):
            E, mI = cfg.num_experts, cfg.moe_intermediate
            L["router"] = {"w": _normal((E, H), 0.02, g, device, dt)}
            if cfg.weight_format == "int8":
                L["exp_gate_up"] = _stack([_int8_linear(2 * mI, H, cfg.group_size, g, device) for _ in range(E)])
                L["exp_down"] = _stack([_int8_linear(H, mI, cfg.group_size, g, device) for _ in range(E)])
            else:
                L["exp_gate_up"] = {"w": _normal((E, 2 * mI, H), 0.02, g, device, dt)}
                L["exp_down"] = {"w": _normal((E, H, mI), 0.02, g, device, dt)}
        else:
            L["gate_up"] = lin(2 * cfg.intermediate, H)
            L["down"] = lin(H, cfg.intermediate)
        layers.append(L)
    final_norm = _normal((H,), 0.1, g, device, dt, mean=1.0)
    return {"layers": layers, "final_norm": final_norm}


def make_rows(cfg: Qwen3Config, n_rows: int, seed: int, device="cpu") -> torch.Tensor:
    """Input hidden rows x [n_rows, hidden], N(0, 1), in the model dtype."""
    return _normal((n_rows, cfg.hidden), 1.0, _gen(seed, device), device, cfg.torch_dtype())


def make_cache_prefill(cfg: Qwen3Config, length: int, seed: int, device="cpu"):
    """Synthetic cache contents for one sequence: post-RoPE K and raw V for
    positions 0..length-1 of every layer, N(0, 1) in the model dtype.
    Returns (K, V), each [layers, kv_heads, length, head_dim]."""
    g = _gen(seed, device)
    shape = (cfg.num_layers, cfg.n_kv_heads, length, cfg.head_dim)
    k = _normal(shape, 1.0, g, device, cfg.torch_dtype())
    v = _normal(shape, 1.0, g, device, cfg.torch_dtype())
    return k, v


def batch_context_lengths(n_seqs: int, lo: int, hi: int, seed: int) -> list[int]:
    """Per-sequence context lengths, integers uniform in [lo, hi]."""
    g = _gen(seed, "cpu")
    return [int(v) for v in torch.randint(lo, hi + 1, (n_seqs,), generator=g)]


def with_sizes(cfg: Qwen3Config, **kw) -> Qwen3Config:
    """A copy of a workload with some sizes changed (for small parity cases)."""
    return replace(cfg, **kw)

"""Helpers shared by the GPU parity tests: move seeded inputs to the device,
run the library and the oracle on the same values, and measure the error
metric max|gpu - oracle| / rms(oracle)."""
import numpy as np
import torch

from oracle import Qwen3Oracle
from qwen3_decoder_layer_gb300 import binding as Q
from qwen3_decoder_layer_gb300 import inputs as I

# Tolerances on max|gpu - oracle| / rms(oracle) over the final-norm output.
TOL = {"fp32": 1e-4, "bf16": 2e-2}


def rel_err(gpu, ref) -> float:
    g = gpu.detach().float().cpu().double().numpy() if hasattr(gpu, "detach") else np.asarray(gpu, float)
    r = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(g - r)) / np.sqrt(np.mean(r * r)))


def to_device(obj, device="cuda"):
    if isinstance(obj, dict):
        return {k: to_device(v, device) for k, v in obj.items()}
    if isinstance(obj, list):
        return [to_device(v, device) for v in obj]
    return obj.to(device)


def make_pair(cfg, seed=None, device_weights=None):
    """(library stack, oracle) on the same seeded weights."""
    w = I.make_weights(cfg, seed=seed, device="cpu") if device_weights is None else device_weights
    wd = to_device(w) if device_weights is None else w
    stack = Q.Qwen3Stack(cfg, wd)
    orc = Qwen3Oracle(cfg, w if device_weights is None else to_device(w, "cpu"))
    return stack, orc


def fill_cache(stack, orc, seq, length, seed):
    """Write the same N(0,1) K/V into both caches at positions 0..length-1."""
    cfg = stack.cfg
    K, V = I.make_cache_prefill(cfg, length, seed=seed, device="cuda")
    for l in range(cfg.num_layers):
        kc, vc = Q.cache_tensors(stack.h, cfg, seq, l)
        kc[:, :length].copy_(K[l])
        vc[:, :length].copy_(V[l])
    torch.cuda.synchronize()
    Q.qwen3_set_length(stack.h, seq, length)
    if orc is not None:
        orc.set_cache(seq, K.cpu(), V.cpu())

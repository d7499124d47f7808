"""Helpers shared by the GPU parity tests: move seeded inputs to the device,
run the library and the oracle on the same values, and check the error metric
max|gpu - oracle| / rms(oracle) of the final-norm output.

Tolerances.  fp32: 1e-4.  bf16: 2e-2, or 2 x the drift between the oracle
and its float32 twin (oracle.Qwen3OracleF32Acc, the same rounding points with
float32 arithmetic between them) on the same inputs, whichever is larger.
The twin term matters only for wide or deep stacks: there any two correct
bf16 implementations disagree by more than 2e-2 (measured: 10-13% max-abs/RMS
after the 28 layers of the 1.7B-shaped stack, 1-2 bf16 ulps of the largest
output on a 3-layer 512-wide stack), so no GPU kernel can meet 2e-2 there; on
the smallest stacks the twin is bit-identical to the oracle and the bound is
2e-2."""
import numpy as np
import torch

from oracle import Qwen3Oracle, Qwen3OracleF32Acc
from qwen3_decoder_layer_gb300 import binding as Q
from qwen3_decoder_layer_gb300 import inputs as I

TOL = {"fp32": 1e-4, "bf16": 2e-2}
TWIN_FACTOR = 2.0


def as_f64(a):
    if hasattr(a, "detach"):
        return a.detach().float().cpu().double().numpy()
    return np.asarray(a, dtype=np.float64)


def rel_err(gpu, ref) -> float:
    g, r = as_f64(gpu), as_f64(ref)
    return float(np.max(np.abs(g - r)) / np.sqrt(np.mean(r * r)))


def to_device(obj, device="cuda"):
    if isinstance(obj, dict):
        return {k: to_device(v, device) for k, v in obj.items()}
    if isinstance(obj, list):
        return [to_device(v, device) for v in obj]
    return obj.to(device)


class Parity:
    """A GPU stack, the oracle and (bf16) the oracle's twin on the same weights.

    step() runs one forward on all of them and records the errors; check()
    asserts the bound described in the module docstring."""

    def __init__(self, cfg, weights=None, seed=None, twin=None, device_weights=None):
        self.cfg = cfg
        w = weights if weights is not None else I.make_weights(cfg, seed=seed, device="cpu")
        if device_weights is None:
            device_weights = to_device(w)
        self.stack = Q.Qwen3Stack(cfg, device_weights)
        self.orc = Qwen3Oracle(cfg, w)
        if twin is None:
            twin = cfg.dtype == "bf16"
        self.twin = Qwen3OracleF32Acc(cfg, w) if twin else None
        self.errs, self.floors = [], []

    def fill_cache(self, seq, length, seed, to_oracle=True):
        """The same N(0,1) K/V at positions 0..length-1 of `seq` on every side
        (on the GPU only when to_oracle is False)."""
        cfg = self.cfg
        K, V = I.make_cache_prefill(cfg, length, seed=seed, device="cuda")
        for l in range(cfg.num_layers):
            kc, vc = Q.cache_tensors(self.stack.h, cfg, seq, l)
            kc[:, :length].copy_(K[l])
            vc[:, :length].copy_(V[l])
        torch.cuda.synchronize()
        Q.qwen3_set_length(self.stack.h, seq, length)
        if not to_oracle:
            return
        Kc, Vc = K.cpu(), V.cpu()
        del K, V
        for o in (self.orc, self.twin):
            if o is not None:
                o.set_cache(seq, Kc, Vc)

    def step(self, x, seq_ids=None, oracle_rows=None):
        """Forward x on the GPU; on the CPU sides forward only `oracle_rows`
        (default all), which must hold every row of the sequences they touch."""
        out = self.stack.forward(x, seq_ids=seq_ids)
        T = x.shape[0]
        sids = list(seq_ids) if seq_ids is not None else [0] * T
        rows = list(range(T)) if oracle_rows is None else list(oracle_rows)
        xs = x[rows].cpu()
        ss = [sids[r] for r in rows]
        ref = self.orc.forward(xs, seq_ids=ss)
        got = as_f64(out[rows])
        self.errs.append(rel_err(got, ref))
        if self.twin is not None:
            self.floors.append(rel_err(self.twin.forward(xs, seq_ids=ss), ref))
        return out, ref

    def bound(self):
        base = TOL[self.cfg.dtype]
        if self.twin is None or not self.floors:
            return base
        return max(base, TWIN_FACTOR * max(self.floors))

    def check(self):
        assert self.errs, "no steps"
        b = self.bound()
        assert max(self.errs) <= b, f"errors {self.errs} above {b} (twin drift {self.floors})"
        return max(self.errs), b

    def close(self):
        self.stack.close()

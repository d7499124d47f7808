"""Helpers shared by the GPU parity tests: move seeded inputs to the device,
run the library and the oracle on the same values, and compare them.

Error metric: max|gpu - oracle| / rms(oracle) of a final-norm output.

Tolerances.

* fp32: 1e-4, at every size (the strict gate).
* bf16, one layer at a time ("layer gate", the primary bf16 claim): each
  layer of a workload, run alone through the C ABI as a one-layer stack whose
  input rows and cache are the oracle's, must match the oracle's same layer to
  2e-2.  The layer's output is read through an RMSNorm with a unit gain (one
  rounding, no gain to round twice).  Per element the bound is
  max(2e-2 * rms, 4 bf16 ulps of the element): the layer ends with two
  roundings (h and pend, each a rounding decision that a float32
  implementation can take the other way when the exact value sits near a tie,
  so their sum can move by two of its ulps), and the read-out divides by the
  row's RMS, a non-power-of-two scale, which can turn two ulps of the sum into
  up to four of the output; the count of elements that need more than 2e-2 is
  reported.  In MoE layers, rows whose expert choice is a near-tie are left
  out of the element comparison (near_tie_rows), counted, and capped at 30%
  (the block itself is held to bit-exact indices on identical inputs by the
  MoE block tests).
* bf16, whole stacks: 2e-2, or TWIN_FACTOR x the drift between the oracle and
  its float32 twin (oracle.Qwen3OracleF32Acc: the same rounding points, float32
  arithmetic between them) on the same inputs, whichever is larger, capped at
  E2E_CAP.  The twin term matters only for deep or wide stacks, where rounding
  decisions that go the other way cascade through the layers (measured: zero
  on the 2-layer 256-wide stack, 10-13% after the 28 layers of the 1.7B-shaped
  stack); TWIN_FACTOR = 2 because the GPU and the twin are two independent
  float32 implementations whose distances from the oracle are draws of the same
  cascade.

Every comparison is recorded in REPORT; conftest prints it at the end of the
session (measured error beside its bound)."""
import numpy as np
import torch

from oracle import Qwen3Oracle, Qwen3OracleF32Acc, moe_layer, rms_norm, rnd
from qwen3_decoder_layer_gb300 import binding as Q
from qwen3_decoder_layer_gb300 import inputs as I

TOL = {"fp32": 1e-4, "bf16": 2e-2}
TWIN_FACTOR = 2.0
E2E_CAP = 0.30
REPORT = []   # (test, what, measured, bound, note)


def report(what, measured, bound, note=""):
    import os
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0].split("::")[-1]
    REPORT.append((test, what, float(measured), float(bound), note))


def as_f64(a):
    if hasattr(a, "detach"):
        return a.detach().float().cpu().double().numpy()
    return np.asarray(a, dtype=np.float64)


def rel_err(gpu, ref) -> float:
    g, r = as_f64(gpu), as_f64(ref)
    return float(np.max(np.abs(g - r)) / np.sqrt(np.mean(r * r)))


def bf16_ulp(v, w=None):
    """Spacing of bf16 values at |v| (8 significant bits); with w, at the
    larger of |v| and |w| (two values on either side of a power of two)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    if w is not None:
        a = np.maximum(a, np.abs(np.asarray(w, dtype=np.float64)))
    a = np.maximum(a, 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def near_tie_rows(y2, router_w, k, rel=1e-2):
    """Rows whose router choice is not decided by the values: the gap between
    the k-th and (k+1)-th largest fp64 logit is below rel * rms(logits).  The
    GPU's router input differs from the oracle's wherever an upstream bf16
    rounding went the other way (up to a fifth of a prefill row's elements,
    one ulp each), which moves a logit by up to ~4e-3 of their rms, so such
    rows may pick another expert on either side."""
    logits = np.asarray(y2, dtype=np.float64) @ np.asarray(router_w, dtype=np.float64).T
    srt = -np.sort(-logits, axis=1)
    margin = srt[:, k - 1] - srt[:, k]
    return margin < rel * np.sqrt(np.mean(logits ** 2, axis=1))


def to_device(obj, device="cuda"):
    if isinstance(obj, dict):
        return {k: to_device(v, device) for k, v in obj.items()}
    if isinstance(obj, list):
        return [to_device(v, device) for v in obj]
    return obj.to(device)


class Parity:
    """A GPU stack, the oracle and (bf16) the oracle's twin on the same weights.

    step() runs one forward on all of them and records the errors; check()
    asserts the whole-stack bound described in the module docstring."""

    def __init__(self, cfg, weights=None, seed=None, twin=None, device_weights=None):
        self.cfg = cfg
        w = weights if weights is not None else I.make_weights(cfg, seed=seed, device="cpu")
        self.w = w
        if device_weights is None:
            device_weights = to_device(w)
        self.wd = device_weights
        self.stack = Q.Qwen3Stack(cfg, device_weights)
        self.orc = Qwen3Oracle(cfg, w)
        if twin is None:
            twin = cfg.dtype == "bf16"
        self.twin = Qwen3OracleF32Acc(cfg, w) if twin else None
        self.errs, self.floors = [], []
        self.gate = None

    def add_layer_gate(self, layers):
        """Hold `layers` to the per-layer bound at every later step."""
        self.gate = LayerGate(self.cfg, self.wd, layers)
        return self.gate

    def fill_cache(self, seq, length, seed, to_oracle=True, to_twin=True):
        """The same N(0,1) K/V at positions 0..length-1 of `seq` on every side
        (on the GPU only when to_oracle is False; not on the twin when to_twin
        is False)."""
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
        for o in (self.orc, self.twin if to_twin else None):
            if o is not None:
                o.set_cache(seq, Kc, Vc)

    def step(self, x, seq_ids=None, oracle_rows=None, twin_rows=None):
        """Forward x on the GPU; on the CPU sides forward only `oracle_rows`
        (default all), which must hold every row of the sequences they touch
        (the twin: `twin_rows`, a subset, default the same rows).  With a layer
        gate, its layers are checked on the same step."""
        out = self.stack.forward(x, seq_ids=seq_ids)
        T = x.shape[0]
        sids = list(seq_ids) if seq_ids is not None else [0] * T
        rows = list(range(T)) if oracle_rows is None else list(oracle_rows)
        xs = x[rows].cpu()
        ss = [sids[r] for r in rows]
        taps = None
        if self.gate is not None:
            self.gate.sync_cache(self.orc, sorted(set(ss)))
            taps = {l: None for l in self.gate.layers}
        ref = self.orc.forward(xs, seq_ids=ss, taps=taps)
        got = as_f64(out[rows])
        self.errs.append(rel_err(got, ref))
        if self.twin is not None:
            trows = rows if twin_rows is None else list(twin_rows)
            pick = [rows.index(r) for r in trows]
            self.floors.append(rel_err(self.twin.forward(x[trows].cpu(), seq_ids=[sids[r] for r in trows]),
                                       ref[pick]))
        if self.gate is not None:
            self.gate.check(taps, x, sids, rows, self.orc)
        return out, ref

    def bound(self):
        base = TOL[self.cfg.dtype]
        if self.twin is None or not self.floors:
            return base
        return min(E2E_CAP, max(base, TWIN_FACTOR * max(self.floors)))

    def check(self):
        assert self.errs, "no steps"
        b = self.bound()
        note = f"twin drift {max(self.floors):.4f}" if self.floors else ""
        report(f"{self.cfg.name} whole stack ({len(self.errs)} steps)", max(self.errs), b, note)
        assert max(self.errs) <= b, f"errors {self.errs} above {b} (twin drift {self.floors})"
        if self.gate is not None:
            self.gate.assert_ok()
        return max(self.errs), b

    def close(self):
        self.stack.close()
        if self.gate is not None:
            self.gate.close()


class LayerGate:
    """One-layer GPU stacks for chosen layers of a workload, fed the oracle's
    input rows of that layer and holding the oracle's cache of that layer; each
    is read out through an RMSNorm with a unit gain and compared with the
    oracle's same layer (module docstring)."""

    def __init__(self, cfg, wd, layers):
        self.cfg = cfg
        self.layers = list(layers)
        self.stacks, self.synced, self.results = {}, {}, []
        dt = cfg.torch_dtype()
        ones = torch.ones(cfg.hidden, dtype=dt, device="cuda")
        for l in self.layers:
            sparse = moe_layer(cfg, l)
            one = I.with_sizes(cfg, num_layers=1, decoder_sparse_step=1, mlp_only_layers=() if sparse else (0,),
                               name=f"{cfg.name}_layer{l}")
            if not sparse and cfg.num_experts == 0:
                one = I.with_sizes(one, mlp_only_layers=())
            self.stacks[l] = (one, Q.Qwen3Stack(one, {"layers": [wd["layers"][l]], "final_norm": ones}))

    def sync_cache(self, orc, seqs):
        """Copy the oracle's cache positions not yet on the GPU (the oracle's own
        K/V of every earlier step) into each one-layer stack."""
        for l, (one, st) in self.stacks.items():
            for s in seqs:
                c = orc._seq(s)
                n, n0 = c["length"], self.synced.get((l, s), 0)
                if n > n0:
                    kc, vc = Q.cache_tensors(st.h, one, s, 0)
                    kc[:, n0:n].copy_(torch.from_numpy(c["K"][l, :, n0:n]).to(kc.dtype))
                    vc[:, n0:n].copy_(torch.from_numpy(c["V"][l, :, n0:n]).to(vc.dtype))
                if n != Q.qwen3_get_length(st.h, s):
                    Q.qwen3_set_length(st.h, s, n)
                self.synced[(l, s)] = n
        torch.cuda.synchronize()

    def check(self, taps, x, sids, rows, orc):
        """Run each gated layer on its oracle input rows (rows outside `rows`
        keep the step's own input; their outputs are not compared).  In a MoE
        layer, rows whose expert choice is a near-tie under the oracle's router
        input (near_tie_rows) are left out of the element comparison: there
        either choice is right, and the index protocol of the MoE block tests
        covers them."""
        cfg = self.cfg
        dt = cfg.torch_dtype()
        for l, (one, st) in self.stacks.items():
            hin = x.clone()
            hin[rows] = torch.from_numpy(taps[l]["h_in"]).to(dt).to("cuda")
            out = st.forward(hin, seq_ids=sids)
            got = as_f64(out[rows])
            hh = rnd(taps[l]["h"] + taps[l]["pend"], cfg.dtype)
            ref = rms_norm(hh, np.ones(cfg.hidden), cfg.rms_eps, cfg.dtype)
            keep = np.ones(len(rows), dtype=bool)
            if moe_layer(cfg, l):
                keep = ~near_tie_rows(taps[l]["y2"], orc.layers[l]["router"]["w"], cfg.top_k)
            r = np.sqrt(np.mean(ref * ref))
            got, ref = got[keep], ref[keep]
            d = np.abs(got - ref)
            if cfg.dtype == "bf16":
                allow = np.maximum(TOL["bf16"] * r, 4 * bf16_ulp(ref, got))
                n_ulp = int(np.sum(d > TOL["bf16"] * r))
            else:
                allow = np.full_like(ref, TOL["fp32"] * r)
                n_ulp = 0
            worst = float(d.max() / r) if d.size else 0.0
            crit = float(np.max(d / allow)) if d.size else 0.0
            self.results.append((l, worst, crit, n_ulp, d.size, int(np.sum(~keep)), len(keep)))
        # the keys this step appended on the GPU are replaced by the oracle's at the next sync_cache

    def assert_ok(self):
        assert self.results, "layer gate ran no step"
        for l in self.layers:
            rs = [r for r in self.results if r[0] == l]
            worst = max(r[1] for r in rs)
            crit = max(r[2] for r in rs)
            n_ulp = sum(r[3] for r in rs)
            n = sum(r[4] for r in rs)
            ties, n_rows = sum(r[5] for r in rs), sum(r[6] for r in rs)
            tol = TOL[self.cfg.dtype]
            note = f"{n_ulp} of {n} elements over {tol} (each within 4 bf16 ulps)" if n_ulp else ""
            if ties:
                note += f"{'; ' if note else ''}{ties} of {n_rows} rows with a near-tie expert choice left out"
            report(f"{self.cfg.name} layer {l} ({len(rs)} steps)", worst, tol, note)
            assert crit <= 1.0, f"layer {l}: max-abs/RMS {worst:.4f}, per-element criterion {crit:.3f} > 1"
            assert ties <= 0.3 * n_rows, f"layer {l}: {ties} of {n_rows} rows are expert near-ties"

    def close(self):
        for one, st in self.stacks.values():
            st.close()

"""Benchmark of the Qwen3 decoder-stack forward on one GB300.

The headline line is batch-1 decode of the Qwen3-1.7B-shaped stack (28
layers, hidden 2048, 16 q / 8 kv heads, head_dim 128, intermediate 6144,
bf16) over a static KV cache prefilled to 4096 positions; the timed steps run
at contexts 4096 .. 4096+K-1 (capacity 8192).  One step = one decode token
through the whole stack (every layer: add+RMSNorm, fused qkv, q/k norm + RoPE +
cache append, attention, o_proj + residual, RMSNorm, fused gate|up + SiLU*up,
down; then the final RMSNorm).

The same run measures the other workloads of the scope table and reports each
under "workloads" with its own roofline, CPU-oracle baseline and end-to-end
number: the 2048-row prefill (and the same rows as 4 x 512 chunks), the
4-layer 128-expert MoE stack's decode at context 2048 and its 1024-row
prefill, 32-sequence int8 decode at contexts uniform in [1024, 16384], and
speculative verify windows (32 sequences x 4 rows).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
    python bench.py --workloads decode            # the headline line only
    python bench.py --layers 2 ...                # a reduced case for profiler captures

Multi-GPU runs are independent replicas (one stack per GPU, no collective on
the data path); the value is all ranks' tokens over the slowest rank's time.
Without torchrun, --gpus N > 1 starts the N ranks itself.  The reference arm
(--impl reference) times the CPU oracle on a bounded sample of the headline
workload.

Timing: W untimed warm-up steps, then K steps between CUDA events on the
launching stream; inputs are resident in HBM and every workload streams more
bytes per step than the 129 MB L2 (weights >= 2.8 GB), so no flush is needed.
Per-kernel times come from a second pass that brackets every launch with CUDA
events, with CUDA graphs and programmatic dependent launch switched off
("serialised"); the roofline's kernel figure uses those, the step figures use
the timed region.
"""
from __future__ import annotations

import argparse
import gc
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tok/s and prefill tok/s per Qwen3 stack; % of HBM / bf16 TC roofline"
UNIT = "tok/s"
CTX0 = 4096
WORKLOADS = ("decode", "prefill", "moe_decode", "moe_prefill", "batched_int8", "verify")
SERIAL = "per-kernel CUDA events around every launch, CUDA graphs and PDL off (serialised launches)"


def _env_int(k, d):
    try:
        return int(os.environ.get(k, d))
    except ValueError:
        return d


def _peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return {}


def _cores():
    return len(os.sched_getaffinity(0))


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = [l for (t, l) in self.lines if self.t0 is not None and self.t0 - 0.05 <= t <= self.t1 + 0.05]
        if not rows:
            rows = [l for (_, l) in self.lines]
        sm, mx, reasons = [], None, set()
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 10:
                continue
            try:
                sm.append(float(f[2]))
                mx = float(f[3])
            except ValueError:
                continue
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                                 f[6:10]):
                if val.lower() == "active":
                    reasons.add(name)
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- algorithmic bytes / FLOPs
def linear_bytes(cfg):
    """Bytes of each weight matrix as stored (int8: codes + bf16 scale and bias per group)."""
    H, KV, D, hid, I_ = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.hidden, cfg.intermediate
    params = {"qkv": (H + 2 * KV) * D * hid, "o": hid * H * D, "gate_up": 2 * I_ * hid, "down": hid * I_}
    if cfg.weight_format == "int8":
        return {k: v + v // cfg.group_size * 4 for k, v in params.items()}
    return {k: 2 * v for k, v in params.items()}


def kv_bytes_per_pos(cfg):
    """K and V bytes of one cached position in one layer."""
    return cfg.n_kv_heads * cfg.head_dim * 2 * 2


def kernel_bytes(cfg, name, rows, ctx_sum):
    """Algorithmic bytes per launch of the decode-path kernels: the weights
    (or the cached K/V) they must read once, plus their activation rows."""
    hid = cfg.hidden
    lb = linear_bytes(cfg)
    act = rows * hid * 2
    if cfg.num_experts:
        mI, E, k = cfg.moe_intermediate, cfg.num_experts, cfg.top_k
        slots = min(rows * k, E)
        extra = {"gemv_router": E * hid * 2 + act,
                 "gemv_expert_gate_up": slots * 2 * mI * hid * 2 + act,
                 "gemv_expert_down": slots * hid * mI * 2 + act}
        if name in extra:
            return extra[name]
    for lin in ("qkv", "o", "gate_up", "down"):
        if name in (f"gemv_{lin}", f"gemm_tc_{lin}", f"gemm_w8tc_{lin}", f"gemm_skinny_{lin}"):
            return lb[lin] + 2 * act
    if name == "attn_decode":
        return ctx_sum * kv_bytes_per_pos(cfg) + rows * (cfg.n_heads + 2 * cfg.n_kv_heads) * cfg.head_dim * 2
    return None


def step_weight_bytes(cfg, rows=1):
    """Weight bytes one decode step must read (MoE: router + the experts the rows can use)."""
    lb = linear_bytes(cfg)
    if cfg.num_experts:
        att = lb["qkv"] + lb["o"]
        mI, hid = cfg.moe_intermediate, cfg.hidden
        used = min(rows * cfg.top_k, cfg.num_experts)
        return cfg.num_layers * (att + cfg.num_experts * hid * 2 + used * 3 * mI * hid * 2)
    return cfg.num_layers * sum(lb.values())


def gemm_flops(cfg, T):
    H, KV, D, hid, I_ = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.hidden, cfg.intermediate
    per = ((H + 2 * KV) * D * hid + hid * H * D + 3 * I_ * hid)
    return 2.0 * per * T * cfg.num_layers


def linear_flops(cfg, T):
    """2 T N K of each linear of one layer (gate|up: both halves)."""
    H, KV, D, hid, I_ = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.hidden, cfg.intermediate
    return {"qkv": 2.0 * T * (H + 2 * KV) * D * hid, "o": 2.0 * T * hid * H * D,
            "gate_up": 2.0 * T * 2 * I_ * hid, "down": 2.0 * T * hid * I_}


# ---------------------------------------------------------------- CPU oracle leg
def _oracle_one_layer(cfg, wl, li):
    """A single-layer oracle with layer li's weights of `wl` (a CPU weight dict)."""
    from oracle import Qwen3Oracle
    from qwen3_decoder_layer_gb300 import inputs as I
    one = I.with_sizes(cfg, num_layers=1, name=cfg.name + "_slice", mlp_only_layers=(),
                       decoder_sparse_step=1)
    return Qwen3Oracle(one, {"layers": [wl["layers"][li]], "final_norm": wl["final_norm"]}), one


def cpu_weights(cfg, n_layers, seed):
    from qwen3_decoder_layer_gb300 import inputs as I
    return I.make_weights(I.with_sizes(cfg, num_layers=n_layers, name=cfg.name), seed=seed, device="cpu")


def oracle_decode_rate(cfg, n_steps, seed, ctxs, layers=(0, 1)):
    """tok/s of the oracle on decode: n_steps single-layer steps, cycling over
    `layers`, each with one row per context in ctxs (its own sequence), scaled
    to the full stack.  Returns (tok/s, sample description)."""
    import numpy as np  # noqa: F401
    from qwen3_decoder_layer_gb300 import inputs as I
    wl = cpu_weights(cfg, max(layers) + 1, seed)
    orcs = {}
    total, done = 0.0, 0
    for step in range(n_steps):
        li = layers[step % len(layers)]
        if li not in orcs:
            o, one = _oracle_one_layer(I.with_sizes(cfg, max_seqs=len(ctxs), capacity=max(ctxs) + n_steps + 1),
                                       wl, li)
            for s, n in enumerate(ctxs):
                K, V = I.make_cache_prefill(one, n, seed=seed + 100 * li + s, device="cpu")
                o.set_cache(s, K, V)
            o.forward(I.make_rows(one, len(ctxs), seed=seed), seq_ids=list(range(len(ctxs))))  # untimed warm-up
            orcs[li] = (o, one)
        o, one = orcs[li]
        x = I.make_rows(one, len(ctxs), seed=seed + 1000 + step)
        for s, n in enumerate(ctxs):
            o.cache[s]["length"] = n
        t = time.perf_counter()
        o.forward(x, seq_ids=list(range(len(ctxs))))
        total += time.perf_counter() - t
        done += 1
    per_layer_step = total / done
    tok_s = len(ctxs) / (per_layer_step * cfg.num_layers)
    desc = (f"{done} single-layer decode steps of {len(ctxs)} row(s) at context(s) "
            f"{ctxs if len(ctxs) <= 4 else f'{min(ctxs)}..{max(ctxs)}'} (layers {list(layers)}), "
            f"fp64 NumPy with {cfg.dtype} rounding emulation, scaled to {cfg.num_layers} layers")
    return tok_s, desc


def oracle_prefill_rate(cfg, rows, seed, layer=0):
    """tok/s of the oracle on a prefill of `rows` rows through one layer, scaled
    to the full stack (attention grows with the row count: a lower bound on the
    oracle's cost per token at longer prefills is not claimed)."""
    from qwen3_decoder_layer_gb300 import inputs as I
    wl = cpu_weights(cfg, layer + 1, seed)
    o, one = _oracle_one_layer(I.with_sizes(cfg, capacity=rows + 1), wl, layer)
    x = I.make_rows(one, rows, seed=seed + 1)
    o.forward(x[:1])   # untimed warm-up (first touch of the weights)
    o.reset()
    t = time.perf_counter()
    o.forward(x)
    dt = time.perf_counter() - t
    return rows / (dt * cfg.num_layers), (f"one {rows}-row prefill through layer {layer} from an empty cache, "
                                          f"fp64 NumPy with {cfg.dtype} rounding emulation, scaled to "
                                          f"{cfg.num_layers} layers")


def cpu_baseline(fn, *a, **k):
    value, desc = fn(*a, **k)
    return {"value": value, "unit": UNIT, "cores": _cores(), "kind": "oracle", "sample": desc}


def run_reference(args):
    """--impl reference: the CPU oracle, as it stands, on the headline workload."""
    from qwen3_decoder_layer_gb300 import inputs as I
    if _env_int("RANK", 0) != 0:
        return
    cfg = I.DENSE_1P7B_DECODE
    oracle_decode_rate(cfg, max(args.warmup, 0), 11, [CTX0])
    tok_s, desc = oracle_decode_rate(cfg, args.steps, 12, [CTX0])
    line = {"metric": METRIC, "value": tok_s, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 / tok_s, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": "Qwen3-1.7B-shaped decode, bf16, batch 1, context 4096, capacity 8192",
                       "global_batch": 1, "seq_len": CTX0, "parallelism": "replicas"},
            "cpu_baseline": {"value": tok_s, "unit": UNIT, "cores": _cores(), "kind": "oracle", "sample": desc},
            "e2e": {"value": tok_s, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU helpers
class Ctx:
    """What every workload needs: the binding, torch, peaks, the stream."""

    def __init__(self):
        import torch
        from qwen3_decoder_layer_gb300 import binding as Q
        from qwen3_decoder_layer_gb300 import inputs as I
        self.torch, self.Q, self.I = torch, Q, I
        p = _peaks()
        self.hbm = p.get("hbm_gbs")
        self.tc_burst = p.get("bf16_tflops")
        self.tc_sust = p.get("bf16_tflops_sustained")
        self.peak_src = "measured" if self.hbm else "fallback"
        self.hbm = self.hbm or 6800.0
        self.tc_burst = self.tc_burst or 1900.0
        self.tc_sust = self.tc_sust or 1700.0


def timed(C, fn, steps, setup=None):
    """ms of `steps` calls of fn(i) between CUDA events on the current stream
    (setup(i), if given, runs before each call, outside nothing: it must only
    enqueue host-side bookkeeping)."""
    torch = C.torch
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(steps):
        fn(i)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def profile_kernels(C, h, fn, warm=1):
    """Per-kernel launches and total ms over one call of fn (serialised)."""
    Q = C.Q
    Q.qwen3_set_option(h, Q.QWEN3_OPT_PROFILE, 1)
    for _ in range(warm):
        fn()
    Q.qwen3_profile_reset(h)
    fn()
    prof = Q.qwen3_profile_read(h)
    Q.qwen3_set_option(h, Q.QWEN3_OPT_PROFILE, 0)
    return prof


def kernels_table(prof):
    total = sum(v[1] for v in prof.values()) or 1.0
    return {k: {"launches": v[0], "total_ms": round(v[1], 4), "share": round(v[1] / total, 4)}
            for k, v in sorted(prof.items(), key=lambda kv: -kv[1][1])}


def _sha(path):
    import hashlib
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def traffic_of(workload, kernel):
    """DRAM bytes per launch from the committed ncu summary (profiles/traffic.txt),
    if the kernel's source is unchanged since the capture; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        f = line.split()
        if len(f) >= 5 and not line.startswith("#") and f[0] == f"{workload}:{kernel}":
            src = os.path.join(ROOT, "qwen3_decoder_layer_gb300", "csrc", f[3])
            if os.path.exists(src) and _sha(src) == f[4]:
                return float(f[1])
    return None


def hbm_roofline(C, prof, cfg, rows, ctx_sum, step_bytes, step_ms, workload=None):
    """Roofline of the dominant kernel with known algorithmic bytes, and of the step."""
    total = sum(v[1] for v in prof.values()) or 1.0
    cands = [(k, v) for k, v in prof.items() if kernel_bytes(cfg, k, rows, ctx_sum)]
    k, (n, ms) = max(cands, key=lambda kv: kv[1][1])
    b = kernel_bytes(cfg, k, rows, ctx_sum)
    avg = ms / n
    ach = b / (avg * 1e-3) / 1e9
    return {"bound": "hbm", "kernel": k, "achieved": ach, "peak": C.hbm, "unit": "GB/s", "frac": ach / C.hbm,
            "traffic": traffic_of(workload, k) if workload else None,
            "algorithmic_bytes_per_launch": b, "avg_launch_ms": avg,
            "kernel_share": ms / total, "timing": SERIAL, "peak_source": f"{C.peak_src} hbm_gbs (burst copy)",
            "step": {"bytes": step_bytes, "achieved_gbs": step_bytes / (step_ms * 1e-3) / 1e9,
                     "frac": step_bytes / (step_ms * 1e-3) / 1e9 / C.hbm}}


def fill_cache(C, stack, cfg, seq, n, seed):
    K, V = C.I.make_cache_prefill(cfg, n, seed=seed, device="cuda")
    for l in range(cfg.num_layers):
        kc, vc = C.Q.cache_tensors(stack.h, cfg, seq, l)
        kc[:, :n].copy_(K[l])
        vc[:, :n].copy_(V[l])
    del K, V


def fill_cache_fast(C, stack, cfg, seq, n, gen):
    for l in range(cfg.num_layers):
        kc, vc = C.Q.cache_tensors(stack.h, cfg, seq, l)
        kc[:, :n].normal_(generator=gen)
        vc[:, :n].normal_(generator=gen)


def decode_workload(C, cfg, ctxs, K, W, rows_per_seq=1, name="decode"):
    """(name: the workload's key in profiles/traffic.txt)"""
    """Steps of `rows_per_seq` rows for each sequence (contexts ctxs, one
    sequence each) through the whole stack: device-timed, end to end, and
    per kernel.  Returns (result dict, stack, timing extras)."""
    torch, Q, I = C.torch, C.Q, C.I
    n_seq = len(ctxs)
    weights = I.make_weights(cfg, seed=I.SEEDS.get(cfg.name, 1234), device="cuda")
    stack = Q.Qwen3Stack(cfg, weights)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(77)
    for s, n in enumerate(ctxs):
        if n_seq == 1:
            fill_cache(C, stack, cfg, s, n, seed=77)
        else:
            fill_cache_fast(C, stack, cfg, s, n, gen)
    R = n_seq * rows_per_seq
    sids = [s for s in range(n_seq) for _ in range(rows_per_seq)]
    xs = I.make_rows(cfg, R * (W + K), seed=99, device="cuda").view(W + K, R, cfg.hidden)
    out = torch.empty(R, cfg.hidden, dtype=xs.dtype, device="cuda")

    def pos(i):
        return [ctxs[s] + i * rows_per_seq + r for s in range(n_seq) for r in range(rows_per_seq)]

    def reset():
        for s, n in enumerate(ctxs):
            Q.qwen3_set_length(stack.h, s, n)

    def step(i):
        Q.qwen3_forward(stack.h, xs[i], sids, pos(i), out)

    reset()
    for i in range(W):
        step(i)
    reset()
    torch.cuda.synchronize()
    launches = Q.qwen3_last_launch_count(stack.h)
    ms = timed(C, step, K)
    # end to end through the public call with host buffers
    x_host = xs.cpu().pin_memory()
    o_host = torch.empty(R, cfg.hidden, dtype=xs.dtype).pin_memory()
    x_dev = torch.empty(R, cfg.hidden, dtype=xs.dtype, device="cuda")
    reset()

    def e2e_step(i):
        x_dev.copy_(x_host[i], non_blocking=True)
        Q.qwen3_forward(stack.h, x_dev, sids, pos(i), out)
        o_host.copy_(out, non_blocking=True)

    e2e_ms = timed(C, e2e_step, K)
    reset()
    prof = profile_kernels(C, stack.h, lambda: (reset(), step(0)))
    reset()
    tok = R
    res = {"value": tok * K / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms / K, "steps": K, "warmup": W,
           "rows_per_step": R, "gpu_launches": int(launches * K),
           "e2e": {"value": tok * K / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": R * cfg.hidden * 2,
                   "d2h_bytes_per_step": R * cfg.hidden * 2},
           "kernels": kernels_table(prof), "kernel_timing": SERIAL}
    ctx_avg_sum = sum(n + (K - 1) / 2.0 * rows_per_seq + (rows_per_seq + 1) / 2.0 for n in ctxs)
    step_bytes = step_weight_bytes(cfg, R) + cfg.num_layers * kv_bytes_per_pos(cfg) * ctx_avg_sum * 1.0
    res["roofline"] = hbm_roofline(C, prof, cfg, R, ctx_avg_sum, step_bytes, ms / K, workload=name)
    res["roofline"]["step"]["note"] = "weights once per step + every sequence's cached K/V once per layer"
    return res, stack, (step, reset)


def prefill_workload(C, cfg, T, K, W, chunks=None):
    torch, Q, I = C.torch, C.Q, C.I
    weights = I.make_weights(cfg, seed=I.SEEDS.get(cfg.name, 1234), device="cuda")
    stack = Q.Qwen3Stack(cfg, weights)
    x = I.make_rows(cfg, T, seed=99, device="cuda")
    out = torch.empty_like(x)

    def one(i):
        Q.qwen3_set_length(stack.h, 0, 0)
        Q.qwen3_forward(stack.h, x, [0] * T, list(range(T)), out)

    for i in range(W):
        one(i)
    runs = []
    for i in range(K):   # each prefill starts from an empty cache (the length reset is host-side)
        runs.append(timed(C, one, 1))
    ms = sorted(runs)[len(runs) // 2]
    launches = Q.qwen3_last_launch_count(stack.h)
    x_host = x.cpu().pin_memory()
    o_host = torch.empty_like(x_host).pin_memory()
    x_dev = torch.empty_like(x)

    def e2e(i):
        x_dev.copy_(x_host, non_blocking=True)
        Q.qwen3_set_length(stack.h, 0, 0)
        Q.qwen3_forward(stack.h, x_dev, [0] * T, list(range(T)), out)
        o_host.copy_(out, non_blocking=True)

    e2e_ms = sorted(timed(C, e2e, 1) for _ in range(K))[K // 2]
    prof = profile_kernels(C, stack.h, lambda: one(0))
    res = {"value": T / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms, "steps": K, "warmup": W,
           "step": f"one {T}-row prefill from an empty cache (median of {K})",
           "gpu_launches": int(launches * K),
           "e2e": {"value": T / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": T * cfg.hidden * 2,
                   "d2h_bytes_per_step": T * cfg.hidden * 2},
           "kernels": kernels_table(prof), "kernel_timing": SERIAL}
    if chunks:
        n = T // chunks

        def chunked(i):
            Q.qwen3_set_length(stack.h, 0, 0)
            for c in range(chunks):
                Q.qwen3_forward(stack.h, x[c * n:(c + 1) * n], [0] * n, list(range(c * n, (c + 1) * n)),
                                out[c * n:(c + 1) * n])

        for i in range(W):
            chunked(i)
        cms = sorted(timed(C, chunked, 1) for _ in range(K))[K // 2]
        res["chunked"] = {"chunks": f"{chunks} x {n}", "value": T / (cms * 1e-3), "unit": UNIT, "ms_per_step": cms}
    return res, stack, prof


# ---------------------------------------------------------------- the workloads
def wl_decode(C, K, W, cpu=True):
    I = C.I
    cfg = _sized(I.DENSE_1P7B_DECODE)
    assert CTX0 + W + K <= cfg.capacity, "steps + warmup exceed the cache capacity"
    res, stack, _ = decode_workload(C, cfg, [CTX0], K, W)
    stack.close()
    res["config"] = {"workload": "Qwen3-1.7B-shaped decode, bf16, batch 1, context 4096..4096+K-1, capacity 8192",
                     "layers": 28, "l2": "inputs larger than L2 (2.8 GB of weights streamed per step)"}
    if cpu:
        res["cpu_baseline"] = cpu_baseline(oracle_decode_rate, cfg, 28, 13, [CTX0])
    return res


def wl_prefill(C, K, W, cpu=True):
    I = C.I
    cfg = _sized(I.DENSE_1P7B_PREFILL)
    T = 2048
    res, stack, prof = prefill_workload(C, cfg, T, K, W, chunks=4)
    stack.close()
    gemm_ms = sum(v[1] for k, v in prof.items() if k.startswith("gemm_tc_"))
    flop = gemm_flops(cfg, T)
    attn_flop = 4.0 * cfg.n_heads * cfg.head_dim * (T * (T + 1) / 2) * cfg.num_layers
    ach = flop / (gemm_ms * 1e-3) / 1e12
    top = max((kv for kv in prof.items() if kv[0].startswith("gemm_tc_")), key=lambda kv: kv[1][1])
    # each linear on its own (the q|k|v launch also applies the q/k RMSNorm,
    # RoPE and cache append in its epilogue)
    per_linear = {}
    for lin, f in linear_flops(cfg, T).items():
        k = next((n for n in prof if n in (f"gemm_tc_{lin}", f"gemm_tc_{lin}_rope")), None)
        if k and prof[k][1] > 0:
            tf = f * prof[k][0] / (prof[k][1] * 1e-3) / 1e12
            per_linear[k] = {"tflops": round(tf, 1), "frac": round(tf / C.tc_burst, 3),
                             "us_per_launch": round(prof[k][1] / prof[k][0] * 1e3, 2)}
    total = sum(v[1] for v in prof.values())
    attn_ms = prof.get("attn_tc", (0, 0.0))[1]
    res["roofline"] = {"bound": "tensor", "kernel": "gemm_tc (the four linears, every layer)", "achieved": ach,
                       "peak": C.tc_burst, "unit": "TFLOP/s", "frac": ach / C.tc_burst, "traffic": None,
                       "flop_per_step": flop, "gemm_ms_per_step": gemm_ms, "timing": SERIAL,
                       "peak_source": f"{C.peak_src} bf16_tflops (burst: each GEMM is timed alone)",
                       "top_kernel": top[0], "kernel_share": top[1][1] / total,
                       "per_linear": per_linear,
                       "attention": {"kernel": "attn_tc", "flop_per_step": attn_flop,
                                     "achieved": attn_flop / (attn_ms * 1e-3) / 1e12 if attn_ms else None,
                                     "note": "causal half only; the tensor cores do 1.5x this (P as hi + lo)"},
                       "step_tflops": (flop + attn_flop) / (res["ms_per_step"] * 1e-3) / 1e12}
    res["config"] = {"workload": "Qwen3-1.7B-shaped prefill, bf16, T=2048 from an empty cache (causal); "
                                 "chunked: the same rows as 4 x 512", "layers": 28}
    if cpu:
        res["cpu_baseline"] = cpu_baseline(oracle_prefill_rate, cfg, 128, 21)
    return res


def wl_moe_decode(C, K, W, cpu=True):
    I = C.I
    cfg = _sized(I.MOE_A3B_4LAYER)
    res, stack, _ = decode_workload(C, cfg, [2048], K, W, name="moe_decode")
    stack.close()
    res["config"] = {"workload": "Qwen3-MoE-shaped decode, bf16, 4 layers, 128 experts top-8, batch 1, "
                                 "context 2048..2048+K-1", "layers": 4}
    if cpu:
        res["cpu_baseline"] = cpu_baseline(oracle_decode_rate, cfg, 8, 31, [2048], layers=(0,))
    return res


def wl_moe_prefill(C, K, W, cpu=True):
    I = C.I
    cfg = _sized(I.MOE_A3B_4LAYER)
    T = 1024
    res, stack, prof = prefill_workload(C, cfg, T, K, W)
    stack.close()
    lb = linear_bytes(cfg)
    mI, hid, E = cfg.moe_intermediate, cfg.hidden, cfg.num_experts
    byts = cfg.num_layers * (lb["qkv"] + lb["o"] + E * hid * 2 + E * 3 * mI * hid * 2)
    flop = 2.0 * T * cfg.num_layers * ((cfg.n_heads + 2 * cfg.n_kv_heads) * cfg.head_dim * hid +
                                       hid * cfg.n_heads * cfg.head_dim + E * hid + cfg.top_k * 3 * mI * hid)
    ms = res["ms_per_step"]
    total = sum(v[1] for v in prof.values())
    top = max(prof.items(), key=lambda kv: kv[1][1])
    res["roofline"] = {"bound": "hbm", "kernel": "whole step", "achieved": byts / (ms * 1e-3) / 1e9,
                       "peak": C.hbm, "unit": "GB/s", "frac": byts / (ms * 1e-3) / 1e9 / C.hbm, "traffic": None,
                       "bytes_per_step": byts, "tflops": flop / (ms * 1e-3) / 1e12,
                       "peak_source": f"{C.peak_src} hbm_gbs", "top_kernel": top[0],
                       "kernel_share": top[1][1] / total, "timing": "device-timed step"}
    res["config"] = {"workload": "Qwen3-MoE-shaped prefill, bf16, 4 layers, 128 experts top-8, T=1024 from an "
                                 "empty cache", "layers": 4}
    if cpu:
        res["cpu_baseline"] = cpu_baseline(oracle_prefill_rate, cfg, 64, 41)
    return res


def wl_batched_int8(C, K, W, cpu=True):
    I = C.I
    cfg = _sized(I.DENSE_1P7B_INT8_B32)
    ctxs = I.batch_context_lengths(32, 1024, 16384, seed=3600)
    assert max(ctxs) + W + K <= cfg.capacity
    res, stack, _ = decode_workload(C, cfg, ctxs, K, W, name="batched_int8")
    stack.close()
    res["config"] = {"workload": "Qwen3-1.7B-shaped batched decode, int8 affine group-64 weights, bf16 "
                                 "activations and KV, 32 sequences at contexts uniform in [1024, 16384]",
                     "layers": 28, "contexts": ctxs}
    if cpu:
        res["cpu_baseline"] = cpu_baseline(oracle_decode_rate, cfg, 2, 51, ctxs[:4])
        res["cpu_baseline"]["sample"] += " (4 of the 32 sequences per step)"
    return res


def wl_verify(C, K, W, cpu=True):
    """Speculative verify windows: depth + 1 = 4 rows for each of 32 sequences."""
    I = C.I
    cfg = _sized(I.with_sizes(I.DENSE_1P7B_DECODE, name="dense_1p7b_decode", max_seqs=32,
                              capacity=4096 + 4 * (W + K) + 8))
    ctxs = I.batch_context_lengths(32, 1024, 4096, seed=3800)
    res, stack, _ = decode_workload(C, cfg, ctxs, K, W, rows_per_seq=4, name="verify")
    stack.close()
    res["config"] = {"workload": "speculative verify windows on the Qwen3-1.7B-shaped stack, bf16: 32 sequences "
                                 "x 4 rows (depth 3) per call at contexts uniform in [1024, 4096]",
                     "layers": 28}
    if cpu:
        res["cpu_baseline"] = cpu_baseline(oracle_decode_rate, cfg, 2, 61, ctxs[:4])
        res["cpu_baseline"]["sample"] += " (one row for each of 4 sequences per step)"
    return res


WL_FN = {"decode": wl_decode, "prefill": wl_prefill, "moe_decode": wl_moe_decode, "moe_prefill": wl_moe_prefill,
         "batched_int8": wl_batched_int8, "verify": wl_verify}
WL_STEPS = {"prefill": 10, "moe_prefill": 10, "moe_decode": 32, "batched_int8": 16, "verify": 16}


LAYERS = 0  # --layers: a reduced profiling case (fewer layers); 0 = the workloads as stated


def _sized(cfg):
    from qwen3_decoder_layer_gb300 import inputs as I
    return I.with_sizes(cfg, num_layers=LAYERS) if LAYERS else cfg


def ranks_max(dist, values, device="cuda"):
    """The maximum over all ranks of each value (the slowest rank's times);
    unchanged with one rank (dist None)."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_rates(K, ms, e2e_ms, world):
    """Whole-job tok/s over the slowest rank's time: every rank decodes K
    tokens (one sequence each), so the job processed K * world tokens."""
    return K * world / (ms * 1e-3), K * world / (e2e_ms * 1e-3)


def run_gpu(args):
    import torch
    from qwen3_decoder_layer_gb300 import binding as Q
    from qwen3_decoder_layer_gb300 import build as B

    rank, world, local = _env_int("RANK", 0), _env_int("WORLD_SIZE", 1), _env_int("LOCAL_RANK", 0)
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    B.build()
    Q.lib()
    global LAYERS
    LAYERS = args.layers
    C = Ctx()
    K, W = args.steps, args.warmup
    cfg = _sized(C.I.DENSE_1P7B_DECODE)
    assert CTX0 + W + K <= cfg.capacity, "steps + warmup exceed the cache capacity"

    # ---- headline: batch-1 decode, replicated on every rank
    res, stack, (step, reset) = decode_workload(C, cfg, [CTX0], K, W)
    # clocks during a repeat of the timed loop
    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else local)
    clocks.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    reset()
    clocks.mark("t0")
    ms = timed(C, step, K)
    t_end = time.time() + 1.0
    while time.time() < t_end:
        reset()
        timed(C, step, min(K, 64))
    clocks.mark("t1")
    clocks.stop()
    stack.close()
    ms, e2e_ms = ranks_max(dist, [ms, K / res["e2e"]["value"] * 1e3])
    value, e2e_value = job_rates(K, ms, e2e_ms, world)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,0.02) weights, N(0,1) cache and inputs)",
        "config": {"workload": "Qwen3-1.7B-shaped decode, bf16, batch 1, context 4096..4096+K-1, capacity 8192",
                   "layers": cfg.num_layers, "hidden": cfg.hidden, "heads": [cfg.n_heads, cfg.n_kv_heads],
                   "head_dim": cfg.head_dim, "intermediate": cfg.intermediate, "global_batch": world,
                   "seq_len": CTX0, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (2.8 GB of weights streamed per step)"},
        "roofline": res["roofline"],
        "kernels": res["kernels"], "kernel_timing": SERIAL,
        "e2e": {**res["e2e"], "value": e2e_value},
        "gpu_launches": res["gpu_launches"],
        "clocks": clocks.summary(),
    }
    if LAYERS:
        line["reduced"] = f"profiling case: {LAYERS} layers per stack, not a measurement of the workloads"
    gc.collect()
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(oracle_decode_rate, cfg, 28, 13, [CTX0])
    # ---- the other workloads (one GPU)
    if world == 1:
        wanted = [w for w in args.workloads.split(",") if w and w != "decode"]
        line["workloads"] = {}
        for wl in wanted:
            try:
                r = WL_FN[wl](C, WL_STEPS.get(wl, K), max(W, 3), cpu=not args.no_cpu_baseline)
            except Exception as ex:  # report and keep measuring the others
                r = {"error": f"{type(ex).__name__}: {ex}"}
            line["workloads"][wl] = r
            gc.collect()
            torch.cuda.empty_cache()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def spawn_replicas(args):
    """--gpus N > 1 without torchrun: start N ranks on this node."""
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling only: every stack with this many layers (the line is marked reduced)")
    ap.add_argument("--workloads", default=",".join(WORKLOADS),
                    help="comma-separated subset of " + ",".join(WORKLOADS) + " (decode is always the headline)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(spawn_replicas(args))
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()

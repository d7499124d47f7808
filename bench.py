"""Benchmark: batch-1 decode of the Qwen3-1.7B-shaped stack (28 layers,
hidden 2048, 16 q / 8 kv heads, head_dim 128, intermediate 6144, bf16) over a
static KV cache prefilled to 4096 positions; the timed steps run at contexts
4096 .. 4096+K-1 (capacity 8192).  One step = one decode token through the
whole stack (every layer: add+RMSNorm, fused qkv, q/k norm + RoPE + cache
append, attention, o_proj + residual, RMSNorm, fused gate|up + SiLU*up, down;
then the final RMSNorm).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
    python bench.py --workload prefill|moe_decode|moe_prefill|batched_int8

The default run is the decode line above.  --workload measures one of the
other workloads on one GPU (2048-row prefill against the bf16 tensor-core
peak; the 4-layer 128-expert MoE stack's decode at context 2048 and its
1024-row prefill, and 32-sequence int8 decode at contexts uniform in
[1024, 16384], against the HBM peak) and prints one JSON line for it.

Multi-GPU runs are independent replicas (one stack per GPU, no collective on
the data path); the value is all ranks' tokens over the slowest rank's time.
The reference arm (--impl reference) times the CPU oracle on a bounded sample
of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
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


# ---------------------------------------------------------------- CPU oracle leg
def oracle_decode_seconds(cfg, layers, n_layer_steps: int, seed: int):
    """Time the CPU oracle on decode tokens through single layers of the stack
    (the bounded sample): layer slices cycle through `layers`, each at context
    CTX0.  Returns (seconds per full 28-layer token, sample description, cores)."""
    import numpy as np  # noqa: F401
    from oracle import Qwen3Oracle
    from qwen3_decoder_layer_gb300 import inputs as I

    one = I.with_sizes(cfg, num_layers=1, name=cfg.name + "_slice")
    slices = [li for li in layers if li != "final_norm"]
    cores = len(os.sched_getaffinity(0))
    total = 0.0
    done = 0
    orcs = {}
    for step in range(n_layer_steps):
        li = slices[step % len(slices)]
        if li not in orcs:
            o = Qwen3Oracle(one, {"layers": [layers[li]], "final_norm": layers["final_norm"]})
            K, V = I.make_cache_prefill(one, CTX0, seed=seed + li, device="cpu")
            o.set_cache(0, K, V)
            orcs[li] = o
        o = orcs[li]
        x = I.make_rows(one, 1, seed=seed + 1000 + step)
        o.cache[0]["length"] = CTX0
        t = time.perf_counter()
        o.forward(x)
        total += time.perf_counter() - t
        done += 1
    per_token = total / done * cfg.num_layers
    desc = (f"{done} single-layer decode steps at context {CTX0} (layers {sorted(orcs)} of "
            f"{cfg.num_layers}, fp64 NumPy, bf16 rounding emulation), scaled to a {cfg.num_layers}-layer token")
    return per_token, desc, cores


def cpu_weights_slices(cfg, seed, which):
    """Weights of a few layers (CPU) for the oracle leg, drawn by the generator."""
    from qwen3_decoder_layer_gb300 import inputs as I
    w = I.make_weights(I.with_sizes(cfg, num_layers=max(which) + 1, name=cfg.name), seed=seed, device="cpu")
    out = {li: w["layers"][li] for li in which}
    out["final_norm"] = w["final_norm"]
    return out


def run_reference(args):
    """--impl reference: the CPU oracle, as it stands, on the same workload."""
    from qwen3_decoder_layer_gb300 import inputs as I
    rank = _env_int("RANK", 0)
    if rank != 0:
        return
    cfg = I.DENSE_1P7B_DECODE
    which = [0, 1]
    layers = cpu_weights_slices(cfg, 5, which)
    # warm-up steps untimed, then K steps; each step is one single-layer slice
    oracle_decode_seconds(cfg, layers, max(args.warmup, 0), seed=11)
    per_tok, desc, cores = oracle_decode_seconds(cfg, layers, args.steps, seed=12)
    value = 1.0 / per_tok
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": per_tok * 1e3 / cfg.num_layers, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": "Qwen3-1.7B-shaped decode, bf16, batch 1, context 4096, capacity 8192",
                       "global_batch": 1, "seq_len": CTX0, "parallelism": "replicas"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm
def _sha(path):
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def _traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's
    source is unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        f = line.split()
        if len(f) >= 4 and f[0] == kernel and not line.startswith("#"):
            src = os.path.join(ROOT, "qwen3_decoder_layer_gb300", "csrc", f[3])
            if len(f) >= 5 and os.path.exists(src) and _sha(src) == f[4]:
                return float(f[1])
    return None


def algorithmic_bytes(cfg, kernel: str, ctx_avg: float):
    """Algorithmic bytes per launch of each decode kernel (weights once, KV once,
    activations negligible but counted)."""
    e = 2
    H, KV, D, hid, I_ = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.hidden, cfg.intermediate
    qkv_rows = (H + 2 * KV) * D
    table = {
        "gemv_qkv": qkv_rows * hid * e + 3 * hid * e + qkv_rows * e,
        "gemv_o": hid * H * D * e + H * D * e + 2 * hid * e,
        "gemv_gate_up": 2 * I_ * hid * e + 2 * hid * e + I_ * e,
        "gemv_down": hid * I_ * e + I_ * e + hid * e,
        "attn_decode": ctx_avg * KV * D * 2 * e + 2 * H * D * e,
        "qk_rope_cache": 2 * qkv_rows * e,
        "add_rmsnorm": 3 * hid * e,
    }
    return table.get(kernel)


def run_gpu(args):
    import torch
    from qwen3_decoder_layer_gb300 import binding as Q
    from qwen3_decoder_layer_gb300 import build as B
    from qwen3_decoder_layer_gb300 import inputs as I

    rank, world, local = _env_int("RANK", 0), _env_int("WORLD_SIZE", 1), _env_int("LOCAL_RANK", 0)
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    B.build()
    cfg = I.DENSE_1P7B_DECODE
    K, W = args.steps, args.warmup
    assert CTX0 + W + K <= cfg.capacity, "steps + warmup exceed the cache capacity"
    weights = I.make_weights(cfg, seed=I.SEEDS[cfg.name], device="cuda")
    stack = Q.Qwen3Stack(cfg, weights)
    kcache, vcache = I.make_cache_prefill(cfg, CTX0, seed=77, device="cuda")
    for l in range(cfg.num_layers):
        kc, vc = Q.cache_tensors(stack.h, cfg, 0, l)
        kc[:, :CTX0].copy_(kcache[l])
        vc[:, :CTX0].copy_(vcache[l])
    del kcache, vcache
    xs = I.make_rows(cfg, W + K, seed=99, device="cuda")
    out = torch.empty(1, cfg.hidden, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()

    def step(i):
        Q.qwen3_forward(stack.h, xs[i:i + 1], [0], [CTX0 + i], out)

    def run_steps(n, off):
        for i in range(n):
            step(off + i)

    # ---- device-timed region (inputs resident in HBM; weights 2.8 GB > L2 each step)
    Q.qwen3_set_length(stack.h, 0, CTX0)
    run_steps(W, 0)
    torch.cuda.synchronize()
    Q.qwen3_set_length(stack.h, 0, CTX0)
    launches_per_step = Q.qwen3_last_launch_count(stack.h)
    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else local)
    clocks.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.mark("t0")
    e0.record(stream)
    for i in range(K):
        Q.qwen3_forward(stack.h, xs[i:i + 1], [0], [CTX0 + i], out)
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.mark("t1")
    ms = e0.elapsed_time(e1)
    if dist:
        t = torch.tensor([ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    # a second, longer pass only for clock samples under load
    Q.qwen3_set_length(stack.h, 0, CTX0)
    clocks.mark("t0")
    t_end = time.time() + 1.0
    while time.time() < t_end:
        Q.qwen3_set_length(stack.h, 0, CTX0)
        run_steps(min(K, 64), 0)
        torch.cuda.synchronize()
    clocks.mark("t1")
    clocks.stop()
    clk = clocks.summary()

    # ---- end to end through the public API with host buffers
    x_host = torch.empty(W + K, 1, cfg.hidden, dtype=torch.bfloat16).pin_memory()
    x_host.copy_(xs.view(W + K, 1, cfg.hidden).cpu())
    o_host = torch.empty(1, cfg.hidden, dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty(1, cfg.hidden, dtype=torch.bfloat16, device="cuda")
    Q.qwen3_set_length(stack.h, 0, CTX0)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    e0.record(stream)
    for i in range(K):
        x_dev.copy_(x_host[i], non_blocking=True)
        Q.qwen3_forward(stack.h, x_dev, [0], [CTX0 + i], out)
        o_host.copy_(out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    if dist:
        t = torch.tensor([e2e_ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_ms = float(t.item())

    # ---- per-kernel durations (events around every launch) over the same K steps
    Q.qwen3_set_option(stack.h, Q.QWEN3_OPT_PROFILE, 1)
    Q.qwen3_set_length(stack.h, 0, CTX0)
    run_steps(2, 0)
    Q.qwen3_profile_reset(stack.h)
    Q.qwen3_set_length(stack.h, 0, CTX0)
    for i in range(K):
        Q.qwen3_forward(stack.h, xs[i:i + 1], [0], [CTX0 + i], out)
    prof = Q.qwen3_profile_read(stack.h)
    Q.qwen3_set_option(stack.h, Q.QWEN3_OPT_PROFILE, 0)
    total_prof = sum(v[1] for v in prof.values())
    top = max(prof.items(), key=lambda kv: kv[1][1])
    kname, (klaunch, kms) = top
    ctx_avg = CTX0 + (K - 1) / 2.0
    bytes_per = algorithmic_bytes(cfg, kname, ctx_avg)
    peaks = _peaks()
    hbm_peak = peaks.get("hbm_gbs")
    peak_src = "measured" if hbm_peak else "fallback"
    hbm_peak = hbm_peak or 6800.0
    avg_ms = kms / klaunch
    achieved = bytes_per / (avg_ms * 1e-3) / 1e9 if bytes_per else None
    # whole-step roofline: algorithmic bytes per token / step time
    step_bytes = (sum(algorithmic_bytes(cfg, k, ctx_avg) for k in
                      ("gemv_qkv", "gemv_o", "gemv_gate_up", "gemv_down", "attn_decode")) * cfg.num_layers)
    tok_s = K / (ms * 1e-3)

    stack.close()
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": tok_s * world, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,0.02) weights, N(0,1) cache and inputs)",
        "config": {"workload": "Qwen3-1.7B-shaped decode, bf16, batch 1, context 4096..4096+K-1, capacity 8192",
                   "layers": cfg.num_layers, "hidden": cfg.hidden, "heads": [cfg.n_heads, cfg.n_kv_heads],
                   "head_dim": cfg.head_dim, "intermediate": cfg.intermediate, "global_batch": world,
                   "seq_len": CTX0, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (2.8 GB of weights streamed per step)"},
        "roofline": {"bound": "hbm", "kernel": kname,
                     "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": (achieved / hbm_peak) if achieved else None,
                     "traffic": _traffic(kname),
                     "algorithmic_bytes_per_launch": bytes_per, "avg_launch_ms": avg_ms,
                     "kernel_share": kms / total_prof, "peak_source": peak_src + " hbm_gbs",
                     "step": {"bytes_per_token": step_bytes,
                              "achieved_gbs": step_bytes * tok_s / 1e9,
                              "frac": step_bytes * tok_s / 1e9 / hbm_peak}},
        "kernels": {k: {"launches": v[0], "total_ms": round(v[1], 4), "share": round(v[1] / total_prof, 4)}
                    for k, v in sorted(prof.items(), key=lambda kv: -kv[1][1])},
        "e2e": {"value": K / (e2e_ms * 1e-3) * world, "unit": UNIT,
                "h2d_bytes_per_step": cfg.hidden * 2, "d2h_bytes_per_step": cfg.hidden * 2},
        "gpu_launches": int(launches_per_step * K),
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        which = [0, 1]
        layers = cpu_weights_slices(cfg, 5, which)
        per_tok, desc, cores = oracle_decode_seconds(cfg, layers, 28, seed=13)
        line["cpu_baseline"] = {"value": 1.0 / per_tok, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": desc}
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


# ---------------------------------------------------------------- other workloads
WORKLOADS = ("decode", "prefill", "moe_decode", "moe_prefill", "batched_int8")


def _linear_params(cfg):
    H, KV, D, hid, I_ = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.hidden, cfg.intermediate
    attn = (H + 2 * KV) * D * hid + hid * H * D
    if cfg.num_experts:
        return attn, hid * cfg.num_experts, 3 * cfg.moe_intermediate * hid
    return attn, 0, 3 * I_ * hid


def run_workload(args):
    """The other workloads of the scope table, each with its own roofline:
    prefill (2048 rows, tensor-core bound), MoE decode / prefill (HBM bound),
    32-sequence int8 decode (HBM bound, KV dominated).  One JSON line each."""
    import statistics

    import torch
    from qwen3_decoder_layer_gb300 import binding as Q
    from qwen3_decoder_layer_gb300 import build as B
    from qwen3_decoder_layer_gb300 import inputs as I

    B.build()
    peaks = _peaks()
    hbm = peaks.get("hbm_gbs") or 6800.0
    tc = peaks.get("bf16_tflops_sustained") or 1700.0
    wl, K, W = args.workload, args.steps, args.warmup
    cfg = {"prefill": I.DENSE_1P7B_PREFILL, "moe_decode": I.MOE_A3B_4LAYER, "moe_prefill": I.MOE_A3B_4LAYER,
           "batched_int8": I.DENSE_1P7B_INT8_B32}[wl]
    # reduced case for profiler captures (fewer layers, one short context): same shapes per layer,
    # a few GB on the device; its line says so and is not a measurement of the workload
    reduced = bool(args.layers or args.ctx)
    if args.layers:
        cfg = I.with_sizes(cfg, num_layers=args.layers)
    if args.ctx and wl in ("moe_decode", "batched_int8"):
        cfg = I.with_sizes(cfg, capacity=args.ctx + W + K + 16)
    weights = I.make_weights(cfg, seed=I.SEEDS[cfg.name], device="cuda")
    stack = Q.Qwen3Stack(cfg, weights)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(4242)
    attn_p, router_p, mlp_p = _linear_params(cfg)
    kv_pos_bytes = cfg.num_layers * cfg.n_kv_heads * cfg.head_dim * 2 * 2  # K and V, bf16, every layer

    def fill(seq, n):
        for l in range(cfg.num_layers):
            kc, vc = Q.cache_tensors(stack.h, cfg, seq, l)
            kc[:, :n].normal_(generator=gen)
            vc[:, :n].normal_(generator=gen)

    if wl == "prefill" or wl == "moe_prefill":
        T = 2048 if wl == "prefill" else 1024
        x = I.make_rows(cfg, T, seed=99, device="cuda")
        out = torch.empty_like(x)
        runs = []
        for i in range(W + K):
            Q.qwen3_set_length(stack.h, 0, 0)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            Q.qwen3_forward(stack.h, x, [0] * T, list(range(T)), out)
            e1.record()
            torch.cuda.synchronize()
            if i >= W:
                runs.append(e0.elapsed_time(e1))
        ms = statistics.median(runs)
        value = T / (ms * 1e-3)
        unit, steps_desc = "tok/s", f"median of {K} {T}-row prefills from an empty cache"
        def run_one():
            Q.qwen3_set_length(stack.h, 0, 0)
            Q.qwen3_forward(stack.h, x, [0] * T, list(range(T)), out)
    else:
        if wl == "moe_decode":
            ctx = [2048]
            n_seq = 1
        else:
            n_seq = cfg.max_seqs
            ctx = I.batch_context_lengths(n_seq, 1024, 16384, seed=3600)
        if args.ctx:
            ctx = [args.ctx] * n_seq
        assert max(ctx) + W + K <= cfg.capacity, "steps + warmup exceed the cache capacity"
        for s_, n in enumerate(ctx):
            fill(s_, n)
        xs = I.make_rows(cfg, n_seq * (W + K), seed=99, device="cuda").view(W + K, n_seq, cfg.hidden)
        out = torch.empty(n_seq, cfg.hidden, dtype=xs.dtype, device="cuda")
        seqs = list(range(n_seq))

        def reset_len():
            for s_, n in enumerate(ctx):
                Q.qwen3_set_length(stack.h, s_, n)

        def step(i):
            Q.qwen3_forward(stack.h, xs[i], seqs, [n + i for n in ctx], out)
        reset_len()
        for i in range(W):
            step(i)
        reset_len()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(K):
            step(i)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / K
        value = n_seq / (ms * 1e-3)
        unit, steps_desc = "tok/s", f"{K} decode steps of {n_seq} row(s)"

        def run_one():
            reset_len()
            step(0)

    # clocks under load, then per-kernel times (events around every launch)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    clocks.mark("t0")
    t_end = time.time() + 1.0
    while time.time() < t_end:
        run_one()
        torch.cuda.synchronize()
    clocks.mark("t1")
    clocks.stop()
    Q.qwen3_set_option(stack.h, Q.QWEN3_OPT_PROFILE, 1)
    run_one()
    Q.qwen3_profile_reset(stack.h)
    run_one()
    prof = Q.qwen3_profile_read(stack.h)
    Q.qwen3_set_option(stack.h, Q.QWEN3_OPT_PROFILE, 0)
    total = sum(v[1] for v in prof.values())
    kernels = {k: {"launches": v[0], "total_ms": round(v[1], 4), "share": round(v[1] / total, 4)}
               for k, v in sorted(prof.items(), key=lambda kv: -kv[1][1])}
    line = {"metric": f"{wl} tok/s", "value": value, "unit": unit, "n_gpus": 1, "steps": K, "warmup": W,
            "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16" if cfg.weight_format != "int8" else
            "bf16 activations, int8 weights", "data": "synthetic (seeded)", "workload": wl,
            "config": {"workload": f"{cfg.name}: {steps_desc}", "layers": cfg.num_layers},
            **({"reduced": "profiling case (--layers / --ctx): not a measurement of the workload"}
               if reduced else {}),
            "kernels": kernels, "clocks": clocks.summary()}
    if wl == "prefill":
        T = 2048
        gemm_flop = 2.0 * (attn_p + mlp_p) * cfg.num_layers * T
        gemm_ms = sum(v[1] for k, v in prof.items() if k.startswith("gemm_")) / 1.0
        attn_flop = 4.0 * cfg.n_heads * cfg.head_dim * (T * (T + 1) / 2) * cfg.num_layers
        line["roofline"] = {"bound": "tensor", "kernel": "gemm_tc (all linears)",
                            "achieved": gemm_flop / (gemm_ms * 1e-3) / 1e12, "peak": tc, "unit": "TFLOP/s",
                            "frac": gemm_flop / (gemm_ms * 1e-3) / 1e12 / tc,
                            "peak_source": "measured bf16_tflops_sustained", "traffic": None,
                            "gemm_flop_per_step": gemm_flop, "gemm_ms_per_step": gemm_ms,
                            "step_tflops": (gemm_flop + attn_flop) / (ms * 1e-3) / 1e12}
    elif wl == "moe_prefill":
        T = 1024
        flop = 2.0 * T * cfg.num_layers * (attn_p + router_p + cfg.top_k * mlp_p)
        byts = 2.0 * cfg.num_layers * (attn_p + router_p + cfg.num_experts * mlp_p)
        line["roofline"] = {"bound": "hbm", "kernel": "whole step", "achieved": byts / (ms * 1e-3) / 1e9,
                            "peak": hbm, "unit": "GB/s", "frac": byts / (ms * 1e-3) / 1e9 / hbm,
                            "peak_source": "measured hbm_gbs", "traffic": None, "bytes_per_step": byts,
                            "tflops": flop / (ms * 1e-3) / 1e12}
    else:
        ctx_avg = [n + (K - 1) / 2.0 for n in ctx]
        if wl == "moe_decode":
            wbytes = 2.0 * cfg.num_layers * (attn_p + router_p + cfg.top_k * mlp_p)
        else:
            params = (attn_p + mlp_p) * cfg.num_layers
            wbytes = params * 1.0 + params / cfg.group_size * 2 * 2
        byts = wbytes + kv_pos_bytes * sum(c + 1 for c in ctx_avg)
        line["roofline"] = {"bound": "hbm", "kernel": "whole step", "achieved": byts / (ms * 1e-3) / 1e9,
                            "peak": hbm, "unit": "GB/s", "frac": byts / (ms * 1e-3) / 1e9 / hbm,
                            "peak_source": "measured hbm_gbs", "traffic": None, "bytes_per_step": byts,
                            "weight_bytes": wbytes}
    stack.close()
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="decode", choices=WORKLOADS,
                    help="decode (default: the headline line) or one of the other scope-table workloads")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling only: run a non-decode workload with this many layers")
    ap.add_argument("--ctx", type=int, default=0,
                    help="profiling only: every sequence of moe_decode / batched_int8 at this context")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = {"decode": 256, "prefill": 10, "moe_decode": 56, "moe_prefill": 10, "batched_int8": 64}[
            args.workload]
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.workload != "decode":
        run_workload(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()

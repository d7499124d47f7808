"""GPU parity of the steps around the stack and of the stack variants the
pages describe beyond the five workloads, each against the oracle:

* embedding rows and the output head (maya2_mlx/backbone.py,
  Backbone.embed_tokens and cb0_logits; a tied head is the embedding table's
  product, @mlx-bun/inference qwen3.ts embed.asLinear);
* the pooled sentence vector (qwen3.ts embedPooled);
* mixed dense / MoE layer schedules and int8 experts (qwen3-moe.ts
  Qwen3MoeDecoderLayer, QuantizedSwitchLinear);
* speculative verify windows: several rows per sequence across many sequences
  in one call (qwen3-moe.ts `verify`: depth + 1 positions per sequence)."""
import numpy as np
import pytest
import torch

from gpu_helpers import E2E_CAP, TOL, TWIN_FACTOR, Parity, as_f64, bf16_ulp, rel_err, report, to_device
from oracle import Qwen3Oracle, Qwen3OracleF32Acc, embed_rows, head_logits, l2_pool_last
from qwen3_decoder_layer_gb300 import binding as Q
from qwen3_decoder_layer_gb300 import inputs as I

pytestmark = pytest.mark.gpu

SMALL_D128 = I.with_sizes(I.TINY_FP32, name="next_d128", dtype="bf16", hidden=512, n_heads=4, n_kv_heads=2,
                          head_dim=128, intermediate=1088, capacity=300, num_layers=3)


def _close(got, ref, dtype, ulps=1):
    """max-abs/RMS within the dtype's bound; bf16 elements may also sit within
    `ulps` bf16 ulps of the oracle (rounding decisions taken the other way)."""
    g, r = as_f64(got), as_f64(ref)
    rms = np.sqrt(np.mean(r * r))
    d = np.abs(g - r)
    allow = TOL[dtype] * rms if dtype == "fp32" else np.maximum(TOL[dtype] * rms, ulps * bf16_ulp(r, g))
    return float(d.max() / rms), bool(np.all(d <= allow))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("T", [1, 3, 9])
def test_embed_and_head(cuda_ok, dtype, T):
    """Rows gathered from a 1000-row table bit-exact; a 2049-wide head (the
    cb0_head shape: ragged against every tile) and a tied head over the table,
    rounded once to the model dtype, then fp32."""
    cfg = I.with_sizes(SMALL_D128, dtype=dtype)
    stack = Q.Qwen3Stack(cfg, I.make_weights(cfg, seed=4000, device="cuda"))
    g = torch.Generator().manual_seed(4001)
    table = torch.randn(1000, cfg.hidden, generator=g).to(cfg.torch_dtype())
    head = (0.02 * torch.randn(2049, cfg.hidden, generator=g)).to(cfg.torch_dtype())
    ids = [int(i) for i in torch.randint(0, 1000, (T,), generator=g)]
    rows = torch.empty(T, cfg.hidden, dtype=cfg.torch_dtype(), device="cuda")
    Q.qwen3_embed(stack.h, table.cuda(), ids, rows)
    torch.cuda.synchronize()
    assert torch.equal(rows.cpu().double(), torch.from_numpy(embed_rows(as_f64(table), ids, dtype)))
    x = I.make_rows(cfg, T, seed=4002)
    for name, W in (("cb0 head 2049", head), ("tied head 1000", table)):
        logits = torch.empty(T, W.shape[0], dtype=torch.float32, device="cuda")
        Q.qwen3_head(stack.h, W.cuda(), x.cuda(), logits)
        torch.cuda.synchronize()
        err, ok = _close(logits, head_logits(as_f64(x), as_f64(W), dtype), dtype)
        report(f"{name}, {T} rows, {dtype}", err, TOL[dtype])
        assert ok, f"{name}: {err}"
    with pytest.raises(Q.Qwen3Error) as e:
        Q.qwen3_embed(stack.h, table.cuda(), [0, 1000], rows[:2])
    assert e.value.status == 1 and "1000" in str(e.value)
    stack.close()


@pytest.mark.parametrize("cfg,T", [(I.TINY_FP32, 16), (I.with_sizes(I.TINY_FP32, dtype="bf16", name="tiny_bf16"), 16),
                                   (SMALL_D128, 37), (SMALL_D128, 3)], ids=["fp32", "bf16", "d128_37", "d128_3"])
def test_embed_pooled(cuda_ok, cfg, T):
    """Last-token L2-normalised sentence vector after a fresh prefill; a second
    call on the same sequence starts over and gives the same vector."""
    w = I.make_weights(cfg, seed=4100)
    stack = Q.Qwen3Stack(cfg, to_device(w))
    x = I.make_rows(cfg, T, seed=4101)
    out = torch.empty(cfg.hidden, dtype=cfg.torch_dtype(), device="cuda")
    Q.qwen3_embed_pooled(stack.h, x.cuda(), 0, out)
    ref = l2_pool_last(Qwen3Oracle(cfg, w).forward(x), cfg.dtype)
    bound = TOL[cfg.dtype]
    if cfg.dtype == "bf16":   # the stack's own bound (gpu_helpers.Parity.bound)
        drift = rel_err(l2_pool_last(Qwen3OracleF32Acc(cfg, w).forward(x), cfg.dtype), ref)
        bound = min(E2E_CAP, max(bound, TWIN_FACTOR * drift))
    err = rel_err(out, ref)
    report(f"pooled vector {cfg.name} T={T}", err, bound)
    assert err <= bound, err
    again = torch.empty_like(out)
    Q.qwen3_embed_pooled(stack.h, x.cuda(), 0, again)
    torch.cuda.synchronize()
    assert torch.equal(out, again) and Q.qwen3_get_length(stack.h, 0) == T
    stack.close()


MIXED = I.with_sizes(I.MOE_A3B_4LAYER, name="mixed_moe", num_layers=4, hidden=256, n_heads=8, n_kv_heads=1,
                     head_dim=64, intermediate=512, num_experts=32, top_k=4, moe_intermediate=128, capacity=128,
                     decoder_sparse_step=2, mlp_only_layers=(3,))


@pytest.mark.parametrize("cfg", [MIXED, I.with_sizes(MIXED, decoder_sparse_step=1, mlp_only_layers=(0, 2),
                                                      name="mixed_moe_b")], ids=["step2_dense3", "step1_dense02"])
@pytest.mark.parametrize("T", [2, 24])
def test_mixed_dense_moe_schedule(cuda_ok, cfg, T):
    """A stack whose layers alternate dense MLPs and MoE blocks by
    decoder_sparse_step and mlp_only_layers: prefill then decode steps."""
    p = Parity(cfg, seed=4200 + T)
    p.step(I.make_rows(cfg, T, seed=4201).cuda())
    for s in range(2):
        p.step(I.make_rows(cfg, 1, seed=4202 + s).cuda())
    p.close()
    p.check()


INT8_MOE = I.with_sizes(MIXED, name="int8_moe", weight_format="int8", group_size=64)


@pytest.mark.parametrize("T", [1, 3, 24, 40])
def test_int8_experts(cuda_ok, T):
    """int8 experts (and int8 attention / dense MLP linears): gathered expert
    GEMVs for few rows, sorted grouped GEMMs from ceil(64 / top_k) rows; the
    expert block alone through qwen3_moe_layer too."""
    p = Parity(INT8_MOE, seed=4300 + T)
    p.step(I.make_rows(INT8_MOE, T, seed=4301).cuda())
    p.step(I.make_rows(INT8_MOE, 1, seed=4302).cuda())
    p.close()
    p.check()
    from test_parity_small import moe_layer_check
    q = Parity(INT8_MOE, seed=4310 + T, twin=False)
    err, clear = moe_layer_check(INT8_MOE, q.stack, q.orc, 1, I.make_rows(INT8_MOE, T, seed=4311).cuda())
    report(f"int8 expert block, {T} rows", err, TOL["bf16"])
    assert clear > 0.9 and err <= TOL["bf16"]
    q.close()


@pytest.mark.parametrize("n_seqs,depth", [(8, 3), (12, 1), (6, 7)])
def test_verify_windows(cuda_ok, n_seqs, depth):
    """depth + 1 rows for each of many sequences in one call, every sequence
    at its own context, then single-row decode of all of them."""
    cfg = I.with_sizes(SMALL_D128, max_seqs=n_seqs, name="verify")
    p = Parity(cfg, seed=4400 + n_seqs)
    rng = np.random.default_rng(4401)
    for s in range(n_seqs):
        p.fill_cache(s, int(rng.integers(5, 200)), seed=4410 + s)
    for step in range(2):
        sids = [s for s in range(n_seqs) for _ in range(depth + 1)]
        p.step(I.make_rows(cfg, len(sids), seed=4420 + step).cuda(), seq_ids=sids)
    p.step(I.make_rows(cfg, n_seqs, seed=4430).cuda(), seq_ids=list(range(n_seqs)))
    p.close()
    p.check()

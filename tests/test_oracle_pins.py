"""Pins for the CPU oracle: checks against things other than the oracle itself
(closed forms, invariants the mathematics fixes, special cases that reduce to a
torch library routine, and an independently written brute-force forward).

Each test names the page and passage it pins (maya2_mlx/backbone.py
``Backbone``; @mlx-bun/inference qwen3-moe.ts ``Qwen3MoeSparseMoeBlock``).
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import (Qwen3Oracle, Qwen3OracleF32Acc, rnd, rms_norm, rope, rope_table, softmax,
                    attention_probs, silu, dequant_affine, router_topk, moe_layer, embed_rows, head_logits,
                    l2_pool_last)
from qwen3_decoder_layer_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

TINY = I.with_sizes(I.TINY_FP32, name="pin_tiny", num_layers=2, hidden=64, n_heads=4,
                    n_kv_heads=2, head_dim=16, intermediate=96, capacity=32)
TINY_MOE = I.with_sizes(TINY, name="pin_tiny_moe", num_experts=8, top_k=2,
                        moe_intermediate=32, rope_theta=1e7)


# ---------------------------------------------------------------- rounding
def test_bf16_rounding_matches_torch_cast():
    """rnd(., 'bf16') is round-to-nearest-even to 8 significant bits: it must
    agree with torch's float32 -> bfloat16 cast on fp32 inputs, ties included."""
    rng = np.random.default_rng(1)
    x = rng.standard_normal(200000).astype(np.float32) * np.float32(3.0)
    # exact ties: bf16 value + half an ulp, for even and odd last kept bits
    bits = (rng.integers(0x3f000000, 0x40ffffff, 5000, dtype=np.uint32) & 0xFFFF0000) | 0x8000
    ties = bits.view(np.float32)
    x = np.concatenate([x, ties, -ties])
    ref = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    assert np.array_equal(rnd(x.astype(np.float64), "bf16"), ref)


def test_fp32_rounding_matches_numpy_cast():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(100000) * 100.0
    assert np.array_equal(rnd(x, "fp32"), x.astype(np.float32).astype(np.float64))


# ---------------------------------------------------------------- RMSNorm
def test_rmsnorm_scale_invariance():
    """RMS(c v) = RMS(v) with eps = 0 (exact mode)."""
    rng = np.random.default_rng(3)
    v = rng.standard_normal((5, 64))
    g = 1 + 0.1 * rng.standard_normal(64)
    base = rms_norm(v, g, 0.0, "exact")
    for c in (1e-3, 7.0, 1e3):
        assert np.max(np.abs(rms_norm(c * v, g, 0.0, "exact") - base)) < 1e-12


def test_rmsnorm_closed_forms():
    """Constant vector a*1 with unit gain gives a / sqrt(a^2 + eps); the hand-worked
    example in tests/golden/closed_forms.json matches; torch's rms_norm agrees."""
    for a in (0.5, -3.0, 1e-3):
        out = rms_norm(np.full(8, a), np.ones(8), 1e-6, "exact")
        assert np.allclose(out, a / math.sqrt(a * a + 1e-6), rtol=0, atol=1e-15)
    gold = json.load(open(os.path.join(GOLDEN, "closed_forms.json")))["rmsnorm"]
    out = rms_norm(np.array(gold["x"]), np.array(gold["gain"]), gold["eps"], "exact")
    assert np.allclose(out, gold["out"], rtol=0, atol=1e-12)
    rng = np.random.default_rng(4)
    v = rng.standard_normal((3, 32))
    g = rng.standard_normal(32)
    ref = F.rms_norm(torch.from_numpy(v), (32,), torch.from_numpy(g), eps=1e-5).numpy()
    assert np.max(np.abs(rms_norm(v, g, 1e-5, "exact") - ref)) < 1e-12


# ---------------------------------------------------------------- RoPE
def _rope_at(x, p, D, theta, prec):
    c, s = rope_table(p + 1, D, theta, prec)
    return rope(x, c[p], s[p], prec)


def test_rope_norm_preservation_and_identity():
    rng = np.random.default_rng(5)
    D = 64
    x = rng.standard_normal(D)
    for p in (0, 1, 17, 500):
        assert abs(np.linalg.norm(_rope_at(x, p, D, 1e6, "exact")) - np.linalg.norm(x)) < 1e-12
    # p = 0 is the identity in every table precision (cos 0 = 1, sin 0 = 0 exactly)
    for prec in ("exact", "fp32", "bf16"):
        xr = rnd(x, prec)
        assert np.array_equal(_rope_at(xr, 0, D, 1e6, prec), xr)


def test_rope_relative_position_identity():
    """<rope(q, m), rope(k, n)> depends only on m - n."""
    rng = np.random.default_rng(6)
    D = 32
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    c, s = rope_table(200, D, 1e4, "exact")
    ref = rope(q, c[9], s[9], "exact") @ rope(k, c[4], s[4], "exact")
    for shift in (1, 30, 150):
        got = rope(q, c[9 + shift], s[9 + shift], "exact") @ rope(k, c[4 + shift], s[4 + shift], "exact")
        assert abs(got - ref) < 1e-10


def test_rope_golden_and_complex_form():
    """Hand-worked D=4, theta=1e4 example (tests/golden/closed_forms.json), and the
    rotate-half rotation equals multiplying (x_i + i x_{i+D/2}) by exp(i p f_i)."""
    gold = json.load(open(os.path.join(GOLDEN, "closed_forms.json")))["rope"]
    out = _rope_at(np.array(gold["x"]), gold["p"], 4, gold["theta"], "exact")
    assert np.allclose(out, gold["out"], rtol=0, atol=1e-12)
    rng = np.random.default_rng(7)
    D, theta, p = 16, 1e6, 37
    x = rng.standard_normal(D)
    f = theta ** (-np.arange(D // 2) * 2.0 / D)
    z = (x[:D // 2] + 1j * x[D // 2:]) * np.exp(1j * p * f)
    assert np.allclose(_rope_at(x, p, D, theta, "exact"), np.concatenate([z.real, z.imag]), atol=1e-12)


def test_rope_bf16_table_uses_rounded_inv_freq():
    """bf16 table: inv_freq rounded to bf16 before the angle (Backbone.__init__)."""
    D, theta, p = 128, 1e6, 4000
    c, s = rope_table(p + 1, D, theta, "bf16")
    inv = rnd(theta ** (-2.0 * np.arange(D // 2) / D), "bf16")
    assert np.array_equal(c[p, :D // 2], rnd(np.cos(p * inv), "bf16"))
    assert np.array_equal(c[p, D // 2:], c[p, :D // 2])
    assert np.array_equal(s[p, D // 2:], s[p, :D // 2])


# ---------------------------------------------------------------- softmax / attention
def test_softmax_rows_sum_to_one_and_masking():
    rng = np.random.default_rng(8)
    s = rng.standard_normal((7, 33)) * 10
    s[:, 20:] = -np.inf
    P = softmax(s)
    assert np.allclose(P.sum(-1), 1.0, atol=1e-14)
    assert np.all(P[:, 20:] == 0)


def test_attention_single_key_returns_v_and_identical_keys_give_mean():
    rng = np.random.default_rng(9)
    q, k = rng.standard_normal(16), rng.standard_normal((1, 16))
    assert np.array_equal(attention_probs(q, k, 0.25), [1.0])
    K = np.tile(rng.standard_normal(16), (10, 1))
    V = rng.standard_normal((10, 16))
    P = attention_probs(q, K, 0.25)
    assert np.allclose(P @ V, V.mean(0), atol=1e-14)


@pytest.mark.parametrize("prec", ["exact", "fp32", "bf16"])
def test_decode_at_position_zero_returns_v_exactly(prec):
    """T=1 at position 0 with one cached key: softmax weight 1, so the attention
    output equals v bit for bit in every precision (q head h reads kv head h//G)."""
    cfg = I.with_sizes(TINY, dtype="bf16" if prec == "bf16" else "fp32")
    w = I.make_weights(cfg, seed=11)
    o = Qwen3Oracle(cfg, w, prec=prec)
    tr = []
    o.forward(I.make_rows(cfg, 1, seed=12), trace=tr)
    G = cfg.n_heads // cfg.n_kv_heads
    for L in tr:
        for h in range(cfg.n_heads):
            assert np.array_equal(L["a"][0, h], L["v"][0, h // G])


def test_gqa_attention_matches_torch_sdpa():
    """One layer's attention (exact mode) against torch's scaled_dot_product_attention
    with the kv heads repeated G times (repeat_kv) and an explicit causal mask."""
    cfg = TINY
    w = I.make_weights(cfg, seed=13)
    o = Qwen3Oracle(cfg, w, prec="exact")
    T = 9
    tr = []
    o.forward(I.make_rows(cfg, T, seed=14), trace=tr)
    G = cfg.n_heads // cfg.n_kv_heads
    for L in tr:
        q = torch.from_numpy(L["q"]).permute(1, 0, 2)[None]          # [1, H, T, D] (post RoPE)
        k = torch.from_numpy(L["k"]).permute(1, 0, 2)[None].repeat_interleave(G, dim=1)
        v = torch.from_numpy(L["v"]).permute(1, 0, 2)[None].repeat_interleave(G, dim=1)
        mask = torch.ones(T, T, dtype=torch.bool).tril()
        a = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=cfg.head_dim ** -0.5)
        assert np.max(np.abs(a[0].permute(1, 0, 2).numpy() - L["a"])) < 1e-12


# ---------------------------------------------------------------- whole stack
def _brute_force(cfg, w, x):
    """Independent fp64 torch forward of a prefill from an empty cache: separate
    q/k/v and gate/up matmuls, complex-number RoPE, full T x T masked attention
    with repeat_kv materialised, torch rms_norm and silu, torch.topk router."""
    d = lambda t: t.detach().double()
    H, KV, D, hid = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.hidden
    T = x.shape[0]
    eps = cfg.rms_eps
    f = cfg.rope_theta ** (-torch.arange(D // 2, dtype=torch.float64) * 2.0 / D)
    ang = torch.arange(T, dtype=torch.float64)[:, None] * f[None]
    rot = torch.polar(torch.ones_like(ang), ang)                           # [T, D/2]

    def rope_c(t):                                                         # t [T, heads, D]
        z = torch.complex(t[..., :D // 2], t[..., D // 2:]) * rot[:, None, :]
        return torch.cat([z.real, z.imag], -1)

    h = d(x)
    for li, L in enumerate(w["layers"]):
        Wqkv = d(L["qkv"]["w"])
        Wq, Wk, Wv = Wqkv[:H * D], Wqkv[H * D:(H + KV) * D], Wqkv[(H + KV) * D:]
        y = F.rms_norm(h, (hid,), d(L["in_norm"]), eps)
        q = F.rms_norm((y @ Wq.T).view(T, H, D), (D,), d(L["q_norm"]), eps)
        k = F.rms_norm((y @ Wk.T).view(T, KV, D), (D,), d(L["k_norm"]), eps)
        v = (y @ Wv.T).view(T, KV, D)
        q, k = rope_c(q), rope_c(k)
        k = k.repeat_interleave(H // KV, dim=1)
        v = v.repeat_interleave(H // KV, dim=1)
        S = torch.einsum("thd,uhd->htu", q, k) / math.sqrt(D)
        S = S.masked_fill(~torch.ones(T, T, dtype=torch.bool).tril(), float("-inf"))
        a = torch.einsum("htu,uhd->thd", torch.softmax(S, -1), v).reshape(T, H * D)
        h = h + a @ d(L["o"]["w"]).T
        y2 = F.rms_norm(h, (hid,), d(L["post_norm"]), eps)
        if "router" in L:                       # the layer's kind from the weights it was given
            mI = cfg.moe_intermediate
            P = torch.softmax(y2 @ d(L["router"]["w"]).T, -1)
            wk, ik = torch.topk(P, cfg.top_k, dim=-1)
            wk = wk / wk.sum(-1, keepdim=True)
            out = torch.zeros_like(h)
            for t in range(T):
                for s in range(cfg.top_k):
                    e = int(ik[t, s])
                    Wgu = d(L["exp_gate_up"]["w"][e])
                    m = F.silu(y2[t] @ Wgu[:mI].T) * (y2[t] @ Wgu[mI:].T)
                    out[t] += wk[t, s] * (m @ d(L["exp_down"]["w"][e]).T)
            h = h + out
        else:
            Wgu = d(L["gate_up"]["w"])
            n = cfg.intermediate
            h = h + (F.silu(y2 @ Wgu[:n].T) * (y2 @ Wgu[n:].T)) @ d(L["down"]["w"]).T
    return F.rms_norm(h, (hid,), d(w["final_norm"]), eps).numpy()


@pytest.mark.parametrize("cfg", [TINY, I.with_sizes(TINY, n_kv_heads=4, name="mha"), TINY_MOE],
                         ids=["gqa", "mha", "moe"])
def test_stack_matches_brute_force(cfg):
    w = I.make_weights(cfg, seed=21)
    x = I.make_rows(cfg, 12, seed=22)
    got = Qwen3Oracle(cfg, w, prec="exact").forward(x)
    assert np.max(np.abs(got - _brute_force(cfg, w, x))) < 1e-12


@pytest.mark.parametrize("cfg", [TINY, TINY_MOE], ids=["dense", "moe"])
def test_chunked_prefill_equals_token_by_token_equals_one_pass(cfg):
    w = I.make_weights(cfg, seed=31)
    x = I.make_rows(cfg, 16, seed=32)
    one = Qwen3Oracle(cfg, w, prec="exact").forward(x)
    o = Qwen3Oracle(cfg, w, prec="exact")
    chunked = np.concatenate([o.forward(x[i:i + 4]) for i in range(0, 16, 4)])
    o = Qwen3Oracle(cfg, w, prec="exact")
    tok = np.concatenate([o.forward(x[i:i + 1]) for i in range(16)])
    assert np.max(np.abs(chunked - one)) < 1e-12
    assert np.max(np.abs(tok - one)) < 1e-12


def test_batched_sequences_are_independent():
    """Rows of different sequences in one forward equal separate forwards."""
    cfg = I.with_sizes(TINY, max_seqs=3)
    w = I.make_weights(cfg, seed=41)
    xs = [I.make_rows(cfg, 5, seed=42 + s) for s in range(3)]
    sep = []
    for s in range(3):
        o = Qwen3Oracle(cfg, w, prec="exact")
        sep.append(o.forward(xs[s][:4]))
        sep.append(o.forward(xs[s][4:5]))
    o = Qwen3Oracle(cfg, w, prec="exact")
    for s in range(3):
        o.forward(xs[s][:4], seq_ids=[s] * 4)
    step = o.forward(torch.cat([xs[s][4:5] for s in range(3)]), seq_ids=[0, 1, 2])
    for s in range(3):
        assert np.max(np.abs(step[s] - sep[2 * s + 1][0])) < 1e-12


def test_capacity_and_position_errors_leave_state_unchanged():
    cfg = TINY
    o = Qwen3Oracle(cfg, I.make_weights(cfg, seed=51), prec="exact")
    o.forward(I.make_rows(cfg, 30, seed=52))
    with pytest.raises(ValueError):
        o.forward(I.make_rows(cfg, 3, seed=53))               # 33 > capacity 32
    assert o.length(0) == 30
    with pytest.raises(ValueError):
        o.forward(I.make_rows(cfg, 1, seed=54), positions=[31])
    assert o.length(0) == 30


# ---------------------------------------------------------------- MoE router / experts
def test_router_weights_sum_to_one_and_ties_go_to_lowest_index():
    rng = np.random.default_rng(61)
    for _ in range(50):
        l = rng.standard_normal(128)
        idx, w, P = router_topk(l, 8, True)
        assert abs(w.sum() - 1) < 1e-14
        assert np.all(np.diff(l[idx]) <= 0)
        assert l[idx].min() >= np.delete(l, idx).max()
    l = np.zeros(16)
    l[[3, 5, 9, 12]] = 2.0                      # four-way tie for the top, k = 3
    idx, _, _ = router_topk(l, 3, True)
    assert list(idx) == [3, 5, 9]
    l = np.array([1.0, 5.0, 1.0, 1.0, 0.0])     # tie for the last slot
    idx, _, _ = router_topk(l, 3, False)
    assert list(idx) == [1, 0, 2]


def test_moe_with_all_experts_is_the_full_softmax_mixture():
    """k = E with renormalisation: sum over all experts of softmax(l)_e * expert_e(x)."""
    cfg = I.with_sizes(TINY_MOE, top_k=8, num_layers=1)
    w = I.make_weights(cfg, seed=71)
    o = Qwen3Oracle(cfg, w, prec="exact")
    y2 = np.random.default_rng(72).standard_normal((3, cfg.hidden))
    pend, idx, wt = o.moe_block(0, y2)
    L = o.layers[0]
    P = softmax(y2 @ L["router"]["w"].astype(np.float64).T)
    ref = np.zeros_like(pend)
    mI = cfg.moe_intermediate
    for e in range(cfg.num_experts):
        Wgu = L["exp_gate_up"]["w"][e].astype(np.float64)
        m = silu(y2 @ Wgu[:mI].T) * (y2 @ Wgu[mI:].T)
        ref += P[:, e:e + 1] * (m @ L["exp_down"]["w"][e].astype(np.float64).T)
    assert np.max(np.abs(pend - ref)) < 1e-12


def test_moe_one_expert_reduces_to_dense_mlp_bitwise():
    """E = 1, k = 1: weight 1, so the MoE block is the dense SwiGLU MLP, rounding for
    rounding, when the expert holds the dense weights (bf16 emulation)."""
    cfg = I.with_sizes(TINY, dtype="bf16", num_layers=1)
    w = I.make_weights(cfg, seed=81)
    mcfg = I.with_sizes(cfg, num_experts=1, top_k=1, moe_intermediate=cfg.intermediate)
    L = w["layers"][0]
    wm = {"final_norm": w["final_norm"], "layers": [dict(L)]}
    wm["layers"][0]["router"] = {"w": torch.ones(1, cfg.hidden, dtype=torch.bfloat16)}
    wm["layers"][0]["exp_gate_up"] = {"w": L["gate_up"]["w"][None]}
    wm["layers"][0]["exp_down"] = {"w": L["down"]["w"][None]}
    y2 = rnd(np.random.default_rng(82).standard_normal((4, cfg.hidden)), "bf16")
    dense = Qwen3Oracle(cfg, w).dense_mlp(Qwen3Oracle(cfg, w).layers[0], y2)
    moe, idx, wt = Qwen3Oracle(mcfg, wm).moe_block(0, y2)
    assert np.array_equal(dense, moe) and np.all(idx == 0) and np.all(wt == 1.0)


# ---------------------------------------------------------------- int8
def test_dequant_affine_closed_forms():
    rng = np.random.default_rng(91)
    codes = rng.integers(0, 256, (3, 128))
    scale = rng.uniform(0.001, 0.01, (3, 2))
    bias = rng.uniform(-1, 1, (3, 2))
    W = dequant_affine(codes, scale, bias, 64)
    for o in range(3):
        for i in range(128):
            assert W[o, i] == scale[o, i // 64] * codes[o, i] + bias[o, i // 64]
    mid = dequant_affine(np.full((2, 64), 128), np.full((2, 1), 0.5), np.full((2, 1), -64.0), 64)
    assert np.all(mid == 0.0)


def test_int8_product_regroups_by_group():
    """The int8 linear y = x W^T with W dequantised per group (the int8 export's
    scale * q + bias) equals, by exact algebra, the per-group form
    sum_g scale[n, g] * (x[:, g] . q[n, g]) + bias[n, g] * sum(x[:, g]) -- the
    form the tensor-core int8 GEMM evaluates.  Pinned with an independent fp64
    einsum over the groups (no call to dequant_affine on that side)."""
    rng = np.random.default_rng(93)
    n_out, k, group, m = 5, 256, 64, 7
    codes = rng.integers(0, 256, (n_out, k))
    scale = rng.uniform(0.001, 0.02, (n_out, k // group))
    bias = rng.uniform(-0.5, 0.5, (n_out, k // group))
    x = rng.standard_normal((m, k))
    y = x @ dequant_affine(codes, scale, bias, group).T
    xg = x.reshape(m, k // group, group)
    qg = codes.reshape(n_out, k // group, group).astype(np.float64)
    regrouped = (np.einsum("mgj,ngj,ng->mn", xg, qg, scale) +
                 np.einsum("mgj,ng->mn", xg, bias))
    assert np.allclose(y, regrouped, rtol=1e-12, atol=1e-12)
    # a dropped bias term or a transposed scale would fail:
    assert not np.allclose(y, np.einsum("mgj,ngj,ng->mn", xg, qg, scale), atol=1e-3)


def test_int8_stack_equals_dense_stack_on_dequantised_weights():
    """An int8 stack is the dense stack run on the dequantised matrices."""
    cfg = I.with_sizes(TINY, dtype="bf16", weight_format="int8", group_size=16)
    w = I.make_weights(cfg, seed=101)
    dense = {"final_norm": w["final_norm"], "layers": []}
    for L in w["layers"]:
        D2 = {}
        for k, v in L.items():
            if isinstance(v, dict) and "scale" in v:
                D2[k] = {"w": torch.from_numpy(dequant_affine(
                    v["w"].numpy(), v["scale"].double().numpy(), v["bias"].double().numpy(), 16))}
            else:
                D2[k] = v
        dense["layers"].append(D2)
    x = I.make_rows(cfg, 6, seed=102)
    a = Qwen3Oracle(cfg, w, prec="exact").forward(x)
    b = Qwen3Oracle(I.with_sizes(cfg, weight_format="dense"), dense, prec="exact").forward(x)
    assert np.max(np.abs(a - b)) < 1e-12


# ---------------------------------------------------------------- mixed dense / MoE stacks
@pytest.mark.parametrize("step,mlp_only,expect", [
    (1, (), [0, 1, 2, 3, 4, 5]),
    (2, (), [1, 3, 5]),
    (2, (3,), [1, 5]),
    (3, (0, 2), [5]),
    (1, (0, 1, 2, 3, 4, 5), []),
])
def test_moe_layer_rule(step, mlp_only, expect):
    """qwen3-moe.ts Qwen3MoeDecoderLayer: a layer is sparse iff it is not in
    mlp_only_layers and (index + 1) % decoder_sparse_step == 0 (enumerated by
    hand for six layers); without experts no layer is sparse."""
    cfg = I.with_sizes(TINY_MOE, num_layers=6, decoder_sparse_step=step, mlp_only_layers=mlp_only)
    assert [i for i in range(6) if moe_layer(cfg, i)] == expect
    assert not any(moe_layer(I.with_sizes(cfg, num_experts=0), i) for i in range(6))


MIXED = I.with_sizes(TINY_MOE, name="pin_mixed", num_layers=4, decoder_sparse_step=2, mlp_only_layers=(3,))


def test_mixed_stack_matches_brute_force():
    """A 4-layer stack with decoder_sparse_step 2 and layer 3 kept dense (only
    layer 1 sparse) equals the brute-force forward, which reads each layer's
    kind from the weights it is given."""
    w = I.make_weights(MIXED, seed=23)
    assert ["router" in L for L in w["layers"]] == [False, True, False, False]
    x = I.make_rows(MIXED, 10, seed=24)
    got = Qwen3Oracle(MIXED, w, prec="exact").forward(x)
    assert np.max(np.abs(got - _brute_force(MIXED, w, x))) < 1e-12


def test_oracle_refuses_weights_of_another_schedule():
    w = I.make_weights(MIXED, seed=25)
    other = I.with_sizes(MIXED, mlp_only_layers=())      # layer 3 would be sparse
    with pytest.raises(ValueError):
        Qwen3Oracle(other, w, prec="exact").forward(I.make_rows(MIXED, 2, seed=26))


def test_int8_experts_equal_dense_experts_on_dequantised_weights():
    """int8 experts (stacked affine-quantised matrices, QuantizedSwitchLinear)
    equal the same MoE stack with each expert matrix dequantised explicitly."""
    cfg = I.with_sizes(TINY_MOE, dtype="bf16", weight_format="int8", group_size=16, name="pin_int8_moe")
    w = I.make_weights(cfg, seed=27)
    dense = {"final_norm": w["final_norm"], "layers": []}
    for L in w["layers"]:
        D2 = {}
        for k, v in L.items():
            if isinstance(v, dict) and "scale" in v:
                codes, sc, bi = v["w"].numpy(), v["scale"].double().numpy(), v["bias"].double().numpy()
                if codes.ndim == 3:
                    mats = [dequant_affine(codes[e], sc[e], bi[e], 16) for e in range(codes.shape[0])]
                    D2[k] = {"w": torch.from_numpy(np.stack(mats))}
                else:
                    D2[k] = {"w": torch.from_numpy(dequant_affine(codes, sc, bi, 16))}
            else:
                D2[k] = v
        dense["layers"].append(D2)
    assert w["layers"][0]["exp_gate_up"]["w"].dtype == torch.uint8
    x = I.make_rows(cfg, 7, seed=28)
    a = Qwen3Oracle(cfg, w, prec="exact").forward(x)
    b = Qwen3Oracle(I.with_sizes(cfg, weight_format="dense"), dense, prec="exact").forward(x)
    assert np.max(np.abs(a - b)) < 1e-12


# ---------------------------------------------------------------- embedding, output head, pooling
def test_embed_rows_is_a_row_gather():
    """Backbone.embed_tokens: the table's rows at the ids (torch's embedding)."""
    rng = np.random.default_rng(111)
    table = torch.from_numpy(rng.standard_normal((50, 24))).to(torch.bfloat16)
    ids = [3, 49, 0, 3, 17]
    ref = F.embedding(torch.tensor(ids), table).double().numpy()
    assert np.array_equal(embed_rows(table.double().numpy(), ids, "bf16"), ref)


def test_head_logits_round_once_then_widen():
    """Backbone.cb0_logits: x W^T in the model dtype, then fp32.  A non-square
    head (2049 outputs, as cb0_head) against torch's float64 linear rounded by
    torch's own bf16 cast; a tied head is the product with the embedding table."""
    rng = np.random.default_rng(112)
    x = rnd(rng.standard_normal((3, 64)), "bf16")
    W = rnd(0.05 * rng.standard_normal((2049, 64)), "bf16")
    got = head_logits(x, W, "bf16")
    ref = F.linear(torch.from_numpy(x), torch.from_numpy(W)).to(torch.bfloat16).float().double().numpy()
    assert got.shape == (3, 2049) and np.array_equal(got, ref)
    table = rnd(rng.standard_normal((40, 64)), "bf16")
    tied = head_logits(x, table, "exact")
    assert np.allclose(tied, np.einsum("th,vh->tv", x, table), rtol=0, atol=1e-12)


def test_l2_pool_last_unit_norm_and_torch_ops():
    """qwen3.ts embedPooled: the last row over its L2 norm.  Exact mode: unit
    norm, parallel to the last row, blind to earlier rows and to the row's
    scale.  bf16: the page's four array operations run as torch bf16 ops."""
    rng = np.random.default_rng(113)
    h = rng.standard_normal((5, 64))
    v = l2_pool_last(h, "exact")
    assert abs(np.linalg.norm(v) - 1) < 1e-14 and np.allclose(v, h[-1] / np.linalg.norm(h[-1]), atol=1e-15)
    h2 = h.copy()
    h2[:-1] = 0
    h2[-1] *= 37.0
    assert np.allclose(l2_pool_last(h2, "exact"), v, atol=1e-14)
    hb = rnd(h, "bf16")
    t = torch.from_numpy(hb[-1]).to(torch.bfloat16)
    sq = torch.square(t)
    ss = torch.sum(sq.float()).to(torch.bfloat16)
    ref = (t / torch.sqrt(ss)).double().numpy()
    assert np.array_equal(l2_pool_last(hb, "bf16"), ref)


# ---------------------------------------------------------------- the float32 twin
def test_twin_steps_equal_oracle_steps_to_float32_precision():
    """Qwen3OracleF32Acc restates each step in float32: on non-square random
    inputs every step equals the oracle's float64 step to float32 precision,
    so a dropped term, a wrong sign or a transposed operand in the twin fails."""
    cfg = I.with_sizes(TINY, dtype="fp32")
    w = I.make_weights(cfg, seed=121)
    o, t = Qwen3Oracle(cfg, w, prec="exact"), Qwen3OracleF32Acc(cfg, w, prec="exact")
    rng = np.random.default_rng(122)
    v = rng.standard_normal((6, 64))
    g = 1 + 0.1 * rng.standard_normal(64)
    rel = lambda a, b: np.max(np.abs(a - b)) / np.max(np.abs(b))
    assert rel(t.rms(v, g), o.rms(v, g)) < 1e-6
    x = rng.standard_normal((6, 4, 16))
    c, s = rope_table(50, 16, 1e4, "exact")
    pos = np.array([0, 3, 9, 17, 33, 49])
    assert rel(t.rope(x, c[pos][:, None], s[pos][:, None]), o.rope(x, c[pos][:, None], s[pos][:, None])) < 1e-6
    q, K, V = rng.standard_normal((3, 16)), rng.standard_normal((11, 16)), rng.standard_normal((11, 16))
    vis = np.arange(11)[None, :] <= np.array([4, 7, 10])[:, None]
    assert rel(t.attend(q, K, V, vis, 0.25), o.attend(q, K, V, vis, 0.25)) < 1e-5
    gg = 4 * rng.standard_normal(100)
    assert rel(t.silu(gg), o.silu(gg)) < 1e-6
    A, B = rng.standard_normal((5, 64)), rng.standard_normal((9, 64))
    assert rel(t._mm(A, B), o._mm(A, B)) < 1e-5


def test_twin_bf16_drift_is_zero_on_the_tiny_stack_and_small_in_fp32():
    """On the 2-layer 256-wide workload the twin's bf16 rounding decisions all
    agree with the oracle's (zero drift); in fp32 its distance is float32 noise."""
    for dtype, bound in (("bf16", 0.0), ("fp32", 2e-6)):
        cfg = I.with_sizes(I.TINY_FP32, dtype=dtype)
        w = I.make_weights(cfg, seed=7)
        o, t = Qwen3Oracle(cfg, w), Qwen3OracleF32Acc(cfg, w)
        for n in (16, 1, 1):
            x = I.make_rows(cfg, n, seed=100 + n)
            a, b = o.forward(x), t.forward(x)
            assert np.max(np.abs(a - b)) / np.sqrt(np.mean(a * a)) <= bound

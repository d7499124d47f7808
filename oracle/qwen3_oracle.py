"""CPU oracle for the Qwen3 decoder-stack forward -- TEST INFRASTRUCTURE ONLY.

This file is the slow, plain, obviously-correct statement of what the CUDA
library computes.  Only the tests, ``__graft_entry__.smoke()`` and bench.py's
CPU-baseline leg may import it; the library never does, and it shares no code
with the library (its only common dependency is the seeded input generator,
which holds no arithmetic of the method).

Sources (page titles as the pages give them):

* maya2_mlx/backbone.py, class ``Backbone`` (module docstring, ``forward``,
  ``_rope``, ``reset``): the dense layer, the static KV cache and the exact
  rounding points ("h = h + pend (one rounding)", "RMSNorm: two roundings",
  "RoPE in fp32 on the cos/sin table, one rounding", "attention over keys
  0..pos (fp32 softmax, one rounding)", "silu in fp32 rounded once").
* @mlx-bun/inference qwen3-moe.ts, ``Qwen3MoeSparseMoeBlock.forward`` and
  ``Qwen3SortedExperts`` / ``Qwen3UnsortedExperts``: router softmax over all
  experts, top-k, renormalisation, SwiGLU experts, weighted sum.
* @mlx-bun/inference qwen3.ts, ``Qwen3Attention.forward``: per-head q/k
  RMSNorm over head_dim before RoPE, GQA.
* rlx_flow/blocks/qwen3_decoder.rs, ``Qwen3DecoderStage::emit``: the same op
  order, stated a second time.

Arithmetic is float64 (numpy).  ``prec`` selects where results are rounded:

* ``"exact"``: never rounded, RoPE table in fp64 -- used for invariants.
* ``"fp32"`` / ``"bf16"``: float64 arithmetic rounded (round-to-nearest-even)
  to the model dtype at exactly the Backbone's rounding points.  The GPU is
  compared against this mode.

Readings taken where the pages are silent:
RMSNorm's "two roundings" = round(x * rsqrt(mean(x^2)+eps)) then
round(that * gain); RoPE table inv_freq_i = theta^(-2i/D) rounded to the table
dtype, angle p*inv_freq in fp64, cos/sin rounded to the table dtype, halves
duplicated; half-split (rotate-half) RoPE; query at position p sees keys 0..p of
its own sequence; q head h uses kv head h // (H/KV); router top-k chosen on the
unrounded router logits with ties to the lowest expert index; the MoE weighted
sum accumulates unrounded and is rounded once; int8 codes are unsigned and
dequantise as scale*q + bias (not rounded); a MoE stack's layer is sparse iff
it is not listed in mlp_only_layers and (index + 1) % decoder_sparse_step == 0.

Parity status: every function here is pinned by a CPU test in
``tests/test_oracle_pins.py``; the only unpinned part is which exact rounding
MLX's own Metal kernels apply inside a fused op (e.g. whether RMSNorm rounds
twice or once), which the pages state but which nothing here can run.
"""
from __future__ import annotations

import numpy as np

PRECS = ("exact", "fp32", "bf16")


# --------------------------------------------------------------------------
# rounding
# --------------------------------------------------------------------------
def rnd(x, prec: str):
    """Round float64 values to ``prec`` (round to nearest, ties to even).

    bf16 keeps 8 significant bits and fp32 24; the value is split as
    m * 2**e with 0.5 <= |m| < 1 and m is rounded to the kept bits with
    numpy's rint (ties to even).  Results stay float64.  Values are assumed to
    be in the normal range of the target type (true for every tensor here)."""
    x = np.asarray(x, dtype=np.float64)
    if prec == "exact":
        return x
    bits = {"fp32": 24, "bf16": 8}[prec]
    m, e = np.frexp(x)
    return np.ldexp(np.rint(np.ldexp(m, bits)), e - bits)


# --------------------------------------------------------------------------
# building blocks
# --------------------------------------------------------------------------
def rms_norm(v, gain, eps: float, prec: str):
    """RMSNorm over the last axis with Qwen3's two roundings (Backbone docstring:
    "y = RMSNorm(h) (mx.fast.rms_norm: Qwen3's two roundings)"):
    n = R(v / sqrt(mean(v^2) + eps)), out = R(n * gain)."""
    v = np.asarray(v, dtype=np.float64)
    ms = np.mean(v * v, axis=-1, keepdims=True)
    n = rnd(v / np.sqrt(ms + eps), prec)
    return rnd(n * np.asarray(gain, dtype=np.float64), prec)


def rope_table(capacity: int, head_dim: int, theta: float, prec: str):
    """cos/sin tables [capacity, head_dim] (Backbone.__init__: "in bf16 it is
    built from the bf16-rounded inv_freq buffer ... stored in bf16; the RoPE
    maths reads it as fp32").  inv_freq_i = theta^(-2i/D) for i < D/2, rounded
    to the table dtype; angle = p * inv_freq in float64; cos and sin rounded to
    the table dtype; the two halves of each row repeat the same frequencies."""
    half = head_dim // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = rnd(theta ** (-2.0 * i / head_dim), prec)
    pos = np.arange(capacity, dtype=np.float64)
    ang = np.outer(pos, inv_freq)
    ang = np.concatenate([ang, ang], axis=1)
    return rnd(np.cos(ang), prec), rnd(np.sin(ang), prec)


def rope(x, cos_p, sin_p, prec: str):
    """Rotate-half RoPE (Backbone._rope): with y1 = x[:D/2], y2 = x[D/2:],
    o1 = y1*c[:D/2] - y2*s[:D/2], o2 = y2*c[D/2:] + y1*s[D/2:], computed in
    wide precision and rounded once.  x [..., D]; cos_p/sin_p broadcast to it."""
    x = np.asarray(x, dtype=np.float64)
    half = x.shape[-1] // 2
    y1, y2 = x[..., :half], x[..., half:]
    o1 = y1 * cos_p[..., :half] - y2 * sin_p[..., :half]
    o2 = y2 * cos_p[..., half:] + y1 * sin_p[..., half:]
    return rnd(np.concatenate([o1, o2], axis=-1), prec)


def softmax(s, axis=-1):
    """Exact (float64) softmax; masked entries may be -inf."""
    s = np.asarray(s, dtype=np.float64)
    m = np.max(s, axis=axis, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=axis, keepdims=True)


def attention_probs(q, keys, scale):
    """Softmax over one query's visible keys: P_u = softmax_u(q . k_u * scale)."""
    return softmax(keys @ q * scale)


def silu(g):
    """silu(g) = g / (1 + exp(-g)), the form Backbone.forward writes out."""
    g = np.asarray(g, dtype=np.float64)
    return g / (1.0 + np.exp(-g))


def dequant_affine(codes, scale, bias, group: int):
    """int8 affine group dequantisation: W[o, i] = scale[o, i//group] * q[o, i]
    + bias[o, i//group], q the unsigned code (0..255); float64, not rounded."""
    q = np.asarray(codes, dtype=np.float64)
    s = np.repeat(np.asarray(scale, dtype=np.float64), group, axis=-1)
    b = np.repeat(np.asarray(bias, dtype=np.float64), group, axis=-1)
    return s * q + b


def router_topk(logits, k: int, norm_topk_prob: bool):
    """Qwen3MoeSparseMoeBlock router on one row of logits [E]:
    P = softmax over all experts; the k experts with the largest logits
    (ties to the lowest index) in (score descending, index ascending) order;
    weights P[idx] / sum(P[idx]) when norm_topk_prob, else P[idx].
    Returns (idx [k] int64, w [k] float64, P [E])."""
    logits = np.asarray(logits, dtype=np.float64)
    P = softmax(logits)
    order = np.argsort(-logits, kind="stable")   # stable: equal logits keep index order
    idx = order[:k]
    w = P[idx]
    if norm_topk_prob:
        w = w / np.sum(w)
    return idx.astype(np.int64), w, P


def moe_layer(cfg, layer: int) -> bool:
    """Which layers of a Qwen3-MoE stack carry the sparse block
    (@mlx-bun/inference qwen3-moe.ts, ``Qwen3MoeDecoderLayer``): a layer is MoE
    iff the model has experts, the layer is not in ``mlp_only_layers``, and
    (index + 1) % decoder_sparse_step == 0; every other layer is the dense MLP."""
    if cfg.num_experts <= 0:
        return False
    if layer in tuple(getattr(cfg, "mlp_only_layers", ())):
        return False
    return (layer + 1) % cfg.decoder_sparse_step == 0


def embed_rows(table, ids, prec: str):
    """Embedding lookup (maya2_mlx/backbone.py, ``Backbone.embed_tokens``: the
    rows of the embedding table at the token ids, in the model dtype)."""
    T = np.asarray(table, dtype=np.float64)
    return rnd(T[np.asarray(ids, dtype=np.int64)], prec)


def head_logits(x, W, prec: str):
    """Output head (maya2_mlx/backbone.py, ``Backbone.cb0_logits``: the product
    with the head's [out, hidden] matrix in the model dtype, then widened to
    fp32).  The product is accumulated in float64 and rounded once to the model
    dtype; the widening to fp32 is exact.  A tied head
    (@mlx-bun/inference qwen3.ts, ``embed.asLinear``) passes the embedding
    table as W."""
    return rnd(np.asarray(x, dtype=np.float64) @ np.asarray(W, dtype=np.float64).T, prec)


def l2_pool_last(h, prec: str):
    """Pooled sentence vector (@mlx-bun/inference qwen3.ts, ``embedPooled``):
    the last row of the final-norm hidden states divided by its L2 norm.  The
    page runs square, sum, sqrt and divide as separate array operations in the
    model dtype, so each result is rounded to it: sq = R(v*v), ss = R(sum sq)
    (the sum itself accumulated wide), n = R(sqrt(ss)), out = R(v / n)."""
    v = np.asarray(h, dtype=np.float64)[-1]
    sq = rnd(v * v, prec)
    ss = rnd(np.sum(sq), prec)
    n = rnd(np.sqrt(ss), prec)
    return rnd(v / n, prec)


# --------------------------------------------------------------------------
# the stack
# --------------------------------------------------------------------------
def _f64(t):
    """torch tensor or array -> float64 numpy (exact for bf16/fp32 values)."""
    if hasattr(t, "detach"):
        t = t.detach().cpu()
        if t.dtype.is_floating_point:
            return t.double().numpy()
        return t.numpy()
    return np.asarray(t)


class Qwen3Oracle:
    """Plain forward of the Qwen3 stack (Backbone.forward) with a static
    per-sequence KV cache (Backbone.reset: K/V per layer [kv_heads, capacity,
    head_dim] in the model dtype, plus a length).

    ``cfg``: a Qwen3Config; ``weights``: the dict from inputs.make_weights
    (torch tensors, any device); ``prec``: "exact" or the model dtype name.
    """

    def __init__(self, cfg, weights, prec: str | None = None):
        self.cfg = cfg
        self.prec = cfg.dtype if prec is None else prec
        assert self.prec in PRECS
        self.layers = []
        for L in weights["layers"]:
            self.layers.append({k: ({kk: _store(vv) for kk, vv in v.items()}
                                    if isinstance(v, dict) else _store(v))
                                for k, v in L.items()})
        self.final_norm = _f64(weights["final_norm"])
        table_prec = "exact" if self.prec == "exact" else cfg.dtype
        self.cos, self.sin = rope_table(cfg.capacity, cfg.head_dim, cfg.rope_theta, table_prec)
        self.cache = {}            # seq -> {"K": [L][KV][cap][D], "V": ..., "length": int}

    # -- weights -----------------------------------------------------------
    def linear_weight(self, lw):
        """The float64 [out, in] matrix of one linear (dequantised if int8)."""
        if "scale" in lw:
            return dequant_affine(lw["w"], lw["scale"], lw["bias"], self.cfg.group_size)
        return lw["w"].astype(np.float64)

    def expert_weight(self, lw, e: int):
        """The float64 [out, in] matrix of expert e of a stacked expert linear
        ([E, out, in]; int8 experts dequantise like any int8 linear, as
        qwen3-moe.ts's QuantizedSwitchLinear stacks quantised expert matrices)."""
        if "scale" in lw:
            return dequant_affine(lw["w"][e], lw["scale"][e], lw["bias"][e], self.cfg.group_size)
        return lw["w"][e].astype(np.float64)

    def matmul(self, x, lw):
        """x [T, in] @ W^T, float64 accumulation (Q.mm), not rounded here."""
        return self._mm(x, self.linear_weight(lw))

    def _mm(self, x, W):
        """x @ W^T for an explicit float64 matrix W [out, in]."""
        return np.asarray(x, dtype=np.float64) @ np.asarray(W, dtype=np.float64).T

    # -- cache ---------------------------------------------------------------
    def _seq(self, s: int):
        if s not in self.cache:
            c = self.cfg
            dt = np.float64 if self.prec == "exact" else np.float32
            shape = (c.num_layers, c.n_kv_heads, c.capacity, c.head_dim)
            self.cache[s] = {"K": np.zeros(shape, dt), "V": np.zeros(shape, dt), "length": 0}
        return self.cache[s]

    def reset(self, seq: int | None = None):
        if seq is None:
            self.cache = {}
        else:
            self.cache.pop(seq, None)

    def set_cache(self, seq: int, K, V):
        """Fill positions 0..n-1 of a sequence's cache (K post-RoPE, V raw),
        K/V [layers, kv_heads, n, head_dim]; the sequence length becomes n."""
        c = self._seq(seq)
        K, V = _f64(K), _f64(V)
        n = K.shape[2]
        c["K"][:, :, :n] = K
        c["V"][:, :, :n] = V
        c["length"] = n

    def length(self, seq: int) -> int:
        return self._seq(seq)["length"]

    # -- one forward -----------------------------------------------------------
    def forward(self, x, seq_ids=None, positions=None, return_moe=False, trace=None, taps=None):
        """x [T, hidden] at the given (sequence, position) of each row ->
        final-norm hidden states [T, hidden] (Backbone.forward).  Rows of a
        sequence must continue that sequence's cache (positions
        length, length+1, ...), as Backbone.forward appends at
        length..length+T-1 and raises on overflow.  If ``trace`` is a list,
        each layer appends a dict of its intermediate tensors.  ``taps`` is a
        dict keyed by layer index: each listed layer stores there the residual
        entering it ("h_in"), the residual after its attention ("h"), the MLP's
        input ("y2") and its output ("pend") -- the pieces a one-layer stack
        needs to reproduce it."""
        cfg, R = self.cfg, (lambda a: rnd(a, self.prec))
        x = _f64(x)
        T = x.shape[0]
        if seq_ids is None:
            seq_ids = [0] * T
        seq_ids = [int(s) for s in seq_ids]
        if positions is None:
            base = {}
            positions = []
            for s in seq_ids:
                p = base.get(s, self.length(s))
                positions.append(p)
                base[s] = p + 1
        positions = [int(p) for p in positions]
        nxt = {}
        for s, p in zip(seq_ids, positions):
            expect = nxt.get(s, self.length(s))
            if p != expect:
                raise ValueError(f"row for sequence {s} at position {p}, expected {expect}")
            if p >= cfg.capacity:
                raise ValueError(f"context {p + 1} exceeds capacity {cfg.capacity}")
            nxt[s] = p + 1

        H, KV, D = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
        G = H // KV
        scale = D ** -0.5
        pos = np.array(positions)
        cos_p, sin_p = self.cos[pos][:, None, :], self.sin[pos][:, None, :]
        moe_trace = []

        h = x
        pend = None
        for li, L in enumerate(self.layers):
            if pend is not None:
                h = R(h + pend)                                   # one rounding
            if taps is not None and li in taps:
                taps[li] = {"h_in": h}
            y = self.rms(h, L["in_norm"])
            qkv = R(self.matmul(y, L["qkv"]))
            q = qkv[:, :H * D].reshape(T, H, D)
            k = qkv[:, H * D:(H + KV) * D].reshape(T, KV, D)
            v = qkv[:, (H + KV) * D:].reshape(T, KV, D)
            q = self.rms(q, L["q_norm"])                            # per head, over D
            k = self.rms(k, L["k_norm"])
            q = self.rope(q, cos_p, sin_p)
            k = self.rope(k, cos_p, sin_p)
            # cache append: post-RoPE k and raw v at each row's position
            for t in range(T):
                c = self._seq(seq_ids[t])
                c["K"][li, :, positions[t]] = k[t]
                c["V"][li, :, positions[t]] = v[t]
            # attention: row at position p of sequence s sees keys 0..p of s
            a = np.empty((T, H, D))
            for s in sorted(set(seq_ids)):
                rows = [t for t in range(T) if seq_ids[t] == s]
                rp = np.array([positions[t] for t in rows])
                n_keys = int(rp.max()) + 1
                c = self._seq(s)
                visible = np.arange(n_keys)[None, :] <= rp[:, None]     # [rows, keys]
                for hh in range(H):
                    j = hh // G                                          # GQA: kv head of q head hh
                    Kj = c["K"][li, j, :n_keys].astype(np.float64)
                    Vj = c["V"][li, j, :n_keys].astype(np.float64)
                    a[rows, hh, :] = R(self.attend(q[rows, hh, :], Kj, Vj, visible, scale))
            h = R(h + R(self.matmul(a.reshape(T, H * D), L["o"])))
            y2 = self.rms(h, L["post_norm"])
            if moe_layer(cfg, li):
                if "router" not in L:
                    raise ValueError(f"layer {li} is a MoE layer but its weights have no router")
                pend, idx, w = self.moe_block(li, y2)
                moe_trace.append((idx, w))
            else:
                if "gate_up" not in L:
                    raise ValueError(f"layer {li} is a dense layer but its weights have no MLP")
                pend = self.dense_mlp(L, y2)
            if taps is not None and li in taps:
                taps[li].update(h=h, pend=pend, y2=y2)
            if trace is not None:
                trace.append({"y": y, "qkv": qkv, "q": q, "k": k, "v": v, "a": a,
                              "h": h, "y2": y2, "pend": pend})
        for t in range(T):
            self._seq(seq_ids[t])["length"] = positions[t] + 1
        out = self.rms(R(h + pend), self.final_norm)
        return (out, moe_trace) if return_moe else out

    # -- the steps, one method each (the twin below restates them in float32)
    def rms(self, v, gain):
        return rms_norm(v, gain, self.cfg.rms_eps, self.prec)

    def rope(self, x, cos_p, sin_p):
        return rope(x, cos_p, sin_p, self.prec)

    def attend(self, q, K, V, visible, scale):
        """Unrounded attention output of query rows q [n, D] over keys K, V
        [m, D] with a visibility mask [n, m]: softmax(q K^T * scale) V."""
        S = np.where(visible, (q @ K.T) * scale, -np.inf)
        return softmax(S, axis=-1) @ V

    def silu(self, g):
        return silu(g)

    def dense_mlp(self, L, y2):
        """gu = R(y2 Wgu^T); act = R(silu(g)) in wide precision; pend = R(R(act*u) Wd^T)
        (Backbone.forward: "act = (g / (1.0 + mx.exp(-g))).astype(self.dt)")."""
        R = lambda a: rnd(a, self.prec)
        I = self.cfg.intermediate
        gu = R(self.matmul(y2, L["gate_up"]))
        act = R(self.silu(gu[:, :I]))
        return R(self.matmul(R(act * gu[:, I:]), L["down"]))

    def moe_block(self, li: int, y2):
        """Qwen3MoeSparseMoeBlock.forward on y2 [T, hidden] -> (pend [T, hidden],
        idx [T, k], w [T, k]).  Router logits stay unrounded; each selected
        expert computes m = R(R(silu(R(y2 Wg^T))) * R(y2 Wu^T)), z = R(m Wd^T);
        pend = R(sum_i w_i z_i)."""
        cfg, R = self.cfg, (lambda a: rnd(a, self.prec))
        L = self.layers[li]
        T = y2.shape[0]
        k, mI = cfg.top_k, cfg.moe_intermediate
        logits = self.matmul(y2, L["router"])
        idx = np.zeros((T, k), np.int64)
        w = np.zeros((T, k))
        for t in range(T):
            idx[t], w[t], _ = router_topk(logits[t], k, cfg.norm_topk_prob)
        z = np.zeros((T, k, cfg.hidden))
        # rows are independent: group the (token, slot) pairs by expert
        for e in np.unique(idx):
            tt, ss = np.nonzero(idx == e)
            xe = y2[tt]
            Wgu = self.expert_weight(L["exp_gate_up"], e)
            g = R(self._mm(xe, Wgu[:mI]))
            u = R(self._mm(xe, Wgu[mI:]))
            m = R(R(self.silu(g)) * u)
            z[tt, ss] = R(self._mm(m, self.expert_weight(L["exp_down"], e)))
        pend = R(np.einsum("tk,tkh->th", w, z))
        return pend, idx, w


class Qwen3OracleF32Acc(Qwen3Oracle):
    """The same forward restated in float32 arithmetic -- NOT a reference.

    Every step the pages state in fp32 (RMSNorm statistics, RoPE, the softmax,
    SiLU) and every weight product (NumPy's float32 GEMM) is computed in
    float32 here, rounding to the model dtype at the same points.  Two correct
    implementations of these rounding points that differ only in how they
    compute between them drift apart: a rounding whose exact value lies within
    the arithmetic error of a tie can go either way, and a one-ulp change in
    one input of a wide projection moves every output of the next one.  The
    distance between this class and Qwen3Oracle on the same inputs measures
    that drift, and sets the envelope the GPU's bf16 results are held to."""

    def _mm(self, x, W):
        return (np.asarray(x, dtype=np.float32) @ np.asarray(W, dtype=np.float32).T).astype(np.float64)

    def rms(self, v, gain):
        v32 = np.asarray(v, dtype=np.float32)
        ms = np.mean(v32 * v32, axis=-1, keepdims=True, dtype=np.float32)
        n = rnd((v32 * (np.float32(1.0) / np.sqrt(ms + np.float32(self.cfg.rms_eps)))).astype(np.float64),
                self.prec)
        return rnd((n.astype(np.float32) * np.asarray(gain, dtype=np.float32)).astype(np.float64), self.prec)

    def rope(self, x, cos_p, sin_p):
        x32 = np.asarray(x, dtype=np.float32)
        c, s_ = cos_p.astype(np.float32), sin_p.astype(np.float32)
        half = x32.shape[-1] // 2
        y1, y2 = x32[..., :half], x32[..., half:]
        o = np.concatenate([y1 * c[..., :half] - y2 * s_[..., :half],
                            y2 * c[..., half:] + y1 * s_[..., half:]], axis=-1)
        return rnd(o.astype(np.float64), self.prec)

    def attend(self, q, K, V, visible, scale):
        S = (np.asarray(q, np.float32) @ np.asarray(K, np.float32).T) * np.float32(scale)
        S = np.where(visible, S, np.float32(-np.inf))
        P = np.exp(S - S.max(axis=-1, keepdims=True))
        out = (P @ np.asarray(V, np.float32)) / P.sum(axis=-1, keepdims=True, dtype=np.float32)
        return out.astype(np.float64)

    def silu(self, g):
        g32 = np.asarray(g, dtype=np.float32)
        return (g32 / (np.float32(1.0) + np.exp(-g32))).astype(np.float64)


def _store(t):
    """Weights are kept in their exact stored values: float32 numpy for
    bf16/fp32 tensors (lossless), the raw integers for int8 codes."""
    if hasattr(t, "detach"):
        t = t.detach().cpu()
        if t.dtype.is_floating_point:
            return t.float().numpy()
        return t.numpy()
    return np.asarray(t)

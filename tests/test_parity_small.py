"""GPU parity on small stacks: the CUDA library through the C ABI against the
CPU oracle, element by element, on the same seeded inputs.  Sizes span several
kernel tiles with ragged tails and cover both the decode (GEMV) and the
prefill (GEMM) plans.  Bounds are those of gpu_helpers (fp32 1e-4; bf16 2e-2
or the measured bf16 drift envelope, which is zero on most of these sizes)."""
import numpy as np
import pytest
import torch

from gpu_helpers import TOL, Parity, bf16_ulp, rel_err, to_device, as_f64
from oracle import Qwen3Oracle
from qwen3_decoder_layer_gb300 import binding as Q
from qwen3_decoder_layer_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TINY_BF16 = I.with_sizes(I.TINY_FP32, name="tiny_bf16", dtype="bf16")
SMALL_D128 = I.with_sizes(I.TINY_FP32, name="small_d128", dtype="bf16", hidden=512, n_heads=4,
                          n_kv_heads=2, head_dim=128, intermediate=1088, capacity=300, num_layers=3)
SMALL_MOE = I.with_sizes(I.MOE_A3B_4LAYER, name="small_moe", num_layers=2, hidden=256, n_heads=8,
                         n_kv_heads=1, head_dim=64, num_experts=32, top_k=4, moe_intermediate=128,
                         capacity=128)
SMALL_INT8 = I.with_sizes(SMALL_D128, name="small_int8", weight_format="int8", group_size=64)


def _prefill_decode(cfg, n_prefill, n_decode, seed):
    p = Parity(cfg, seed=seed)
    p.step(I.make_rows(cfg, n_prefill, seed=seed + 1).cuda())
    for s in range(n_decode):
        p.step(I.make_rows(cfg, 1, seed=seed + 100 + s).cuda())
    p.close()
    return p.check()


def test_tiny_fp32_prefill_then_decode(cuda_ok):
    """The tiny fp32 workload exactly: 16-row prefill, then 16 single-row decode steps."""
    _prefill_decode(I.TINY_FP32, 16, 16, seed=1000)


def test_tiny_bf16_prefill_then_decode(cuda_ok):
    _prefill_decode(TINY_BF16, 16, 8, seed=1100)


@pytest.mark.parametrize("n_prefill", [1, 3, 4, 5, 37, 130])
def test_d128_row_counts(cuda_ok, n_prefill):
    """Row counts around the GEMV/GEMM switch (4|5), ragged GEMM tiles (37, 130),
    head_dim 128, three layers, then decode steps."""
    _prefill_decode(SMALL_D128, n_prefill, 3, seed=1200 + n_prefill)


@pytest.mark.parametrize("n_prefill", [4, 37])
def test_fp32_d128_strict(cuda_ok, n_prefill):
    _prefill_decode(I.with_sizes(SMALL_D128, dtype="fp32"), n_prefill, 3, seed=1300 + n_prefill)


TC_CFG = I.with_sizes(SMALL_D128, name="tc_d128", intermediate=1024, capacity=400)


@pytest.mark.parametrize("T", [40, 128, 130, 256])
def test_tensor_core_gemm_prefill(cuda_ok, T):
    """Prefill with every linear on the tcgen05 GEMM (T=130 leaves a ragged
    2-row tile; T=40 and 128 fit one row tile, where o_proj, gate|up and down
    split k over the SMs and a second kernel adds the partial tiles): within
    the bound of the oracle, and within the same bound of the CUDA-core GEMM
    path run on the same inputs."""
    w = I.make_weights(TC_CFG, seed=1350 + T)
    wd = to_device(w)
    x = I.make_rows(TC_CFG, T, seed=1351).cuda()
    p = Parity(TC_CFG, weights=w, device_weights=wd)
    tc, _ = p.step(x)
    p.check()
    simt = Q.Qwen3Stack(TC_CFG, wd)
    Q.qwen3_set_option(simt.h, Q.QWEN3_OPT_TENSOR_CORES, 0)
    ref_simt = simt.forward(x)
    assert rel_err(tc, ref_simt) <= p.bound()
    assert Q.qwen3_device_error(p.stack.h) == 0
    simt.close()
    p.close()


QKV_CFG = I.with_sizes(SMALL_D128, name="qkv_rope_d128", hidden=1024, n_heads=16, n_kv_heads=8,
                       intermediate=1024, capacity=1300, num_layers=1)


def test_qkv_rope_epilogue_ragged(cuda_ok):
    """1220 rows: 10 row tiles (the last one 68 rows) x 16 column tiles fill a
    wave, so the q/k RMSNorm, RoPE and cache append run in the q|k|v GEMM's
    epilogue; against the oracle, and the cached keys and values against the
    CUDA-core path's."""
    T = 1220
    w = I.make_weights(QKV_CFG, seed=1370)
    wd = to_device(w)
    x = I.make_rows(QKV_CFG, T, seed=1371).cuda()
    p = Parity(QKV_CFG, weights=w, device_weights=wd)
    tc, _ = p.step(x)
    p.check()
    simt = Q.Qwen3Stack(QKV_CFG, wd)
    Q.qwen3_set_option(simt.h, Q.QWEN3_OPT_TENSOR_CORES, 0)
    ref_simt = simt.forward(x)
    torch.cuda.synchronize()
    k_tc, v_tc = Q.cache_tensors(p.stack.h, QKV_CFG, 0, 0)
    k_ref, v_ref = Q.cache_tensors(simt.h, QKV_CFG, 0, 0)
    # two GPU paths with different fp32 summation orders: each element within
    # 2e-2 of the rms or 4 bf16 ulps of itself (a rounding step apart)
    for got, ref in ((tc, ref_simt), (k_tc[:, :T], k_ref[:, :T]), (v_tc[:, :T], v_ref[:, :T])):
        g, r = as_f64(got), as_f64(ref)
        allow = np.maximum(TOL["bf16"] * np.sqrt(np.mean(r * r)), 4 * bf16_ulp(r, g))
        assert np.all(np.abs(g - r) <= allow)
    assert Q.qwen3_device_error(p.stack.h) == 0
    simt.close()
    p.close()


def test_chunked_prefill_matches_one_pass(cuda_ok):
    """One 96-row prefill, four 24-row chunks and 96 single rows: each against the
    oracle, and the chunked GPU run against the one-pass GPU run."""
    cfg = SMALL_D128
    w = I.make_weights(cfg, seed=1400)
    wd = to_device(w)
    x = I.make_rows(cfg, 96, seed=1401).cuda()
    runs = [Parity(cfg, weights=w, device_weights=wd) for _ in range(3)]
    one, _ = runs[0].step(x)
    chunks = torch.cat([runs[1].step(x[i:i + 24])[0] for i in range(0, 96, 24)])
    toks = torch.cat([runs[2].step(x[i:i + 1])[0] for i in range(96)])
    for p in runs:
        p.check()
        p.close()
    assert rel_err(chunks, one) <= runs[0].bound()
    assert rel_err(toks, one) <= runs[0].bound()


def test_batched_sequences_with_cached_context(cuda_ok):
    """Several sequences at different lengths in one decode call, then a
    multi-row call that mixes sequences (3 rows of one, 2 of another)."""
    cfg = I.with_sizes(SMALL_D128, max_seqs=4)
    p = Parity(cfg, seed=1500)
    for s, n in enumerate([7, 150, 64, 250]):
        p.fill_cache(s, n, seed=1510 + s)
    for step in range(3):
        p.step(I.make_rows(cfg, 4, seed=1520 + step).cuda(), seq_ids=[0, 1, 2, 3])
    p.step(I.make_rows(cfg, 5, seed=1530).cuda(), seq_ids=[2, 2, 2, 0, 0])
    p.close()
    p.check()


@pytest.mark.parametrize("T", [1, 3, 24])
def test_moe_stack(cuda_ok, T):
    """MoE layers: unsorted (gathered GEMV) experts for few rows, sorted grouped
    GEMMs from ceil(64/top_k) rows."""
    p = Parity(SMALL_MOE, seed=1600 + T)
    p.step(I.make_rows(SMALL_MOE, T, seed=1601).cuda())
    p.step(I.make_rows(SMALL_MOE, 1, seed=1602).cuda())
    p.close()
    p.check()


def moe_layer_check(cfg, stack, orc, layer, y):
    """Run qwen3_moe_layer on y and compare with the oracle's MoE block: top-k
    experts bit-exact wherever the k-th / (k+1)-th logit margin exceeds
    1e-4 * rms(logits) (others must be a valid top-k within that margin);
    weights to 1e-5; the block output within the bf16 bound."""
    T = y.shape[0]
    out = torch.empty_like(y)
    idx = torch.empty(T, cfg.top_k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, cfg.top_k, dtype=torch.float32, device="cuda")
    Q.qwen3_moe_layer(stack.h, layer, y, out, idx, w)
    torch.cuda.synchronize()
    yd = as_f64(y)
    pend, ridx, rw = orc.moe_block(layer, yd)
    logits = yd @ orc.layers[layer]["router"]["w"].astype(np.float64).T
    srt = -np.sort(-logits, axis=1)
    margin = srt[:, cfg.top_k - 1] - srt[:, cfg.top_k]
    tol = 1e-4 * np.sqrt(np.mean(logits ** 2, axis=1))
    clear = margin > tol
    gi = idx.cpu().numpy()
    assert np.array_equal(gi[clear], ridx[clear])
    for t in np.nonzero(~clear)[0]:           # near-ties: any valid top-k set
        kth = srt[t, cfg.top_k - 1]
        assert np.all(logits[t, gi[t]] >= kth - tol[t])
        assert len(set(gi[t])) == cfg.top_k
    assert np.max(np.abs(w.cpu().numpy()[clear] - rw[clear])) < 1e-5
    return rel_err(out, pend), clear.mean()


@pytest.mark.parametrize("T", [2, 40])
def test_moe_layer_indices_bit_exact(cuda_ok, T):
    p = Parity(SMALL_MOE, seed=1700 + T, twin=False)
    err, clear = moe_layer_check(SMALL_MOE, p.stack, p.orc, 0, I.make_rows(SMALL_MOE, T, seed=1701).cuda())
    assert clear > 0.9 and err <= TOL["bf16"]
    p.close()


def test_moe_exact_tie_goes_to_lower_index(cuda_ok):
    """Experts 5, 9 and 20 get identical router rows, so their logits are
    bitwise equal on the GPU; 5 must be chosen before 9 and 20."""
    cfg = I.with_sizes(SMALL_MOE, num_layers=1)
    w = I.make_weights(cfg, seed=1800)
    r = w["layers"][0]["router"]["w"]
    r[9] = r[5]
    r[20] = r[5]
    stack = Q.Qwen3Stack(cfg, to_device(w))
    y = I.make_rows(cfg, 64, seed=1801).cuda()
    idx = torch.empty(64, cfg.top_k, dtype=torch.int32, device="cuda")
    wt = torch.empty(64, cfg.top_k, dtype=torch.float32, device="cuda")
    Q.qwen3_moe_layer(stack.h, 0, y, torch.empty_like(y), idx, wt)
    seen = 0
    for row in idx.cpu().numpy():
        s = list(row)
        for e in (9, 20):
            if e in s:
                seen += 1
                assert 5 in s and s.index(5) < s.index(e)
    assert seen > 0
    stack.close()


@pytest.mark.parametrize("n_prefill", [2, 9, 24, 40])
def test_int8_weights(cuda_ok, n_prefill):
    """int8 weights through every linear path: the decode GEMV (2 rows), the
    tensor-core int8 GEMM for up to 32 rows (9, 24; the intermediate size 1088
    leaves a ragged last tile, and the narrow linears split K over CTAs) and
    the tiled skinny GEMM (40 rows), then two decode steps."""
    _prefill_decode(SMALL_INT8, n_prefill, 2, seed=1900 + n_prefill)


@pytest.mark.parametrize("n_prefill", [9, 24])
def test_int8_weights_cuda_cores(cuda_ok, n_prefill):
    """The same rows with tensor cores switched off: the CUDA-core int8 GEMM."""
    p = Parity(SMALL_INT8, seed=1950 + n_prefill)
    Q.qwen3_set_option(p.stack.h, Q.QWEN3_OPT_TENSOR_CORES, 0)
    p.step(I.make_rows(SMALL_INT8, n_prefill, seed=1951 + n_prefill).cuda())
    p.step(I.make_rows(SMALL_INT8, 1, seed=1952 + n_prefill).cuda())
    p.close()
    p.check()


@pytest.mark.parametrize("opts", [{"CUDA_GRAPHS": 0, "PDL": 0}, {"CUDA_GRAPHS": 0}, {"PDL": 0},
                                  {"L2_PREFETCH": 1}, {"L2_PREFETCH": 2}, {"GEMV_CORESIDENT": 1}],
                         ids=["direct", "direct_pdl", "graph_no_pdl", "prefetch1", "prefetch2", "coresident"])
def test_launch_options_do_not_change_results(cuda_ok, opts):
    """CUDA-graph replay, programmatic dependent launch, L2 prefetch and the
    GEMV block size change scheduling only: results are bitwise equal to the
    default; options switched on a live handle take effect (its captured
    graphs are dropped)."""
    cfg = SMALL_D128
    wd = to_device(I.make_weights(cfg, seed=2000))
    xs = [I.make_rows(cfg, n, seed=2001 + i).cuda() for i, n in enumerate([9, 1, 1, 2, 1])]
    outs = []
    for o in [{}, opts]:
        s = Q.Qwen3Stack(cfg, wd)
        s.forward(xs[0])                       # a graph-free prefill, then switch on the live handle
        Q.qwen3_reset(s.h, 0)
        for k, v in o.items():
            Q.qwen3_set_option(s.h, getattr(Q, "QWEN3_OPT_" + k), v)
        outs.append([s.forward(x).clone() for x in xs])
        s.close()
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_errors_leave_state_unchanged(cuda_ok):
    """Capacity overflow, a position gap, a bad or split sequence: each returns its
    status before any launch, the lengths stay put, the output is untouched, and
    the next valid call still matches the oracle."""
    cfg = I.with_sizes(TINY_BF16, capacity=20, max_seqs=2)
    p = Parity(cfg, seed=2100)
    p.step(I.make_rows(cfg, 18, seed=2101).cuda())
    out = torch.zeros(3, cfg.hidden, dtype=torch.bfloat16, device="cuda")
    x3 = I.make_rows(cfg, 3, seed=2102).cuda()
    cases = [([0, 0, 0], [18, 19, 20], 3), ([0, 0, 0], [17, 18, 19], 4), ([0, 2, 0], [18, 0, 19], 5),
             ([0, 1, 0], [18, 0, 19], 5)]
    for sids, pos, status in cases:
        with pytest.raises(Q.Qwen3Error) as e:
            Q.qwen3_forward(p.stack.h, x3, sids, pos, out)
        assert e.value.status == status
        assert Q.qwen3_get_length(p.stack.h, 0) == 18 and Q.qwen3_get_length(p.stack.h, 1) == 0
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0
    p.step(I.make_rows(cfg, 2, seed=2103).cuda())
    assert Q.qwen3_get_length(p.stack.h, 0) == 20
    p.close()
    p.check()


def test_fill_to_capacity_then_overflow(cuda_ok):
    cfg = I.with_sizes(TINY_BF16, capacity=24)
    p = Parity(cfg, seed=2150)
    p.step(I.make_rows(cfg, 23, seed=2151).cuda())
    p.step(I.make_rows(cfg, 1, seed=2152).cuda())          # position 23: the last one
    with pytest.raises(Q.Qwen3Error) as e:
        p.stack.forward(I.make_rows(cfg, 1, seed=2153).cuda())
    assert e.value.status == 3
    p.close()
    p.check()


def test_reset_then_reuse(cuda_ok):
    cfg = TINY_BF16
    wd = to_device(I.make_weights(cfg, seed=2200))
    stack = Q.Qwen3Stack(cfg, wd)
    x = I.make_rows(cfg, 6, seed=2201).cuda()
    first = stack.forward(x).clone()
    stack.forward(I.make_rows(cfg, 3, seed=2202).cuda())
    Q.qwen3_reset(stack.h, 0)
    assert Q.qwen3_get_length(stack.h, 0) == 0
    assert torch.equal(stack.forward(x), first)
    stack.close()


@pytest.mark.parametrize("cfg", [SMALL_D128, I.with_sizes(SMALL_D128, dtype="fp32"), SMALL_MOE],
                         ids=["bf16", "fp32", "moe_g8"])
@pytest.mark.parametrize("cluster", [1, 0])
def test_decode_attention_cluster_and_split_k(cuda_ok, cfg, cluster):
    """Decode attention of few query blocks runs on thread-block clusters
    (partials merged through distributed shared memory) unless switched off
    (split-K with the global merge): both against the oracle, at contexts
    from one key to a few hundred, one to four rows per sequence."""
    cfg = I.with_sizes(cfg, max_seqs=3, capacity=400)
    p = Parity(cfg, seed=2400 + cluster)
    Q.qwen3_set_option(p.stack.h, Q.QWEN3_OPT_CLUSTER_ATTENTION, cluster)
    p.step(I.make_rows(cfg, 1, seed=2401).cuda(), seq_ids=[0])                       # one key
    p.fill_cache(1, 333, seed=2402)
    p.fill_cache(2, 64, seed=2403)
    for i, sids in enumerate([[1], [2], [0, 1], [1, 1, 1], [0, 1, 2], [2, 2, 2, 2], [1]]):
        p.step(I.make_rows(cfg, len(sids), seed=2410 + i).cuda(), seq_ids=sids)
    p.close()
    p.check()

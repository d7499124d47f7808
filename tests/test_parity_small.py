"""GPU parity on small stacks: the CUDA library through the C ABI against the
CPU oracle, element by element, on the same seeded inputs.  Sizes span several
kernel tiles with ragged tails and cover both the decode (GEMV) and the
prefill (GEMM) plans.

Error metric: max|gpu - oracle| / rms(oracle) of the final-norm output,
<= 1e-4 in fp32 and <= 2e-2 in bf16."""
import numpy as np
import pytest
import torch

from gpu_helpers import TOL, fill_cache, make_pair, rel_err
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


def _run_prefill_decode(cfg, n_prefill, n_decode, seed):
    stack, orc = make_pair(cfg, seed=seed)
    errs = []
    x = I.make_rows(cfg, n_prefill, seed=seed + 1).cuda()
    out = stack.forward(x)
    errs.append(rel_err(out, orc.forward(x.cpu())))
    for s in range(n_decode):
        x = I.make_rows(cfg, 1, seed=seed + 100 + s).cuda()
        out = stack.forward(x)
        errs.append(rel_err(out, orc.forward(x.cpu())))
    stack.close()
    return errs


def test_tiny_fp32_prefill_then_decode(cuda_ok):
    """The tiny fp32 workload exactly: 16-row prefill, then 16 single-row decode steps."""
    errs = _run_prefill_decode(I.TINY_FP32, 16, 16, seed=1000)
    assert max(errs) <= TOL["fp32"], errs


def test_tiny_bf16_prefill_then_decode(cuda_ok):
    errs = _run_prefill_decode(TINY_BF16, 16, 8, seed=1100)
    assert max(errs) <= TOL["bf16"], errs


@pytest.mark.parametrize("n_prefill", [1, 3, 4, 5, 37, 130])
def test_d128_row_counts(cuda_ok, n_prefill):
    """Row counts around the GEMV/GEMM switch (4|5), a ragged GEMM tile (37, 130),
    head_dim 128, three layers, then decode steps."""
    errs = _run_prefill_decode(SMALL_D128, n_prefill, 3, seed=1200 + n_prefill)
    assert max(errs) <= TOL["bf16"], errs


def test_fp32_d128_strict(cuda_ok):
    cfg = I.with_sizes(SMALL_D128, dtype="fp32")
    errs = _run_prefill_decode(cfg, 37, 3, seed=1300)
    assert max(errs) <= TOL["fp32"], errs


def test_chunked_prefill_matches_one_pass(cuda_ok):
    cfg = SMALL_D128
    w = I.make_weights(cfg, seed=1400)
    from gpu_helpers import to_device
    wd = to_device(w)
    x = I.make_rows(cfg, 96, seed=1401).cuda()
    a = Q.Qwen3Stack(cfg, wd)
    one = a.forward(x)
    b = Q.Qwen3Stack(cfg, wd)
    chunks = torch.cat([b.forward(x[i:i + 24]) for i in range(0, 96, 24)])
    c = Q.Qwen3Stack(cfg, wd)
    toks = torch.cat([c.forward(x[i:i + 1]) for i in range(96)])
    ref = Qwen3Oracle(cfg, w).forward(x.cpu())
    assert rel_err(one, ref) <= TOL["bf16"]
    assert rel_err(chunks, ref) <= TOL["bf16"]
    assert rel_err(toks, ref) <= TOL["bf16"]
    assert rel_err(chunks, one.float().cpu().double().numpy()) <= TOL["bf16"]
    for s in (a, b, c):
        s.close()


def test_batched_sequences_with_cached_context(cuda_ok):
    """Several sequences at different lengths in one decode call (and a
    multi-row verify-style call), against the oracle."""
    cfg = I.with_sizes(SMALL_D128, max_seqs=4)
    stack, orc = make_pair(cfg, seed=1500)
    lens = [7, 150, 64, 250]
    for s, n in enumerate(lens):
        fill_cache(stack, orc, s, n, seed=1510 + s)
    for step in range(3):
        x = I.make_rows(cfg, 4, seed=1520 + step).cuda()
        out = stack.forward(x, seq_ids=[0, 1, 2, 3])
        assert rel_err(out, orc.forward(x.cpu(), seq_ids=[0, 1, 2, 3])) <= TOL["bf16"]
    # three rows for sequence 2 and two for sequence 0 in one call
    x = I.make_rows(cfg, 5, seed=1530).cuda()
    sids = [2, 2, 2, 0, 0]
    out = stack.forward(x, seq_ids=sids)
    assert rel_err(out, orc.forward(x.cpu(), seq_ids=sids)) <= TOL["bf16"]
    stack.close()


@pytest.mark.parametrize("T", [1, 3, 24])
def test_moe_stack(cuda_ok, T):
    """MoE layers: unsorted (gathered GEMV) experts for few rows, sorted grouped
    GEMMs from ceil(64/top_k) rows."""
    stack, orc = make_pair(SMALL_MOE, seed=1600 + T)
    x = I.make_rows(SMALL_MOE, T, seed=1601).cuda()
    assert rel_err(stack.forward(x), orc.forward(x.cpu())) <= TOL["bf16"]
    x = I.make_rows(SMALL_MOE, 1, seed=1602).cuda()
    assert rel_err(stack.forward(x), orc.forward(x.cpu())) <= TOL["bf16"]
    stack.close()


@pytest.mark.parametrize("T", [2, 40])
def test_moe_layer_indices_bit_exact(cuda_ok, T):
    """qwen3_moe_layer: top-k experts equal the oracle's wherever the k-th / (k+1)-th
    logit margin exceeds 1e-4 * rms(logits) (expected: every row)."""
    cfg = SMALL_MOE
    stack, orc = make_pair(cfg, seed=1700 + T)
    y = I.make_rows(cfg, T, seed=1701).cuda()
    out = torch.empty_like(y)
    idx = torch.empty(T, cfg.top_k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, cfg.top_k, dtype=torch.float32, device="cuda")
    Q.qwen3_moe_layer(stack.h, 0, y, out, idx, w)
    torch.cuda.synchronize()
    pend, ridx, rw = orc.moe_block(0, y.cpu().double().numpy())
    logits = y.cpu().double().numpy() @ orc.layers[0]["router"]["w"].astype(np.float64).T
    srt = -np.sort(-logits, axis=1)
    margin = srt[:, cfg.top_k - 1] - srt[:, cfg.top_k]
    clear = margin > 1e-4 * np.sqrt(np.mean(logits ** 2, axis=1))
    assert clear.mean() > 0.9
    assert np.array_equal(idx.cpu().numpy()[clear], ridx[clear])
    assert np.max(np.abs(w.cpu().numpy()[clear] - rw[clear])) < 1e-5
    assert rel_err(out, pend) <= TOL["bf16"]
    stack.close()


def test_moe_exact_tie_goes_to_lower_index(cuda_ok):
    """Two experts with identical router rows give bitwise-equal logits on the
    GPU; the lower index must be chosen first."""
    cfg = I.with_sizes(SMALL_MOE, num_layers=1)
    w = I.make_weights(cfg, seed=1800)
    r = w["layers"][0]["router"]["w"]
    r[9] = r[5]
    r[20] = r[5]
    from gpu_helpers import to_device
    stack = Q.Qwen3Stack(cfg, to_device(w))
    y = I.make_rows(cfg, 64, seed=1801).cuda()
    idx = torch.empty(64, cfg.top_k, dtype=torch.int32, device="cuda")
    wt = torch.empty(64, cfg.top_k, dtype=torch.float32, device="cuda")
    Q.qwen3_moe_layer(stack.h, 0, y, torch.empty_like(y), idx, wt)
    got = idx.cpu().numpy()
    for row in got:
        s = list(row)
        for e in (9, 20):
            if e in s:
                assert 5 in s and s.index(5) < s.index(e)
    stack.close()


@pytest.mark.parametrize("n_prefill", [2, 40])
def test_int8_weights(cuda_ok, n_prefill):
    errs = _run_prefill_decode(SMALL_INT8, n_prefill, 2, seed=1900 + n_prefill)
    assert max(errs) <= TOL["bf16"], errs


@pytest.mark.parametrize("graphs,pdl", [(0, 0), (0, 1), (1, 0)])
def test_launch_options_do_not_change_results(cuda_ok, graphs, pdl):
    """CUDA-graph replay and programmatic dependent launch change scheduling only."""
    cfg = SMALL_D128
    from gpu_helpers import to_device
    wd = to_device(I.make_weights(cfg, seed=2000))
    xs = [I.make_rows(cfg, n, seed=2001 + i).cuda() for i, n in enumerate([9, 1, 1, 2, 1])]
    outs = []
    for opt in [(1, 1), (graphs, pdl)]:
        s = Q.Qwen3Stack(cfg, wd)
        Q.qwen3_set_option(s.h, Q.QWEN3_OPT_CUDA_GRAPHS, opt[0])
        Q.qwen3_set_option(s.h, Q.QWEN3_OPT_PDL, opt[1])
        outs.append([s.forward(x).clone() for x in xs])
        s.close()
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_errors_leave_state_unchanged(cuda_ok):
    """Capacity overflow, a position gap, a bad or split sequence: each returns its
    status before any launch, the lengths stay put, and the next valid call
    still matches the oracle."""
    cfg = I.with_sizes(TINY_BF16, capacity=20, max_seqs=2)
    stack, orc = make_pair(cfg, seed=2100)
    x = I.make_rows(cfg, 18, seed=2101).cuda()
    stack.forward(x)
    orc.forward(x.cpu())
    out = torch.zeros(3, cfg.hidden, dtype=torch.bfloat16, device="cuda")
    x3 = I.make_rows(cfg, 3, seed=2102).cuda()
    cases = [([0, 0, 0], [18, 19, 20], 3), ([0, 0, 0], [17, 18, 19], 4), ([0, 2, 0], [18, 0, 19], 5),
             ([0, 1, 0], [18, 0, 19], 5)]
    for sids, pos, status in cases:
        with pytest.raises(Q.Qwen3Error) as e:
            Q.qwen3_forward(stack.h, x3, sids, pos, out)
        assert e.value.status == status
        assert Q.qwen3_get_length(stack.h, 0) == 18 and Q.qwen3_get_length(stack.h, 1) == 0
    assert torch.count_nonzero(out) == 0
    x2 = I.make_rows(cfg, 2, seed=2103).cuda()
    assert rel_err(stack.forward(x2), orc.forward(x2.cpu())) <= TOL["bf16"]
    assert Q.qwen3_get_length(stack.h, 0) == 20
    stack.close()


def test_reset_then_reuse(cuda_ok):
    cfg = TINY_BF16
    stack, _ = make_pair(cfg, seed=2200)
    x = I.make_rows(cfg, 6, seed=2201).cuda()
    first = stack.forward(x).clone()
    stack.forward(I.make_rows(cfg, 3, seed=2202).cuda())
    Q.qwen3_reset(stack.h, 0)
    assert Q.qwen3_get_length(stack.h, 0) == 0
    assert torch.equal(stack.forward(x), first)
    stack.close()

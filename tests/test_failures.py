"""Bounds and failure handling on the GPU, without faulting or hanging it:

* nothing reads a sequence's cache past its length: with NaN written into
  every position a sequence does not hold, every kernel path gives results
  bitwise equal to a run over a zeroed cache (this stands in for a memory
  checker);
* an allocation that fails (injected through QWEN3_OPT_FAIL_ALLOC) returns
  QWEN3_E_OOM before any state changes, and the next call works;
* a bounded device wait that runs out records its code for
  qwen3_device_error and the context stays usable."""
import numpy as np
import pytest
import torch

from gpu_helpers import Parity, to_device
from qwen3_decoder_layer_gb300 import binding as Q
from qwen3_decoder_layer_gb300 import inputs as I

pytestmark = pytest.mark.gpu

SMALL_D128 = I.with_sizes(I.TINY_FP32, name="fail_d128", dtype="bf16", hidden=512, n_heads=4, n_kv_heads=2,
                          head_dim=128, intermediate=1024, capacity=400, num_layers=3, max_seqs=3)
SMALL_MOE = I.with_sizes(I.MOE_A3B_4LAYER, name="fail_moe", num_layers=2, hidden=256, n_heads=8, n_kv_heads=1,
                         head_dim=64, num_experts=32, top_k=4, moe_intermediate=128, capacity=200, max_seqs=3)


def _poison(stack, cfg):
    """NaN in every cache position of every sequence and layer."""
    nan = float("nan")
    for s in range(cfg.max_seqs):
        for l in range(cfg.num_layers):
            k, v = Q.cache_tensors(stack.h, cfg, s, l)
            k.fill_(nan)
            v.fill_(nan)
    torch.cuda.synchronize()


def _script(cfg, seed):
    """Calls touching every attention path: a ragged prefill (tensor-core
    attention for bf16, 130 rows = a 2-row last tile), decode rows of one and
    of several sequences, a verify window, a second prefill chunk."""
    g = lambda n, k: I.make_rows(cfg, n, seed=seed + k).cuda()
    return [(g(130, 1), [0] * 130), (g(1, 2), [0]), (g(37, 3), [1] * 37), (g(2, 4), [0, 1]),
            (g(8, 5), [0] * 4 + [1] * 4), (g(9, 6), [2] * 9), (g(3, 7), [0, 1, 2]), (g(1, 8), [2])]


@pytest.mark.parametrize("cfg", [SMALL_D128, I.with_sizes(SMALL_D128, dtype="fp32", name="fail_f32"),
                                 I.with_sizes(SMALL_D128, weight_format="int8", group_size=64, name="fail_int8"),
                                 SMALL_MOE], ids=["bf16", "fp32", "int8", "moe"])
def test_nan_in_the_cache_tail_is_never_read(cuda_ok, cfg):
    wd = to_device(I.make_weights(cfg, seed=5000))
    clean, dirty = Q.Qwen3Stack(cfg, wd), Q.Qwen3Stack(cfg, wd)
    _poison(dirty, cfg)
    for x, sids in _script(cfg, 5001):
        a, b = clean.forward(x, seq_ids=sids), dirty.forward(x, seq_ids=sids)
        torch.cuda.synchronize()
        assert not torch.isnan(b).any(), f"NaN reached the output ({len(sids)} rows)"
        assert torch.equal(a, b), f"{len(sids)} rows: results depend on the cache past the length"
    assert Q.qwen3_device_error(dirty.h) == 0
    clean.close()
    dirty.close()


def test_nan_tail_after_a_synthetic_prefix(cuda_ok):
    """A cache filled through qwen3_cache_view to a length, NaN beyond it."""
    cfg = I.with_sizes(SMALL_D128, max_seqs=1)
    wd = to_device(I.make_weights(cfg, seed=5100))
    K, V = I.make_cache_prefill(cfg, 250, seed=5101, device="cuda")
    outs = []
    for poison in (False, True):
        st = Q.Qwen3Stack(cfg, wd)
        if poison:
            _poison(st, cfg)
        for l in range(cfg.num_layers):
            k, v = Q.cache_tensors(st.h, cfg, 0, l)
            k[:, :250].copy_(K[l])
            v[:, :250].copy_(V[l])
        Q.qwen3_set_length(st.h, 0, 250)
        outs.append([st.forward(I.make_rows(cfg, n, seed=5102 + n).cuda()).clone() for n in (1, 3, 20, 1)])
        st.close()
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_injected_allocation_failure(cuda_ok):
    """The workspace grows on first use; making that allocation fail returns
    QWEN3_E_OOM with lengths unchanged, and the call succeeds once the hook is
    off.  The same for the MoE block and the pooled vector."""
    cfg = SMALL_MOE
    p = Parity(cfg, seed=5200)
    x = I.make_rows(cfg, 20, seed=5201).cuda()
    for n in (1, 3):
        Q.qwen3_set_option(p.stack.h, Q.QWEN3_OPT_FAIL_ALLOC, n)
        with pytest.raises(Q.Qwen3Error) as e:
            Q.qwen3_forward(p.stack.h, x, [0] * 20, list(range(20)), torch.empty_like(x))
        assert e.value.status == 6 and "injected" in str(e.value)
        assert Q.qwen3_get_length(p.stack.h, 0) == 0
    Q.qwen3_set_option(p.stack.h, Q.QWEN3_OPT_FAIL_ALLOC, 0)
    p.step(x)
    p.step(I.make_rows(cfg, 1, seed=5202).cuda())
    p.close()
    p.check()
    st = Q.Qwen3Stack(cfg, to_device(I.make_weights(cfg, seed=5203)))
    y = I.make_rows(cfg, 50, seed=5204).cuda()
    idx = torch.empty(50, cfg.top_k, dtype=torch.int32, device="cuda")
    w = torch.empty(50, cfg.top_k, dtype=torch.float32, device="cuda")
    Q.qwen3_set_option(st.h, Q.QWEN3_OPT_FAIL_ALLOC, 1)
    with pytest.raises(Q.Qwen3Error) as e:
        Q.qwen3_moe_layer(st.h, 0, y, torch.empty_like(y), idx, w)
    assert e.value.status == 6
    Q.qwen3_set_option(st.h, Q.QWEN3_OPT_FAIL_ALLOC, 1)
    with pytest.raises(Q.Qwen3Error) as e:
        Q.qwen3_embed_pooled(st.h, y[:10], 1, torch.empty(cfg.hidden, dtype=y.dtype, device="cuda"))
    assert e.value.status == 6
    Q.qwen3_moe_layer(st.h, 0, y, torch.empty_like(y), idx, w)
    torch.cuda.synchronize()
    st.close()


def test_bounded_wait_gives_up_and_reports(cuda_ok):
    """A kernel waiting for data nothing delivers gives up after its bounded
    wait, records its code and returns: qwen3_device_error reports it once,
    and the stack still computes the right thing afterwards."""
    cfg = I.with_sizes(SMALL_D128, max_seqs=1)
    p = Parity(cfg, seed=5300)
    p.step(I.make_rows(cfg, 5, seed=5301).cuda())
    assert Q.qwen3_device_error(p.stack.h) == 0
    Q.qwen3_selftest_bounded_wait(p.stack.h)
    assert Q.qwen3_device_error(p.stack.h) == 99
    assert Q.qwen3_device_error(p.stack.h) == 0          # read once, then cleared
    p.step(I.make_rows(cfg, 1, seed=5302).cuda())
    p.step(I.make_rows(cfg, 6, seed=5303).cuda())
    assert Q.qwen3_device_error(p.stack.h) == 0
    p.close()
    p.check()

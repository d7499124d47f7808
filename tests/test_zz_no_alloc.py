"""qwen3_moe_layer_static, the MoE block for callers that must not allocate
device memory, against qwen3_moe_layer.

The static variant keeps all of its scratch in one fixed array inside the
library, so callers whose memory is fully reserved up front, or owned by
another allocator, can still run the MoE block.  These tests call it through
the C ABI twice in a row -- the second call finds the first call's leftovers
in the shared array -- and check that:

* it runs the same kernels as qwen3_moe_layer (the same launch count, the
  tensor-core grouped expert GEMMs included), so its results are bitwise
  equal to qwen3_moe_layer's;
* it allocates nothing: after a first call, further calls of other row counts
  leave the device's free memory and the handle's workspace as they were;
* rows past the array's limit are refused before any work is enqueued.

The file is named to be collected last.
"""
import pytest
import torch

from qwen3_decoder_layer_gb300 import binding as Q
from qwen3_decoder_layer_gb300 import inputs as I

pytestmark = pytest.mark.gpu

SMALL = I.with_sizes(I.MOE_A3B_4LAYER, name="static_small_moe", num_layers=1, hidden=256, n_heads=8,
                     n_kv_heads=1, head_dim=64, num_experts=32, top_k=4, moe_intermediate=128, capacity=64)
FULL_1L = I.with_sizes(I.MOE_A3B_4LAYER, name="static_moe_1layer", num_layers=1, capacity=64)


def _run(fn, stack, cfg, y):
    T = y.shape[0]
    out = torch.empty_like(y)
    idx = torch.empty(T, cfg.top_k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, cfg.top_k, dtype=torch.float32, device="cuda")
    fn(stack.h, 0, y, out, idx, w)
    return out, idx, w, Q.qwen3_last_launch_count(stack.h)


def _two_calls_match(cfg, seed, rows):
    stack = Q.Qwen3Stack(cfg, I.make_weights(cfg, seed=seed, device="cuda"))
    try:
        ys = [I.make_rows(cfg, T, seed=seed + 1 + n).cuda() for n, T in enumerate(rows)]
        static = [_run(Q.qwen3_moe_layer_static, stack, cfg, y) for y in ys]  # back to back
        ref = [_run(Q.qwen3_moe_layer, stack, cfg, y) for y in ys]
        torch.cuda.synchronize()
        for (o_s, i_s, w_s, n_s), (o_r, i_r, w_r, n_r) in zip(static, ref):
            assert n_s == n_r, "the static variant launched other kernels"
            assert torch.equal(i_s, i_r) and torch.equal(w_s, w_r)
            assert torch.equal(o_s, o_r)
    finally:
        stack.close()


@pytest.mark.parametrize("rows", [(3, 3), (2, 40), (40, 1)])
def test_static_scratch_matches_workspace_path(cuda_ok, rows):
    """Few rows (gathered expert GEMVs) and many rows (sorted grouped GEMMs)."""
    _two_calls_match(SMALL, 2100 + sum(rows), rows)


@pytest.mark.parametrize("rows", [(1, 4), (64, 91)])
def test_static_scratch_full_size_moe(cuda_ok, rows):
    """128 experts, top-8, hidden 2048: 91 rows is the most the 4 MiB array holds."""
    _two_calls_match(FULL_1L, 2200 + sum(rows), rows)


def test_static_scratch_allocates_nothing(cuda_ok):
    stack = Q.Qwen3Stack(FULL_1L, I.make_weights(FULL_1L, seed=2250, device="cuda"))
    try:
        ys = [I.make_rows(FULL_1L, T, seed=2252 + T).cuda() for T in (1, 5, 17, 64, 91)]
        for y in ys:   # first use of each kernel (lazy module loading may take device memory once)
            _run(Q.qwen3_moe_layer_static, stack, FULL_1L, y)
        torch.cuda.synchronize()
        free0, ws0 = torch.cuda.mem_get_info()[0], Q.qwen3_workspace_bytes(stack.h)
        ys = ys[::-1] + ys
        for y in ys:
            _run(Q.qwen3_moe_layer_static, stack, FULL_1L, y)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0
        assert Q.qwen3_workspace_bytes(stack.h) == ws0
    finally:
        stack.close()


def test_static_scratch_rejects_too_many_rows(cuda_ok):
    stack = Q.Qwen3Stack(FULL_1L, I.make_weights(FULL_1L, seed=2300, device="cuda"))
    try:
        with pytest.raises(Q.Qwen3Error) as ei:
            _run(Q.qwen3_moe_layer_static, stack, FULL_1L, I.make_rows(FULL_1L, 92, seed=2301).cuda())
        assert Q.STATUS[ei.value.status] == "QWEN3_E_ARG" and "at most 91 rows" in str(ei.value)
        # the refused call enqueued nothing; the next one works
        y = I.make_rows(FULL_1L, 2, seed=2302).cuda()
        o_s, i_s, _, _ = _run(Q.qwen3_moe_layer_static, stack, FULL_1L, y)
        o_r, i_r, _, _ = _run(Q.qwen3_moe_layer, stack, FULL_1L, y)
        torch.cuda.synchronize()
        assert torch.equal(i_s, i_r) and torch.equal(o_s, o_r)
    finally:
        stack.close()

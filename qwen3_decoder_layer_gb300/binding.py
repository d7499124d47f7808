"""Thin ctypes binding of the C ABI in include/qwen3.h.

Functions carry the C names and only marshal arguments (torch tensors become
device pointers, Python lists become int32 host arrays, the current torch
stream becomes the cudaStream_t).  All computation happens in
libqwen3_gb300.so; if the library is missing this module raises -- there is no
Python or CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libqwen3_gb300.so")

QWEN3_OK = 0
STATUS = {0: "QWEN3_OK", 1: "QWEN3_E_ARG", 2: "QWEN3_E_DTYPE", 3: "QWEN3_E_CAPACITY",
          4: "QWEN3_E_POSITION", 5: "QWEN3_E_SEQ", 6: "QWEN3_E_OOM", 7: "QWEN3_E_CUDA",
          8: "QWEN3_E_UNSUPPORTED", 9: "QWEN3_E_DEVICE"}
QWEN3_OPT_CUDA_GRAPHS, QWEN3_OPT_PROFILE, QWEN3_OPT_PDL, QWEN3_OPT_TENSOR_CORES = 1, 2, 3, 4
QWEN3_OPT_L2_PREFETCH = 5
QWEN3_OPT_FAIL_ALLOC = 7
QWEN3_OPT_CLUSTER_ATTENTION = 8
QWEN3_OPT_GEMV_CORESIDENT = 9


class Qwen3Error(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


class qwen3_config(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("n_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("intermediate", ctypes.c_int32),
                ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_double),
                ("capacity", ctypes.c_int32), ("max_seqs", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("weight_format", ctypes.c_int32),
                ("group_size", ctypes.c_int32), ("num_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("moe_intermediate", ctypes.c_int32),
                ("norm_topk_prob", ctypes.c_int32), ("decoder_sparse_step", ctypes.c_int32),
                ("mlp_only_layers", ctypes.POINTER(ctypes.c_int32)),
                ("n_mlp_only_layers", ctypes.c_int32)]


class qwen3_linear(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("bias", ctypes.c_void_p)]


class qwen3_layer_weights(ctypes.Structure):
    _fields_ = [("in_norm", ctypes.c_void_p), ("post_norm", ctypes.c_void_p),
                ("q_norm", ctypes.c_void_p), ("k_norm", ctypes.c_void_p),
                ("qkv", qwen3_linear), ("o", qwen3_linear), ("gate_up", qwen3_linear),
                ("down", qwen3_linear), ("router", ctypes.c_void_p),
                ("exp_gate_up", qwen3_linear), ("exp_down", qwen3_linear)]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_PI32 = ctypes.POINTER(ctypes.c_int32)
_SIGS = {
    "qwen3_check_config": (_I32, [ctypes.POINTER(qwen3_config)]),
    "qwen3_create": (_I32, [ctypes.POINTER(qwen3_config), ctypes.POINTER(qwen3_layer_weights), _P,
                            ctypes.POINTER(_P)]),
    "qwen3_destroy": (None, [_P]),
    "qwen3_reset": (_I32, [_P, _I32, _P]),
    "qwen3_forward": (_I32, [_P, _P, _I32, _PI32, _PI32, _P, _P]),
    "qwen3_moe_layer": (_I32, [_P, _I32, _P, _I32, _P, _P, _P, _P]),
    "qwen3_moe_layer_static": (_I32, [_P, _I32, _P, _I32, _P, _P, _P, _P]),
    "qwen3_embed": (_I32, [_P, _P, _I32, _PI32, _I32, _P, _P]),
    "qwen3_head": (_I32, [_P, _P, _I32, _P, _I32, _P, _P]),
    "qwen3_embed_pooled": (_I32, [_P, _P, _I32, _I32, _P, _P]),
    "qwen3_workspace_bytes": (_I32, [_P, ctypes.POINTER(ctypes.c_int64)]),
    "qwen3_cache_view": (_I32, [_P, _I32, _I32, ctypes.POINTER(_P), ctypes.POINTER(_P)]),
    "qwen3_set_length": (_I32, [_P, _I32, _I32]),
    "qwen3_get_length": (_I32, [_P, _I32, _PI32]),
    "qwen3_set_option": (_I32, [_P, _I32, ctypes.c_int64]),
    "qwen3_profile_read": (_I32, [_P, _I32, ctypes.POINTER(ctypes.c_char_p),
                                  ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_double),
                                  _PI32]),
    "qwen3_profile_reset": (_I32, [_P]),
    "qwen3_last_launch_count": (ctypes.c_int64, [_P]),
    "qwen3_device_error": (_I32, [_P, _PI32]),
    "qwen3_selftest_bounded_wait": (_I32, [_P, _P]),
    "qwen3_last_error": (ctypes.c_char_p, [_P]),
    "qwen3_status_string": (ctypes.c_char_p, [_I32]),
}

_lib = None


def lib():
    """Load libqwen3_gb300.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m qwen3_decoder_layer_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(h, st):
    if st != QWEN3_OK:
        msg = lib().qwen3_last_error(h).decode() if h else ""
        raise Qwen3Error(st, msg or lib().qwen3_status_string(st).decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def make_config(cfg) -> qwen3_config:
    """qwen3_config from an inputs.Qwen3Config."""
    c = qwen3_config()
    for f in ("num_layers", "hidden", "n_heads", "n_kv_heads", "head_dim", "intermediate",
              "capacity", "max_seqs", "group_size", "num_experts", "top_k", "moe_intermediate",
              "decoder_sparse_step"):
        setattr(c, f, int(getattr(cfg, f)))
    c.rms_eps = float(cfg.rms_eps)
    c.rope_theta = float(cfg.rope_theta)
    c.dtype = {"fp32": 0, "bf16": 1}.get(cfg.dtype, 99)
    c.weight_format = {"dense": 0, "int8": 1}[cfg.weight_format]
    c.norm_topk_prob = int(bool(cfg.norm_topk_prob))
    dense = [int(i) for i in getattr(cfg, "mlp_only_layers", ())]
    c._mlp_only = (ctypes.c_int32 * max(len(dense), 1))(*dense)   # kept alive with the struct
    c.mlp_only_layers = ctypes.cast(c._mlp_only, ctypes.POINTER(ctypes.c_int32)) if dense else None
    c.n_mlp_only_layers = len(dense)
    return c


def qwen3_check_config(cfg) -> int:
    c = cfg if isinstance(cfg, qwen3_config) else make_config(cfg)
    return lib().qwen3_check_config(ctypes.byref(c))


def qwen3_create(cfg, weights: dict):
    """Create a handle from a config and the weight dict of inputs.make_weights
    (tensors on the current CUDA device).  Returns the opaque handle."""
    c = cfg if isinstance(cfg, qwen3_config) else make_config(cfg)
    n = len(weights["layers"])
    arr = (qwen3_layer_weights * n)()
    for i, L in enumerate(weights["layers"]):
        w = arr[i]
        w.in_norm, w.post_norm = _ptr(L["in_norm"]), _ptr(L["post_norm"])
        w.q_norm, w.k_norm = _ptr(L["q_norm"]), _ptr(L["k_norm"])
        for name in ("qkv", "o", "gate_up", "down"):
            if name in L:
                lw = L[name]
                setattr(w, name, qwen3_linear(_ptr(lw["w"]), _ptr(lw.get("scale")), _ptr(lw.get("bias"))))
        if "router" in L:
            w.router = _ptr(L["router"]["w"])
            for name in ("exp_gate_up", "exp_down"):
                lw = L[name]
                setattr(w, name, qwen3_linear(_ptr(lw["w"]), _ptr(lw.get("scale")), _ptr(lw.get("bias"))))
    h = ctypes.c_void_p()
    st = lib().qwen3_create(ctypes.byref(c), arr, _ptr(weights["final_norm"]), ctypes.byref(h))
    if st != QWEN3_OK:
        raise Qwen3Error(st, lib().qwen3_status_string(st).decode())
    return h


def qwen3_destroy(h) -> None:
    lib().qwen3_destroy(h)


def qwen3_reset(h, seq_id: int = -1, stream=None) -> None:
    _check(h, lib().qwen3_reset(h, seq_id, _stream(stream)))


def qwen3_forward(h, x, seq_ids, positions, out, stream=None) -> None:
    T = int(x.shape[0])
    sid = (ctypes.c_int32 * T)(*[int(s) for s in seq_ids])
    pos = (ctypes.c_int32 * T)(*[int(p) for p in positions])
    _check(h, lib().qwen3_forward(h, _ptr(x), T, sid, pos, _ptr(out), _stream(stream)))


def qwen3_moe_layer(h, layer: int, y, out, topk_idx, topk_w, stream=None) -> None:
    _check(h, lib().qwen3_moe_layer(h, layer, _ptr(y), int(y.shape[0]), _ptr(out), _ptr(topk_idx),
                                    _ptr(topk_w), _stream(stream)))


def qwen3_moe_layer_static(h, layer: int, y, out, topk_idx, topk_w, stream=None) -> None:
    """qwen3_moe_layer with its scratch in the library's fixed device array
    (no allocation; T bounded by that array's size)."""
    _check(h, lib().qwen3_moe_layer_static(h, layer, _ptr(y), int(y.shape[0]), _ptr(out), _ptr(topk_idx),
                                           _ptr(topk_w), _stream(stream)))


def qwen3_embed(h, table, ids, out, stream=None) -> None:
    """out[t] = table[ids[t]] (ids: a list of host ints)."""
    n = len(ids)
    arr = (ctypes.c_int32 * n)(*[int(i) for i in ids])
    _check(h, lib().qwen3_embed(h, _ptr(table), int(table.shape[0]), arr, n, _ptr(out), _stream(stream)))


def qwen3_head(h, w, x, logits, stream=None) -> None:
    """logits fp32 [T, n_out] = fp32(R(x w^T))."""
    _check(h, lib().qwen3_head(h, _ptr(w), int(w.shape[0]), _ptr(x), int(x.shape[0]), _ptr(logits),
                               _stream(stream)))


def qwen3_embed_pooled(h, x, seq: int, out, stream=None) -> None:
    """out [hidden] = the last row's final-norm hidden state over its L2 norm,
    after running the T rows of x from position 0 of sequence `seq`."""
    _check(h, lib().qwen3_embed_pooled(h, _ptr(x), int(x.shape[0]), int(seq), _ptr(out), _stream(stream)))


def qwen3_workspace_bytes(h) -> int:
    n = ctypes.c_int64()
    _check(h, lib().qwen3_workspace_bytes(h, ctypes.byref(n)))
    return n.value


def qwen3_cache_view(h, seq: int, layer: int):
    k, v = ctypes.c_void_p(), ctypes.c_void_p()
    _check(h, lib().qwen3_cache_view(h, seq, layer, ctypes.byref(k), ctypes.byref(v)))
    return k.value, v.value


def qwen3_set_length(h, seq: int, length: int) -> None:
    _check(h, lib().qwen3_set_length(h, seq, length))


def qwen3_get_length(h, seq: int) -> int:
    n = ctypes.c_int32()
    _check(h, lib().qwen3_get_length(h, seq, ctypes.byref(n)))
    return n.value


def qwen3_set_option(h, option: int, value: int) -> None:
    _check(h, lib().qwen3_set_option(h, option, value))


def qwen3_profile_read(h) -> dict:
    """{kernel name: (launches, total ms)} since the last reset (synchronises)."""
    cnt = ctypes.c_int32()
    _check(h, lib().qwen3_profile_read(h, -1, None, None, None, ctypes.byref(cnt)))
    out = {}
    for i in range(cnt.value):
        name, n, ms = ctypes.c_char_p(), ctypes.c_int64(), ctypes.c_double()
        _check(h, lib().qwen3_profile_read(h, i, ctypes.byref(name), ctypes.byref(n), ctypes.byref(ms),
                                           None))
        out[name.value.decode()] = (n.value, ms.value)
    return out


def qwen3_profile_reset(h) -> None:
    _check(h, lib().qwen3_profile_reset(h))


def qwen3_last_launch_count(h) -> int:
    return int(lib().qwen3_last_launch_count(h))


def qwen3_device_error(h) -> int:
    """0, or the code a kernel recorded when it gave up a bounded wait."""
    code = ctypes.c_int32()
    st = lib().qwen3_device_error(h, ctypes.byref(code))
    if st not in (QWEN3_OK, 9):
        _check(h, st)
    return code.value


def qwen3_selftest_bounded_wait(h, stream=None) -> None:
    _check(h, lib().qwen3_selftest_bounded_wait(h, _stream(stream)))


def qwen3_last_error(h) -> str:
    return lib().qwen3_last_error(h).decode()


def qwen3_status_string(st: int) -> str:
    return lib().qwen3_status_string(st).decode()


def cache_tensors(h, cfg, seq: int, layer: int):
    """torch views [n_kv_heads, capacity, head_dim] of one (sequence, layer)
    cache slab (library-owned memory; valid until qwen3_destroy)."""
    k, v = qwen3_cache_view(h, seq, layer)
    n = cfg.n_kv_heads * cfg.capacity * cfg.head_dim
    dt = cfg.torch_dtype()
    return _wrap(k, n, dt).view(cfg.n_kv_heads, cfg.capacity, cfg.head_dim), \
        _wrap(v, n, dt).view(cfg.n_kv_heads, cfg.capacity, cfg.head_dim)


def _wrap(ptr: int, numel: int, dtype) -> torch.Tensor:
    """A torch tensor over library-owned device memory (no copy, no ownership)."""
    class _Iface:
        pass
    o = _Iface()
    typestr = {torch.bfloat16: "<i2", torch.float32: "<f4"}[dtype]
    o.__cuda_array_interface__ = {"shape": (numel,), "typestr": typestr, "data": (ptr, False),
                                  "version": 2}
    t = torch.as_tensor(o, device="cuda")
    return t.view(dtype) if dtype == torch.bfloat16 else t


class Qwen3Stack:
    """A handle plus the weight tensors it borrows (kept alive here)."""

    def __init__(self, cfg, weights: dict):
        self.cfg = cfg
        self.weights = weights
        self.h = qwen3_create(cfg, weights)

    def forward(self, x, seq_ids=None, positions=None, out=None, stream=None):
        T = x.shape[0]
        if seq_ids is None:
            seq_ids = [0] * T
        if positions is None:
            base, positions = {}, []
            for s in seq_ids:
                p = base.get(s, qwen3_get_length(self.h, s))
                positions.append(p)
                base[s] = p + 1
        if out is None:
            out = torch.empty_like(x)
        qwen3_forward(self.h, x, seq_ids, positions, out, stream)
        return out

    def close(self):
        if self.h:
            qwen3_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

"""ctypes binding of libzb (``include/zb.h``): same names, argument marshalling only.

Tensors are passed as ``torch.Tensor`` (their ``data_ptr()`` is handed to the
library) or as plain integer device addresses.  Every compute step runs in the
library's CUDA kernels; nothing here computes.  A missing library raises: there
is no fallback.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

c_void_p = ctypes.c_void_p
c_int32 = ctypes.c_int32
c_size_t = ctypes.c_size_t
c_float = ctypes.c_float

ZB_OK = 0
STATUS_NAMES = {
    0: "ZB_OK", -1: "ZB_ERR_ARG", -2: "ZB_ERR_SHAPE", -3: "ZB_ERR_ORDER", -4: "ZB_ERR_STASH_FULL",
    -5: "ZB_ERR_NO_MB", -6: "ZB_ERR_CUDA", -7: "ZB_ERR_DEVICE_TIMEOUT", -8: "ZB_ERR_CAPACITY",
    -9: "ZB_ERR_DEVICE", -10: "ZB_ERR_WORKSPACE",
}
SCHED = {"1f1b": 0, "zbh1": 1, "gpipe": 2, "zb2p": 3}
LAYER_KINDS = {"linear": 0, "mlp": 1, "transformer": 2}


class ZBError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        self.name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{where}: {self.name}")


class zb_op(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_uint8), ("pad", ctypes.c_uint8 * 3), ("mb", c_int32)]


class zb_stage_config(ctypes.Structure):
    _fields_ = [("kind", c_int32), ("n_layers", c_int32), ("hidden", c_int32), ("ffn", c_int32),
                ("n_heads", c_int32), ("n_kv_heads", c_int32), ("head_dim", c_int32), ("eps", c_float),
                ("max_tokens", c_int32), ("max_inflight", c_int32), ("attention", c_int32), ("seq_len", c_int32)]


class zb_kernel_stats(ctypes.Structure):
    _fields_ = [("launches", c_int32), ("pad", c_int32), ("ms", ctypes.c_double), ("flops", ctypes.c_double),
                ("bytes", ctypes.c_double)]


KERNEL_CLASSES = ["gemm_forward", "gemm_backward_input", "gemm_backward_weight", "row_backward_input",
                  "row_backward_weight", "row_forward", "attn_forward", "attn_backward", "stash_copy"]
ATTENTION_KINDS = {"standin": 0, "causal": 1}


class zb_layer_params(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("w_qkv", "dw_qkv", "w_o", "dw_o", "w_gu", "dw_gu", "w_down",
                                        "dw_down", "gamma1", "dgamma1", "gamma2", "dgamma2", "w", "dw")]


_SIGS = {
    "zb_status_string": (ctypes.c_char_p, [c_int32]),
    "zb_version": (c_int32, []),
    "zb_schedule": (c_int32, [c_int32, c_int32, c_int32, c_int32, ctypes.POINTER(zb_op), c_int32,
                              ctypes.POINTER(c_int32)]),
    "zb_schedule_bubble": (c_int32, [c_int32, c_int32, c_int32, ctypes.POINTER(c_int32),
                                     ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]),
    "zb_schedule_window_idle": (c_int32, [c_int32, c_int32, c_int32, ctypes.POINTER(ctypes.c_int64),
                                          ctypes.POINTER(ctypes.c_double)]),
    "zb_schedule_search": (c_int32, [c_int32] * 7 + [ctypes.POINTER(zb_op), c_int32, ctypes.POINTER(c_int32),
                                     ctypes.POINTER(c_int32), ctypes.POINTER(ctypes.c_int64)]),
    "zb_op_linear_forward": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32,
                                       c_void_p]),
    "zb_op_backward_input": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32, c_void_p]),
    "zb_op_backward_input_swiglu": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_int32,
                                              c_int32, c_void_p]),
    "zb_op_backward_input_rmsnorm": (c_int32, [c_void_p] * 8 + [c_int32, c_int32, c_int32, c_void_p]),
    "zb_op_backward_input_attention": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32,
                                                 c_int32, c_void_p]),
    "zb_op_backward_weight": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32, c_void_p]),
    "zb_op_backward_weight_group": (c_int32, [c_int32, ctypes.POINTER(c_void_p), ctypes.POINTER(c_void_p),
                                              ctypes.POINTER(c_void_p), c_int32, ctypes.POINTER(c_int32),
                                              ctypes.POINTER(c_int32), c_void_p]),
    "zb_op_rmsnorm_backward_gamma_scratch_bytes": (c_size_t, [c_int32, c_int32]),
    "zb_op_rmsnorm_backward_gamma": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_int32,
                                               c_void_p, c_size_t, c_void_p]),
    "zb_op_rmsnorm_backward_gamma_noalloc_max_floats": (c_size_t, []),
    "zb_op_rmsnorm_backward_gamma_noalloc": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_int32,
                                                       c_void_p]),
    "zb_op_rmsnorm_forward": (c_int32, [c_void_p, c_void_p, c_float, c_void_p, c_void_p, c_int32, c_int32,
                                        c_void_p]),
    "zb_op_swiglu_forward": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_void_p]),
    "zb_op_attention_forward": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32, c_void_p]),
    "zb_op_attention_stat_stride": (c_int32, [c_int32]),
    "zb_op_attention_causal_forward": (c_int32, [c_void_p, c_void_p, c_void_p] + [c_int32] * 5 + [c_void_p]),
    "zb_op_attention_causal_backward": (c_int32, [c_void_p] * 6 + [c_int32] * 5 + [c_void_p]),
    "zb_device_status": (c_int32, [c_void_p, c_int32, ctypes.POINTER(c_int32)]),
    "zb_selftest_wait_timeout": (c_int32, [c_int32, c_void_p]),
    "zb_stage_workspace_bytes": (c_size_t, [ctypes.POINTER(zb_stage_config)]),
    "zb_stage_create": (c_int32, [ctypes.POINTER(zb_stage_config), ctypes.POINTER(zb_layer_params), c_void_p,
                                  c_size_t, ctypes.POINTER(c_void_p)]),
    "zb_stage_destroy": (c_int32, [c_void_p]),
    "zb_stage_forward": (c_int32, [c_void_p, c_int32, c_void_p, c_int32, c_void_p, c_void_p]),
    "zb_backward_input": (c_int32, [c_void_p, c_int32, c_void_p, c_void_p, c_void_p]),
    "zb_backward_weight": (c_int32, [c_void_p, c_int32, c_void_p]),
    "zb_wgrad_flush": (c_int32, [c_void_p, c_void_p]),
    "zb_stage_sync": (c_int32, [c_void_p, c_void_p]),
    "zb_stage_stats": (c_int32, [c_void_p, ctypes.POINTER(c_int32), ctypes.POINTER(c_int32),
                                 ctypes.POINTER(c_size_t)]),
    "zb_stage_stash_view": (c_int32, [c_void_p, c_int32, c_int32, c_int32, ctypes.POINTER(c_void_p),
                                      ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64),
                                      ctypes.POINTER(c_int32)]),
    "zb_stage_set_tracing": (c_int32, [c_void_p, c_int32]),
    "zb_stage_read_tracing": (c_int32, [c_void_p, ctypes.POINTER(zb_kernel_stats), c_int32]),
}

_LIB = None


def lib():
    """The loaded libzb (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"{_build.LIB} is missing: build it with __graft_entry__.build()")
        handle = ctypes.CDLL(_build.LIB)
        for name, (res, args) in _SIGS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = handle
    return _LIB


def declared_symbols():
    return list(_SIGS)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if s is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status, where):
    if status != ZB_OK:
        raise ZBError(status, where)


# ---------------------------------------------------------------- misc / schedule


def zb_status_string(status):
    return lib().zb_status_string(status).decode()


def zb_version():
    return lib().zb_version()


def zb_schedule(kind, stage, p, m):
    """F/B/W order of one stage: list of ("F" | "B" | "W", mb)."""
    n = c_int32(0)
    buf = (zb_op * (3 * m))()
    _check(lib().zb_schedule(SCHED[kind], stage, p, m, buf, 3 * m, ctypes.byref(n)), "zb_schedule")
    return [(chr(buf[i].kind), buf[i].mb) for i in range(n.value)]


def zb_schedule_raw(kind, stage, p, m, cap):
    """Low-level form: (status, n_out, ops) without raising."""
    n = c_int32(-1)
    buf = (zb_op * max(cap, 1))()
    st = lib().zb_schedule(kind, stage, p, m, buf if cap > 0 else None, cap, ctypes.byref(n))
    return st, n.value, [(chr(buf[i].kind), buf[i].mb) for i in range(min(max(n.value, 0), cap))]


def zb_schedule_search(stage, p, m, mem_limit, t_f, t_b, t_w):
    """(order of `stage`, chosen ceiling, makespan) of the memory-limited search."""
    arr = (zb_op * (3 * m))()
    n = c_int32(0)
    limit = c_int32(0)
    span = ctypes.c_int64(0)
    _check(lib().zb_schedule_search(stage, p, m, mem_limit, t_f, t_b, t_w, arr, 3 * m, ctypes.byref(n),
                                    ctypes.byref(limit), ctypes.byref(span)), "zb_schedule_search")
    return [(chr(arr[i].kind), arr[i].mb) for i in range(n.value)], limit.value, span.value


def zb_schedule_bubble(kind, p, m):
    """(makespan, idle / compute, idle / wall) of the unit-time pipeline model."""
    span = c_int32(0)
    a = ctypes.c_double(0)
    b = ctypes.c_double(0)
    _check(lib().zb_schedule_bubble(SCHED[kind], p, m, ctypes.byref(span), ctypes.byref(a), ctypes.byref(b)),
           "zb_schedule_bubble")
    return span.value, a.value, b.value


def zb_schedule_window_idle(kind, p, m):
    """(idle units, idle / compute) inside each stage's own window, summed over stages."""
    n = ctypes.c_int64(0)
    f = ctypes.c_double(0)
    _check(lib().zb_schedule_window_idle(SCHED[kind], p, m, ctypes.byref(n), ctypes.byref(f)),
           "zb_schedule_window_idle")
    return n.value, f.value


# ---------------------------------------------------------------- per-step ops


def zb_op_linear_forward(x, w, residual, y, tokens, in_features, out_features, stream=None):
    _check(lib().zb_op_linear_forward(_ptr(x), _ptr(w), _ptr(residual), _ptr(y), tokens, in_features,
                                      out_features, _stream(stream)), "zb_op_linear_forward")


def zb_op_backward_input(dy, w, dx, tokens, in_features, out_features, stream=None):
    _check(lib().zb_op_backward_input(_ptr(dy), _ptr(w), _ptr(dx), tokens, in_features, out_features,
                                      _stream(stream)), "zb_op_backward_input")


def zb_op_backward_input_swiglu(dy, w_down, gu, dgu, tokens, hidden, ffn, stream=None):
    _check(lib().zb_op_backward_input_swiglu(_ptr(dy), _ptr(w_down), _ptr(gu), _ptr(dgu), tokens, hidden, ffn,
                                             _stream(stream)), "zb_op_backward_input_swiglu")


def zb_op_backward_input_rmsnorm(dy, w, x, rstd, gamma, dres, dn, dx, tokens, hidden, out_features, stream=None):
    _check(lib().zb_op_backward_input_rmsnorm(_ptr(dy), _ptr(w), _ptr(x), _ptr(rstd), _ptr(gamma), _ptr(dres),
                                              _ptr(dn), _ptr(dx), tokens, hidden, out_features, _stream(stream)),
           "zb_op_backward_input_rmsnorm")


def zb_op_backward_input_attention(dh, w_o, dqkv, tokens, n_heads, n_kv_heads, head_dim, stream=None):
    _check(lib().zb_op_backward_input_attention(_ptr(dh), _ptr(w_o), _ptr(dqkv), tokens, n_heads, n_kv_heads,
                                                head_dim, _stream(stream)), "zb_op_backward_input_attention")


def zb_op_backward_weight(dy, x, dw, tokens, in_features, out_features, stream=None):
    _check(lib().zb_op_backward_weight(_ptr(dy), _ptr(x), _ptr(dw), tokens, in_features, out_features,
                                       _stream(stream)), "zb_op_backward_weight")


def zb_op_backward_weight_group(dys, xs, dws, tokens, in_features, out_features, stream=None):
    n = len(dys)
    ptrs = lambda ts: (c_void_p * n)(*[_ptr(t) for t in ts])  # noqa: E731
    ints = lambda vs: (c_int32 * n)(*vs)  # noqa: E731
    _check(lib().zb_op_backward_weight_group(n, ptrs(dys), ptrs(xs), ptrs(dws), tokens, ints(in_features),
                                             ints(out_features), _stream(stream)), "zb_op_backward_weight_group")


def zb_op_rmsnorm_backward_gamma_scratch_bytes(tokens, hidden):
    return lib().zb_op_rmsnorm_backward_gamma_scratch_bytes(tokens, hidden)


def zb_op_rmsnorm_backward_gamma(dn, x, rstd, dgamma, tokens, hidden, scratch, scratch_bytes, stream=None):
    _check(lib().zb_op_rmsnorm_backward_gamma(_ptr(dn), _ptr(x), _ptr(rstd), _ptr(dgamma), tokens, hidden,
                                              _ptr(scratch), scratch_bytes, _stream(stream)),
           "zb_op_rmsnorm_backward_gamma")


def zb_op_rmsnorm_backward_gamma_noalloc_max_floats():
    return lib().zb_op_rmsnorm_backward_gamma_noalloc_max_floats()


def zb_op_rmsnorm_backward_gamma_noalloc(dn, x, rstd, dgamma, tokens, hidden, stream=None):
    """Gamma-gradient reduction without caller scratch (see include/zb.h for its limits)."""
    _check(lib().zb_op_rmsnorm_backward_gamma_noalloc(_ptr(dn), _ptr(x), _ptr(rstd), _ptr(dgamma), tokens, hidden,
                                                      _stream(stream)), "zb_op_rmsnorm_backward_gamma_noalloc")


def zb_op_rmsnorm_forward(x, gamma, eps, n, rstd, tokens, hidden, stream=None):
    _check(lib().zb_op_rmsnorm_forward(_ptr(x), _ptr(gamma), eps, _ptr(n), _ptr(rstd), tokens, hidden,
                                       _stream(stream)), "zb_op_rmsnorm_forward")


def zb_op_swiglu_forward(gu, s, tokens, ffn, stream=None):
    _check(lib().zb_op_swiglu_forward(_ptr(gu), _ptr(s), tokens, ffn, _stream(stream)), "zb_op_swiglu_forward")


def zb_op_attention_forward(qkv, a, tokens, n_heads, n_kv_heads, head_dim, stream=None):
    _check(lib().zb_op_attention_forward(_ptr(qkv), _ptr(a), tokens, n_heads, n_kv_heads, head_dim,
                                         _stream(stream)), "zb_op_attention_forward")


def zb_op_attention_stat_stride(tokens):
    return lib().zb_op_attention_stat_stride(tokens)


def zb_op_attention_causal_forward(qkv, a, lse, tokens, n_heads, n_kv_heads, head_dim, seq_len=0, stream=None):
    _check(lib().zb_op_attention_causal_forward(_ptr(qkv), _ptr(a), _ptr(lse), tokens, n_heads, n_kv_heads,
                                                head_dim, seq_len, _stream(stream)),
           "zb_op_attention_causal_forward")


def zb_op_attention_causal_backward(qkv, a, da, lse, dvec, dqkv, tokens, n_heads, n_kv_heads, head_dim,
                                    seq_len=0, stream=None):
    _check(lib().zb_op_attention_causal_backward(_ptr(qkv), _ptr(a), _ptr(da), _ptr(lse), _ptr(dvec), _ptr(dqkv),
                                                 tokens, n_heads, n_kv_heads, head_dim, seq_len, _stream(stream)),
           "zb_op_attention_causal_backward")


def zb_device_status(stream=None, reset=False):
    """(status, code): status is ZB_OK or ZB_ERR_DEVICE_TIMEOUT; never raises on a timeout."""
    code = c_int32(0)
    st = lib().zb_device_status(_stream(stream), 1 if reset else 0, ctypes.byref(code))
    if st not in (ZB_OK, -7):
        raise ZBError(st, "zb_device_status")
    return st, code.value


def zb_selftest_wait_timeout(limit_us, stream=None):
    _check(lib().zb_selftest_wait_timeout(limit_us, _stream(stream)), "zb_selftest_wait_timeout")


# ---------------------------------------------------------------- stage


def make_config(kind, n_layers, hidden, ffn, n_heads=0, n_kv_heads=0, head_dim=0, eps=1e-5, max_tokens=128,
                max_inflight=1, attention="standin", seq_len=0):
    return zb_stage_config(LAYER_KINDS[kind], n_layers, hidden, ffn, n_heads, n_kv_heads, head_dim, eps,
                           max_tokens, max_inflight, ATTENTION_KINDS[attention], seq_len)


def zb_stage_workspace_bytes(cfg):
    return lib().zb_stage_workspace_bytes(ctypes.byref(cfg))


def zb_stage_create(cfg, layers, workspace, workspace_bytes):
    """layers: list of dicts name -> tensor / int pointer (names of zb_layer_params)."""
    arr = (zb_layer_params * len(layers))()
    for i, d in enumerate(layers):
        for k, v in d.items():
            setattr(arr[i], k, _ptr(v))
    handle = c_void_p(0)
    _check(lib().zb_stage_create(ctypes.byref(cfg), arr, _ptr(workspace), workspace_bytes, ctypes.byref(handle)),
           "zb_stage_create")
    return handle.value


def zb_stage_destroy(st):
    _check(lib().zb_stage_destroy(st), "zb_stage_destroy")


def zb_stage_forward(st, mb, x, tokens, y, stream=None):
    _check(lib().zb_stage_forward(st, mb, _ptr(x), tokens, _ptr(y), _stream(stream)), "zb_stage_forward")


def zb_backward_input(st, mb, dy, dx, stream=None):
    _check(lib().zb_backward_input(st, mb, _ptr(dy), _ptr(dx), _stream(stream)), "zb_backward_input")


def zb_backward_weight(st, mb, stream=None):
    _check(lib().zb_backward_weight(st, mb, _stream(stream)), "zb_backward_weight")


def zb_wgrad_flush(st, stream=None):
    _check(lib().zb_wgrad_flush(st, _stream(stream)), "zb_wgrad_flush")


def zb_stage_sync(st, stream=None):
    _check(lib().zb_stage_sync(st, _stream(stream)), "zb_stage_sync")


def zb_stage_stats(st):
    a, b, c = c_int32(0), c_int32(0), c_size_t(0)
    _check(lib().zb_stage_stats(st, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)), "zb_stage_stats")
    return a.value, b.value, c.value


STASH_TENSORS = ["x", "rstd1", "n1", "a", "h", "rstd2", "n2", "gu", "s", "dy", "dn2", "dh", "dqkv", "dn1", "qkv",
                 "lse"]


def zb_stage_stash_view(st, mb, layer, tensor):
    """(device address, rows, cols, element bytes) of one stashed tensor; `tensor` is a name of
    STASH_TENSORS or its index."""
    idx = STASH_TENSORS.index(tensor) if isinstance(tensor, str) else int(tensor)
    ptr, rows, cols, eb = c_void_p(0), ctypes.c_int64(0), ctypes.c_int64(0), c_int32(0)
    _check(lib().zb_stage_stash_view(st, mb, layer, idx, ctypes.byref(ptr), ctypes.byref(rows), ctypes.byref(cols),
                                     ctypes.byref(eb)), "zb_stage_stash_view")
    return ptr.value or 0, rows.value, cols.value, eb.value


def zb_stage_set_tracing(st, enable):
    _check(lib().zb_stage_set_tracing(st, 1 if enable else 0), "zb_stage_set_tracing")


def zb_stage_read_tracing(st, reset=True):
    """dict kernel class -> {"launches", "ms", "flops", "bytes"} of the launches recorded so far."""
    arr = (zb_kernel_stats * len(KERNEL_CLASSES))()
    _check(lib().zb_stage_read_tracing(st, arr, 1 if reset else 0), "zb_stage_read_tracing")
    return {name: {"launches": arr[i].launches, "ms": arr[i].ms, "flops": arr[i].flops, "bytes": arr[i].bytes}
            for i, name in enumerate(KERNEL_CLASSES)}

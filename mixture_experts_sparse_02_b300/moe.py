"""Python binding of libmoe (include/moe.h): argument marshalling only.

Every call takes torch tensors on the current CUDA device (or plain integer addresses) and
forwards their data pointers to the C ABI; all computation happens in the library's CUDA
kernels.  Importing this module fails if libmoe.so has not been built: there is no CPU or
PyTorch fallback.  With the environment variable MOE_LIBRARY=debug it loads the
bounds-checking build libmoe_debug.so instead (same calls; see build.py).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
_DEBUG = os.environ.get("MOE_LIBRARY", "") == "debug"
LIB_PATH = os.path.join(_HERE, "libmoe_debug.so" if _DEBUG else "libmoe.so")

if not os.path.exists(LIB_PATH):
    raise ImportError("%s is missing; build it with `python -m mixture_experts_sparse_02_b300.build%s`"
                      % (LIB_PATH, " --debug-bounds" if _DEBUG else ""))
_lib = ctypes.CDLL(LIB_PATH)

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, MOE_ERR_DEVICE = range(6)
MOE_F32, MOE_BF16 = 0, 1
MOE_SOFTMAX_TOPK_RENORM, MOE_SIGMOID_TOPK_NORM, MOE_SOFTMAX_TOPK_PLAIN, MOE_EXPERT_CHOICE = 0, 1, 2, 3
SCORING = {"softmax": MOE_SOFTMAX_TOPK_RENORM, "sigmoid": MOE_SIGMOID_TOPK_NORM,
           "softmax_norenorm": MOE_SOFTMAX_TOPK_PLAIN, "expert_choice": MOE_EXPERT_CHOICE}
MOE_NUM_STAGES = 6
STAGE_NAMES = ("route", "dispatch", "experts_w12", "experts_w3", "shared", "combine")


class MoEConfig(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("scoring", ctypes.c_int32), ("n_shared", ctypes.c_int32),
                ("d_ff_shared", ctypes.c_int32), ("capacity_factor", ctypes.c_float)]


class MoEError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (call, status_string(status), status))


_P = ctypes.c_void_p
_CFG = ctypes.POINTER(MoEConfig)
_SZ = ctypes.c_size_t
_I = ctypes.c_int


def _sig(name, args, res=_I):
    f = getattr(_lib, name)
    f.argtypes = args
    f.restype = res
    return f


_workspace_bytes = _sig("moe_workspace_bytes", [_CFG], _SZ)
_route = _sig("moe_route", [_CFG, _P, _P, _P, _P, _P, _P, _P, _SZ, _P])
_dispatch = _sig("moe_dispatch", [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P])
_experts = _sig("moe_experts", [_CFG, _P, _P, _P, _P, _P, _P, _P, _SZ, _P])
_combine = _sig("moe_combine", [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P])
_forward = _sig("moe_forward", [_CFG] + [_P] * 14 + [_SZ, _P])
_forward_profiled = _sig("moe_forward_profiled", [_CFG] + [_P] * 14 + [_SZ, _P, _P])
_forward_host = _sig("moe_forward_host", [_CFG] + [_P] * 12 + [_SZ, _P])
_forward_host_async = _sig("moe_forward_host_async", [_CFG] + [_P] * 12 + [_SZ, _P])
_get_device_error = _sig("moe_get_device_error", [_P, ctypes.POINTER(ctypes.c_uint32)])
_last_launch_count = _sig("moe_last_launch_count", [], ctypes.c_int32)
_status_string = _sig("moe_status_string", [_I], ctypes.c_char_p)
_dispatch_static = _sig("moe_dispatch_static", [_CFG, _P, _P, _P, _P, _P, _P, _P, _P])
_update_sel_bias = _sig("moe_update_sel_bias", [_CFG, _P, ctypes.c_float, _P, _P])
_route_ec = _sig("moe_route_expert_choice", [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P])
_combine_ec = _sig("moe_combine_expert_choice", [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P])
_test_pipeline_fault = _sig("moe_test_pipeline_fault", [ctypes.c_uint64])
_load_stats = _sig("moe_load_stats", [_CFG, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P, _P, _SZ, _P])
DISPATCH_STATIC_SCRATCH_BYTES = 1 << 20

EXPORTS = ("moe_workspace_bytes", "moe_route", "moe_dispatch", "moe_experts", "moe_combine",
           "moe_forward", "moe_forward_profiled", "moe_forward_host", "moe_forward_host_async", "moe_get_device_error",
           "moe_last_launch_count", "moe_status_string", "moe_dispatch_static", "moe_update_sel_bias",
           "moe_load_stats", "moe_route_expert_choice", "moe_combine_expert_choice", "moe_test_pipeline_fault")


def status_string(status: int) -> str:
    return _status_string(int(status)).decode()


def config(T: int, d: int, d_ff: int, E: int, k: int, dtype: str = "bf16", scoring: str = "softmax",
           n_shared: int = 0, d_ff_shared: int = 0, capacity_factor: float = 0.0) -> MoEConfig:
    return MoEConfig(T, d, d_ff, E, k, MOE_BF16 if dtype == "bf16" else MOE_F32, SCORING[scoring],
                     n_shared, d_ff_shared, capacity_factor)


def config_from_shape(shape, T: Optional[int] = None) -> MoEConfig:
    """MoEConfig from any object with T, d, d_ff, E, k, dtype, scoring, n_shared, d_ff_shared
    (and optionally capacity_factor)."""
    return config(shape.T if T is None else T, shape.d, shape.d_ff, shape.E, shape.k, shape.dtype,
                  shape.scoring, shape.n_shared, shape.d_ff_shared, getattr(shape, "capacity_factor", 0.0))


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, call: str):
    if status != MOE_OK:
        raise MoEError(status, call)


def workspace_bytes(cfg: MoEConfig) -> int:
    return int(_workspace_bytes(ctypes.byref(cfg)))


def route(cfg, x, W_g, topk_idx, topk_gate, logit_bias=None, sel_bias=None, ws=None, ws_bytes=None, stream=None):
    nb = ws.numel() * ws.element_size() if ws_bytes is None and ws is not None else (ws_bytes or 0)
    _check(_route(ctypes.byref(cfg), _ptr(x), _ptr(W_g), _ptr(logit_bias), _ptr(sel_bias), _ptr(topk_idx),
                  _ptr(topk_gate), _ptr(ws), nb, _stream(stream)), "moe_route")


def dispatch(cfg, topk_idx, x, counts, offsets, perm_tok, inv_pos, x_perm, ws, ws_bytes=None, stream=None):
    nb = ws.numel() * ws.element_size() if ws_bytes is None and ws is not None else (ws_bytes or 0)
    _check(_dispatch(ctypes.byref(cfg), _ptr(topk_idx), _ptr(x), _ptr(counts), _ptr(offsets), _ptr(perm_tok),
                     _ptr(inv_pos), _ptr(x_perm), _ptr(ws), nb, _stream(stream)), "moe_dispatch")


def dispatch_static(cfg, topk_idx, x, counts, offsets, perm_tok, inv_pos, x_perm, stream=None):
    """moe_dispatch without a workspace: for callers that cannot allocate device memory; the
    scratch is a fixed 1 MiB array inside the library (size limit and sharing rules in moe.h)."""
    _check(_dispatch_static(ctypes.byref(cfg), _ptr(topk_idx), _ptr(x), _ptr(counts), _ptr(offsets), _ptr(perm_tok),
                            _ptr(inv_pos), _ptr(x_perm), _stream(stream)), "moe_dispatch_static")


def route_expert_choice(cfg, x, W_g, offsets, perm_tok, gate, pos_of, logit_bias=None, ws=None, ws_bytes=None,
                        stream=None):
    """Expert choice: every expert's m tokens (offsets = e*m, perm_tok, gate by position, pos_of [T][E])."""
    nb = ws.numel() * ws.element_size() if ws_bytes is None and ws is not None else (ws_bytes or 0)
    _check(_route_ec(ctypes.byref(cfg), _ptr(x), _ptr(W_g), _ptr(logit_bias), _ptr(offsets), _ptr(perm_tok),
                     _ptr(gate), _ptr(pos_of), _ptr(ws), nb, _stream(stream)), "moe_route_expert_choice")


def combine_expert_choice(cfg, y_perm, gate, pos_of, y, x=None, Ws1=None, Ws2=None, Ws3=None, ws=None, ws_bytes=None,
                          stream=None):
    nb = ws.numel() * ws.element_size() if ws_bytes is None and ws is not None else (ws_bytes or 0)
    _check(_combine_ec(ctypes.byref(cfg), _ptr(y_perm), _ptr(gate), _ptr(pos_of), _ptr(x), _ptr(Ws1), _ptr(Ws2),
                       _ptr(Ws3), _ptr(y), _ptr(ws), nb, _stream(stream)), "moe_combine_expert_choice")


def load_stats(cfg, x, W_g, counts, alpha, f, P, summary, logit_bias=None, ws=None, ws_bytes=None, stream=None):
    """Per-expert f (routed fraction), P (mean score), and summary = [L_aux, max/mean load]."""
    nb = ws.numel() * ws.element_size() if ws_bytes is None and ws is not None else (ws_bytes or 0)
    _check(_load_stats(ctypes.byref(cfg), _ptr(x), _ptr(W_g), _ptr(logit_bias), _ptr(counts), float(alpha), _ptr(f),
                       _ptr(P), _ptr(summary), _ptr(ws), nb, _stream(stream)), "moe_load_stats")


def update_sel_bias(cfg, counts, gamma, sel_bias, stream=None):
    """One step of the selection-bias controller: sel_bias[e] -= gamma where counts[e] is above
    the share T*k/E, += gamma where below (in place, float32)."""
    _check(_update_sel_bias(ctypes.byref(cfg), _ptr(counts), float(gamma), _ptr(sel_bias), _stream(stream)),
           "moe_update_sel_bias")


def experts(cfg, x_perm, offsets, W1, W2, W3, y_perm, ws, ws_bytes=None, stream=None):
    nb = ws.numel() * ws.element_size() if ws_bytes is None and ws is not None else (ws_bytes or 0)
    _check(_experts(ctypes.byref(cfg), _ptr(x_perm), _ptr(offsets), _ptr(W1), _ptr(W2), _ptr(W3), _ptr(y_perm),
                    _ptr(ws), nb, _stream(stream)), "moe_experts")


def combine(cfg, y_perm, inv_pos, topk_gate, y, x=None, Ws1=None, Ws2=None, Ws3=None, ws=None, ws_bytes=None,
            stream=None):
    nb = ws.numel() * ws.element_size() if ws_bytes is None and ws is not None else (ws_bytes or 0)
    _check(_combine(ctypes.byref(cfg), _ptr(y_perm), _ptr(inv_pos), _ptr(topk_gate), _ptr(x), _ptr(Ws1), _ptr(Ws2),
                    _ptr(Ws3), _ptr(y), _ptr(ws), nb, _stream(stream)), "moe_combine")


def forward(cfg, x, W_g, W1, W2, W3, y, ws, logit_bias=None, sel_bias=None, Ws1=None, Ws2=None, Ws3=None,
            topk_idx_out=None, counts_out=None, ws_bytes=None, stream=None, events: Optional[Sequence] = None):
    """The whole layer.  `events`: optional MOE_NUM_STAGES + 1 torch.cuda.Event objects recorded
    at the stage boundaries."""
    nb = ws.numel() * ws.element_size() if ws_bytes is None and ws is not None else (ws_bytes or 0)
    args = [ctypes.byref(cfg), _ptr(x), _ptr(W_g), _ptr(logit_bias), _ptr(sel_bias), _ptr(W1), _ptr(W2), _ptr(W3),
            _ptr(Ws1), _ptr(Ws2), _ptr(Ws3), _ptr(y), _ptr(topk_idx_out), _ptr(counts_out), _ptr(ws), nb,
            _stream(stream)]
    if events is None:
        _check(_forward(*args), "moe_forward")
    else:
        handles = []
        for e in events:
            if e is not None and not e.cuda_event:
                e.record()          # torch creates its CUDA event lazily, on the first record
            handles.append(e.cuda_event if e is not None else None)
        arr = (ctypes.c_void_p * (MOE_NUM_STAGES + 1))(*handles)
        _check(_forward_profiled(*args, ctypes.cast(arr, ctypes.c_void_p)), "moe_forward_profiled")


def forward_host(cfg, x_host, W_g, W1, W2, W3, y_host, ws, logit_bias=None, sel_bias=None, Ws1=None, Ws2=None,
                 Ws3=None, ws_bytes=None, stream=None):
    """The whole layer with x and y in host memory (pinned CPU tensors give the fastest copies)."""
    nb = ws.numel() * ws.element_size() if ws_bytes is None and ws is not None else (ws_bytes or 0)
    _check(_forward_host(ctypes.byref(cfg), _ptr(x_host), _ptr(W_g), _ptr(logit_bias), _ptr(sel_bias), _ptr(W1),
                         _ptr(W2), _ptr(W3), _ptr(Ws1), _ptr(Ws2), _ptr(Ws3), _ptr(y_host), _ptr(ws), nb,
                         _stream(stream)), "moe_forward_host")


def forward_host_async(cfg, x_host, W_g, W1, W2, W3, y_host, ws, logit_bias=None, sel_bias=None, Ws1=None, Ws2=None,
                       Ws3=None, ws_bytes=None, stream=None):
    """forward_host without the final wait: y_host is ready once `stream` reaches the end of
    the call (synchronise or record an event)."""
    nb = ws.numel() * ws.element_size() if ws_bytes is None and ws is not None else (ws_bytes or 0)
    _check(_forward_host_async(ctypes.byref(cfg), _ptr(x_host), _ptr(W_g), _ptr(logit_bias), _ptr(sel_bias),
                               _ptr(W1), _ptr(W2), _ptr(W3), _ptr(Ws1), _ptr(Ws2), _ptr(Ws3), _ptr(y_host), _ptr(ws),
                               nb, _stream(stream)), "moe_forward_host_async")


def get_device_error(stream=None) -> int:
    """Waits for the stream, returns and clears the device error word (0 = no error)."""
    w = ctypes.c_uint32(0)
    st = _get_device_error(_stream(stream), ctypes.byref(w))
    if st not in (MOE_OK, MOE_ERR_DEVICE):
        raise MoEError(st, "moe_get_device_error")
    return int(w.value)


def test_pipeline_fault(wait_limit_ns: int):
    """Testing aid: starve the next grouped tensor-core GEMM launch (its waits run out after
    wait_limit_ns and it reports through the device error word)."""
    _check(_test_pipeline_fault(int(wait_limit_ns)), "moe_test_pipeline_fault")


def last_launch_count() -> int:
    return int(_last_launch_count())

"""Python binding of the B300 MoE-layer C ABI (include/moe.h).

Argument marshalling only: every step of the layer runs in the CUDA library
``_lib/libmoe_b300.so`` (built by ``expert_dispatch_top_b300.build``).  There
is no CPU or PyTorch fallback: if the library is missing, every call raises.

The functions keep the C names (moe_route, moe_dispatch, moe_expert_ffn,
moe_combine, moe_layer_forward, ...) and take torch tensors on the current
CUDA device; work is enqueued on ``torch.cuda.current_stream()`` unless a
``stream`` is given.  ``MoeLayer`` bundles a config with its buffers for the
common "whole layer" call.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# MOE_B300_CHECKED=1 loads the range-checked debugging build instead.
LIB_PATH = os.path.join(_PKG, "_lib", "libmoe_b300_checked.so"
                        if os.environ.get("MOE_B300_CHECKED") == "1" else "libmoe_b300.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_TIMEOUT, \
    MOE_ERR_NONFINITE, MOE_ERR_BOUNDS = range(7)
MOE_DTYPE_F32, MOE_DTYPE_BF16 = 0, 1
MOE_SCORE_SOFTMAX, MOE_SCORE_SIGMOID = 0, 1
MOE_ACT_GELU, MOE_ACT_SWIGLU, MOE_ACT_IDENTITY = 0, 1, 2
MOE_DEV_GEMM_TIMEOUT, MOE_DEV_BAD_INDEX, MOE_DEV_COPY_TIMEOUT, MOE_DEV_NONFINITE, MOE_DEV_BOUNDS = \
    0x2, 0x4, 0x8, 0x10, 0x20

_ACTS = {"gelu": MOE_ACT_GELU, "swiglu": MOE_ACT_SWIGLU, "identity": MOE_ACT_IDENTITY}
_SCORES = {"softmax": MOE_SCORE_SOFTMAX, "sigmoid": MOE_SCORE_SIGMOID}
_DTYPES = {"f32": MOE_DTYPE_F32, "bf16": MOE_DTYPE_BF16, torch.float32: MOE_DTYPE_F32,
           torch.bfloat16: MOE_DTYPE_BF16}


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


class moe_config(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("R", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("act_dtype", ctypes.c_int32),
                ("score", ctypes.c_int32), ("renorm", ctypes.c_int32),
                ("capacity_factor", ctypes.c_float), ("capacity", ctypes.c_int32),
                ("act", ctypes.c_int32), ("add_residual", ctypes.c_int32),
                ("max_ranks", ctypes.c_int32)]


class moe_buffers(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("topk_idx", "topk_gate", "slot_row", "row_token", "expert_counts",
                 "expert_offsets", "rank_counts", "rank_splits", "n_dropped", "xp", "h", "yp",
                 "shared_h", "shared_out")]


_lib = None


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"CUDA library not built: {LIB_PATH} "
                          "(run python -m expert_dispatch_top_b300.build)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, cfgp, i32 = ctypes.c_void_p, ctypes.POINTER(moe_config), ctypes.c_int
    lib.moe_status_string.argtypes = [i32]
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_check_config.argtypes = [cfgp]
    lib.moe_check_config.restype = i32
    lib.moe_workspace_size.argtypes = [cfgp]
    lib.moe_workspace_size.restype = ctypes.c_size_t
    lib.moe_capacity.argtypes = [cfgp]
    lib.moe_capacity.restype = ctypes.c_int64
    lib.moe_max_rows.argtypes = [cfgp]
    lib.moe_max_rows.restype = ctypes.c_int64
    lib.moe_route.argtypes = [cfgp] + [vp] * 8
    lib.moe_route.restype = i32
    lib.moe_dispatch.argtypes = [cfgp] + [vp] * 12
    lib.moe_dispatch.restype = i32
    lib.moe_test_expert_ffn_stall.argtypes = [cfgp] + [vp] * 4 + [ctypes.c_int32, ctypes.c_uint32,
                                                                vp, vp]
    lib.moe_test_expert_ffn_stall.restype = i32
    lib.moe_dispatch_noalloc.argtypes = [cfgp] + [vp] * 12
    lib.moe_dispatch_noalloc.restype = i32
    lib.moe_expert_ffn.argtypes = [cfgp] + [vp] * 13
    lib.moe_expert_ffn.restype = i32
    lib.moe_combine.argtypes = [cfgp] + [vp] * 7
    lib.moe_combine.restype = i32
    lib.moe_layer_forward.argtypes = [cfgp] + [vp] * 8 + [ctypes.POINTER(moe_buffers), vp, vp, vp]
    lib.moe_layer_forward.restype = i32
    lib.moe_layer_forward_host.argtypes = [cfgp] + [vp] * 9 + [ctypes.POINTER(moe_buffers), vp, vp,
                                                              vp, vp]
    lib.moe_layer_forward_host.restype = i32
    lib.moe_route_backward.argtypes = [cfgp] + [vp] * 10
    lib.moe_route_backward.restype = i32
    lib.moe_combine_backward.argtypes = [cfgp] + [vp] * 7
    lib.moe_combine_backward.restype = i32
    lib.moe_dispatch_backward.argtypes = [cfgp] + [vp] * 4
    lib.moe_dispatch_backward.restype = i32
    lib.moe_expert_ffn_backward_scratch_size.argtypes = [cfgp, i32]
    lib.moe_expert_ffn_backward_scratch_size.restype = ctypes.c_size_t
    lib.moe_expert_ffn_backward.argtypes = [cfgp] + [vp] * 9 + [ctypes.c_size_t, vp, vp]
    lib.moe_expert_ffn_backward.restype = i32
    lib.moe_update_sel_bias.argtypes = [cfgp, vp, vp, ctypes.c_float, vp]
    lib.moe_update_sel_bias.restype = i32
    lib.moe_read_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp]
    lib.moe_read_device_status.restype = i32
    lib.moe_build_checked.argtypes = []
    lib.moe_build_checked.restype = i32
    lib.moe_launch_count.argtypes = []
    lib.moe_launch_count.restype = ctypes.c_uint64
    _lib = lib
    return lib


def library():
    """The loaded ctypes library (raises ImportError if it is not built)."""
    return _load()


def status_string(status: int) -> str:
    return _load().moe_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoeError(status, where)


def _p(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def make_config(T, d, E, k, R, d_ff=0, n_shared=0, dtype="bf16", score="softmax", renorm=True,
                capacity_factor=0.0, capacity=0, act="swiglu", add_residual=False,
                max_ranks=0) -> moe_config:
    return moe_config(int(T), int(d), int(E), int(k), int(R), int(d_ff), int(n_shared),
                      _DTYPES[dtype], _SCORES[score], int(bool(renorm)), float(capacity_factor),
                      int(capacity), _ACTS[act], int(bool(add_residual)), int(max_ranks))


def config_from_workload(w, T: Optional[int] = None, add_residual: Optional[bool] = None,
                         capacity: int = 0) -> moe_config:
    """moe_config of a workload description (any object with the Workload fields)."""
    return make_config(w.T if T is None else T, w.d, w.E, w.k, w.R, w.d_ff, w.n_shared, w.dtype,
                       w.score, w.renorm, w.capacity_factor, capacity, w.act,
                       w.add_residual if add_residual is None else add_residual,
                       getattr(w, "max_ranks", 0))


def moe_check_config(cfg: moe_config) -> int:
    return int(_load().moe_check_config(ctypes.byref(cfg)))


def moe_workspace_size(cfg: moe_config) -> int:
    return int(_load().moe_workspace_size(ctypes.byref(cfg)))


def moe_capacity(cfg: moe_config) -> int:
    return int(_load().moe_capacity(ctypes.byref(cfg)))


def moe_max_rows(cfg: moe_config) -> int:
    return int(_load().moe_max_rows(ctypes.byref(cfg)))


def alloc_workspace(cfg: moe_config, device=None) -> torch.Tensor:
    n = moe_workspace_size(cfg)
    if n == 0:
        raise MoeError(moe_check_config(cfg) or MOE_ERR_INVALID_ARG, "moe_workspace_size")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def moe_route(cfg, x, w_router, logit_bias, sel_bias, topk_idx, topk_gate, ws, stream=None):
    _check(_load().moe_route(ctypes.byref(cfg), _p(x), _p(w_router), _p(logit_bias), _p(sel_bias),
                             _p(topk_idx), _p(topk_gate), _p(ws), _stream(stream)), "moe_route")


def moe_dispatch(cfg, x, topk_idx, xp, row_token, slot_row, expert_counts, expert_offsets,
                 rank_counts, rank_splits, n_dropped, ws, stream=None):
    _check(_load().moe_dispatch(ctypes.byref(cfg), _p(x), _p(topk_idx), _p(xp), _p(row_token),
                                _p(slot_row), _p(expert_counts), _p(expert_offsets),
                                _p(rank_counts), _p(rank_splits), _p(n_dropped), _p(ws),
                                _stream(stream)), "moe_dispatch")


def moe_test_expert_ffn_stall(cfg, xp, expert_offsets, w_up, h, stall_kb, wait_limit_us, ws,
                              stream=None):
    """Failure-detection hook: the FFN up projection with one pipeline stage
    never loaded; the bounded wait runs out and sets MOE_DEV_GEMM_TIMEOUT."""
    _check(_load().moe_test_expert_ffn_stall(ctypes.byref(cfg), _p(xp), _p(expert_offsets),
                                             _p(w_up), _p(h), int(stall_kb), int(wait_limit_us),
                                             _p(ws), _stream(stream)), "moe_test_expert_ffn_stall")


def moe_dispatch_noalloc(cfg, x, topk_idx, xp, row_token, slot_row, expert_counts, expert_offsets,
                         rank_counts, rank_splits, n_dropped, device_status=None, stream=None):
    """moe_dispatch with its scratch in the library's fixed device array (no
    workspace argument, nothing allocated); for callers that cannot allocate."""
    _check(_load().moe_dispatch_noalloc(ctypes.byref(cfg), _p(x), _p(topk_idx), _p(xp),
                                        _p(row_token), _p(slot_row), _p(expert_counts),
                                        _p(expert_offsets), _p(rank_counts), _p(rank_splits),
                                        _p(n_dropped), _p(device_status), _stream(stream)),
           "moe_dispatch_noalloc")


def moe_expert_ffn(cfg, xp, expert_offsets, w_up, w_down, h, yp, shared_x=None, shared_up=None,
                   shared_down=None, shared_h=None, shared_out=None, ws=None, stream=None):
    _check(_load().moe_expert_ffn(ctypes.byref(cfg), _p(xp), _p(expert_offsets), _p(w_up),
                                  _p(w_down), _p(h), _p(yp), _p(shared_x), _p(shared_up),
                                  _p(shared_down), _p(shared_h), _p(shared_out), _p(ws),
                                  _stream(stream)), "moe_expert_ffn")


def moe_combine(cfg, yp, slot_row, topk_gate, shared_out, x_residual, y, stream=None):
    _check(_load().moe_combine(ctypes.byref(cfg), _p(yp), _p(slot_row), _p(topk_gate),
                               _p(shared_out), _p(x_residual), _p(y), _stream(stream)),
           "moe_combine")


def moe_layer_forward(cfg, x, w_router, logit_bias, sel_bias, w_up, w_down, shared_up, shared_down,
                      buffers: moe_buffers, y, ws, stream=None):
    _check(_load().moe_layer_forward(ctypes.byref(cfg), _p(x), _p(w_router), _p(logit_bias),
                                     _p(sel_bias), _p(w_up), _p(w_down), _p(shared_up),
                                     _p(shared_down), ctypes.byref(buffers), _p(y), _p(ws),
                                     _stream(stream)), "moe_layer_forward")


def moe_route_backward(cfg, x, w_router, logit_bias, topk_idx, d_gate, d_logits, dx=None,
                       d_w_router=None, d_logit_bias=None, stream=None):
    """Backward of the router through its gates: d_logits [T,E] fp32 and, when
    given, dx [T,d], d_w_router [E,d] and d_logit_bias [E]."""
    _check(_load().moe_route_backward(ctypes.byref(cfg), _p(x), _p(w_router), _p(logit_bias),
                                      _p(topk_idx), _p(d_gate), _p(d_logits), _p(dx),
                                      _p(d_w_router), _p(d_logit_bias), _stream(stream)),
           "moe_route_backward")


def moe_layer_forward_host(cfg, x_host, x_dev, w_router, logit_bias, sel_bias, w_up, w_down,
                           shared_up, shared_down, buffers: moe_buffers, y_dev, y_host, ws,
                           stream=None):
    """The layer with host input and output (x_host, y_host: CPU tensors, pinned for
    asynchronous copies); x_dev, y_dev: device staging tensors [T, d]."""
    _check(_load().moe_layer_forward_host(ctypes.byref(cfg), _p(x_host), _p(x_dev), _p(w_router),
                                          _p(logit_bias), _p(sel_bias), _p(w_up), _p(w_down),
                                          _p(shared_up), _p(shared_down), ctypes.byref(buffers),
                                          _p(y_dev), _p(y_host), _p(ws), _stream(stream)),
           "moe_layer_forward_host")


def moe_combine_backward(cfg, dy, yp, slot_row, topk_gate, d_yp, d_gate, stream=None):
    """Reverse of the combine exchange: d_yp rows and gate gradients."""
    _check(_load().moe_combine_backward(ctypes.byref(cfg), _p(dy), _p(yp), _p(slot_row),
                                        _p(topk_gate), _p(d_yp), _p(d_gate), _stream(stream)),
           "moe_combine_backward")


def moe_dispatch_backward(cfg, d_xp, slot_row, dx, stream=None):
    """Reverse of the dispatch exchange: dx[t] = sum of its kept rows' gradients."""
    _check(_load().moe_dispatch_backward(ctypes.byref(cfg), _p(d_xp), _p(slot_row), _p(dx),
                                         _stream(stream)), "moe_dispatch_backward")


def moe_expert_ffn_backward_scratch_size(cfg, weight_grads=True) -> int:
    return int(_load().moe_expert_ffn_backward_scratch_size(ctypes.byref(cfg), int(bool(weight_grads))))


def moe_expert_ffn_backward(cfg, xp, expert_offsets, w_up, w_down, d_yp, d_xp, d_w_up, d_w_down,
                            scratch, ws, stream=None):
    """Backward through the expert FFNs: d_xp and (when not None) the weight
    gradients d_w_up, d_w_down; scratch is a uint8 device tensor of at least
    moe_expert_ffn_backward_scratch_size bytes."""
    nbytes = 0 if scratch is None else scratch.numel() * scratch.element_size()
    _check(_load().moe_expert_ffn_backward(ctypes.byref(cfg), _p(xp), _p(expert_offsets), _p(w_up),
                                           _p(w_down), _p(d_yp), _p(d_xp), _p(d_w_up),
                                           _p(d_w_down), _p(scratch), ctypes.c_size_t(nbytes),
                                           _p(ws), _stream(stream)), "moe_expert_ffn_backward")


def moe_update_sel_bias(cfg, expert_counts, sel_bias, gamma, stream=None):
    """Bias-based balancing step on the device: sel_bias -= gamma for experts
    above the even share T*k/E, += gamma below it (in place)."""
    _check(_load().moe_update_sel_bias(ctypes.byref(cfg), _p(expert_counts), _p(sel_bias),
                                       ctypes.c_float(gamma), _stream(stream)),
           "moe_update_sel_bias")


def moe_build_checked() -> bool:
    """True if the loaded library is the range-checked debugging build."""
    return bool(_load().moe_build_checked())


def moe_launch_count() -> int:
    """Kernel launches the library has enqueued since it loaded (all threads)."""
    return int(_load().moe_launch_count())


def moe_read_device_status(ws, stream=None) -> int:
    out = ctypes.c_uint32(0)
    _check(_load().moe_read_device_status(_p(ws), ctypes.byref(out), _stream(stream)),
           "moe_read_device_status")
    return int(out.value)


@dataclass
class LayerBuffers:
    """Every buffer of one layer call, allocated with torch on one device."""
    topk_idx: torch.Tensor
    topk_gate: torch.Tensor
    slot_row: torch.Tensor
    row_token: torch.Tensor
    expert_counts: torch.Tensor
    expert_offsets: torch.Tensor
    rank_counts: torch.Tensor
    rank_splits: torch.Tensor
    n_dropped: torch.Tensor
    xp: torch.Tensor
    h: Optional[torch.Tensor]
    yp: Optional[torch.Tensor]
    shared_h: Optional[torch.Tensor]
    shared_out: Optional[torch.Tensor]
    y: torch.Tensor
    ws: torch.Tensor

    def c_struct(self) -> moe_buffers:
        return moe_buffers(*[_p(getattr(self, n)) for n, _ in moe_buffers._fields_])


def alloc_buffers(cfg: moe_config, device="cuda") -> LayerBuffers:
    dt = torch.float32 if cfg.act_dtype == MOE_DTYPE_F32 else torch.bfloat16
    T, d, E, k, R, f = cfg.T, cfg.d, cfg.E, cfg.k, cfg.R, cfg.d_ff
    rows = max(moe_max_rows(cfg), 1)
    ident = cfg.act == MOE_ACT_IDENTITY
    i32 = dict(dtype=torch.int32, device=device)
    return LayerBuffers(
        topk_idx=torch.empty((T, k), **i32), topk_gate=torch.empty((T, k), dtype=torch.float32,
                                                                    device=device),
        slot_row=torch.empty((T, k), **i32), row_token=torch.empty((rows,), **i32),
        expert_counts=torch.empty((E,), **i32), expert_offsets=torch.empty((E + 1,), **i32),
        rank_counts=torch.empty((R,), **i32), rank_splits=torch.empty((R, R), **i32),
        n_dropped=torch.empty((1,), **i32),
        xp=torch.empty((rows, d), dtype=dt, device=device),
        h=None if ident else torch.empty((rows, f), dtype=dt, device=device),
        yp=None if ident else torch.empty((rows, d), dtype=dt, device=device),
        shared_h=torch.empty((T, f), dtype=dt, device=device) if cfg.n_shared else None,
        shared_out=torch.empty((T, d), dtype=dt, device=device) if cfg.n_shared else None,
        y=torch.empty((T, d), dtype=dt, device=device),
        ws=alloc_workspace(cfg, device))


class MoeLayer:
    """One MoE layer: a config, its weights and its buffers; ``forward(x)``
    runs route -> dispatch -> expert FFN -> combine through moe_layer_forward."""

    def __init__(self, cfg: moe_config, w_router, w_up=None, w_down=None, shared_up=None,
                 shared_down=None, logit_bias=None, sel_bias=None, device="cuda"):
        self.cfg = cfg
        self.w_router, self.w_up, self.w_down = w_router, w_up, w_down
        self.shared_up, self.shared_down = shared_up, shared_down
        self.logit_bias, self.sel_bias = logit_bias, sel_bias
        self.buf = alloc_buffers(cfg, device)
        self._cbuf = self.buf.c_struct()

    def forward(self, x, stream=None) -> torch.Tensor:
        moe_layer_forward(self.cfg, x, self.w_router, self.logit_bias, self.sel_bias, self.w_up,
                          self.w_down, self.shared_up, self.shared_down, self._cbuf, self.buf.y,
                          self.buf.ws, stream)
        return self.buf.y

    __call__ = forward

    def forward_host(self, x_host, y_host, x_dev=None, stream=None):
        """Host x in, host y out through moe_layer_forward_host (x_dev: an optional
        device staging tensor; the layer's own y buffer receives the result on the
        device).  Returns y_host."""
        if x_dev is None:
            if getattr(self, "_x_dev", None) is None:
                self._x_dev = torch.empty_like(self.buf.y)
            x_dev = self._x_dev
        moe_layer_forward_host(self.cfg, x_host, x_dev, self.w_router, self.logit_bias,
                               self.sel_bias, self.w_up, self.w_down, self.shared_up,
                               self.shared_down, self._cbuf, self.buf.y, y_host, self.buf.ws,
                               stream)
        return y_host

    def device_status(self) -> int:
        return moe_read_device_status(self.buf.ws)


__all__ = [n for n in dir() if n.startswith(("moe_", "MOE_", "Moe", "make_", "alloc_", "config_"))] + \
    ["library", "status_string", "LayerBuffers", "LIB_PATH"]

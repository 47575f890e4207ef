"""Thin ctypes binding of libmoe.so (include/moe.h).

Argument marshalling only: torch tensors are checked for device, dtype,
contiguity and size, and passed to the C ABI as raw pointers on the current
CUDA stream.  Every step of the MoE layer runs in the library's kernels; if
the library is missing this module raises at import, there is no fallback.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import torch

from . import workloads as W

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_DEVICE = range(5)
MOE_DEV_OK, MOE_DEV_BAD_EXPERT_ID, MOE_DEV_TIMEOUT, MOE_DEV_BAD_ROW, MOE_DEV_BAD_OFFSETS = range(5)

EXPORTS = ("moe_version", "moe_status_string", "moe_last_error", "moe_capacity", "moe_workspace_size",
           "moe_route", "moe_balance_bias_update", "moe_dispatch", "moe_dispatch_noalloc", "moe_expert_ffn",
           "moe_shared_ffn", "moe_combine", "moe_layer_forward", "moe_get_device_status", "moe_combine_backward",
           "moe_route_backward", "moe_expert_ffn_backward", "moe_dispatch_backward", "moe_router_input_backward",
           "moe_layer_backward", "moe_quantize_fp8", "moe_dispatch_fp8", "moe_expert_ffn_fp8",
           "moe_layer_forward_fp8", "moe_expert_ffn_gather", "moe_router_pack_size", "moe_pack_router",
           "moe_route_packed")


class MoeError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_name(status)}: {message}")
        self.status = status


class moe_config(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("h", ctypes.c_int32), ("E", ctypes.c_int32), ("k", ctypes.c_int32),
                ("d_e", ctypes.c_int32), ("capacity_factor", ctypes.c_float), ("capacity", ctypes.c_int32),
                ("score_fn", ctypes.c_int32), ("renorm", ctypes.c_int32), ("noisy", ctypes.c_int32),
                ("priority", ctypes.c_int32), ("dtype", ctypes.c_int32), ("n_shared", ctypes.c_int32),
                ("d_shared", ctypes.c_int32), ("n_group", ctypes.c_int32), ("topk_group", ctypes.c_int32)]


_P = ctypes.c_void_p


class moe_layer_args(ctypes.Structure):
    _fields_ = [(n, _P) for n in (
        "U", "W_r", "b_r", "W_noise", "eps", "W_gate", "W_up", "W_down", "logits_out", "idx", "gate",
        "counts_routed", "counts_kept", "offsets", "slot_row", "row_token", "n_dropped", "X", "act", "Y",
        "out", "f", "P", "aux", "z_loss", "sel_bias", "W_gate_shared", "W_up_shared", "W_down_shared",
        "act_shared", "Y_shared", "W_r_packed")]


class moe_fp8_args(ctypes.Structure):
    _fields_ = [(n, _P) for n in ("X8", "x_scale", "W_gate8", "W_up8", "s_gate", "s_up")]


class moe_layer_grads(ctypes.Structure):
    _fields_ = ([("dO", _P), ("w_aux", ctypes.c_float), ("w_z", ctypes.c_float)] +
                [(n, _P) for n in ("d_gate", "dY", "dH", "d_act", "dG", "dUp", "dX", "dU_router", "d_act_shared",
                                   "dG_shared", "dUp_shared", "dX_shared", "dU", "dW_gate", "dW_up", "dW_down",
                                   "dW_r", "db_r", "dW_noise", "dW_gate_shared", "dW_up_shared", "dW_down_shared")])


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmoe.so is not built ({LIB_PATH}); run "
                          "`python -m mixture_experts_layer_84_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    S, I64, SZ = ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    cfgp = ctypes.POINTER(moe_config)
    lib.moe_version.restype = ctypes.c_char_p
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_status_string.argtypes = [S]
    lib.moe_last_error.restype = ctypes.c_char_p
    lib.moe_capacity.restype = S
    lib.moe_capacity.argtypes = [cfgp, ctypes.POINTER(I64)]
    lib.moe_workspace_size.restype = S
    lib.moe_workspace_size.argtypes = [cfgp, ctypes.POINTER(SZ)]
    lib.moe_route.restype = S
    lib.moe_route.argtypes = [cfgp] + [_P] * 10 + [_P, _P]
    lib.moe_router_pack_size.restype = S
    lib.moe_router_pack_size.argtypes = [cfgp, ctypes.POINTER(SZ)]
    lib.moe_pack_router.restype = S
    lib.moe_pack_router.argtypes = [cfgp, _P, _P, _P, _P]
    lib.moe_route_packed.restype = S
    lib.moe_route_packed.argtypes = [cfgp] + [_P] * 10
    lib.moe_balance_bias_update.restype = S
    lib.moe_balance_bias_update.argtypes = [cfgp, _P, ctypes.c_float, _P, _P]
    lib.moe_shared_ffn.restype = S
    lib.moe_shared_ffn.argtypes = [cfgp] + [_P] * 6 + [_P, _P]
    lib.moe_dispatch.restype = S
    lib.moe_dispatch.argtypes = [cfgp] + [_P] * 9 + [_P, _P]
    lib.moe_dispatch_noalloc.restype = S
    lib.moe_dispatch_noalloc.argtypes = [cfgp] + [_P] * 10 + [_P]
    lib.moe_expert_ffn.restype = S
    lib.moe_expert_ffn.argtypes = [cfgp] + [_P] * 7 + [_P, _P]
    lib.moe_combine.restype = S
    lib.moe_combine.argtypes = [cfgp] + [_P] * 11 + [_P, _P]
    lib.moe_combine_backward.restype = S
    lib.moe_combine_backward.argtypes = [cfgp] + [_P] * 6 + [_P, _P]
    lib.moe_route_backward.restype = S
    lib.moe_route_backward.argtypes = [cfgp, _P, _P, _P, _P, ctypes.c_float, ctypes.c_float, _P, _P]
    lib.moe_expert_ffn_backward.restype = S
    lib.moe_expert_ffn_backward.argtypes = [cfgp] + [_P] * 14 + [_P, _P]
    lib.moe_dispatch_backward.restype = S
    lib.moe_dispatch_backward.argtypes = [cfgp] + [_P] * 4 + [_P, _P]
    lib.moe_router_input_backward.restype = S
    lib.moe_router_input_backward.argtypes = [cfgp] + [_P] * 9 + [_P, _P]
    lib.moe_layer_backward.restype = S
    lib.moe_layer_backward.argtypes = [cfgp, ctypes.POINTER(moe_layer_args), ctypes.POINTER(moe_layer_grads), _P, _P]
    lib.moe_layer_forward.restype = S
    lib.moe_layer_forward.argtypes = [cfgp, ctypes.POINTER(moe_layer_args), _P, _P]
    lib.moe_expert_ffn_gather.restype = S
    lib.moe_expert_ffn_gather.argtypes = [cfgp] + [_P] * 8 + [_P, _P]
    lib.moe_quantize_fp8.restype = S
    lib.moe_quantize_fp8.argtypes = [I64, ctypes.c_int32, _P, _P, _P, _P]
    lib.moe_dispatch_fp8.restype = S
    lib.moe_dispatch_fp8.argtypes = [cfgp] + [_P] * 10 + [_P, _P]
    lib.moe_expert_ffn_fp8.restype = S
    lib.moe_expert_ffn_fp8.argtypes = [cfgp] + [_P] * 10 + [_P, _P]
    lib.moe_layer_forward_fp8.restype = S
    lib.moe_layer_forward_fp8.argtypes = [cfgp, ctypes.POINTER(moe_layer_args), ctypes.POINTER(moe_fp8_args), _P,
                                          _P]
    lib.moe_get_device_status.restype = S
    lib.moe_get_device_status.argtypes = [_P, _P, ctypes.POINTER(ctypes.c_int32)]
    return lib


lib = _load()


def status_name(status: int) -> str:
    return lib.moe_status_string(int(status)).decode()


def version() -> str:
    return lib.moe_version().decode()


def _check(status: int) -> None:
    if status != MOE_OK:
        raise MoeError(status, lib.moe_last_error().decode())


def config(T, h, E, k, d_e, *, capacity_factor=0.0, capacity=0, score_fn=W.SOFTMAX, renorm=True, noisy=False,
           priority=W.PRIORITY_CHOICE_MAJOR, dtype=W.BF16, n_shared=0, d_shared=0, n_group=0,
           topk_group=0) -> moe_config:
    return moe_config(int(T), int(h), int(E), int(k), int(d_e), float(capacity_factor), int(capacity),
                      int(score_fn), int(bool(renorm)), int(bool(noisy)), int(priority), int(dtype), int(n_shared),
                      int(d_shared), int(n_group), int(topk_group))


def config_of(w: W.Workload, **override) -> moe_config:
    kw = dict(capacity_factor=w.capacity_factor, capacity=w.capacity, score_fn=w.score_fn, renorm=w.renorm,
              noisy=w.noisy, priority=w.priority, dtype=w.dtype, n_shared=w.n_shared, d_shared=w.d_shared,
              n_group=w.n_group, topk_group=w.topk_group)
    kw.update(override)
    T = kw.pop("T", w.T)
    return config(T, w.h, w.E, w.k, w.d_e, **kw)


def capacity(cfg: moe_config) -> int:
    c = ctypes.c_int64()
    _check(lib.moe_capacity(ctypes.byref(cfg), ctypes.byref(c)))
    return c.value


def workspace_size(cfg: moe_config) -> int:
    n = ctypes.c_size_t()
    _check(lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def _act_dtype(cfg: moe_config):
    return torch.bfloat16 if cfg.dtype == W.BF16 else torch.float32


def _ptr(t: Optional[torch.Tensor], name: str, dtype=None, numel: Optional[int] = None) -> Optional[int]:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name}: must be a CUDA tensor (got {t.device})")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name}: {t.numel()} elements, need {numel}")
    return t.data_ptr() if t.numel() > 0 else None


def _stream(stream) -> Optional[int]:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream if s.cuda_stream else None


def new_workspace(cfg: moe_config, device="cuda") -> torch.Tensor:
    """A zero-filled workspace of moe_workspace_size() bytes (256-byte aligned by the allocator)."""
    return torch.zeros(max(workspace_size(cfg), 256), dtype=torch.uint8, device=device)


def moe_route(cfg, U, W_r, b_r, W_noise, eps, logits_in, logits_out, idx, gate, ws, stream=None, sel_bias=None):
    dt = _act_dtype(cfg)
    T, E, k, h = cfg.T, cfg.E, cfg.k, cfg.h
    _check(lib.moe_route(ctypes.byref(cfg), _ptr(U, "U", dt, T * h) if logits_in is None else None,
                         _ptr(W_r, "W_r", dt, h * E) if logits_in is None else None,
                         _ptr(b_r, "b_r", torch.float32, E), _ptr(sel_bias, "sel_bias", torch.float32, E),
                         _ptr(W_noise, "W_noise", dt, h * E),
                         _ptr(eps, "eps", torch.float32, T * E), _ptr(logits_in, "logits_in", torch.float32, T * E),
                         _ptr(logits_out, "logits_out", torch.float32, T * E), _ptr(idx, "idx", torch.int32, T * k),
                         _ptr(gate, "gate", torch.float32, T * k), _ptr(ws, "ws"), _stream(stream)))


def moe_dispatch(cfg, U, idx, counts_routed, counts_kept, offsets, slot_row, row_token, X, n_dropped, ws,
                 stream=None):
    dt = _act_dtype(cfg)
    T, E, k, h = cfg.T, cfg.E, cfg.k, cfg.h
    _check(lib.moe_dispatch(ctypes.byref(cfg), _ptr(U, "U", dt, T * h), _ptr(idx, "idx", torch.int32, T * k),
                            _ptr(counts_routed, "counts_routed", torch.int32, E),
                            _ptr(counts_kept, "counts_kept", torch.int32, E),
                            _ptr(offsets, "offsets", torch.int32, E + 1),
                            _ptr(slot_row, "slot_row", torch.int32, T * k),
                            _ptr(row_token, "row_token", torch.int32, T * k), _ptr(X, "X", dt, T * k * h),
                            _ptr(n_dropped, "n_dropped", torch.int64, 1), _ptr(ws, "ws"), _stream(stream)))


def moe_dispatch_noalloc(cfg, U, idx, counts_routed, counts_kept, offsets, slot_row, row_token, X, n_dropped,
                         status=None, stream=None):
    """moe_dispatch without a workspace: the histogram scratch is the library's static device array."""
    dt = _act_dtype(cfg)
    T, E, k, h = cfg.T, cfg.E, cfg.k, cfg.h
    _check(lib.moe_dispatch_noalloc(ctypes.byref(cfg), _ptr(U, "U", dt, T * h),
                                    _ptr(idx, "idx", torch.int32, T * k),
                                    _ptr(counts_routed, "counts_routed", torch.int32, E),
                                    _ptr(counts_kept, "counts_kept", torch.int32, E),
                                    _ptr(offsets, "offsets", torch.int32, E + 1),
                                    _ptr(slot_row, "slot_row", torch.int32, T * k),
                                    _ptr(row_token, "row_token", torch.int32, T * k), _ptr(X, "X", dt, T * k * h),
                                    _ptr(n_dropped, "n_dropped", torch.int64, 1),
                                    _ptr(status, "status", torch.int32, 1), _stream(stream)))


def router_pack_size(cfg: moe_config) -> int:
    n = ctypes.c_size_t()
    _check(lib.moe_router_pack_size(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def moe_pack_router(cfg, W_r, W_noise, stream=None) -> Optional[torch.Tensor]:
    """The router weights packed once for the tensor-core router ([N, h] bf16), or None when the
    config's router reads W_r as it is."""
    n = router_pack_size(cfg)
    if n == 0:
        return None
    dt = _act_dtype(cfg)
    out = torch.empty(n // 2, dtype=torch.bfloat16, device=W_r.device)
    _check(lib.moe_pack_router(ctypes.byref(cfg), _ptr(W_r, "W_r", dt, cfg.h * cfg.E),
                               _ptr(W_noise, "W_noise", dt, cfg.h * cfg.E) if cfg.noisy else None,
                               _ptr(out, "W_r_packed"), _stream(stream)))
    return out


def moe_route_packed(cfg, U, W_r_packed, b_r, eps, logits_out, idx, gate, ws, stream=None, sel_bias=None):
    dt = _act_dtype(cfg)
    T, E, k, h = cfg.T, cfg.E, cfg.k, cfg.h
    _check(lib.moe_route_packed(ctypes.byref(cfg), _ptr(U, "U", dt, T * h), _ptr(W_r_packed, "W_r_packed"),
                                _ptr(b_r, "b_r", torch.float32, E), _ptr(sel_bias, "sel_bias", torch.float32, E),
                                _ptr(eps, "eps", torch.float32, T * E) if cfg.noisy else None,
                                _ptr(logits_out, "logits_out", torch.float32, T * E),
                                _ptr(idx, "idx", torch.int32, T * k), _ptr(gate, "gate", torch.float32, T * k),
                                _ptr(ws, "ws"), _stream(stream)))


def moe_balance_bias_update(cfg, counts_routed, u, bias, stream=None):
    """bias += u * sign(mean(counts) - counts), in place on the device."""
    _check(lib.moe_balance_bias_update(ctypes.byref(cfg), _ptr(counts_routed, "counts_routed", torch.int32, cfg.E),
                                       float(u), _ptr(bias, "bias", torch.float32, cfg.E), _stream(stream)))


def moe_shared_ffn(cfg, U, W_gate_sh, W_up_sh, W_down_sh, act_sh, Y_sh, ws, stream=None):
    dt = _act_dtype(cfg)
    T, h, ns, ds = cfg.T, cfg.h, cfg.n_shared, cfg.d_shared
    _check(lib.moe_shared_ffn(ctypes.byref(cfg), _ptr(U, "U", dt, T * h), _ptr(W_gate_sh, "W_gate_sh", dt, ns * ds * h),
                              _ptr(W_up_sh, "W_up_sh", dt, ns * ds * h), _ptr(W_down_sh, "W_down_sh", dt, ns * h * ds),
                              _ptr(act_sh, "act_sh", dt, ns * T * ds), _ptr(Y_sh, "Y_sh", dt, ns * T * h), _ptr(ws, "ws"),
                              _stream(stream)))


def moe_expert_ffn(cfg, X, offsets, W_gate, W_up, W_down, act, Y, ws, stream=None):
    dt = _act_dtype(cfg)
    T, E, k, h, d = cfg.T, cfg.E, cfg.k, cfg.h, cfg.d_e
    _check(lib.moe_expert_ffn(ctypes.byref(cfg), _ptr(X, "X", dt, T * k * h),
                              _ptr(offsets, "offsets", torch.int32, E + 1), _ptr(W_gate, "W_gate", dt, E * d * h),
                              _ptr(W_up, "W_up", dt, E * d * h), _ptr(W_down, "W_down", dt, E * h * d),
                              _ptr(act, "act", dt, T * k * d), _ptr(Y, "Y", dt, T * k * h), _ptr(ws, "ws"),
                              _stream(stream)))


def moe_combine(cfg, U, Y, slot_row, gate, counts_routed, out, f, P, aux, ws, stream=None, z_loss=None,
                Y_shared=None):
    dt = _act_dtype(cfg)
    T, E, k, h = cfg.T, cfg.E, cfg.k, cfg.h
    _check(lib.moe_combine(ctypes.byref(cfg), _ptr(U, "U", dt, T * h), _ptr(Y, "Y", dt, T * k * h),
                           _ptr(Y_shared, "Y_shared", dt, cfg.n_shared * T * h),
                           _ptr(slot_row, "slot_row", torch.int32, T * k), _ptr(gate, "gate", torch.float32, T * k),
                           _ptr(counts_routed, "counts_routed", torch.int32, E), _ptr(out, "out", dt, T * h),
                           _ptr(f, "f", torch.float32, E), _ptr(P, "P", torch.float32, E),
                           _ptr(aux, "aux", torch.float32, 1), _ptr(z_loss, "z_loss", torch.float32, 1),
                           _ptr(ws, "ws"), _stream(stream)))


def moe_combine_backward(cfg, dO, Y, slot_row, gate, d_gate, dY, ws, stream=None):
    dt = _act_dtype(cfg)
    T, k, h = cfg.T, cfg.k, cfg.h
    _check(lib.moe_combine_backward(ctypes.byref(cfg), _ptr(dO, "dO", dt, T * h), _ptr(Y, "Y", dt, T * k * h),
                                    _ptr(slot_row, "slot_row", torch.int32, T * k),
                                    _ptr(gate, "gate", torch.float32, T * k),
                                    _ptr(d_gate, "d_gate", torch.float32, T * k), _ptr(dY, "dY", dt, T * k * h),
                                    _ptr(ws, "ws"), _stream(stream)))


def moe_route_backward(cfg, logits, idx, d_gate, counts_routed, w_aux, w_z, dH, stream=None):
    T, E, k = cfg.T, cfg.E, cfg.k
    _check(lib.moe_route_backward(ctypes.byref(cfg), _ptr(logits, "logits", torch.float32, T * E),
                                  _ptr(idx, "idx", torch.int32, T * k), _ptr(d_gate, "d_gate", torch.float32, T * k),
                                  _ptr(counts_routed, "counts_routed", torch.int32, E), float(w_aux), float(w_z),
                                  _ptr(dH, "dH", torch.float32, T * E), _stream(stream)))


def moe_expert_ffn_backward(cfg, X, offsets, W_gate, W_up, W_down, act, dY, d_act, dG, dUp, dX, dW_gate, dW_up,
                            dW_down, ws, stream=None):
    dt = _act_dtype(cfg)
    T, E, k, h, d = cfg.T, cfg.E, cfg.k, cfg.h, cfg.d_e
    f32 = torch.float32
    _check(lib.moe_expert_ffn_backward(
        ctypes.byref(cfg), _ptr(X, "X", dt, T * k * h), _ptr(offsets, "offsets", torch.int32, E + 1),
        _ptr(W_gate, "W_gate", dt, E * d * h), _ptr(W_up, "W_up", dt, E * d * h), _ptr(W_down, "W_down", dt, E * h * d),
        _ptr(act, "act", dt, T * k * d), _ptr(dY, "dY", dt, T * k * h), _ptr(d_act, "d_act", dt, T * k * d),
        _ptr(dG, "dG", dt, T * k * d), _ptr(dUp, "dUp", dt, T * k * d), _ptr(dX, "dX", dt, T * k * h),
        _ptr(dW_gate, "dW_gate", f32, E * d * h), _ptr(dW_up, "dW_up", f32, E * d * h),
        _ptr(dW_down, "dW_down", f32, E * h * d), _ptr(ws, "ws"), _stream(stream)))


def moe_dispatch_backward(cfg, dO, dX, slot_row, dU, ws, stream=None):
    dt = _act_dtype(cfg)
    T, k, h = cfg.T, cfg.k, cfg.h
    _check(lib.moe_dispatch_backward(ctypes.byref(cfg), _ptr(dO, "dO", dt, T * h), _ptr(dX, "dX", dt, T * k * h),
                                     _ptr(slot_row, "slot_row", torch.int32, T * k), _ptr(dU, "dU", dt, T * h),
                                     _ptr(ws, "ws"), _stream(stream)))


@dataclasses.dataclass
class LayerBuffers:
    """Device buffers for every output of one layer forward (capacity-sized X, act, Y)."""
    idx: torch.Tensor
    gate: torch.Tensor
    logits: Optional[torch.Tensor]
    counts_routed: torch.Tensor
    counts_kept: torch.Tensor
    offsets: torch.Tensor
    slot_row: torch.Tensor
    row_token: torch.Tensor
    n_dropped: torch.Tensor
    X: torch.Tensor
    act: torch.Tensor
    Y: torch.Tensor
    out: torch.Tensor
    f: torch.Tensor
    P: torch.Tensor
    aux: torch.Tensor
    z_loss: torch.Tensor
    act_shared: Optional[torch.Tensor]
    Y_shared: Optional[torch.Tensor]
    ws: torch.Tensor

    @staticmethod
    def allocate(cfg: moe_config, device="cuda", with_logits: bool = False, with_X: bool = True) -> "LayerBuffers":
        """with_X=False leaves X empty (the FP8 layer dispatches into FP8Rows instead)."""
        dt = _act_dtype(cfg)
        T, E, k, h, d = cfg.T, cfg.E, cfg.k, cfg.h, cfg.d_e
        i32, f32 = torch.int32, torch.float32
        return LayerBuffers(
            idx=torch.empty((T, k), dtype=i32, device=device), gate=torch.empty((T, k), dtype=f32, device=device),
            logits=torch.empty((T, E), dtype=f32, device=device) if with_logits else None,
            counts_routed=torch.empty(E, dtype=i32, device=device),
            counts_kept=torch.empty(E, dtype=i32, device=device),
            offsets=torch.empty(E + 1, dtype=i32, device=device),
            slot_row=torch.empty(T * k, dtype=i32, device=device),
            row_token=torch.empty(T * k, dtype=i32, device=device),
            n_dropped=torch.empty(1, dtype=torch.int64, device=device),
            X=torch.empty((T * k if with_X else 0, h), dtype=dt, device=device),
            act=torch.empty((T * k, d), dtype=dt, device=device),
            Y=torch.empty((T * k, h), dtype=dt, device=device), out=torch.empty((T, h), dtype=dt, device=device),
            f=torch.empty(E, dtype=f32, device=device), P=torch.empty(E, dtype=f32, device=device),
            aux=torch.empty(1, dtype=f32, device=device), z_loss=torch.empty(1, dtype=f32, device=device),
            act_shared=torch.empty((cfg.n_shared, T, cfg.d_shared), dtype=dt, device=device) if cfg.n_shared else None,
            Y_shared=torch.empty((cfg.n_shared, T, h), dtype=dt, device=device) if cfg.n_shared else None,
            ws=new_workspace(cfg, device))


def moe_layer_forward(cfg, U, W_r, b_r, W_noise, eps, W_gate, W_up, W_down, bufs: LayerBuffers, stream=None,
                      sel_bias=None, shared=None, W_r_packed=None):
    """The whole layer.  sel_bias: [E] loss-free selection bias; shared: (W_gate_sh, W_up_sh, W_down_sh);
    W_r_packed: the router weights from moe_pack_router (None: packed on each call)."""
    a = layer_args(cfg, U, W_r, b_r, W_noise, eps, W_gate, W_up, W_down, bufs, sel_bias, shared, W_r_packed)
    _check(lib.moe_layer_forward(ctypes.byref(cfg), ctypes.byref(a), _ptr(bufs.ws, "ws"), _stream(stream)))


def layer_args(cfg, U, W_r, b_r, W_noise, eps, W_gate, W_up, W_down, bufs: LayerBuffers, sel_bias=None,
               shared=None, W_r_packed=None) -> moe_layer_args:
    """The moe_layer_args of one layer (inputs, weights and every buffer of `bufs`)."""
    dt = _act_dtype(cfg)
    T, E, k, h, d = cfg.T, cfg.E, cfg.k, cfg.h, cfg.d_e
    ns, ds = cfg.n_shared, cfg.d_shared
    if ns and shared is None:
        raise ValueError("cfg.n_shared > 0 needs the shared experts' weights")
    sg, su, sd = shared if ns else (None, None, None)
    a = moe_layer_args(
        U=_ptr(U, "U", dt, T * h), W_r=_ptr(W_r, "W_r", dt, h * E), b_r=_ptr(b_r, "b_r", torch.float32, E),
        W_noise=_ptr(W_noise, "W_noise", dt, h * E), eps=_ptr(eps, "eps", torch.float32, T * E),
        W_gate=_ptr(W_gate, "W_gate", dt, E * d * h), W_up=_ptr(W_up, "W_up", dt, E * d * h),
        W_down=_ptr(W_down, "W_down", dt, E * h * d),
        logits_out=_ptr(bufs.logits, "logits", torch.float32, T * E),
        idx=_ptr(bufs.idx, "idx", torch.int32, T * k), gate=_ptr(bufs.gate, "gate", torch.float32, T * k),
        counts_routed=_ptr(bufs.counts_routed, "counts_routed", torch.int32, E),
        counts_kept=_ptr(bufs.counts_kept, "counts_kept", torch.int32, E),
        offsets=_ptr(bufs.offsets, "offsets", torch.int32, E + 1),
        slot_row=_ptr(bufs.slot_row, "slot_row", torch.int32, T * k),
        row_token=_ptr(bufs.row_token, "row_token", torch.int32, T * k),
        n_dropped=_ptr(bufs.n_dropped, "n_dropped", torch.int64, 1),
        X=_ptr(bufs.X, "X", dt, T * k * h) if bufs.X.numel() else None, act=_ptr(bufs.act, "act", dt, T * k * d),
        Y=_ptr(bufs.Y, "Y", dt, T * k * h), out=_ptr(bufs.out, "out", dt, T * h),
        f=_ptr(bufs.f, "f", torch.float32, E), P=_ptr(bufs.P, "P", torch.float32, E),
        aux=_ptr(bufs.aux, "aux", torch.float32, 1), z_loss=_ptr(bufs.z_loss, "z_loss", torch.float32, 1),
        sel_bias=_ptr(sel_bias, "sel_bias", torch.float32, E),
        W_gate_shared=_ptr(sg, "W_gate_shared", dt, ns * ds * h), W_up_shared=_ptr(su, "W_up_shared", dt, ns * ds * h),
        W_down_shared=_ptr(sd, "W_down_shared", dt, ns * h * ds),
        act_shared=_ptr(bufs.act_shared, "act_shared", dt, ns * T * ds) if ns else None,
        Y_shared=_ptr(bufs.Y_shared, "Y_shared", dt, ns * T * h) if ns else None,
        W_r_packed=_ptr(W_r_packed, "W_r_packed"))
    return a


def moe_expert_ffn_gather(cfg, U, row_token, offsets, W_gate, W_up, W_down, act, Y, ws, stream=None):
    """moe_expert_ffn on X[r] = U[row_token[r]] without materialising X (bf16)."""
    T, E, k, h, d = cfg.T, cfg.E, cfg.k, cfg.h, cfg.d_e
    bf = torch.bfloat16
    _check(lib.moe_expert_ffn_gather(ctypes.byref(cfg), _ptr(U, "U", bf, T * h),
                                     _ptr(row_token, "row_token", torch.int32, T * k),
                                     _ptr(offsets, "offsets", torch.int32, E + 1),
                                     _ptr(W_gate, "W_gate", bf, E * d * h), _ptr(W_up, "W_up", bf, E * d * h),
                                     _ptr(W_down, "W_down", bf, E * h * d), _ptr(act, "act", bf, T * k * d),
                                     _ptr(Y, "Y", bf, T * k * h), _ptr(ws, "ws"), _stream(stream)))


# ---- FP8 dispatch and up-projection ----------------------------------------------------------

def moe_quantize_fp8(src, dst, scale, stream=None):
    """src [rows, cols] bf16 -> dst [rows, cols] uint8 E4M3 codes, scale [rows] float32 (powers of two)."""
    if src.dim() != 2:
        raise ValueError("src: expected a [rows, cols] tensor")
    rows, cols = int(src.shape[0]), int(src.shape[1])
    _check(lib.moe_quantize_fp8(rows, cols, _ptr(src, "src", torch.bfloat16, rows * cols),
                                _ptr(dst, "dst", torch.uint8, rows * cols), _ptr(scale, "scale", torch.float32, rows),
                                _stream(stream)))


@dataclasses.dataclass
class FP8Weights:
    """The gate and up weights as E4M3 codes [E, d_e, h] with one scale per row [E * d_e]."""
    W_gate8: torch.Tensor
    W_up8: torch.Tensor
    s_gate: torch.Tensor
    s_up: torch.Tensor

    @staticmethod
    def quantize(W_gate: torch.Tensor, W_up: torch.Tensor, stream=None) -> "FP8Weights":
        E, d, h = W_gate.shape
        dev = W_gate.device
        w = FP8Weights(torch.empty((E, d, h), dtype=torch.uint8, device=dev),
                       torch.empty((E, d, h), dtype=torch.uint8, device=dev),
                       torch.empty(E * d, dtype=torch.float32, device=dev),
                       torch.empty(E * d, dtype=torch.float32, device=dev))
        moe_quantize_fp8(W_gate.reshape(E * d, h), w.W_gate8, w.s_gate, stream)
        moe_quantize_fp8(W_up.reshape(E * d, h), w.W_up8, w.s_up, stream)
        return w


@dataclasses.dataclass
class FP8Rows:
    """The dispatched token rows as E4M3 codes [T*k, h] with their scales [T*k]."""
    X8: torch.Tensor
    x_scale: torch.Tensor

    @staticmethod
    def allocate(cfg: moe_config, device="cuda") -> "FP8Rows":
        return FP8Rows(torch.empty((cfg.T * cfg.k, cfg.h), dtype=torch.uint8, device=device),
                       torch.empty(cfg.T * cfg.k, dtype=torch.float32, device=device))


def moe_dispatch_fp8(cfg, U, idx, counts_routed, counts_kept, offsets, slot_row, row_token, X8, x_scale, n_dropped,
                     ws, stream=None):
    T, E, k, h = cfg.T, cfg.E, cfg.k, cfg.h
    _check(lib.moe_dispatch_fp8(ctypes.byref(cfg), _ptr(U, "U", torch.bfloat16, T * h),
                                _ptr(idx, "idx", torch.int32, T * k),
                                _ptr(counts_routed, "counts_routed", torch.int32, E),
                                _ptr(counts_kept, "counts_kept", torch.int32, E),
                                _ptr(offsets, "offsets", torch.int32, E + 1),
                                _ptr(slot_row, "slot_row", torch.int32, T * k),
                                _ptr(row_token, "row_token", torch.int32, T * k),
                                _ptr(X8, "X8", torch.uint8, T * k * h), _ptr(x_scale, "x_scale", torch.float32, T * k),
                                _ptr(n_dropped, "n_dropped", torch.int64, 1), _ptr(ws, "ws"), _stream(stream)))


def moe_expert_ffn_fp8(cfg, X8, x_scale, offsets, w8: FP8Weights, W_down, act, Y, ws, stream=None):
    T, E, k, h, d = cfg.T, cfg.E, cfg.k, cfg.h, cfg.d_e
    _check(lib.moe_expert_ffn_fp8(ctypes.byref(cfg), _ptr(X8, "X8", torch.uint8, T * k * h),
                                  _ptr(x_scale, "x_scale", torch.float32, T * k),
                                  _ptr(offsets, "offsets", torch.int32, E + 1),
                                  _ptr(w8.W_gate8, "W_gate8", torch.uint8, E * d * h),
                                  _ptr(w8.W_up8, "W_up8", torch.uint8, E * d * h),
                                  _ptr(w8.s_gate, "s_gate", torch.float32, E * d),
                                  _ptr(w8.s_up, "s_up", torch.float32, E * d),
                                  _ptr(W_down, "W_down", torch.bfloat16, E * h * d),
                                  _ptr(act, "act", torch.bfloat16, T * k * d), _ptr(Y, "Y", torch.bfloat16, T * k * h),
                                  _ptr(ws, "ws"), _stream(stream)))


def moe_layer_forward_fp8(cfg, U, W_r, b_r, W_noise, eps, w8: FP8Weights, W_down, bufs: LayerBuffers, rows: FP8Rows,
                          stream=None, sel_bias=None, shared=None, W_r_packed=None):
    """The whole layer with the FP8 dispatch and up-projection (bufs.X is not used)."""
    a = layer_args(cfg, U, W_r, b_r, W_noise, eps, None, None, W_down, bufs, sel_bias, shared, W_r_packed)
    T, E, k, h, d = cfg.T, cfg.E, cfg.k, cfg.h, cfg.d_e
    f = moe_fp8_args(X8=_ptr(rows.X8, "X8", torch.uint8, T * k * h),
                     x_scale=_ptr(rows.x_scale, "x_scale", torch.float32, T * k),
                     W_gate8=_ptr(w8.W_gate8, "W_gate8", torch.uint8, E * d * h),
                     W_up8=_ptr(w8.W_up8, "W_up8", torch.uint8, E * d * h),
                     s_gate=_ptr(w8.s_gate, "s_gate", torch.float32, E * d),
                     s_up=_ptr(w8.s_up, "s_up", torch.float32, E * d))
    _check(lib.moe_layer_forward_fp8(ctypes.byref(cfg), ctypes.byref(a), ctypes.byref(f), _ptr(bufs.ws, "ws"),
                                     _stream(stream)))


@dataclasses.dataclass
class GradBuffers:
    """Scratch and outputs of one layer backward (bf16 configs)."""
    d_gate: torch.Tensor
    dY: torch.Tensor
    dH: torch.Tensor
    d_act: torch.Tensor
    dG: torch.Tensor
    dUp: torch.Tensor
    dX: torch.Tensor
    dU_router: torch.Tensor
    dU: torch.Tensor
    dW_gate: torch.Tensor
    dW_up: torch.Tensor
    dW_down: torch.Tensor
    dW_r: torch.Tensor
    db_r: torch.Tensor
    dW_noise: Optional[torch.Tensor]
    d_act_shared: Optional[torch.Tensor]
    dG_shared: Optional[torch.Tensor]
    dUp_shared: Optional[torch.Tensor]
    dX_shared: Optional[torch.Tensor]
    dW_gate_shared: Optional[torch.Tensor]
    dW_up_shared: Optional[torch.Tensor]
    dW_down_shared: Optional[torch.Tensor]

    @staticmethod
    def allocate(cfg: moe_config, device="cuda") -> "GradBuffers":
        dt = _act_dtype(cfg)
        T, E, k, h, d, ns, ds = cfg.T, cfg.E, cfg.k, cfg.h, cfg.d_e, cfg.n_shared, cfg.d_shared
        f32 = torch.float32

        def z(*shape, dtype=dt):
            return torch.empty(shape, dtype=dtype, device=device)
        return GradBuffers(
            d_gate=z(T, k, dtype=f32), dY=z(T * k, h), dH=z(T, E, dtype=f32), d_act=z(T * k, d), dG=z(T * k, d),
            dUp=z(T * k, d), dX=z(T * k, h), dU_router=z(T, h), dU=z(T, h), dW_gate=z(E, d, h, dtype=f32),
            dW_up=z(E, d, h, dtype=f32), dW_down=z(E, h, d, dtype=f32), dW_r=z(h, E, dtype=f32),
            db_r=z(E, dtype=f32), dW_noise=z(h, E, dtype=f32) if cfg.noisy else None,
            d_act_shared=z(T, ds) if ns else None, dG_shared=z(T, ds) if ns else None,
            dUp_shared=z(T, ds) if ns else None, dX_shared=z(ns, T, h) if ns else None,
            dW_gate_shared=z(ns, ds, h, dtype=f32) if ns else None, dW_up_shared=z(ns, ds, h, dtype=f32) if ns else None,
            dW_down_shared=z(ns, h, ds, dtype=f32) if ns else None)


def moe_layer_backward(cfg, U, W_r, b_r, W_noise, eps, W_gate, W_up, W_down, bufs: LayerBuffers, dO,
                       grads: GradBuffers, w_aux=0.0, w_z=0.0, stream=None, sel_bias=None, shared=None):
    """The whole backward for <dO, out> + w_aux E sum f P + w_z L_z; `bufs` must hold the forward's
    tensors (allocated with with_logits=True)."""
    if bufs.logits is None:
        raise ValueError("the backward needs the forward's logits (LayerBuffers.allocate(with_logits=True))")
    a = layer_args(cfg, U, W_r, b_r, W_noise, eps, W_gate, W_up, W_down, bufs, sel_bias, shared)
    dt = _act_dtype(cfg)
    g = moe_layer_grads(dO=_ptr(dO, "dO", dt, cfg.T * cfg.h), w_aux=float(w_aux), w_z=float(w_z),
                        **{f.name: _ptr(getattr(grads, f.name), f.name) for f in dataclasses.fields(grads)})
    _check(lib.moe_layer_backward(ctypes.byref(cfg), ctypes.byref(a), ctypes.byref(g), _ptr(bufs.ws, "ws"),
                                  _stream(stream)))


def moe_get_device_status(ws: torch.Tensor, stream=None) -> int:
    """Synchronises the stream and returns (and clears) the workspace's device status code."""
    code = ctypes.c_int32()
    st = lib.moe_get_device_status(_ptr(ws, "ws"), _stream(stream), ctypes.byref(code))
    if st not in (MOE_OK, MOE_ERR_DEVICE):
        _check(st)
    return code.value

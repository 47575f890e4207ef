"""Plain CPU oracle of the single-GPU MoE layer: the Python face of oracle/moe_oracle.cpp.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU legs import or run
this module; the MoE library never does, and the two share no code.  Every step of the method is
computed in moe_oracle.cpp (plain C++ loops, double accumulation, OpenMP over independent rows);
this module only marshals arguments: it makes host copies of the inputs in their own float type
(float64, float32 or bfloat16, widened exactly in C++), allocates the outputs, calls the library
through ctypes and returns numpy arrays.

The sources and the readings the oracle follows are listed in the header of moe_oracle.cpp.
Every function is pinned by the `-m "not gpu"` tests (worked examples of the pages, closed forms,
invariants, brute force and textbook special cases).

`Oracle(path)` loads one build of the library; the module-level functions are those of the
default build, oracle/libmoe_oracle.so, compiled from moe_oracle.cpp with g++ when it is missing
or older than its source.
"""
from __future__ import annotations

import ctypes

import numpy as np

from .build_oracle import CXXFLAGS, LIB, SRC, build  # noqa: F401

SOFTMAX = 0
SIGMOID = 1
CHOICE_MAJOR = 0
TOKEN_MAJOR = 1
E4M3_MAX = 448.0

_DT_F64, _DT_F32, _DT_BF16 = 0, 1, 2


def f64(a) -> np.ndarray:
    """Exact float64 copy of a numpy array or (CPU/GPU) torch tensor of any float type."""
    if hasattr(a, "detach"):
        import torch
        a = a.detach().to("cpu")
        if a.dtype in (torch.bfloat16, torch.float16):
            a = a.to(torch.float32)
        a = a.numpy()
    return np.asarray(a, dtype=np.float64)


# ------------------------------------------------------------------------------ marshalling

class _In:
    """A host copy of an input in its own float type (float64, float32 or bfloat16; anything else
    becomes float64), kept alive while the C call runs."""

    def __init__(self, x):
        self.keep, self.ptr, self.dt = None, None, _DT_F64
        if x is None:
            return
        if hasattr(x, "detach"):
            import torch
            t = x.detach()
            if t.device.type != "cpu":
                t = t.cpu()
            t = t.contiguous()
            if t.dtype == torch.bfloat16:
                self.dt = _DT_BF16
            elif t.dtype == torch.float32:
                self.dt = _DT_F32
            elif t.dtype != torch.float64:
                t = t.to(torch.float64)
            self.keep, self.ptr, self.shape = t, t.data_ptr(), tuple(t.shape)
            return
        a = np.ascontiguousarray(x)
        if a.dtype == np.float32:
            self.dt = _DT_F32
        elif a.dtype != np.float64:
            a = np.ascontiguousarray(a, dtype=np.float64)
        self.keep, self.ptr, self.shape = a, a.ctypes.data, a.shape


def _d(x) -> np.ndarray:
    return np.ascontiguousarray(f64(x))


def _i(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x), dtype=np.int64)


def _p(a):
    return None if a is None else a.ctypes.data


_P, _I64, _I32, _F64, _F32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_float
_SIGNATURES = {
    "orc_threads": (_I32, []),
    "orc_set_threads": (None, [_I32]),
    "orc_softplus": (None, [_I64, _P, _P]),
    "orc_round_f32": (None, [_I64, _P, _P]),
    "orc_router_logits": (None, [_I64, _I32, _I32] + [_P, _I32] * 5 + [_P]),
    "orc_scores": (None, [_I64, _I32, _P, _I32, _P]),
    "orc_topk": (None, [_I64, _I32, _P, _I32, _P, _P]),
    "orc_group_scores": (None, [_I64, _I32, _P, _I32, _I32, _P]),
    "orc_group_limited_mask": (None, [_I64, _I32, _P, _I32, _I32, _I32, _P]),
    "orc_gates": (None, [_I64, _I32, _I32, _P, _P, _I32, _P]),
    "orc_route": (None, [_I64, _I32, _P, _I32, _I32, _I32, _P, _I32, _I32] + [_P] * 6),
    "orc_capacity": (_I64, [_I64, _I32, _I32, _F32, _I64]),
    "orc_dispatch": (_I64, [_I64, _I32, _I32, _P, _I64, _I32] + [_P] * 6),
    "orc_permute": (None, [_I64, _I32, _P, _I32, _P, _P]),
    "orc_expert_rows": (None, [_I64, _I32, _I32, _P] + [_P, _I32, _I64] * 3 + [_I32, _I32, _P, _P]),
    "orc_expert_ffn": (None, [_I64, _I32, _I32, _I32, _P, _P] + [_P, _I32] * 3 + [_I32, _P, _P]),
    "orc_e4m3_round": (None, [_I64, _P, _P]),
    "orc_e4m3_bits": (None, [_I64, _P, _P]),
    "orc_pow2_scale_exponents": (None, [_I64, _P, _P]),
    "orc_quantize_rows_fp8": (None, [_I64, _I64, _P, _I32, _P, _P]),
    "orc_dequantize_rows_fp8": (None, [_I64, _I64, _P, _P, _P]),
    "orc_shared_ffn": (None, [_I32, _I64, _I32, _I32] + [_P, _I32] * 4 + [_P]),
    "orc_combine": (None, [_I64, _I32, _I32, _P, _I32, _P, _P, _P, _I32, _P, _P]),
    "orc_load_stats": (None, [_I32, _I64, _F64, _P, _P, _I32, _P, _P, _P]),
    "orc_z_loss": (_F64, [_I64, _I32, _P]),
    "orc_balance_bias_update": (None, [_I32, _P, _P, _F64, _P]),
    "orc_topk_margins": (None, [_I64, _I32, _P, _I32, _P]),
    "orc_group_margins": (None, [_I64, _I32, _P, _I32, _I32, _I32, _P]),
    "orc_layer_forward": (None, [_I64, _I32, _I32, _I32, _I32, _I32, _I32, _F32, _I64, _I32] + [_P, _I32] * 5 +
                          [_P] + [_P, _I32] * 3 + [_P, _I32, _I32, _I32, _I32] + [_P, _I32] * 3 + [_I32] +
                          [_P] * 23),
    "orc_sampled_combine": (None, [_I64, _I32, _I32, _P, _P, _P, _P, _I32, _P, _P]),
    "orc_combine_backward": (None, [_I64, _I32, _I32, _I64] + [_P] * 6),
    "orc_gate_backward": (None, [_I64, _I32, _I32, _P, _P, _P, _I32, _I32, _P]),
    "orc_aux_loss_grad": (None, [_I64, _I32, _P, _P, _I32, _P]),
    "orc_z_loss_grad": (None, [_I64, _I32, _P, _P]),
    "orc_router_backward": (None, [_I64, _I32, _I32, _P, _P, _P, _P, _I32, _I32, _F64, _F64, _P]),
    "orc_swiglu_backward": (None, [_I64, _I32, _I32, _P] + [_P, _I32, _I64] * 3 + [_P] * 8),
    "orc_expert_ffn_backward": (None, [_I64, _I32, _I32, _I32, _P, _P] + [_P, _I32] * 3 + [_P] * 8),
    "orc_dispatch_backward": (None, [_I64, _I32, _I32, _P, _P, _P, _P]),
    "orc_router_input_backward": (None, [_I64, _I32, _I32, _P, _I32, _P, _I32, _P, _P, _I32, _P, _I32] + [_P] * 4),
    "orc_layer_backward": (None, [_I64, _I32, _I32, _I32, _I32, _I32, _I32, _F64, _F64] + [_P, _I32] * 7 +
                           [_I32, _I32] + [_P, _I32] * 3 + [_P] * 4 + [_I64] + [_P] * 22),
}

STAGES = ("router_logits", "selection", "dispatch", "experts", "shared_experts", "combine", "statistics")


# ------------------------------------------------------------------------------ the oracle

class Oracle:
    """One build of the oracle library, with the method's steps as numpy-returning functions."""

    SOFTMAX, SIGMOID, CHOICE_MAJOR, TOKEN_MAJOR, E4M3_MAX = SOFTMAX, SIGMOID, CHOICE_MAJOR, TOKEN_MAJOR, E4M3_MAX
    STAGES = STAGES

    def __init__(self, path: str):
        self.path = path
        self.lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(self.lib, name)
            fn.restype, fn.argtypes = res, args

    def threads(self) -> int:
        """OpenMP threads the oracle's parallel loops use."""
        return int(self.lib.orc_threads())

    def set_threads(self, n: int) -> None:
        """Sets the OpenMP thread count of the oracle's parallel loops (results do not depend on it)."""
        self.lib.orc_set_threads(int(n))

    # ---------------------------------------------------------------- router
    def softplus(self, x) -> np.ndarray:
        x = _d(x)
        out = np.empty_like(x)
        self.lib.orc_softplus(x.size, _p(x), _p(out))
        return out

    def router_logits(self, U, W_r, b_r=None, W_noise=None, eps=None) -> np.ndarray:
        """H = U W_r (+ b_r) (+ eps * Softplus(U W_noise)), float64 [T, E]."""
        u, w, b, wn, ep = _In(U), _In(W_r), _In(b_r), _In(W_noise), _In(eps)
        T, h = u.shape
        E = w.shape[1]
        H = np.empty((T, E))
        self.lib.orc_router_logits(T, h, E, u.ptr, u.dt, w.ptr, w.dt, b.ptr, b.dt, wn.ptr, wn.dt, ep.ptr, ep.dt,
                                   _p(H))
        return H

    def round_f32(self, H) -> np.ndarray:
        H = _d(H)
        out = np.empty_like(H)
        self.lib.orc_round_f32(H.size, _p(H), _p(out))
        return out

    def topk_select(self, H32, k: int, allowed=None) -> np.ndarray:
        key = _d(H32)
        T, E = key.shape
        al = None if allowed is None else np.ascontiguousarray(np.asarray(allowed, dtype=bool).astype(np.uint8))
        idx = np.empty((T, k), dtype=np.int64)
        self.lib.orc_topk(T, E, _p(key), k, _p(al), _p(idx))
        return idx.astype(np.int32)

    def group_scores(self, aff, n_group: int, r: int) -> np.ndarray:
        aff = _d(aff)
        T, E = aff.shape
        out = np.empty((T, n_group))
        self.lib.orc_group_scores(T, E, _p(aff), n_group, r, _p(out))
        return out

    def group_limited_mask(self, aff, n_group: int, topk_group: int, k: int) -> np.ndarray:
        aff = _d(aff)
        T, E = aff.shape
        out = np.empty((T, E), dtype=np.uint8)
        self.lib.orc_group_limited_mask(T, E, _p(aff), n_group, topk_group, k, _p(out))
        return out.astype(bool)

    def scores(self, H, score_fn: int) -> np.ndarray:
        if score_fn not in (SOFTMAX, SIGMOID):
            raise ValueError("score_fn")
        H = _d(H)
        T, E = H.shape
        s = np.empty_like(H)
        self.lib.orc_scores(T, E, _p(H), score_fn, _p(s))
        return s

    def gates(self, s, idx, renorm: bool) -> np.ndarray:
        s, idx = _d(s), _i(idx)
        T, E = s.shape
        k = idx.shape[1]
        g = np.empty((T, k))
        self.lib.orc_gates(T, E, k, _p(s), _p(idx), int(bool(renorm)), _p(g))
        return g

    def route(self, H, k: int, score_fn: int, renorm: bool, sel_bias=None, n_group: int = 1,
              topk_group: int = 1) -> dict:
        """logits (rounded to float32), idx, s, gate, sel_key and (n_group > 1) the allowed mask."""
        if score_fn not in (SOFTMAX, SIGMOID):
            raise ValueError("score_fn")
        H = _d(H)
        T, E = H.shape
        sb = None if sel_bias is None else _d(sel_bias)
        groups = n_group is not None and n_group > 1
        out = dict(logits=np.empty((T, E)), s=np.empty((T, E)), sel_key=np.empty((T, E)),
                   allowed=np.empty((T, E), dtype=np.uint8) if groups else None,
                   idx=np.empty((T, k), dtype=np.int64), gate=np.empty((T, k)))
        self.lib.orc_route(T, E, _p(H), k, score_fn, int(bool(renorm)), _p(sb), n_group if groups else 1,
                           topk_group if groups else 1, _p(out["logits"]), _p(out["s"]), _p(out["sel_key"]),
                           _p(out["allowed"]), _p(out["idx"]), _p(out["gate"]))
        out["idx"] = out["idx"].astype(np.int32)
        if groups:
            out["allowed"] = out["allowed"].astype(bool)
        return out

    # ---------------------------------------------------------------- capacity and dispatch
    def capacity(self, T: int, E: int, k: int, capacity_factor: float, override: int = 0) -> int:
        return int(self.lib.orc_capacity(int(T), int(E), int(k), float(capacity_factor), int(override)))

    def dispatch(self, idx, E: int, C: int, priority: int = CHOICE_MAJOR) -> dict:
        """counts_routed, counts_kept [E], offsets [E+1], slot, slot_row [T*k] (-1 = dropped),
        row_token [A], n_dropped, C."""
        if priority not in (CHOICE_MAJOR, TOKEN_MAJOR):
            raise ValueError("priority")
        idx = _i(idx)
        T, k = idx.shape
        o = dict(counts_routed=np.empty(E, dtype=np.int64), counts_kept=np.empty(E, dtype=np.int64),
                 offsets=np.empty(E + 1, dtype=np.int64), slot=np.empty(T * k, dtype=np.int64),
                 slot_row=np.empty(T * k, dtype=np.int64), row_token=np.full(T * k, -1, dtype=np.int64))
        dropped = self.lib.orc_dispatch(T, k, E, _p(idx), int(C), priority, _p(o["counts_routed"]),
                                        _p(o["counts_kept"]), _p(o["offsets"]), _p(o["slot"]), _p(o["slot_row"]),
                                        _p(o["row_token"]))
        o["row_token"] = o["row_token"][:int(o["offsets"][E])].copy()
        o["n_dropped"], o["C"] = int(dropped), int(C)
        return o

    def permute(self, U, row_token) -> np.ndarray:
        u, rt = _In(U), _i(row_token)
        h = u.shape[1]
        X = np.empty((rt.size, h))
        self.lib.orc_permute(rt.size, h, u.ptr, u.dt, _p(rt), _p(X))
        return X

    # ---------------------------------------------------------------- experts
    def _expert_rows(self, x, Wg_e, Wu_e, Wd_e, fp8_x=False, fp8_w=False):
        x = _d(x)
        g, u, d_ = _In(Wg_e), _In(Wu_e), _In(Wd_e)
        n, h = x.shape
        d = g.shape[0]
        y, a = np.empty((n, h)), np.empty((n, d))
        self.lib.orc_expert_rows(n, h, d, _p(x), g.ptr, g.dt, 0, u.ptr, u.dt, 0, d_.ptr, d_.dt, 0, int(fp8_x),
                                 int(fp8_w), _p(y), _p(a))
        return y, a

    def swiglu(self, x, W_gate_e, W_up_e, W_down_e):
        """One expert on rows x [n, h]: (W_down (SiLU(W_gate x) * W_up x) [n, h], the activation [n, d_e])."""
        return self._expert_rows(x, W_gate_e, W_up_e, W_down_e)

    def expert_ffn(self, X, offsets, W_gate, W_up, W_down, d_e: int):
        """(Y, act): the grouped FFN over the expert segments of X."""
        X, off = _d(X), _i(offsets)
        g, u, d_ = _In(W_gate), _In(W_up), _In(W_down)
        A, h = X.shape
        E = off.size - 1
        Y, act = np.empty((A, h)), np.empty((A, d_e))
        self.lib.orc_expert_ffn(A, h, d_e, E, _p(X), _p(off), g.ptr, g.dt, u.ptr, u.dt, d_.ptr, d_.dt, 0, _p(Y),
                                _p(act))
        return Y, act

    # ---------------------------------------------------------------- FP8
    def e4m3_round(self, x):
        scalar = np.ndim(x) == 0
        x = _d(x)
        out = np.empty_like(x)
        self.lib.orc_e4m3_round(x.size, _p(x), _p(out))
        return float(out.reshape(-1)[0]) if scalar else out

    def e4m3_bits(self, v) -> np.ndarray:
        v = _d(v)
        out = np.empty(v.shape, dtype=np.uint8)
        self.lib.orc_e4m3_bits(v.size, _p(v), _p(out))
        return out

    def pow2_scale_exponents(self, amax) -> np.ndarray:
        a = _d(amax)
        out = np.empty(a.shape, dtype=np.int64)
        self.lib.orc_pow2_scale_exponents(a.size, _p(a), _p(out))
        return out

    def quantize_rows_fp8(self, A):
        """Row-wise E4M3 with one power-of-two scale per row: (codes [n, c], s [n]), A ~ codes * 2^s."""
        a = _In(A)
        n, c = a.shape
        codes, s = np.empty((n, c)), np.empty(n, dtype=np.int64)
        self.lib.orc_quantize_rows_fp8(n, c, a.ptr, a.dt, _p(codes), _p(s))
        return codes, s

    def dequantize_rows_fp8(self, codes, s) -> np.ndarray:
        codes, s = _d(codes), _i(s)
        n, c = codes.shape
        out = np.empty_like(codes)
        self.lib.orc_dequantize_rows_fp8(n, c, _p(codes), _p(s), _p(out))
        return out

    def fp8_weights(self, W) -> np.ndarray:
        """[E, d, h] weights as the FP8 up-projection sees them: each row quantised and dequantised."""
        shape = tuple(W.shape)
        flat = W.reshape(-1, shape[-1])
        return self.dequantize_rows_fp8(*self.quantize_rows_fp8(flat)).reshape(shape)

    # ---------------------------------------------------------------- shared experts, combine, statistics
    def shared_ffn(self, U, W_gate_sh, W_up_sh, W_down_sh) -> np.ndarray:
        """Y_sh [N_s, T, h]: each shared expert's SwiGLU FFN on every token."""
        u, g, up, d_ = _In(U), _In(W_gate_sh), _In(W_up_sh), _In(W_down_sh)
        T, h = u.shape
        n_s, d = g.shape[0], g.shape[1]
        Y = np.empty((n_s, T, h))
        self.lib.orc_shared_ffn(n_s, T, h, d, u.ptr, u.dt, g.ptr, g.dt, up.ptr, up.dt, d_.ptr, d_.dt, _p(Y))
        return Y

    def combine(self, U, Y, slot_row, gate, k: int, Y_shared=None) -> np.ndarray:
        """out_t = u_t + sum_s Y_shared[s, t] + sum_j g_{j,t} Y[row of (t, j)], kept pairs, j ascending."""
        u, Y, sr, g = _In(U), _d(Y), _i(slot_row), _d(gate)
        T, h = u.shape
        ysh = None if Y_shared is None else _d(Y_shared)
        n_s = 0 if ysh is None else ysh.shape[0]
        out = np.empty((T, h))
        self.lib.orc_combine(T, h, k, u.ptr, u.dt, _p(Y), _p(sr), _p(g), n_s, _p(ysh), _p(out))
        return out

    def load_stats(self, counts_routed, s, T: int, k, score_fn: int) -> dict:
        """f_i, P_i, E * sum_i f_i P_i and MaxVio."""
        c, s = _d(counts_routed), _d(s)
        E = c.size
        f, P, sc = np.empty(E), np.empty(E), np.empty(2)
        self.lib.orc_load_stats(E, int(T), float(k), _p(c), _p(s), score_fn, _p(f), _p(P), _p(sc))
        return dict(f=f, P=P, aux=float(sc[0]), maxvio=float(sc[1]))

    def router_z_loss(self, H) -> float:
        H = _d(H)
        if H.ndim == 1:
            H = H.reshape(1, -1)
        T, E = H.shape
        return float(self.lib.orc_z_loss(T, E, _p(H)))

    def balance_bias_update(self, b, counts_routed, u: float) -> np.ndarray:
        b, c = _d(b), _d(counts_routed)
        out = np.empty_like(b)
        self.lib.orc_balance_bias_update(b.size, _p(b), _p(c), float(u), _p(out))
        return out

    def topk_margins(self, H32, k: int) -> np.ndarray:
        """Smallest gap between adjacent values among each row's k+1 largest (keeps the tests' routing
        decisions away from ties)."""
        H = _d(H32)
        T, E = H.shape
        out = np.empty(T)
        self.lib.orc_topk_margins(T, E, _p(H), k, _p(out))
        return out

    def group_margins(self, aff, n_group: int, topk_group: int, k: int) -> np.ndarray:
        """Per token, the gap between the topk_group-th and the next group score (inf when every group
        is kept)."""
        a = _d(aff)
        T, E = a.shape
        out = np.empty(T)
        self.lib.orc_group_margins(T, E, _p(a), n_group, topk_group, k, _p(out))
        return out

    # ---------------------------------------------------------------- the whole layer
    def layer_forward(self, inp, *, T, h, E, k, d_e, score_fn, renorm, capacity_factor, capacity_override=0,
                      priority=CHOICE_MAJOR, logits=None, sel_bias=None, shared=None, n_group=1, topk_group=1,
                      fp8=False) -> dict:
        """The full single-GPU MoE layer forward, stage by stage.

        `inp` carries U, W_r, b_r, W_noise, eps, W_gate, W_up, W_down (numpy or torch).  `logits`
        given: the router GEMM is skipped and those logits are used.  `sel_bias` [E]: loss-free
        selection bias; `shared` = (W_gate_sh, W_up_sh, W_down_sh): shared experts; n_group > 1:
        group-limited routing; fp8: E4M3 dispatch and up-projection (X holds the dequantised rows,
        "U_codes", "U_s" the quantised U).  "seconds" holds each stage's wall time (STAGES order).
        """
        if score_fn not in (SOFTMAX, SIGMOID) or priority not in (CHOICE_MAJOR, TOKEN_MAJOR):
            raise ValueError("score_fn / priority")
        T, h, E, k, d_e = int(T), int(h), int(E), int(k), int(d_e)
        U, Wr, br = _In(inp.U), _In(inp.W_r), _In(inp.b_r)
        Wn, ep = _In(inp.W_noise), _In(inp.eps)
        Wg, Wu, Wd = _In(inp.W_gate), _In(inp.W_up), _In(inp.W_down)
        H = None if logits is None else _d(logits)
        sb = None if sel_bias is None else _d(sel_bias)
        n_s, d_s = 0, 0
        Sg = Su = Sd = _In(None)
        if shared is not None:
            Sg, Su, Sd = (_In(x) for x in shared)
            n_s, d_s = Sg.shape[0], Sg.shape[1]
        groups = n_group is not None and n_group > 1
        Tk = T * k
        o = dict(logits=np.empty((T, E)), s=np.empty((T, E)), sel_key=np.empty((T, E)),
                 allowed=np.empty((T, E), dtype=np.uint8) if groups else None,
                 idx=np.empty((T, k), dtype=np.int64), gate=np.empty((T, k)),
                 counts_routed=np.empty(E, dtype=np.int64), counts_kept=np.empty(E, dtype=np.int64),
                 offsets=np.empty(E + 1, dtype=np.int64), slot=np.empty(Tk, dtype=np.int64),
                 slot_row=np.empty(Tk, dtype=np.int64), row_token=np.full(Tk, -1, dtype=np.int64),
                 X=np.empty((Tk, h)), act=np.empty((Tk, d_e)), Y=np.empty((Tk, h)),
                 Y_shared=np.empty((n_s, T, h)) if n_s else None, out=np.empty((T, h)),
                 f=np.empty(E), P=np.empty(E),
                 U_codes=np.empty((T, h)) if fp8 else None, U_s=np.empty(T, dtype=np.int64) if fp8 else None)
        scal, sec = np.empty(5), np.empty(len(STAGES))
        self.lib.orc_layer_forward(
            T, h, E, k, d_e, score_fn, int(bool(renorm)), float(capacity_factor), int(capacity_override or 0),
            priority, U.ptr, U.dt, Wr.ptr, Wr.dt, br.ptr, br.dt, Wn.ptr, Wn.dt, ep.ptr, ep.dt, _p(H), Wg.ptr, Wg.dt,
            Wu.ptr, Wu.dt, Wd.ptr, Wd.dt, _p(sb), n_group if groups else 1, topk_group if groups else 1, n_s, d_s,
            Sg.ptr, Sg.dt, Su.ptr, Su.dt, Sd.ptr, Sd.dt, int(bool(fp8)),
            *(_p(o[n]) for n in ("logits", "s", "sel_key", "allowed", "idx", "gate", "counts_routed", "counts_kept",
                                 "offsets", "slot", "slot_row", "row_token", "X", "act", "Y", "Y_shared", "out",
                                 "f", "P", "U_codes", "U_s")),
            _p(scal), _p(sec))
        A = int(o["offsets"][E])
        o["idx"] = o["idx"].astype(np.int32)
        if groups:
            o["allowed"] = o["allowed"].astype(bool)
        for n in ("row_token", "X", "act", "Y"):
            o[n] = o[n][:A].copy()
        o.update(C=int(scal[0]), n_dropped=int(scal[1]), aux=float(scal[2]), maxvio=float(scal[3]),
                 z_loss=float(scal[4]), seconds=dict(zip(STAGES, sec.tolist())))
        if not fp8:
            del o["U_codes"], o["U_s"]
        return o

    def sampled_outputs(self, inp, tokens, idx, gate, slot_row, k: int, shared=None, fp8=False) -> dict:
        """out rows (and the Y rows they use) for a sample of tokens of a full-size layer.

        Each kept pair's Y row is one expert applied to one token row; the pairs are grouped by
        expert so that each expert's weights are copied to the host once.  `shared` adds the shared
        experts; `fp8` gives the experts E4M3 token rows and gate/up weight rows.
        Returns {"out": [n, h], "Y": {row: [h]}}.
        """
        tokens = [int(t) for t in tokens]
        idx, g, sr = _i(idx), _d(gate), _i(slot_row).reshape(-1, k)
        n = len(tokens)
        if n == 0:
            return dict(out=np.zeros((0, 0)), Y={})
        if hasattr(inp.U, "detach"):
            import torch
            u = _d(inp.U[torch.as_tensor(tokens, device=inp.U.device)])
        else:
            u = _d(np.asarray(inp.U)[tokens])
        h = u.shape[1]
        y = np.zeros((n, k, h))
        by_expert = {}
        for i, t in enumerate(tokens):
            for j in range(k):
                if sr[t, j] >= 0:
                    by_expert.setdefault(int(idx[t, j]), []).append((i, j))
        for e, pairs in sorted(by_expert.items()):
            ye, _ = self._expert_rows(u[[i for i, _ in pairs]], inp.W_gate[e], inp.W_up[e], inp.W_down[e],
                                      fp8_x=fp8, fp8_w=fp8)
            for (i, j), row in zip(pairs, ye):
                y[i, j] = row
        n_s, ysh = 0, None
        if shared is not None:
            n_s = len(shared[0])
            ysh = np.stack([self._expert_rows(u, shared[0][s], shared[1][s], shared[2][s])[0] for s in range(n_s)])
        sub_sr = np.ascontiguousarray(sr[tokens])
        sub_g = np.ascontiguousarray(g.reshape(-1, k)[tokens])
        out = np.empty((n, h))
        self.lib.orc_sampled_combine(n, h, k, _p(u), _p(y), _p(sub_sr), _p(sub_g), n_s, _p(ysh), _p(out))
        rows = {int(sub_sr[i, j]): y[i, j] for i in range(n) for j in range(k) if sub_sr[i, j] >= 0}
        return dict(out=out, Y=rows)

    # ---------------------------------------------------------------- backward
    def combine_backward(self, dO, Y, slot_row, gate, k: int) -> dict:
        """d_gate [T, k] = dO_t . Y[row] (0 when dropped), dY [A, h] = g dO_t."""
        dO, Y, sr, g = _d(dO), _d(Y), _i(slot_row), _d(gate)
        T, h = dO.shape
        A = Y.shape[0]
        d_gate, dY = np.empty((T, k)), np.empty((A, h))
        self.lib.orc_combine_backward(T, h, k, A, _p(dO), _p(Y), _p(sr), _p(g), _p(d_gate), _p(dY))
        return dict(d_gate=d_gate, dY=dY)

    def gate_backward(self, H32, idx, d_gate, score_fn: int, renorm: bool) -> np.ndarray:
        H, idx, dg = _d(H32), _i(idx), _d(d_gate)
        T, E = H.shape
        k = idx.shape[1]
        dg = np.ascontiguousarray(dg.reshape(T, k))
        dH = np.empty((T, E))
        self.lib.orc_gate_backward(T, E, k, _p(H), _p(idx), _p(dg), score_fn, int(bool(renorm)), _p(dH))
        return dH

    def aux_loss_grad(self, H32, f, score_fn: int) -> np.ndarray:
        H, f = _d(H32), _d(f)
        T, E = H.shape
        out = np.empty((T, E))
        self.lib.orc_aux_loss_grad(T, E, _p(H), _p(f), score_fn, _p(out))
        return out

    def z_loss_grad(self, H32) -> np.ndarray:
        H = _d(H32)
        T, E = H.shape
        out = np.empty((T, E))
        self.lib.orc_z_loss_grad(T, E, _p(H), _p(out))
        return out

    def router_backward(self, H32, idx, d_gate, f, score_fn: int, renorm: bool, w_aux: float = 0.0,
                        w_z: float = 0.0) -> np.ndarray:
        """dL/dH for L = (the loss through the gates) + w_aux E sum f P + w_z L_z."""
        H, idx, dg, f = _d(H32), _i(idx), _d(d_gate), _d(f)
        T, E = H.shape
        k = idx.shape[1]
        dg = np.ascontiguousarray(dg.reshape(T, k))
        dH = np.empty((T, E))
        self.lib.orc_router_backward(T, E, k, _p(H), _p(idx), _p(dg), _p(f), score_fn, int(bool(renorm)),
                                     float(w_aux), float(w_z), _p(dH))
        return dH

    def swiglu_backward(self, x, W_gate_e, W_up_e, W_down_e, dy) -> dict:
        x, dy = _d(x), _d(dy)
        g, u, d_ = _In(W_gate_e), _In(W_up_e), _In(W_down_e)
        n, h = x.shape
        d = g.shape[0]
        o = dict(d_act=np.empty((n, d)), dG=np.empty((n, d)), dUp=np.empty((n, d)), dx=np.empty((n, h)),
                 dW_gate=np.empty((d, h)), dW_up=np.empty((d, h)), dW_down=np.empty((h, d)))
        self.lib.orc_swiglu_backward(n, h, d, _p(x), g.ptr, g.dt, 0, u.ptr, u.dt, 0, d_.ptr, d_.dt, 0, _p(dy),
                                     *(_p(o[m]) for m in ("d_act", "dG", "dUp", "dx", "dW_gate", "dW_up", "dW_down")))
        return o

    def expert_ffn_backward(self, X, offsets, W_gate, W_up, W_down, dY, d_e: int) -> dict:
        X, off, dY = _d(X), _i(offsets), _d(dY)
        g, u, d_ = _In(W_gate), _In(W_up), _In(W_down)
        A, h = X.shape
        E = off.size - 1
        o = dict(d_act=np.empty((A, d_e)), dG=np.empty((A, d_e)), dUp=np.empty((A, d_e)), dX=np.empty((A, h)),
                 dW_gate=np.empty((E, d_e, h)), dW_up=np.empty((E, d_e, h)), dW_down=np.empty((E, h, d_e)))
        self.lib.orc_expert_ffn_backward(A, h, d_e, E, _p(X), _p(off), g.ptr, g.dt, u.ptr, u.dt, d_.ptr, d_.dt,
                                         _p(dY), *(_p(o[m]) for m in ("d_act", "dG", "dUp", "dX", "dW_gate",
                                                                       "dW_up", "dW_down")))
        return o

    def dispatch_backward(self, dO, dX, slot_row, k: int) -> np.ndarray:
        dO, dX, sr = _d(dO), _d(dX), _i(slot_row)
        T, h = dO.shape
        dU = np.empty((T, h))
        self.lib.orc_dispatch_backward(T, h, k, _p(dO), _p(dX), _p(sr), _p(dU))
        return dU

    def router_input_backward(self, U, W_r, dH, W_noise=None, eps=None) -> dict:
        u, w, dH = _In(U), _In(W_r), _d(dH)
        wn, ep = _In(W_noise), _In(eps)
        T, h = u.shape
        E = w.shape[1]
        o = dict(dU=np.empty((T, h)), dW_r=np.empty((h, E)), db_r=np.empty(E),
                 dW_noise=np.empty((h, E)) if W_noise is not None else None)
        self.lib.orc_router_input_backward(T, h, E, u.ptr, u.dt, w.ptr, w.dt, _p(dH), wn.ptr, wn.dt, ep.ptr, ep.dt,
                                           _p(o["dU"]), _p(o["dW_r"]), _p(o["db_r"]), _p(o["dW_noise"]))
        return o

    def layer_backward(self, inp, fwd: dict, dO, *, k: int, d_e: int, score_fn: int, renorm: bool,
                       w_aux: float = 0.0, w_z: float = 0.0) -> dict:
        """Gradients of L = <dO, out> + w_aux E sum_i f_i P_i + w_z L_z through the whole layer, with
        the routing decisions held fixed.  `fwd` is layer_forward's result."""
        U, Wr, Wn, ep = _In(inp.U), _In(inp.W_r), _In(inp.W_noise), _In(inp.eps)
        Wg, Wu, Wd = _In(inp.W_gate), _In(inp.W_up), _In(inp.W_down)
        shared = getattr(inp, "shared", None)
        n_s, d_s = 0, 0
        Sg = Su = Sd = _In(None)
        if shared is not None:
            Sg, Su, Sd = (_In(x) for x in shared)
            n_s, d_s = Sg.shape[0], Sg.shape[1]
        T, h = U.shape
        E = Wr.shape[1]
        logits, idx, sr, g = _d(fwd["logits"]), _i(fwd["idx"]), _i(fwd["slot_row"]), _d(fwd["gate"])
        X, Y, off, f = _d(fwd["X"]), _d(fwd["Y"]), _i(fwd["offsets"]), _d(fwd["f"])
        dO = _d(dO)
        A = X.shape[0]
        o = dict(dU=np.empty((T, h)), d_gate=np.empty((T, k)), dY=np.empty((A, h)), dH=np.empty((T, E)),
                 dW_r=np.empty((h, E)), db_r=np.empty(E),
                 dW_noise=np.empty((h, E)) if inp.W_noise is not None else None,
                 d_act=np.empty((A, d_e)), dG=np.empty((A, d_e)), dUp=np.empty((A, d_e)), dX=np.empty((A, h)),
                 dW_gate=np.empty((E, d_e, h)), dW_up=np.empty((E, d_e, h)), dW_down=np.empty((E, h, d_e)),
                 dW_gate_sh=np.empty((n_s, d_s, h)) if n_s else None, dW_up_sh=np.empty((n_s, d_s, h)) if n_s else None,
                 dW_down_sh=np.empty((n_s, h, d_s)) if n_s else None)
        self.lib.orc_layer_backward(
            T, h, E, k, d_e, score_fn, int(bool(renorm)), float(w_aux), float(w_z), U.ptr, U.dt, Wr.ptr, Wr.dt,
            Wn.ptr, Wn.dt, ep.ptr, ep.dt, Wg.ptr, Wg.dt, Wu.ptr, Wu.dt, Wd.ptr, Wd.dt, n_s, d_s, Sg.ptr, Sg.dt,
            Su.ptr, Su.dt, Sd.ptr, Sd.dt, _p(logits), _p(idx), _p(sr), _p(g), A, _p(X), _p(Y), _p(off), _p(f), _p(dO),
            *(_p(o[m]) for m in ("dU", "d_gate", "dY", "dH", "dW_r", "db_r", "dW_noise", "d_act", "dG", "dUp", "dX",
                                 "dW_gate", "dW_up", "dW_down", "dW_gate_sh", "dW_up_sh", "dW_down_sh")))
        if not n_s:
            del o["dW_gate_sh"], o["dW_up_sh"], o["dW_down_sh"]
        return o


# ------------------------------------------------------------------------------ the default build

default = Oracle(build())

_EXPORTS = ("threads", "set_threads", "softplus", "router_logits", "round_f32", "topk_select", "group_scores",
            "group_limited_mask", "scores", "gates", "route", "capacity", "dispatch", "permute", "swiglu",
            "expert_ffn", "e4m3_round", "e4m3_bits", "pow2_scale_exponents", "quantize_rows_fp8",
            "dequantize_rows_fp8", "fp8_weights", "shared_ffn", "combine", "load_stats", "router_z_loss",
            "balance_bias_update", "topk_margins", "group_margins", "layer_forward", "sampled_outputs",
            "combine_backward", "gate_backward", "aux_loss_grad", "z_loss_grad", "router_backward",
            "swiglu_backward", "expert_ffn_backward", "dispatch_backward", "router_input_backward",
            "layer_backward")
for _name in _EXPORTS:
    globals()[_name] = getattr(default, _name)

__all__ = ["Oracle", "build", "f64", "default", "SOFTMAX", "SIGMOID", "CHOICE_MAJOR", "TOKEN_MAJOR", "E4M3_MAX",
           "STAGES", *_EXPORTS]

"""Shared pieces of the GPU parity tests: margin-safe inputs, error measures.

The oracle decides every expected value; the library's outputs are only ever
compared against it (or against properties that hold at any size).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from mixture_experts_layer_84_b300 import synth
from mixture_experts_layer_84_b300 import workloads as W

# Output tolerances: normwise max relative error max|a-b| / max|b|.
TOL = {W.F32: 1e-5, W.BF16: 2e-2}
LOGIT_TOL = 1e-5     # float32 logits, gates and statistics on both dtypes
MARGIN = 1e-3        # every adjacent gap among the top-(k+1) logits of a token
ULP_BITS = {W.F32: 23, W.BF16: 7}


def f64(x):
    return oracle.f64(x)


def normwise(a, b) -> float:
    a, b = f64(a), f64(b)
    if a.size == 0:
        return 0.0
    den = float(np.max(np.abs(b)))
    num = float(np.max(np.abs(a - b)))
    return num / den if den > 0 else num


def delta_error(out, U, out_ref, dtype) -> float:
    """Normwise error of the expert contribution out - U against the oracle's.

    The layer output is rounded once to its dtype at the scale of |out| (the
    residual dominates it), so one unit in the last place of out is allowed
    per element before the error is measured against max |out_ref - U|.
    """
    o, u, ref = f64(out), f64(U), f64(out_ref)
    d, dref = o - u, ref - u
    mag = np.maximum(np.abs(ref), np.finfo(np.float64).tiny)
    ulp = 2.0 ** (np.floor(np.log2(mag)) - ULP_BITS[dtype])
    excess = np.maximum(np.abs(d - dref) - ulp, 0.0)
    if excess.size == 0:
        return 0.0
    den = float(np.max(np.abs(dref)))
    return float(np.max(excess)) / den if den > 0 else float(np.max(excess))


def logits_of(w: W.Workload, inp, rows=None) -> np.ndarray:
    if rows is None:
        return oracle.router_logits(inp.U, inp.W_r, inp.b_r, inp.W_noise, inp.eps)
    r = torch.as_tensor(rows, device=inp.U.device)
    return oracle.router_logits(inp.U[r], inp.W_r, inp.b_r, inp.W_noise,
                                None if inp.eps is None else inp.eps[r])


def route_of(w: W.Workload, H, sel_bias=None) -> dict:
    """The oracle's routing of logits H under workload w (selection bias, expert groups)."""
    return oracle.route(H, w.k, w.score_fn, w.renorm, sel_bias, w.n_group, w.topk_group)


def selection_margins(w: W.Workload, H, sel_bias=None) -> np.ndarray:
    """Per token, the smallest gap that decides its routing: adjacent gaps among the top-(k+1)
    selection keys (the logits, or score + selection bias) of the experts it may use, and with
    expert groups the gap between the last kept and the first dropped group score."""
    r = route_of(w, H, sel_bias)
    key = r["sel_key"]
    if r["allowed"] is None:
        return oracle.topk_margins(key, w.k)
    m = oracle.topk_margins(np.where(r["allowed"], key, -np.inf), w.k)
    aff = r["s"] if sel_bias is None else key
    return np.minimum(m, oracle.group_margins(aff, w.n_group, w.topk_group, w.k))


def margin_inputs(w: W.Workload, seed: int = 0, device="cuda", experts: bool = True, max_rounds: int = 40):
    """Layer inputs whose tokens all keep a routing margin >= MARGIN (in float64): see
    selection_margins.

    Tokens that violate it get fresh U (and eps) rows; returns (inputs, float64 logits).
    """
    inp = synth.generate(w, seed, device, experts=experts)
    H = logits_of(w, inp)
    for attempt in range(max_rounds):
        bad = np.nonzero(selection_margins(w, H, inp.sel_bias) < MARGIN)[0]
        if bad.size == 0:
            return inp, H
        synth.redraw_rows(inp, torch.as_tensor(bad, dtype=torch.int64), seed, attempt)
        H[bad] = logits_of(w, inp, bad)
    raise RuntimeError(f"could not reach the top-k margin for {w.name}")


def check_routing_and_dispatch(w, bufs, H, sel_bias=None):
    r = route_of(w, H, sel_bias)
    C = oracle.capacity(w.T, w.E, w.k, w.capacity_factor, w.capacity)
    d = oracle.dispatch(r["idx"], w.E, C, w.priority)
    A = int(d["offsets"][-1])
    if bufs.logits is not None:
        assert normwise(bufs.logits, H) <= LOGIT_TOL
    assert np.array_equal(bufs.idx.cpu().numpy(), r["idx"])
    assert normwise(bufs.gate, r["gate"]) <= LOGIT_TOL
    assert np.array_equal(bufs.counts_routed.cpu().numpy(), d["counts_routed"])
    assert np.array_equal(bufs.counts_kept.cpu().numpy(), d["counts_kept"])
    assert np.array_equal(bufs.offsets.cpu().numpy(), d["offsets"])
    assert np.array_equal(bufs.slot_row.cpu().numpy(), d["slot_row"])
    assert np.array_equal(bufs.row_token[:A].cpu().numpy(), d["row_token"])
    assert int(bufs.n_dropped.item()) == d["n_dropped"]
    st = oracle.load_stats(d["counts_routed"], r["s"], w.T, w.k, w.score_fn)
    assert normwise(bufs.f, st["f"]) <= 1e-6
    assert normwise(bufs.P, st["P"]) <= LOGIT_TOL
    assert abs(float(bufs.aux.item()) - st["aux"]) <= LOGIT_TOL * max(1.0, abs(st["aux"]))
    zl = oracle.router_z_loss(r["logits"])
    assert abs(float(bufs.z_loss.item()) - zl) <= LOGIT_TOL * max(1.0, abs(zl))
    return r, d, A

"""moe_combine against the oracle: gate-weighted un-permute with the residual, and the
load statistics (f, P, aux) from the router's per-block sums."""
import pytest
import torch

import oracle
from gpu_helpers import LOGIT_TOL, TOL, delta_error, normwise
from mixture_experts_layer_84_b300 import _lib as L
from mixture_experts_layer_84_b300 import synth
from mixture_experts_layer_84_b300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("w", W.SMALL, ids=lambda w: w.name)
def test_combine_and_stats(w):
    T, E, k, h = w.T, w.E, w.k, w.h
    logits = synth.random_logits(T, E, seed=21, scale=1.5, tie_fraction=0.0)
    cfg = L.config_of(w)
    ws = L.new_workspace(cfg)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, k), dtype=torch.float32, device="cuda")
    L.moe_route(cfg, None, None, None, None, None, logits.cuda(), None, idx, gate, ws)  # leaves the P sums in ws
    r = oracle.route(oracle.f64(logits), k, w.score_fn, w.renorm)
    C = oracle.capacity(T, E, k, w.capacity_factor, w.capacity)
    d = oracle.dispatch(r["idx"], E, C, w.priority)
    U = synth.random_rows(T, h, 5, "U", "cuda", w.torch_dtype)
    Y = synth.random_rows(T * k, h, 6, "Y", "cuda", w.torch_dtype)
    slot_row = torch.as_tensor(d["slot_row"], dtype=torch.int32, device="cuda")
    counts = torch.as_tensor(d["counts_routed"], dtype=torch.int32, device="cuda")
    out = torch.empty((T, h), dtype=w.torch_dtype, device="cuda")
    f = torch.empty(E, dtype=torch.float32, device="cuda")
    P = torch.empty(E, dtype=torch.float32, device="cuda")
    aux = torch.empty(1, dtype=torch.float32, device="cuda")
    z = torch.empty(1, dtype=torch.float32, device="cuda")
    L.moe_combine(cfg, U, Y, slot_row, gate, counts, out, f, P, aux, ws, z_loss=z)
    assert L.moe_get_device_status(ws) == 0
    ref = oracle.combine(U, Y, d["slot_row"], r["gate"], k)
    tol = TOL[w.dtype]
    assert normwise(out, ref) <= tol
    assert delta_error(out, U, ref, w.dtype) <= tol
    st = oracle.load_stats(d["counts_routed"], r["s"], T, k, w.score_fn)
    assert normwise(f, st["f"]) <= 1e-6
    assert normwise(P, st["P"]) <= LOGIT_TOL
    assert abs(float(aux.item()) - st["aux"]) <= LOGIT_TOL * max(1.0, abs(st["aux"]))
    zl = oracle.router_z_loss(r["logits"])
    assert abs(float(z.item()) - zl) <= LOGIT_TOL * max(1.0, abs(zl))


def test_combine_bad_rows_flagged_and_skipped():
    T, E, k, h = 64, 4, 2, 64
    cfg = L.config(T, h, E, k, 64, capacity_factor=0.0, dtype=W.BF16)
    ws = L.new_workspace(cfg)
    U = synth.random_rows(T, h, 5, "U", "cuda", torch.bfloat16)
    Y = synth.random_rows(T * k, h, 6, "Y", "cuda", torch.bfloat16)
    slot_row = torch.arange(T * k, dtype=torch.int32, device="cuda")
    slot_row[5] = T * k + 3
    slot_row[8] = -2
    gate = torch.full((T, k), 0.5, dtype=torch.float32, device="cuda")
    counts = torch.full((E,), T * k // E, dtype=torch.int32, device="cuda")
    out = torch.empty((T, h), dtype=torch.bfloat16, device="cuda")
    f, P, aux = (torch.empty(n, dtype=torch.float32, device="cuda") for n in (E, E, 1))
    L.moe_combine(cfg, U, Y, slot_row, gate, counts, out, f, P, aux, ws)
    assert L.moe_get_device_status(ws) == L.MOE_DEV_BAD_ROW
    sr = slot_row.cpu().numpy().copy()
    sr[5] = -1
    sr[8] = -1
    ref = oracle.combine(U, Y, sr, gate.cpu().numpy(), k)
    assert normwise(out, ref) <= TOL[W.BF16]

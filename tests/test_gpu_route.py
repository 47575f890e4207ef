"""moe_route against the oracle: bit-exact selection, gates and logits within tolerance."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import LOGIT_TOL, margin_inputs, normwise
from mixture_experts_layer_84_b300 import _lib as L
from mixture_experts_layer_84_b300 import synth
from mixture_experts_layer_84_b300 import workloads as W

pytestmark = pytest.mark.gpu

SM, SG = W.SOFTMAX, W.SIGMOID

# stage mode: both sides get the same float32 logits (with exact ties planted)
STAGE = [
    (300, 8, 2, SM, True), (257, 5, 3, SG, True), (100, 64, 6, SM, True), (64, 256, 8, SG, True),
    (50, 128, 1, SM, False), (33, 1024, 16, SM, True), (10, 1, 1, SM, True), (40, 16, 16, SG, True),
    (129, 12, 4, SM, False), (0, 8, 2, SM, True), (1000, 300, 5, SG, True),
]


@pytest.mark.parametrize("T,E,k,score_fn,renorm", STAGE)
def test_route_stage_mode(T, E, k, score_fn, renorm):
    logits = synth.random_logits(T, E, seed=T + E, scale=2.0)
    cfg = L.config(T, 8, E, k, 8, score_fn=score_fn, renorm=renorm, dtype=W.F32)
    idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    gate = torch.full((T, k), -7.0, dtype=torch.float32, device="cuda")
    ws = L.new_workspace(cfg)
    L.moe_route(cfg, None, None, None, None, None, logits.cuda(), None, idx, gate, ws)
    assert L.moe_get_device_status(ws) == 0
    r = oracle.route(oracle.f64(logits), k, score_fn, renorm)
    assert np.array_equal(idx.cpu().numpy(), r["idx"])
    assert normwise(gate, r["gate"]) <= LOGIT_TOL
    if renorm and T > 0:
        assert np.allclose(gate.sum(1).cpu().numpy(), 1.0, atol=1e-6)


def test_route_stage_mode_all_equal_row():
    T, E, k = 4, 32, 5
    logits = torch.zeros((T, E), dtype=torch.float32)
    logits[1, 7] = 1.0
    cfg = L.config(T, 8, E, k, 8, dtype=W.F32)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, k), dtype=torch.float32, device="cuda")
    L.moe_route(cfg, None, None, None, None, None, logits.cuda(), None, idx, gate, L.new_workspace(cfg))
    got = idx.cpu().tolist()
    assert got[0] == [0, 1, 2, 3, 4] and got[1] == [7, 0, 1, 2, 3]


EXTRA = [
    W.Workload("route_e5_bf16", T=300, h=136, E=5, k=2, d_e=8, dtype=W.BF16, score_fn=SM, renorm=True,
               noisy=False, capacity_factor=1.0),
    W.Workload("route_e1024_bf16", T=200, h=256, E=1024, k=16, d_e=8, dtype=W.BF16, score_fn=SG, renorm=True,
               noisy=False, capacity_factor=1.0, bias="normal"),
    W.Workload("route_e12_f32", T=97, h=64, E=12, k=3, d_e=8, dtype=W.F32, score_fn=SM, renorm=False,
               noisy=True, capacity_factor=1.0),
    W.Workload("route_e512_noisy", T=150, h=520, E=512, k=4, d_e=8, dtype=W.BF16, score_fn=SM, renorm=False,
               noisy=True, capacity_factor=1.0, bias="zipf"),
]


@pytest.mark.parametrize("w", W.SMALL + EXTRA + [W.MIXTRAL, W.SWITCH, W.DSV3, W.STRESS], ids=lambda w: w.name)
def test_route_end_to_end(w):
    inp, H = margin_inputs(w, seed=1, experts=False)
    cfg = L.config_of(w)
    T, E, k = w.T, w.E, w.k
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, k), dtype=torch.float32, device="cuda")
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    ws = L.new_workspace(cfg)
    L.moe_route(cfg, inp.U, inp.W_r, inp.b_r, inp.W_noise, inp.eps, None, logits, idx, gate, ws)
    assert L.moe_get_device_status(ws) == 0
    r = oracle.route(H, k, w.score_fn, w.renorm)
    assert normwise(logits, H) <= LOGIT_TOL
    assert np.array_equal(idx.cpu().numpy(), r["idx"])
    assert normwise(gate, r["gate"]) <= LOGIT_TOL

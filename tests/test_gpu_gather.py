"""The dispatch's row copy fused into the first expert GEMM (moe_expert_ffn_gather, and
moe_layer_forward with X == NULL): bit-identical to the path that materialises X, which the
other tests hold against the oracle; plus the oracle directly on a few shapes."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import TOL, margin_inputs, normwise
from mixture_experts_layer_84_b300 import _lib as L
from mixture_experts_layer_84_b300 import synth
from mixture_experts_layer_84_b300 import workloads as W

pytestmark = pytest.mark.gpu

SHAPES = [
    W.MIXTRAL_SMALL, W.DSV3_SMALL, W.STRESS_SMALL, W.SWITCH_SMALL,
    # K tail of 8 columns (h = 136) and an output-column tail
    W.Workload("gather_tails", T=333, h=136, E=6, k=2, d_e=200, dtype=W.BF16, score_fn=W.SOFTMAX, renorm=True,
               noisy=False, capacity_factor=0.0),
    W.Workload("gather_many_small", T=700, h=320, E=96, k=3, d_e=384, dtype=W.BF16, score_fn=W.SIGMOID,
               renorm=True, noisy=False, capacity_factor=0.0),
    W.Workload("gather_capacity_drops", T=1500, h=256, E=16, k=4, d_e=256, dtype=W.BF16, score_fn=W.SOFTMAX,
               renorm=True, noisy=False, capacity_factor=0.5),
]


def _dispatch(w, inp, idx):
    cfg = L.config_of(w)
    bufs = L.LayerBuffers.allocate(cfg)
    L.moe_dispatch(cfg, inp.U, idx, bufs.counts_routed, bufs.counts_kept, bufs.offsets, bufs.slot_row,
                   bufs.row_token, bufs.X, bufs.n_dropped, bufs.ws)
    return cfg, bufs


@pytest.mark.parametrize("tiles", ["single", "pair"])
@pytest.mark.parametrize("w", SHAPES, ids=lambda w: w.name)
@pytest.mark.parametrize("zipf", [0.0, 1.2])
def test_expert_ffn_gather_matches_materialised(w, zipf, tiles, monkeypatch):
    monkeypatch.setenv("MOE_FFN_TILES", tiles)
    inp = synth.generate(w, seed=2, device="cuda")
    idx = synth.random_routing(w.T, w.E, w.k, seed=21, zipf_s=zipf).cuda()
    cfg, bufs = _dispatch(w, inp, idx)
    L.moe_expert_ffn(cfg, bufs.X, bufs.offsets, inp.W_gate, inp.W_up, inp.W_down, bufs.act, bufs.Y, bufs.ws)
    act2, Y2 = torch.full_like(bufs.act, 7.0), torch.full_like(bufs.Y, 7.0)
    L.moe_expert_ffn_gather(cfg, inp.U, bufs.row_token, bufs.offsets, inp.W_gate, inp.W_up, inp.W_down, act2, Y2,
                            bufs.ws)
    assert L.moe_get_device_status(bufs.ws) == 0
    A = int(bufs.offsets[-1].item())
    assert torch.equal(act2[:A], bufs.act[:A])
    assert torch.equal(Y2[:A], bufs.Y[:A])
    if w.T * w.h * w.d_e <= 333 * 320 * 400:  # the oracle on the smaller shapes
        offsets = bufs.offsets.cpu().numpy()
        X = oracle.f64(inp.U)[bufs.row_token[:A].cpu().numpy()]
        Y, act = oracle.expert_ffn(X, offsets, inp.W_gate.cpu(), inp.W_up.cpu(), inp.W_down.cpu(), w.d_e)
        assert normwise(act2[:A], act) <= TOL[W.BF16]
        assert normwise(Y2[:A], Y) <= TOL[W.BF16]


@pytest.mark.parametrize("w", [W.MIXTRAL_SMALL, W.DSV3_SHARED_SMALL, W.STRESS_SMALL, W.SWITCH_SMALL, W.MIXTRAL,
                               W.STRESS], ids=lambda w: w.name)
def test_layer_forward_without_X_matches(w):
    """moe_layer_forward with X == NULL gives the same bits as with X, small and full size."""
    inp, _ = margin_inputs(w, seed=0) if w.T <= 4096 else (synth.generate(w, 0, "cuda"), None)
    cfg = L.config_of(w)
    outs = []
    for with_X in (True, False):
        bufs = L.LayerBuffers.allocate(cfg, with_X=with_X)
        L.moe_layer_forward(cfg, inp.U, inp.W_r, inp.b_r, inp.W_noise, inp.eps, inp.W_gate, inp.W_up, inp.W_down,
                            bufs, sel_bias=inp.sel_bias, shared=inp.shared)
        assert L.moe_get_device_status(bufs.ws) == 0
        outs.append(bufs)
    a, b = outs
    A = int(a.offsets[-1].item())
    for name in ("idx", "gate", "slot_row", "offsets", "out", "aux", "P"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    assert torch.equal(a.act[:A], b.act[:A]) and torch.equal(a.Y[:A], b.Y[:A])


def test_gather_bad_row_ids_set_the_status():
    """row_token entries outside [0, T) read row 0 and set MOE_DEV_BAD_ROW (no access outside U)."""
    w = W.MIXTRAL_SMALL
    inp = synth.generate(w, seed=3, device="cuda")
    idx = synth.random_routing(w.T, w.E, w.k, seed=5).cuda()
    cfg, bufs = _dispatch(w, inp, idx)
    bad = bufs.row_token.clone()
    bad[3] = w.T + 5
    bad[10] = -2
    L.moe_expert_ffn_gather(cfg, inp.U, bad, bufs.offsets, inp.W_gate, inp.W_up, inp.W_down, bufs.act, bufs.Y,
                            bufs.ws)
    assert L.moe_get_device_status(bufs.ws) == L.MOE_DEV_BAD_ROW
    assert L.moe_get_device_status(bufs.ws) == 0  # reading the status clears it


def test_layer_without_X_needs_bf16():
    w = W.TINY_FP32
    inp = synth.generate(w, seed=0, device="cuda")
    cfg = L.config_of(w)
    bufs = L.LayerBuffers.allocate(cfg, with_X=False)
    with pytest.raises(L.MoeError, match="bf16"):
        L.moe_layer_forward(cfg, inp.U, inp.W_r, inp.b_r, inp.W_noise, inp.eps, inp.W_gate, inp.W_up, inp.W_down,
                            bufs)

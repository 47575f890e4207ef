"""The fused tensor-core router (bf16, E or 2E <= 256 logit columns) against the oracle, on shapes
chosen to reach every cluster size (1, 2, 4, 8 CTAs per 128-token tile), both CTA sizes (256 threads,
and 512 when one CTA fills an SM), ragged last tiles (CTAs of a cluster with no rows), h not a
multiple of 64, several selection passes per CTA, the noisy router,
group-limited routing with a selection bias, k = 16; and the router from weights packed once
(moe_pack_router) against the one that packs them on each call, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import LOGIT_TOL, check_routing_and_dispatch, margin_inputs, normwise
from mixture_experts_layer_84_b300 import _lib as L
from mixture_experts_layer_84_b300 import workloads as W

pytestmark = pytest.mark.gpu

SM, SG = W.SOFTMAX, W.SIGMOID


def _w(name, T, h, E, k, score, renorm=True, noisy=False, bias="none", **kw):
    return W.Workload(name, T=T, h=h, E=E, k=k, d_e=16, dtype=W.BF16, score_fn=score, renorm=renorm, noisy=noisy,
                      capacity_factor=1.0, bias=bias, **kw)


FUSED = [
    _w("cs8_ragged_tile", 130, 1032, 8, 2, SM),                        # 2 tiles; 2 rows in the last: 7 idle CTAs
    _w("cs4_noisy", 500, 768, 64, 4, SM, renorm=False, noisy=True, bias="zipf"),
    _w("cs2_sigmoid_groups_bias", 1000, 256, 32, 4, SG, bias="normal", sel_bias="normal", n_group=4, topk_group=2),
    _w("cs1_one_pass_512", 2000, 192, 128, 3, SM),                     # 128 rows in one pass (512 threads, 4 lanes)
    _w("cs4_e256_k16", 300, 512, 256, 16, SG),
    _w("e5_narrow", 260, 640, 5, 2, SM, bias="normal"),
    _w("noisy_e128_one_pass", 700, 320, 128, 1, SM, renorm=False, noisy=True, bias="zipf"),
    # more CTAs than SMs: the 256-thread kernel, 128 rows in two passes of 64 tokens
    _w("e128_many_tiles_256_threads", 19200, 128, 128, 2, SM),
]


def _run(w, inp, packed=None):
    cfg = L.config_of(w)
    bufs = L.LayerBuffers.allocate(cfg, with_logits=True)
    L.moe_layer_forward(cfg, inp.U, inp.W_r, inp.b_r, inp.W_noise, inp.eps, inp.W_gate, inp.W_up, inp.W_down, bufs,
                        sel_bias=inp.sel_bias, shared=inp.shared, W_r_packed=packed)
    assert L.moe_get_device_status(bufs.ws) == 0
    return bufs


@pytest.mark.parametrize("w", FUSED, ids=lambda w: w.name)
def test_fused_router_against_the_oracle(w):
    inp, H = margin_inputs(w, seed=2)
    bufs = _run(w, inp)
    check_routing_and_dispatch(w, bufs, H, inp.sel_bias)
    # the same layer from router weights packed once: identical bits
    packed = L.moe_pack_router(L.config_of(w), inp.W_r, inp.W_noise)
    assert packed is not None
    b2 = _run(w, inp, packed)
    for name in ("logits", "idx", "gate", "slot_row", "P", "aux", "z_loss", "out"):
        assert torch.equal(getattr(bufs, name), getattr(b2, name)), name


@pytest.mark.parametrize("w", [W.MIXTRAL, W.SWITCH, W.DSV3, W.STRESS], ids=lambda w: w.name)
def test_route_packed_full_size(w):
    """moe_route_packed at full size (the launch configuration the benchmark times) against the
    oracle, and against moe_route bit for bit."""
    inp, H = margin_inputs(w, seed=3, experts=False)
    cfg = L.config_of(w)
    T, E, k = w.T, w.E, w.k
    ws = L.new_workspace(cfg)
    packed = L.moe_pack_router(cfg, inp.W_r, inp.W_noise)
    outs = []
    for use_packed in (True, False):
        idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
        gate = torch.empty((T, k), dtype=torch.float32, device="cuda")
        logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
        if use_packed:
            L.moe_route_packed(cfg, inp.U, packed, inp.b_r, inp.eps, logits, idx, gate, ws)
        else:
            L.moe_route(cfg, inp.U, inp.W_r, inp.b_r, inp.W_noise, inp.eps, None, logits, idx, gate, ws)
        assert L.moe_get_device_status(ws) == 0
        outs.append((idx, gate, logits))
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
    idx, gate, logits = outs[0]
    r = oracle.route(H, k, w.score_fn, w.renorm)
    assert normwise(logits, H) <= LOGIT_TOL
    assert np.array_equal(idx.cpu().numpy(), r["idx"])
    assert normwise(gate, r["gate"]) <= LOGIT_TOL


def test_pack_router_layout():
    """Row n < E of the packed matrix is column n of W_r, rows E .. 2E-1 (noisy) the columns of
    W_noise, the rest zero, N = 2E rounded up to 16."""
    w = _w("pack", 64, 136, 5, 2, SM, noisy=True)
    cfg = L.config_of(w)
    W_r = torch.randn((w.h, w.E), device="cuda").bfloat16()
    W_n = torch.randn((w.h, w.E), device="cuda").bfloat16()
    packed = L.moe_pack_router(cfg, W_r, W_n)
    N = 16
    assert packed.numel() == N * w.h
    P = packed.view(N, w.h)
    assert torch.equal(P[:5], W_r.t()) and torch.equal(P[5:10], W_n.t())
    assert not P[10:].any()


def test_pack_router_refused_where_unused():
    cfg = L.config(64, 128, 8, 2, 16, dtype=W.F32)
    assert L.router_pack_size(cfg) == 0
    assert L.moe_pack_router(cfg, None, None) is None

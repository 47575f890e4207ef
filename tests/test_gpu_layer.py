"""moe_layer_forward end to end against the oracle.

Oracle-sized workloads are compared element by element on every output.  The
full-size workloads run in the launch configuration the benchmark times; the
routing, dispatch and statistics are compared on every token, the output and
expert rows on a sample of tokens the oracle evaluates one by one, and the
permutation through properties that hold at any size.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import TOL, check_routing_and_dispatch, delta_error, margin_inputs, normwise
from mixture_experts_layer_84_b300 import _lib as L
from mixture_experts_layer_84_b300 import synth
from mixture_experts_layer_84_b300 import workloads as W

pytestmark = pytest.mark.gpu


def run_layer(w, inp, with_logits=True):
    cfg = L.config_of(w)
    bufs = L.LayerBuffers.allocate(cfg, with_logits=with_logits)
    L.moe_layer_forward(cfg, inp.U, inp.W_r, inp.b_r, inp.W_noise, inp.eps, inp.W_gate, inp.W_up, inp.W_down, bufs,
                        sel_bias=inp.sel_bias, shared=inp.shared)
    code = L.moe_get_device_status(bufs.ws)
    assert code == 0, f"device status {code}"
    return cfg, bufs


EDGE = [
    W.MIXTRAL_SMALL.replace(name="mixtral_small_token_major", priority=W.PRIORITY_TOKEN_MAJOR),
    # the literal reading of the capacity, ceil(CF * T / E), through the override
    W.MIXTRAL_SMALL.replace(name="mixtral_small_literal_capacity", capacity=-(-int(1.25 * 700) // 8)),
    W.STRESS_SMALL.replace(name="stress_small_capacity_1", capacity=1),
    W.Workload("one_expert_bf16", T=300, h=256, E=1, k=1, d_e=128, dtype=W.BF16, score_fn=W.SOFTMAX,
               renorm=True, noisy=False, capacity_factor=0.0),
    W.Workload("k_equals_E_bf16", T=257, h=128, E=4, k=4, d_e=256, dtype=W.BF16, score_fn=W.SIGMOID,
               renorm=True, noisy=False, capacity_factor=1.0),
    W.Workload("tails_bf16", T=333, h=136, E=6, k=2, d_e=200, dtype=W.BF16, score_fn=W.SOFTMAX, renorm=True,
               noisy=True, capacity_factor=1.1, bias="zipf"),
    W.Workload("tiny_noisy_f32", T=200, h=64, E=8, k=2, d_e=96, dtype=W.F32, score_fn=W.SOFTMAX, renorm=False,
               noisy=True, capacity_factor=1.0, bias="zipf"),
]


EDGE += [
    W.DSV3_SHARED_SMALL,
    # two shared experts, softmax router with a selection bias, float32
    W.Workload("shared2_bias_f32", T=150, h=64, E=6, k=2, d_e=48, dtype=W.F32, score_fn=W.SOFTMAX, renorm=True,
               noisy=False, capacity_factor=1.0, n_shared=2, d_shared=40, sel_bias="normal"),
    W.Workload("shared2_bias_bf16", T=413, h=192, E=12, k=3, d_e=136, dtype=W.BF16, score_fn=W.SIGMOID,
               renorm=False, noisy=True, capacity_factor=1.3, n_shared=2, d_shared=200, sel_bias="normal"),
    # group-limited routing: DS-V3's 8 groups, 4 kept, without a selection bias; softmax with
    # groups of 16 that straddle the selection lanes' expert chunks, and a capacity limit
    W.DSV3_SMALL.replace(name="dsv3_small_groups", n_group=8, topk_group=4),
    W.STRESS_SMALL.replace(name="stress_small_groups", n_group=4, topk_group=2, capacity_factor=1.25),
]


@pytest.mark.parametrize("w", W.SMALL + EDGE, ids=lambda w: w.name)
def test_layer_small(w):
    inp, H = margin_inputs(w, seed=0)
    cfg, bufs = run_layer(w, inp)
    r, d, A = check_routing_and_dispatch(w, bufs, H, inp.sel_bias)
    ref = oracle.layer_forward(inp, T=w.T, h=w.h, E=w.E, k=w.k, d_e=w.d_e, score_fn=w.score_fn, renorm=w.renorm,
                               capacity_factor=w.capacity_factor, capacity_override=w.capacity,
                               priority=w.priority, logits=H, sel_bias=inp.sel_bias, shared=inp.shared,
                               n_group=w.n_group, topk_group=w.topk_group)
    tol = TOL[w.dtype]
    assert torch.equal(bufs.X[:A], inp.U[bufs.row_token[:A].long()])
    assert normwise(bufs.act[:A], ref["act"]) <= tol
    assert normwise(bufs.Y[:A], ref["Y"]) <= tol
    assert normwise(bufs.out, ref["out"]) <= tol
    assert delta_error(bufs.out, inp.U, ref["out"], w.dtype) <= tol
    if w.n_shared:
        assert normwise(bufs.Y_shared, ref["Y_shared"]) <= tol
    # tokens whose every pair was dropped keep exactly their residual (plus the shared experts)
    sr = bufs.slot_row.view(w.T, w.k)
    gone = torch.all(sr < 0, dim=1)
    if bool(gone.any()) and not w.n_shared:
        assert torch.equal(bufs.out[gone], inp.U[gone])


def test_layer_empty_batch():
    w = W.MIXTRAL_SMALL.replace(name="empty", T=0)
    inp = synth.generate(w, 0, "cuda")
    cfg, bufs = run_layer(w, inp)
    assert bufs.counts_routed.tolist() == [0] * w.E
    assert bufs.offsets.tolist() == [0] * (w.E + 1)
    assert int(bufs.n_dropped.item()) == 0
    assert bufs.f.tolist() == [0.0] * w.E and bufs.P.tolist() == [0.0] * w.E
    assert float(bufs.aux.item()) == 0.0
    assert float(bufs.z_loss.item()) == 0.0


def test_layer_deterministic():
    w = W.STRESS_SMALL
    inp, H = margin_inputs(w, seed=3)
    _, b1 = run_layer(w, inp)
    _, b2 = run_layer(w, inp)
    for name in ("idx", "gate", "slot_row", "offsets", "act", "Y", "out", "P", "aux", "logits"):
        assert torch.equal(getattr(b1, name), getattr(b2, name)), name


SAMPLE = {"mixtral_bf16": 64, "switch_noisy_bf16": 64, "dsv3_bf16": 16, "stress_bf16": 48, "tiny_fp32": 64,
          "dsv3_shared_bf16": 16}


@pytest.mark.parametrize("w", W.FULL + W.EXTENDED, ids=lambda w: w.name)
def test_layer_full_size_sampled(w):
    inp, H = margin_inputs(w, seed=0)
    cfg, bufs = run_layer(w, inp, with_logits=True)
    r, d, A = check_routing_and_dispatch(w, bufs, H, inp.sel_bias)
    # permutation property on every kept row, on the device
    assert torch.equal(bufs.X[:A], inp.U[bufs.row_token[:A].long()])
    rng = np.random.default_rng(0)
    n = SAMPLE[w.name]
    toks = np.unique(np.concatenate([[0, w.T - 1], rng.choice(w.T, size=n, replace=False)]))
    sr = d["slot_row"].reshape(w.T, w.k)
    dropped = np.nonzero(np.any(sr < 0, axis=1))[0]
    if dropped.size:
        toks = np.unique(np.concatenate([toks, dropped[:4]]))
    smp = oracle.sampled_outputs(inp, toks, r["idx"], r["gate"], d["slot_row"], w.k, shared=inp.shared)
    tol = TOL[w.dtype]
    tt = torch.as_tensor(toks, device="cuda")
    assert normwise(bufs.out[tt], smp["out"]) <= tol
    assert delta_error(bufs.out[tt], inp.U[tt], smp["out"], w.dtype) <= tol
    rows = sorted(smp["Y"])
    assert normwise(bufs.Y[torch.as_tensor(rows, device="cuda")], np.stack([smp["Y"][i] for i in rows])) <= tol


@pytest.mark.parametrize("w", [W.MIXTRAL, W.DSV3, W.SWITCH, W.STRESS], ids=lambda w: w.name)
def test_layer_full_size_sampled_swapped_tiles(w, monkeypatch):
    """The full-size layers again with the expert GEMMs on the weights-as-M pair kernel."""
    monkeypatch.setenv("MOE_FFN_TILES", "swab")
    test_layer_full_size_sampled(w)


@pytest.mark.parametrize("w", [W.MIXTRAL_SMALL, W.DSV3_SHARED_SMALL, EDGE[-1]], ids=lambda w: w.name)
def test_layer_small_swapped_tiles(w, monkeypatch):
    monkeypatch.setenv("MOE_FFN_TILES", "swab")
    test_layer_small(w)

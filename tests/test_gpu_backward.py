"""Backward of the router side against the oracle: the combine (gate gradients and the gradient
into the expert outputs) and the router logits (gates, aux loss, z-loss)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import LOGIT_TOL, TOL, normwise
from mixture_experts_layer_84_b300 import _lib as L
from mixture_experts_layer_84_b300 import synth
from mixture_experts_layer_84_b300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,h,E,k,C,dtype", [(700, 512, 8, 2, 200, W.BF16), (333, 136, 6, 3, 0, W.BF16),
                                             (123, 72, 5, 2, 40, W.F32), (4096, 1024, 64, 6, 300, W.BF16)])
def test_combine_backward(T, h, E, k, C, dtype):
    tdt = torch.bfloat16 if dtype == W.BF16 else torch.float32
    idx = synth.random_routing(T, E, k, seed=T, zipf_s=0.8).numpy()
    d = oracle.dispatch(idx, E, C if C else T)
    A = int(d["offsets"][-1])
    dO = synth.random_rows(T, h, 1, "U", "cuda", tdt)
    Y = synth.random_rows(T * k, h, 2, "Y", "cuda", tdt)
    gate = synth.random_gates(T, k, seed=3, device="cuda")
    slot_row = torch.as_tensor(d["slot_row"], dtype=torch.int32, device="cuda")
    cfg = L.config(T, h, E, k, 8, capacity=C, dtype=dtype)
    d_gate = torch.full((T, k), 9.0, dtype=torch.float32, device="cuda")
    dY = torch.full((T * k, h), 7.0, dtype=tdt, device="cuda")
    ws = L.new_workspace(cfg)
    L.moe_combine_backward(cfg, dO, Y, slot_row, gate, d_gate, dY, ws)
    assert L.moe_get_device_status(ws) == 0
    ref = oracle.combine_backward(dO, Y, d["slot_row"], gate, k)
    assert normwise(d_gate, ref["d_gate"]) <= LOGIT_TOL
    assert np.all(d_gate.cpu().numpy()[d["slot_row"].reshape(T, k) < 0] == 0.0)
    kept = np.sort(d["slot_row"][d["slot_row"] >= 0])
    kt = torch.as_tensor(kept, device="cuda")
    assert normwise(dY[kt], ref["dY"][kept]) <= TOL[dtype]
    untouched = np.setdiff1d(np.arange(T * k), kept)
    if untouched.size:
        assert torch.all(dY[torch.as_tensor(untouched, device="cuda")] == 7.0)


@pytest.mark.parametrize("E,k,score_fn,renorm", [(8, 2, W.SOFTMAX, True), (64, 6, W.SOFTMAX, True),
                                                 (128, 1, W.SOFTMAX, False), (256, 8, W.SIGMOID, True),
                                                 (32, 4, W.SIGMOID, False), (1000, 16, W.SOFTMAX, True)])
@pytest.mark.parametrize("w_aux,w_z", [(0.0, 0.0), (0.01, 0.001), (1.0, 1.0)])
def test_route_backward(E, k, score_fn, renorm, w_aux, w_z):
    T = 300
    H = synth.random_logits(T, E, seed=E + k, scale=2.0, tie_fraction=0.1)
    r = oracle.route(oracle.f64(H), k, score_fn, renorm)
    counts = np.bincount(r["idx"].reshape(-1), minlength=E)
    d_gate = synth.normal((T, k), 1.0, seed=E, stream="gates", device="cpu", dtype=torch.float32)
    cfg = L.config(T, 8, E, k, 8, score_fn=score_fn, renorm=renorm, dtype=W.F32)
    dH = torch.full((T, E), 5.0, dtype=torch.float32, device="cuda")
    L.moe_route_backward(cfg, H.cuda(), torch.as_tensor(r["idx"], dtype=torch.int32, device="cuda"), d_gate.cuda(),
                         torch.as_tensor(counts, dtype=torch.int32, device="cuda"), w_aux, w_z, dH)
    torch.cuda.synchronize()
    f = counts / (T * k)
    want = oracle.router_backward(oracle.f64(H), r["idx"], oracle.f64(d_gate), f, score_fn, renorm, w_aux, w_z)
    assert normwise(dH, want) <= LOGIT_TOL


def test_route_backward_under_selection_bias():
    """With a loss-free selection bias the gates are still the scores, so the gate gradient is the
    same function of the (biased) selection."""
    T, E, k = 200, 64, 4
    H = synth.random_logits(T, E, seed=5, scale=2.0, tie_fraction=0.0)
    b = synth.normal((E,), 0.05, seed=5, stream="sel_bias", device="cpu", dtype=torch.float32)
    r = oracle.route(oracle.f64(H), k, W.SIGMOID, True, oracle.f64(b))
    d_gate = synth.normal((T, k), 1.0, seed=6, stream="gates", device="cpu", dtype=torch.float32)
    cfg = L.config(T, 8, E, k, 8, score_fn=W.SIGMOID, renorm=True, dtype=W.F32)
    dH = torch.empty((T, E), dtype=torch.float32, device="cuda")
    L.moe_route_backward(cfg, H.cuda(), torch.as_tensor(r["idx"], dtype=torch.int32, device="cuda"), d_gate.cuda(),
                         None, 0.0, 0.0, dH)
    torch.cuda.synchronize()
    want = oracle.gate_backward(oracle.f64(H), r["idx"], oracle.f64(d_gate), W.SIGMOID, True)
    assert normwise(dH, want) <= LOGIT_TOL


EXPERT_BWD = [
    # T, h, E, k, d_e, capacity (0: unbounded), routing skew
    (700, 512, 8, 2, 640, 0, 0.0),      # several 128-row tiles per expert, 64-row K tails in the weight grads
    (333, 136, 6, 2, 200, 0, 1.2),      # h and d_e off the 64/128 grid, skewed segments
    (300, 256, 96, 3, 384, 0, 0.0),     # many small segments (a few rows each), some experts empty
    (64, 128, 4, 1, 128, 10, 0.0),      # capacity-limited: every segment shorter than one k-block
]


@pytest.mark.parametrize("T,h,E,k,d_e,C,zipf", EXPERT_BWD)
def test_expert_ffn_backward(T, h, E, k, d_e, C, zipf):
    w = W.Workload("bwd", T=T, h=h, E=E, k=k, d_e=d_e, dtype=W.BF16, score_fn=W.SOFTMAX, renorm=True, noisy=False,
                   capacity_factor=0.0, capacity=C)
    inp = synth.generate(w, seed=7, device="cuda")
    idx = synth.random_routing(T, E, k, seed=8, zipf_s=zipf).numpy()
    d = oracle.dispatch(idx, E, C if C else T)
    A = int(d["offsets"][-1])
    Tk = T * k
    X = torch.zeros((Tk, h), dtype=torch.bfloat16, device="cuda")
    X[:A] = inp.U[torch.as_tensor(d["row_token"], device="cuda")]
    offsets = torch.as_tensor(d["offsets"], dtype=torch.int32, device="cuda")
    cfg = L.config_of(w)
    ws = L.new_workspace(cfg)
    act = torch.zeros((Tk, d_e), dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros((Tk, h), dtype=torch.bfloat16, device="cuda")
    L.moe_expert_ffn(cfg, X, offsets, inp.W_gate, inp.W_up, inp.W_down, act, Y, ws)
    dY = torch.full((Tk, h), float("nan"), dtype=torch.bfloat16, device="cuda")  # rows >= A must not be read
    dY[:A] = synth.random_rows(A, h, 9, "Y", "cuda", torch.bfloat16)
    bufs = {n: torch.full((Tk, d_e), 7.0, dtype=torch.bfloat16, device="cuda") for n in ("d_act", "dG", "dUp")}
    dX = torch.full((Tk, h), 7.0, dtype=torch.bfloat16, device="cuda")
    dW = {n: torch.full(s, 7.0, dtype=torch.float32, device="cuda")
          for n, s in (("dW_gate", (E, d_e, h)), ("dW_up", (E, d_e, h)), ("dW_down", (E, h, d_e)))}
    L.moe_expert_ffn_backward(cfg, X, offsets, inp.W_gate, inp.W_up, inp.W_down, act, dY, bufs["d_act"], bufs["dG"],
                              bufs["dUp"], dX, dW["dW_gate"], dW["dW_up"], dW["dW_down"], ws)
    assert L.moe_get_device_status(ws) == 0
    ref = oracle.expert_ffn_backward(X[:A], d["offsets"], inp.W_gate, inp.W_up, inp.W_down, dY[:A], d_e)
    tol = TOL[W.BF16]
    for n in ("d_act", "dG", "dUp"):
        assert normwise(bufs[n][:A], ref[n]) <= tol, n
    assert normwise(dX[:A], ref["dX"]) <= tol
    for n in ("dW_gate", "dW_up", "dW_down"):
        assert normwise(dW[n], ref[n]) <= tol, n
        # per expert too, so that a small expert cannot hide behind a large one
        for e in range(E):
            if d["offsets"][e + 1] > d["offsets"][e]:
                assert normwise(dW[n][e], ref[n][e]) <= tol, (n, e)
            else:
                assert torch.all(dW[n][e] == 0.0), (n, e)
    assert torch.all(dX[A:] == 7.0)


@pytest.mark.parametrize("dtype", [W.BF16, W.F32])
def test_dispatch_backward(dtype):
    T, h, E, k = 500, 264, 16, 3
    tdt = torch.bfloat16 if dtype == W.BF16 else torch.float32
    idx = synth.random_routing(T, E, k, seed=3, zipf_s=1.0).numpy()
    d = oracle.dispatch(idx, E, 60)
    dO = synth.random_rows(T, h, 1, "U", "cuda", tdt)
    dX = synth.random_rows(T * k, h, 2, "X", "cuda", tdt)
    dU = torch.empty((T, h), dtype=tdt, device="cuda")
    cfg = L.config(T, h, E, k, 8, capacity=60, dtype=dtype)
    ws = L.new_workspace(cfg)
    L.moe_dispatch_backward(cfg, dO, dX, torch.as_tensor(d["slot_row"], dtype=torch.int32, device="cuda"), dU, ws)
    assert L.moe_get_device_status(ws) == 0
    ref = oracle.dispatch_backward(dO, dX, d["slot_row"], k)
    assert normwise(dU, ref) <= TOL[dtype]


LAYER_BWD = [W.MIXTRAL_SMALL, W.SWITCH_SMALL, W.DSV3_SHARED_SMALL, W.STRESS_SMALL,
             W.Workload("bwd_shared2_softmax_norenorm", T=333, h=192, E=12, k=3, d_e=136, dtype=W.BF16,
                        score_fn=W.SOFTMAX, renorm=False, noisy=False, capacity_factor=1.2, bias="normal",
                        n_shared=2, d_shared=200)]


@pytest.mark.parametrize("w", LAYER_BWD, ids=lambda w: w.name)
def test_layer_backward(w):
    """moe_layer_backward against the oracle's layer_backward (itself pinned to torch autograd):
    every input and weight gradient, with the balance loss and the z-loss in the objective."""
    from gpu_helpers import margin_inputs
    inp, H = margin_inputs(w, seed=2)
    cfg = L.config_of(w)
    bufs = L.LayerBuffers.allocate(cfg, with_logits=True)
    L.moe_layer_forward(cfg, inp.U, inp.W_r, inp.b_r, inp.W_noise, inp.eps, inp.W_gate, inp.W_up, inp.W_down, bufs,
                        sel_bias=inp.sel_bias, shared=inp.shared)
    dO = synth.random_rows(w.T, w.h, 11, "Y", "cuda", torch.bfloat16)
    grads = L.GradBuffers.allocate(cfg)
    w_aux, w_z = 0.5, 0.05
    L.moe_layer_backward(cfg, inp.U, inp.W_r, inp.b_r, inp.W_noise, inp.eps, inp.W_gate, inp.W_up, inp.W_down, bufs,
                         dO, grads, w_aux=w_aux, w_z=w_z, sel_bias=inp.sel_bias, shared=inp.shared)
    assert L.moe_get_device_status(bufs.ws) == 0
    fwd = oracle.layer_forward(inp, T=w.T, h=w.h, E=w.E, k=w.k, d_e=w.d_e, score_fn=w.score_fn, renorm=w.renorm,
                               capacity_factor=w.capacity_factor, capacity_override=w.capacity, priority=w.priority,
                               logits=H, sel_bias=inp.sel_bias, shared=inp.shared, n_group=w.n_group,
                               topk_group=w.topk_group)
    ref = oracle.layer_backward(inp, fwd, dO, k=w.k, d_e=w.d_e, score_fn=w.score_fn, renorm=w.renorm, w_aux=w_aux,
                                w_z=w_z)
    tol = TOL[W.BF16]
    names = ["dU", "dH", "dW_gate", "dW_up", "dW_down", "dW_r", "db_r"]
    if w.noisy:
        names.append("dW_noise")
    if w.n_shared:
        names += ["dW_gate_shared", "dW_up_shared", "dW_down_shared"]
    for n in names:
        refn = ref[n[:-len("_shared")] + "_sh" if n.endswith("_shared") else n]
        assert normwise(getattr(grads, n), refn) <= tol, n


@pytest.mark.parametrize("E,noisy", [(6, False), (5, True), (8, False)])
def test_router_input_backward_narrow_rows(E, noisy):
    """The router's weight gradients [h, E] with E not a multiple of 4 (rows of E floats take the
    plain-store epilogue; multiples of 4 the TMA-store one) against the oracle."""
    import ctypes
    T, h = 300, 192
    w = W.Workload("rb", T=T, h=h, E=E, k=2, d_e=64, dtype=W.BF16, score_fn=W.SOFTMAX, renorm=True, noisy=noisy,
                   capacity_factor=0.0)
    inp = synth.generate(w, seed=4, device="cuda", experts=False)
    dH = synth.normal((T, E), 1.0, 3, "logits", "cuda", torch.float32)
    cfg = L.config_of(w)
    dU = torch.empty((T, h), dtype=torch.bfloat16, device="cuda")
    dW_r = torch.full((h, E), 7.0, dtype=torch.float32, device="cuda")
    dW_n = torch.full((h, E), 7.0, dtype=torch.float32, device="cuda") if noisy else None
    db = torch.empty(E, dtype=torch.float32, device="cuda")
    ws = L.new_workspace(cfg)
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    st = L.lib.moe_router_input_backward(ctypes.byref(cfg), P(inp.U), P(inp.W_r), P(inp.W_noise), P(inp.eps), P(dH),
                                         P(dU), P(dW_r), P(dW_n), P(db), P(ws), None)
    assert st == L.MOE_OK, L.lib.moe_last_error().decode()
    assert L.moe_get_device_status(ws) == 0
    # the library rounds dH (and dN) to bf16 for the tensor-core products
    ref = oracle.router_input_backward(inp.U, inp.W_r, oracle.f64(dH.bfloat16()), inp.W_noise, inp.eps)
    err = normwise(dW_r, ref["dW_r"])
    assert err <= 2e-2, err
    if noisy:
        err = normwise(dW_n, ref["dW_noise"])
        assert err <= 2e-2, err

"""moe_expert_ffn against the oracle: the grouped SwiGLU over ragged expert segments
(tcgen05 for bf16, CUDA cores for float32)."""
import pytest
import torch

import oracle
from gpu_helpers import TOL, normwise
from mixture_experts_layer_84_b300 import _lib as L
from mixture_experts_layer_84_b300 import synth
from mixture_experts_layer_84_b300 import workloads as W

pytestmark = pytest.mark.gpu

EDGE = [
    # h and d_e off the 64/128 grid: K tails and an output-column tail
    W.Workload("ffn_tails_bf16", T=333, h=136, E=6, k=2, d_e=200, dtype=W.BF16, score_fn=W.SOFTMAX, renorm=True,
               noisy=False, capacity_factor=0.0),
    W.Workload("ffn_one_expert_bf16", T=300, h=256, E=1, k=1, d_e=128, dtype=W.BF16, score_fn=W.SOFTMAX,
               renorm=True, noisy=False, capacity_factor=0.0),
    W.Workload("ffn_many_small_bf16", T=700, h=320, E=96, k=3, d_e=384, dtype=W.BF16, score_fn=W.SIGMOID,
               renorm=True, noisy=False, capacity_factor=0.0),
    W.Workload("ffn_tails_f32", T=123, h=72, E=5, k=2, d_e=40, dtype=W.F32, score_fn=W.SOFTMAX, renorm=True,
               noisy=False, capacity_factor=0.0),
    # segments longer than the weights (~1000 rows against 2 x 72 gate|up and 192 down rows): both
    # GEMMs take column tiles fastest, with ragged row, column and K tails
    W.Workload("ffn_long_segments_bf16", T=1500, h=192, E=3, k=2, d_e=72, dtype=W.BF16, score_fn=W.SOFTMAX,
               renorm=True, noisy=False, capacity_factor=0.0),
]


def segments(w, seed, zipf):
    idx = synth.random_routing(w.T, w.E, w.k, seed=seed, zipf_s=zipf).numpy()
    C = oracle.capacity(w.T, w.E, w.k, w.capacity_factor, w.capacity)
    return oracle.dispatch(idx, w.E, C, w.priority)


@pytest.mark.parametrize("tiles", ["single", "pair", "swab"])
@pytest.mark.parametrize("w", W.SMALL + EDGE, ids=lambda w: w.name)
@pytest.mark.parametrize("zipf", [0.0, 1.2])
def test_expert_ffn(w, zipf, tiles, monkeypatch, order=None):
    """The three bf16 kernels (128-row tiles on one CTA, 256-row tiles on a CTA pair, and weight
    rows as M with tokens as N on a CTA pair) against the oracle."""
    if w.dtype == W.F32 and tiles != "single":
        pytest.skip("float32 runs on the CUDA cores")
    monkeypatch.setenv("MOE_FFN_TILES", tiles)
    if order:
        monkeypatch.setenv("MOE_FFN_ORDER", order)
    inp = synth.generate(w, seed=2, device="cuda")
    d = segments(w, seed=9, zipf=zipf)
    A = int(d["offsets"][-1])
    Tk = w.T * w.k
    X = torch.zeros((Tk, w.h), dtype=w.torch_dtype, device="cuda")
    X[:A] = inp.U[torch.as_tensor(d["row_token"], device="cuda")]
    offsets = torch.as_tensor(d["offsets"], dtype=torch.int32, device="cuda")
    act = torch.full((Tk, w.d_e), 7.0, dtype=w.torch_dtype, device="cuda")
    Y = torch.full((Tk, w.h), 7.0, dtype=w.torch_dtype, device="cuda")
    cfg = L.config_of(w)
    ws = L.new_workspace(cfg)
    L.moe_expert_ffn(cfg, X, offsets, inp.W_gate, inp.W_up, inp.W_down, act, Y, ws)
    assert L.moe_get_device_status(ws) == 0
    Y_ref, act_ref = oracle.expert_ffn(X[:A], d["offsets"], inp.W_gate, inp.W_up, inp.W_down, w.d_e)
    tol = TOL[w.dtype]
    assert normwise(act[:A], act_ref) <= tol
    assert normwise(Y[:A], Y_ref) <= tol
    # per expert as well, so a small expert cannot hide behind a large one
    for e in range(w.E):
        lo, hi = int(d["offsets"][e]), int(d["offsets"][e + 1])
        if hi > lo:
            assert normwise(Y[lo:hi], Y_ref[lo:hi]) <= tol, e
    # rows >= A are not written
    assert torch.all(Y[A:] == 7.0) and torch.all(act[A:] == 7.0)


@pytest.mark.parametrize("order", ["rows", "cols"])
@pytest.mark.parametrize("tiles", ["single", "pair"])
@pytest.mark.parametrize("w", [EDGE[0], EDGE[-1]], ids=lambda w: w.name)
def test_expert_ffn_tile_orders(w, tiles, order, monkeypatch):
    """Both tile orders (row tiles or column tiles fastest inside an expert) on both row-tiled
    kernels, with ragged row, column and K tails."""
    test_expert_ffn(w, 1.2, tiles, monkeypatch, order=order)


@pytest.mark.parametrize("l2", ["none", "first"])
def test_expert_ffn_l2_hints(l2, monkeypatch):
    """The L2 hint modes kept for measurement change nothing but the cache policy."""
    monkeypatch.setenv("MOE_FFN_L2", l2)
    test_expert_ffn(EDGE[-1], 1.2, "pair", monkeypatch, order="cols")


@pytest.mark.parametrize("dtype,tiles", [(W.BF16, "single"), (W.BF16, "pair"), (W.BF16, "swab"), (W.F32, "single")])
def test_expert_ffn_rejects_inconsistent_offsets(dtype, tiles, monkeypatch):
    monkeypatch.setenv("MOE_FFN_TILES", tiles)
    w = W.Workload("bad", T=64, h=64, E=4, k=2, d_e=64, dtype=dtype, score_fn=0, renorm=True, noisy=False,
                   capacity_factor=0.0)
    inp = synth.generate(w, seed=2, device="cuda")
    Tk = w.T * w.k
    X = torch.zeros((Tk, w.h), dtype=w.torch_dtype, device="cuda")
    act = torch.full((Tk, w.d_e), 7.0, dtype=w.torch_dtype, device="cuda")
    Y = torch.full((Tk, w.h), 7.0, dtype=w.torch_dtype, device="cuda")
    cfg = L.config_of(w)
    ws = L.new_workspace(cfg)
    for bad in ([0, 10, 5, 20, 30], [0, 10, 20, 30, Tk + 1], [-4, 10, 20, 30, 40]):
        offsets = torch.tensor(bad, dtype=torch.int32, device="cuda")
        L.moe_expert_ffn(cfg, X, offsets, inp.W_gate, inp.W_up, inp.W_down, act, Y, ws)
        assert L.moe_get_device_status(ws) == L.MOE_DEV_BAD_OFFSETS
        assert torch.all(Y == 7.0) and torch.all(act == 7.0)


@pytest.mark.parametrize("tiles", ["single", "pair"])
@pytest.mark.parametrize("T,h,n_shared,d_shared,dtype", [(600, 512, 1, 384, W.BF16), (1100, 256, 2, 200, W.BF16),
                                                         (130, 64, 2, 40, W.F32), (1, 128, 1, 64, W.BF16)])
def test_shared_ffn(T, h, n_shared, d_shared, dtype, tiles, monkeypatch):
    """moe_shared_ffn: every shared expert's SwiGLU on every token, against the oracle."""
    if dtype == W.F32 and tiles == "pair":
        pytest.skip("float32 runs on the CUDA cores")
    monkeypatch.setenv("MOE_FFN_TILES", tiles)
    w = W.Workload("shared", T=T, h=h, E=4, k=1, d_e=64, dtype=dtype, score_fn=W.SOFTMAX, renorm=True, noisy=False,
                   capacity_factor=0.0, n_shared=n_shared, d_shared=d_shared)
    inp = synth.generate(w, seed=5, device="cuda")
    cfg = L.config_of(w)
    act = torch.empty((n_shared, T, d_shared), dtype=w.torch_dtype, device="cuda")
    Y = torch.full((n_shared, T, h), 7.0, dtype=w.torch_dtype, device="cuda")
    ws = L.new_workspace(cfg)
    L.moe_shared_ffn(cfg, inp.U, inp.W_gate_sh, inp.W_up_sh, inp.W_down_sh, act, Y, ws)
    assert L.moe_get_device_status(ws) == 0
    ref = oracle.shared_ffn(inp.U, *inp.shared)
    for i in range(n_shared):
        assert normwise(Y[i], ref[i]) <= TOL[dtype], i

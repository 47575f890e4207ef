"""The FP8 dispatch and up-projection against the oracle.

Codes and scales are compared bit for bit (both sides take the same exact
power-of-two scaling of the same bf16 inputs and round to nearest even);
act, Y and out within the bf16 tolerance of the oracle's exact products of
the dequantised values.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import TOL, delta_error, margin_inputs, normwise, route_of
from mixture_experts_layer_84_b300 import _lib as L
from mixture_experts_layer_84_b300 import synth
from mixture_experts_layer_84_b300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_BF16 = TOL[W.BF16]


def _codes_and_scales(A):
    codes, s = oracle.quantize_rows_fp8(A)
    return oracle.e4m3_bits(codes), np.ldexp(1.0, s)


@pytest.mark.parametrize("rows,cols", [(1, 8), (37, 136), (300, 4096), (5, 7168), (0, 64)])
def test_quantize_rows_bitexact(rows, cols):
    """Rows at very different magnitudes (1e-30 .. 1e30), an all-zero row and exact powers of two."""
    x = synth.random_rows(rows, cols, seed=cols, stream="X", device="cpu", dtype=torch.float32)
    if rows:
        mags = torch.logspace(-30, 30, rows, dtype=torch.float64).to(torch.float32)
        x = x * mags[:, None]
        x[0, 0] = 448.0 if rows > 2 else x[0, 0]
        if rows > 3:
            x[1] = 0.0
            x[2, :] = 2.0 ** -3
    xb = x.to(torch.bfloat16)
    dst = torch.full((rows, cols), 0xAA, dtype=torch.uint8, device="cuda")
    scale = torch.full((rows,), -1.0, dtype=torch.float32, device="cuda")
    L.moe_quantize_fp8(xb.cuda(), dst, scale)
    torch.cuda.synchronize()
    codes, sc = _codes_and_scales(xb)
    assert np.array_equal(dst.cpu().numpy(), codes.reshape(rows, cols))
    assert np.array_equal(scale.cpu().numpy().astype(np.float64), sc)


@pytest.mark.parametrize("T,E,k,C,h", [(700, 8, 2, 220, 512), (3000, 64, 6, 300, 256), (4096, 256, 8, 0, 7168),
                                       (1, 1, 1, 1, 16)])
def test_dispatch_fp8_bitexact(T, E, k, C, h):
    """Routing metadata identical to moe_dispatch; X8[row] the codes of U[row_token[row]]."""
    idx = synth.random_routing(T, E, k, seed=T + E, zipf_s=0.7).cuda()
    U = synth.random_rows(T, h, seed=5, stream="U", device="cuda", dtype=torch.bfloat16)
    cfg = L.config(T, h, E, k, 16, capacity=C, capacity_factor=0.0)
    i32 = dict(dtype=torch.int32, device="cuda")
    out = {n: torch.full((m,), -5, **i32) for n, m in (("counts_routed", E), ("counts_kept", E), ("offsets", E + 1),
                                                       ("slot_row", T * k), ("row_token", T * k))}
    nd = torch.full((1,), -5, dtype=torch.int64, device="cuda")
    rows = L.FP8Rows.allocate(cfg)
    ws = L.new_workspace(cfg)
    L.moe_dispatch_fp8(cfg, U, idx, out["counts_routed"], out["counts_kept"], out["offsets"], out["slot_row"],
                       out["row_token"], rows.X8, rows.x_scale, nd, ws)
    assert L.moe_get_device_status(ws) == 0
    d = oracle.dispatch(idx.cpu().numpy(), E, C if C > 0 else T, W.PRIORITY_CHOICE_MAJOR)
    A = int(d["offsets"][-1])
    for n in ("counts_routed", "counts_kept", "offsets", "slot_row"):
        assert np.array_equal(out[n].cpu().numpy(), d[n]), n
    assert np.array_equal(out["row_token"][:A].cpu().numpy(), d["row_token"])
    assert int(nd.item()) == d["n_dropped"]
    codes, sc = _codes_and_scales(U.cpu())
    rt = d["row_token"]
    assert np.array_equal(rows.X8[:A].cpu().numpy(), codes[rt])
    assert np.array_equal(rows.x_scale[:A].cpu().numpy().astype(np.float64), sc[rt])


FFN = [
    W.MIXTRAL_SMALL,
    W.DSV3_SMALL,
    # K tail (h = 272: two full 128-element stages and one of 16) and an output-column tail
    W.Workload("fp8_tails", T=333, h=272, E=6, k=2, d_e=200, dtype=W.BF16, score_fn=W.SOFTMAX, renorm=True,
               noisy=False, capacity_factor=0.0),
    W.Workload("fp8_many_small", T=700, h=320, E=96, k=3, d_e=384, dtype=W.BF16, score_fn=W.SIGMOID,
               renorm=True, noisy=False, capacity_factor=0.0),
]


@pytest.mark.parametrize("tiles", ["single", "swab"])
@pytest.mark.parametrize("w", FFN, ids=lambda w: w.name)
@pytest.mark.parametrize("zipf", [0.0, 1.2])
def test_expert_ffn_fp8(w, zipf, tiles, monkeypatch):
    """Weights quantised on the GPU (bit-exact against the oracle), the dispatch's FP8 rows, then
    act and Y against the oracle's SwiGLU on the dequantised rows and weights; the FP8 gate|up
    GEMM on the single-CTA kernel and on the weights-as-M pair kernel."""
    monkeypatch.setenv("MOE_FFN_TILES", tiles)
    inp = synth.generate(w, seed=1, device="cuda")
    idx = synth.random_routing(w.T, w.E, w.k, seed=9, zipf_s=zipf).cuda()
    cfg = L.config_of(w)
    w8 = L.FP8Weights.quantize(inp.W_gate, inp.W_up)
    torch.cuda.synchronize()
    for q, s, Wt in ((w8.W_gate8, w8.s_gate, inp.W_gate), (w8.W_up8, w8.s_up, inp.W_up)):
        codes, sc = _codes_and_scales(Wt.reshape(-1, w.h).cpu())
        assert np.array_equal(q.reshape(-1, w.h).cpu().numpy(), codes)
        assert np.array_equal(s.cpu().numpy().astype(np.float64), sc)
    bufs = L.LayerBuffers.allocate(cfg, with_X=False)
    rows = L.FP8Rows.allocate(cfg)
    L.moe_dispatch_fp8(cfg, inp.U, idx, bufs.counts_routed, bufs.counts_kept, bufs.offsets, bufs.slot_row,
                       bufs.row_token, rows.X8, rows.x_scale, bufs.n_dropped, bufs.ws)
    L.moe_expert_ffn_fp8(cfg, rows.X8, rows.x_scale, bufs.offsets, w8, inp.W_down, bufs.act, bufs.Y, bufs.ws)
    assert L.moe_get_device_status(bufs.ws) == 0
    offsets = bufs.offsets.cpu().numpy()
    A = int(offsets[-1])
    X = oracle.dequantize_rows_fp8(*oracle.quantize_rows_fp8(inp.U.cpu()))[bufs.row_token[:A].cpu().numpy()]
    Y, act = oracle.expert_ffn(X, offsets, oracle.fp8_weights(inp.W_gate.cpu()), oracle.fp8_weights(inp.W_up.cpu()),
                               inp.W_down.cpu(), w.d_e)
    assert normwise(bufs.act[:A], act) <= TOL_BF16
    assert normwise(bufs.Y[:A], Y) <= TOL_BF16


def _run_layer_fp8(w, inp):
    cfg = L.config_of(w)
    bufs = L.LayerBuffers.allocate(cfg, with_logits=True, with_X=False)
    rows = L.FP8Rows.allocate(cfg)
    w8 = L.FP8Weights.quantize(inp.W_gate, inp.W_up)
    L.moe_layer_forward_fp8(cfg, inp.U, inp.W_r, inp.b_r, inp.W_noise, inp.eps, w8, inp.W_down, bufs, rows,
                            sel_bias=inp.sel_bias, shared=inp.shared)
    assert L.moe_get_device_status(bufs.ws) == 0
    return bufs, rows


LAYER = [W.MIXTRAL_SMALL, W.SWITCH_SMALL, W.DSV3_SHARED_SMALL, W.STRESS_SMALL]


@pytest.mark.parametrize("w", LAYER, ids=lambda w: w.name)
def test_layer_forward_fp8(w):
    inp, H = margin_inputs(w, seed=0)
    bufs, rows = _run_layer_fp8(w, inp)
    ref = oracle.layer_forward(inp, T=w.T, h=w.h, E=w.E, k=w.k, d_e=w.d_e, score_fn=w.score_fn, renorm=w.renorm,
                               capacity_factor=w.capacity_factor, capacity_override=w.capacity, priority=w.priority,
                               logits=H, sel_bias=inp.sel_bias, shared=inp.shared, n_group=w.n_group,
                               topk_group=w.topk_group, fp8=True)
    assert np.array_equal(bufs.idx.cpu().numpy(), ref["idx"])
    assert np.array_equal(bufs.slot_row.cpu().numpy(), ref["slot_row"])
    A = int(ref["offsets"][-1])
    assert np.array_equal(rows.X8[:A].cpu().numpy(), oracle.e4m3_bits(ref["U_codes"])[ref["row_token"]])
    assert normwise(bufs.act[:A], ref["act"]) <= TOL_BF16
    assert normwise(bufs.Y[:A], ref["Y"]) <= TOL_BF16
    assert normwise(bufs.out, ref["out"]) <= TOL_BF16
    assert delta_error(bufs.out, inp.U, ref["out"], W.BF16) <= TOL_BF16


def test_layer_forward_fp8_full_size_sampled():
    """Mixtral-shaped layer at full size: sampled tokens against the oracle's FP8 experts."""
    w = W.MIXTRAL
    inp, H = margin_inputs(w, seed=0)
    bufs, rows = _run_layer_fp8(w, inp)
    r = route_of(w, H, inp.sel_bias)
    assert np.array_equal(bufs.idx.cpu().numpy(), r["idx"])
    # the drops and slots come from the oracle's own dispatch, checked against the library first
    C = oracle.capacity(w.T, w.E, w.k, w.capacity_factor, w.capacity)
    d = oracle.dispatch(r["idx"], w.E, C, w.priority)
    assert np.array_equal(bufs.slot_row.cpu().numpy(), d["slot_row"])
    assert np.array_equal(bufs.offsets.cpu().numpy(), d["offsets"])
    toks = np.unique(np.concatenate([[0, w.T - 1], np.random.default_rng(0).choice(w.T, size=24, replace=False)]))
    dropped = np.nonzero(np.any(d["slot_row"].reshape(w.T, w.k) < 0, axis=1))[0]
    if dropped.size:
        toks = np.unique(np.concatenate([toks, dropped[:4]]))
    smp = oracle.sampled_outputs(inp, toks, r["idx"], r["gate"], d["slot_row"], w.k, fp8=True)
    tt = torch.as_tensor(toks, device="cuda")
    assert normwise(bufs.out[tt], smp["out"]) <= TOL_BF16
    assert delta_error(bufs.out[tt], inp.U[tt], smp["out"], W.BF16) <= TOL_BF16

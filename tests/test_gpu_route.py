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


@pytest.mark.parametrize("score_fn", [SM, SG])
def test_route_stage_mode_masked_experts(score_fn):
    """Logits of -inf (masked experts) are valid input: they rank last, ties to the lower id,
    and get zero weight, as in the oracle."""
    T, E, k = 70, 24, 6
    logits = synth.random_logits(T, E, seed=11, scale=2.0, tie_fraction=0.0)
    logits[:, 3::4] = -float("inf")
    logits[5, :] = -float("inf")
    logits[5, 7] = 0.25
    cfg = L.config(T, 8, E, k, 8, score_fn=score_fn, renorm=True, dtype=W.F32)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ws = L.new_workspace(cfg)
    L.moe_route(cfg, None, None, None, None, None, logits.cuda(), None, idx, gate, ws)
    assert L.moe_get_device_status(ws) == 0
    r = oracle.route(oracle.f64(logits), k, score_fn, True)
    assert np.array_equal(idx.cpu().numpy(), r["idx"])
    assert normwise(gate, r["gate"]) <= LOGIT_TOL
    assert idx[5].tolist() == [7, 0, 1, 2, 3, 4]


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


@pytest.mark.parametrize("w", [W.MIXTRAL_SMALL, W.SWITCH_SMALL, W.DSV3_SMALL], ids=lambda w: w.name)
def test_route_repeated_calls_on_one_workspace(w):
    """The tensor-core router splits h over several CTAs per token tile; the CTA that finishes a
    tile last adds the slices up, using per-tile counters kept in the workspace.  Repeated calls
    on one workspace must give identical results (the counters return to zero), and the P sums
    it leaves behind must match the oracle."""
    inp, H = margin_inputs(w, seed=4, experts=False)
    cfg = L.config_of(w)
    T, E, k = w.T, w.E, w.k
    ws = L.new_workspace(cfg)
    outs = []
    for _ in range(3):
        idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
        gate = torch.empty((T, k), dtype=torch.float32, device="cuda")
        L.moe_route(cfg, inp.U, inp.W_r, inp.b_r, inp.W_noise, inp.eps, None, None, idx, gate, ws)
        assert L.moe_get_device_status(ws) == 0
        outs.append((idx, gate))
    for idx, gate in outs[1:]:
        assert torch.equal(idx, outs[0][0]) and torch.equal(gate, outs[0][1])
    r = oracle.route(H, k, w.score_fn, w.renorm)
    assert np.array_equal(outs[0][0].cpu().numpy(), r["idx"])
    # the statistics read the router's per-tile score sums from the same workspace
    counts = torch.as_tensor(np.bincount(r["idx"].reshape(-1), minlength=E), dtype=torch.int32, device="cuda")
    f, P, aux = (torch.empty(n, dtype=torch.float32, device="cuda") for n in (E, E, 1))
    U0 = torch.zeros((T, w.h), dtype=w.torch_dtype, device="cuda")
    Y0 = torch.zeros((T * k, w.h), dtype=w.torch_dtype, device="cuda")
    sr = torch.full((T * k,), -1, dtype=torch.int32, device="cuda")
    out = torch.empty((T, w.h), dtype=w.torch_dtype, device="cuda")
    z = torch.empty(1, dtype=torch.float32, device="cuda")
    L.moe_combine(cfg, U0, Y0, sr, outs[0][1], counts, out, f, P, aux, ws, z_loss=z)
    assert L.moe_get_device_status(ws) == 0
    st = oracle.load_stats(np.bincount(r["idx"].reshape(-1), minlength=E), r["s"], T, k, w.score_fn)
    assert normwise(P, st["P"]) <= LOGIT_TOL
    assert abs(float(aux.item()) - st["aux"]) <= LOGIT_TOL * max(1.0, abs(st["aux"]))
    zl = oracle.router_z_loss(H)
    assert abs(float(z.item()) - zl) <= LOGIT_TOL * max(1.0, abs(zl))


@pytest.mark.parametrize("T,E,k,score_fn,renorm", [(300, 8, 2, SG, True), (257, 256, 8, SG, True),
                                                   (180, 64, 6, SM, True), (90, 128, 1, SM, False),
                                                   (60, 1024, 16, SG, False)])
def test_route_loss_free_selection_bias(T, E, k, score_fn, renorm):
    """Loss-free balancing: top-k on score + bias, gates from the scores.  Both sides get the same
    float32 logits; the rows whose selection keys keep a margin of 1e-4 (a few float32 ulps of a
    score, well above the float32 score rounding) must select exactly what the oracle selects,
    and every row's gates must be the scores of the experts it selected."""
    logits = synth.random_logits(T, E, seed=T + E + 1, scale=2.0, tie_fraction=0.0)
    bias = synth.normal((E,), 0.05, seed=E, stream="sel_bias", device="cpu", dtype=torch.float32)
    cfg = L.config(T, 8, E, k, 8, score_fn=score_fn, renorm=renorm, dtype=W.F32)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ws = L.new_workspace(cfg)
    L.moe_route(cfg, None, None, None, None, None, logits.cuda(), None, idx, gate, ws, sel_bias=bias.cuda())
    assert L.moe_get_device_status(ws) == 0
    r = oracle.route(oracle.f64(logits), k, score_fn, renorm, oracle.f64(bias))
    ok = oracle.topk_margins(r["sel_key"], k) >= 1e-4
    assert ok.mean() > 0.5
    got = idx.cpu().numpy()
    assert np.array_equal(got[ok], r["idx"][ok])
    # gates: the (renormalised) scores of whatever was selected
    sel = np.take_along_axis(r["s"], got.astype(np.int64), axis=1)
    want = sel / sel.sum(axis=1, keepdims=True) if renorm else sel
    assert normwise(gate, want) <= LOGIT_TOL


GROUPED = [  # T, E, k, n_group, topk_group, score_fn, renorm, selection bias
    (300, 256, 8, 8, 4, SG, True, True),     # DS-V3's groups with the loss-free bias (lane = group)
    (257, 256, 8, 8, 4, SG, True, False),
    (180, 64, 6, 4, 2, SM, True, False),     # 2 lanes per token, 4 groups of 16
    (150, 96, 4, 6, 2, SM, True, True),      # 4 lanes of 24 experts, groups of 16 straddle them
    (100, 12, 4, 3, 2, SM, False, True),     # one lane per token
    (90, 1024, 16, 32, 8, SG, True, False),  # 32 groups of 32, one per lane
    (77, 40, 3, 20, 3, SG, False, False),    # groups of 2, r = 1
    (64, 32, 2, 32, 2, SG, True, False),     # groups of one expert
    (0, 256, 8, 8, 4, SG, True, False),
]


@pytest.mark.parametrize("T,E,k,n_group,topk_group,score_fn,renorm,bias", GROUPED)
def test_route_group_limited(T, E, k, n_group, topk_group, score_fn, renorm, bias):
    """Group-limited routing on the same float32 logits on both sides.  Rows whose group scores
    and kept-expert keys keep a margin of 1e-4 (far above float32 score rounding) select exactly
    what the oracle selects; every row uses at most topk_group groups and distinct experts, with
    gates equal to the scores of what it selected.  The constant rows (all group scores tied)
    keep the lowest groups and then the lowest ids."""
    logits = synth.random_logits(T, E, seed=T + E + 5, scale=2.0, tie_fraction=0.0)
    b = synth.normal((E,), 0.05, seed=E + 1, stream="sel_bias", device="cpu", dtype=torch.float32) if bias else None
    cfg = L.config(T, 8, E, k, 8, score_fn=score_fn, renorm=renorm, dtype=W.F32, n_group=n_group,
                   topk_group=topk_group)
    idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    gate = torch.full((T, k), -7.0, dtype=torch.float32, device="cuda")
    ws = L.new_workspace(cfg)
    L.moe_route(cfg, None, None, None, None, None, logits.cuda(), None, idx, gate, ws,
                sel_bias=None if b is None else b.cuda())
    assert L.moe_get_device_status(ws) == 0
    if T == 0:
        return
    bb = None if b is None else oracle.f64(b)
    r = oracle.route(oracle.f64(logits), k, score_fn, renorm, bb, n_group, topk_group)
    key = r["sel_key"]
    aff = r["s"] if b is None else key
    ok = ((oracle.group_margins(aff, n_group, topk_group, k) >= 1e-4)
          & (oracle.topk_margins(np.where(r["allowed"], key, -np.inf), k) >= 1e-4))
    assert ok.mean() > 0.5
    got = idx.cpu().numpy()
    assert np.array_equal(got[ok], r["idx"][ok])
    groups = got // (E // n_group)
    assert all(len(set(g)) <= topk_group for g in groups.tolist())
    assert all(len(set(row)) == k for row in got.tolist())
    assert got.min() >= 0 and got.max() < E
    sel = np.take_along_axis(r["s"], got.astype(np.int64), axis=1)
    want = sel / sel.sum(axis=1, keepdims=True) if renorm else sel
    assert normwise(gate, want) <= LOGIT_TOL
    if T >= 4 and b is None:  # random_logits makes the last two rows constant
        assert got[-1].tolist() == list(range(k)) == r["idx"][-1].tolist()


@pytest.mark.parametrize("E", [8, 256, 1000])
def test_balance_bias_update(E):
    counts = torch.as_tensor(np.random.default_rng(E).integers(0, 50, size=E), dtype=torch.int32)
    counts[0] = int(counts.sum() - counts[0]) // (E - 1) if E > 1 else counts[0]
    bias = synth.normal((E,), 0.1, seed=E, stream="sel_bias", device="cpu", dtype=torch.float32)
    cfg = L.config(64, 8, E, 1, 8, dtype=W.F32)
    b = bias.cuda()
    L.moe_balance_bias_update(cfg, counts.cuda(), 0.001, b)
    torch.cuda.synchronize()
    want = oracle.balance_bias_update(oracle.f64(bias), counts.numpy(), 0.001)
    # float32 add of +-u: within one float32 rounding of the float64 update
    assert np.max(np.abs(oracle.f64(b) - want)) <= 1e-7
    step = np.sign(oracle.f64(b) - oracle.f64(bias))
    assert np.array_equal(step, np.sign(want - oracle.f64(bias)))

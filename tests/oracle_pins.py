"""Pins that tie the oracle to what the pages and the mathematics fix.

Each pin takes the oracle module and raises AssertionError when the oracle
disagrees with a printed worked example, a closed form, an invariant, a brute
force on tiny inputs or a textbook special case.  test_oracle_pins runs them on
the oracle; test_oracle_sensitivity plants one plausible mistake at a time in
the oracle and checks that some pin fails.
"""
from __future__ import annotations

import itertools
import json
import math
import os
import types

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name: str) -> dict:
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


def _inputs(**kw):
    return types.SimpleNamespace(**kw)


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- gates

def pin_gate_worked_example(O):
    """Top-2 scores 0.80 and 0.49 normalise to 0.62 and 0.38 (sigmoid router, E=8)."""
    g = golden("gate_worked_example.json")
    s_top = np.array(g["top_scores"])
    others = np.array([0.30, 0.22, 0.15, 0.10, 0.05, 0.02])
    s = np.concatenate([others[:3], [s_top[1]], others[3:], [s_top[0]]])  # shuffled positions
    H = np.log(s / (1 - s))[None, :]                                      # sigmoid^-1
    r = O.route(H, g["k"], O.SIGMOID, True)
    assert list(r["idx"][0]) == [len(s) - 1, 3], r["idx"]
    assert np.allclose(np.round(r["gate"][0], 2), g["gates_2dp"]), r["gate"]
    exact = s_top / s_top.sum()
    assert np.allclose(r["gate"][0], exact, atol=1e-6), (r["gate"], exact)


def pin_topk_then_softmax_identity(O):
    """Softmax then renormalise over the selected == softmax over the selected logits only."""
    rng = _rng(1)
    H = rng.normal(size=(64, 16)) * 2
    k = 4
    r = O.route(H, k, O.SOFTMAX, True)
    sel = np.take_along_axis(r["logits"], r["idx"].astype(np.int64), 1)
    direct = np.exp(sel - sel.max(1, keepdims=True))
    direct /= direct.sum(1, keepdims=True)
    assert np.allclose(r["gate"], direct, rtol=1e-12, atol=1e-14)


def pin_gate_sums(O):
    """Renormalised gates sum to 1; unrenormalised softmax gates sum below 1 and equal the scores."""
    rng = _rng(2)
    H = rng.normal(size=(50, 12))
    for fn in (O.SOFTMAX, O.SIGMOID):
        r = O.route(H, 3, fn, True)
        assert np.allclose(r["gate"].sum(1), 1.0, atol=1e-12)
    r = O.route(H, 3, O.SOFTMAX, False)
    assert np.all(r["gate"].sum(1) < 1.0)
    # with no renormalisation the gate is the softmax probability itself
    p = np.exp(r["logits"]) / np.exp(r["logits"]).sum(1, keepdims=True)
    assert np.allclose(r["gate"], np.take_along_axis(p, r["idx"].astype(np.int64), 1), atol=1e-12)


def pin_sigmoid_scores(O):
    """Sigmoid scores are independent per expert: s = 1/(1+e^-x); s(0) = 1/2; s(ln 3) = 3/4."""
    H = np.array([[0.0, math.log(3.0), -math.log(3.0)]])
    s = O.scores(H, O.SIGMOID)
    assert np.allclose(s, [[0.5, 0.75, 0.25]], atol=1e-15)
    s2 = O.scores(np.array([[0.0, math.log(3.0), 5.0]]), O.SIGMOID)
    assert np.allclose(s2[0, :2], s[0, :2], atol=1e-15)


def pin_softmax_bf16_example(O):
    """Ten logits of 128 and one of 128.5: 0.142; after bf16 rounding 128.5 -> 128: 1/11 = 0.091."""
    import torch
    g = golden("softmax_bf16_example.json")
    H = np.array([g["logits"]], dtype=np.float64)
    s = O.scores(H, O.SOFTMAX)
    assert round(float(s[0, -1]), g["printed_decimals"]) == g["softmax_of_last"]
    Hb = torch.tensor(H, dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    sb = O.scores(Hb, O.SOFTMAX)
    assert round(float(sb[0, -1]), g["printed_decimals"]) == g["softmax_of_last_after_bf16"]
    assert abs(sb[0, -1] - 1 / 11) < 1e-15


# ---------------------------------------------------------------- router

def pin_router_logits_small(O):
    """H = U W_r on hand-computed integers, plus bias; the noisy term is eps*ln2 when U W_noise = 0."""
    U = np.array([[1.0, 2.0], [3.0, 4.0]])
    W = np.array([[1.0, 0.0, 2.0], [0.0, 1.0, 3.0]])
    H = O.router_logits(U, W)
    assert np.array_equal(H, [[1, 2, 8], [3, 4, 18]])
    b = np.array([0.5, -1.0, 0.0])
    assert np.array_equal(O.router_logits(U, W, b), [[1.5, 1, 8], [3.5, 3, 18]])
    eps = np.array([[1.0, -2.0, 0.5], [0.0, 1.0, 1.0]])
    Hn = O.router_logits(U, W, None, np.zeros((2, 3)), eps)
    assert np.allclose(Hn - H, eps * math.log(2.0), atol=1e-15)


def pin_softplus(O):
    """Softplus closed forms: ln 2 at 0, x + ln(1+e^-x) for x > 0, e^x-ish far left, no overflow."""
    x = np.array([0.0, 1.0, -1.0, 50.0, -50.0, 800.0])
    sp = O.softplus(x)
    assert abs(sp[0] - math.log(2)) < 1e-15
    assert abs(sp[1] - math.log(1 + math.e)) < 1e-14
    assert abs(sp[2] - math.log(1 + 1 / math.e)) < 1e-15
    assert abs(sp[3] - 50.0) < 1e-14 and abs(sp[4] - math.exp(-50)) < 1e-30
    assert sp[5] == 800.0


def pin_topk_bruteforce(O):
    """Top-k against sorting every row by (-value, expert id), on small integers with many ties."""
    rng = _rng(3)
    for E, k in ((5, 2), (8, 3), (16, 16), (1, 1), (12, 1)):
        H = rng.integers(-3, 4, size=(40, E)).astype(np.float64)
        idx = O.topk_select(H, k)
        for t in range(H.shape[0]):
            ref = sorted(range(E), key=lambda e: (-H[t, e], e))[:k]
            assert list(idx[t]) == ref, (E, k, t, H[t], idx[t], ref)


def pin_route_selects_on_float32_logits(O):
    """Routing rounds the logits to float32 first (the library's logits are float32): 1 + 2^-30
    rounds to 1, so it ties with a logit of 1 and the lower expert id wins; the rounded logits
    are returned."""
    H = np.array([[1.0, 1.0 + 2.0 ** -30, 0.5], [0.25, 1.0 + 2.0 ** -22, 1.0]])
    r = O.route(H, 1, O.SOFTMAX, False)
    assert r["idx"].tolist() == [[0], [1]]
    assert r["logits"][0, 1] == 1.0 and r["logits"][1, 1] == 1.0 + 2.0 ** -22


def pin_topk_ties(O):
    """Exact ties go to the lower expert id, for membership and for rank order."""
    H = np.array([[1.0, 3.0, 3.0, 2.0, 3.0],
                  [0.0, 0.0, 0.0, 0.0, 0.0],
                  [-1.0, 5.0, -1.0, -1.0, 5.0]])
    idx = O.topk_select(H, 3)
    assert idx.tolist() == [[1, 2, 4], [0, 1, 2], [1, 4, 0]]


# ---------------------------------------------------------------- capacity / dispatch

def pin_capacity_examples(O):
    g = golden("capacity_examples.json")
    s, l = g["small"], g["large"]
    assert O.capacity(s["T"], s["E"], s["k"], s["CF"]) == s["C"]
    assert O.capacity(l["T"], l["E"], l["k"], l["CF"]) == l["C"]
    assert l["T"] * l["k"] // l["E"] == l["balanced_load"]
    # ceil of a non-integer load: 10 tokens, 4 experts, top-1, CF 1 -> 2.5 -> 3; CF 1.1 -> 2.75 -> 3
    assert O.capacity(10, 4, 1, 1.0) == 3
    assert O.capacity(10, 4, 1, 1.1) == 3
    assert O.capacity(700, 8, 2, 1.25) == 219      # 218.75
    assert O.capacity(16, 4, 2, 0.0) == 16         # no limit: C = T
    assert O.capacity(16, 4, 2, 1.0, override=5) == 5


def pin_dispatch_small_example(O):
    """T=12, E=4, k=1, CF=1: C=3; the expert with 5 tokens drops its last 2 (token order)."""
    g = golden("capacity_examples.json")["small"]
    # expert 0 ("expert 1" of the example) gets 5 tokens, experts 1, 2 get 3, expert 3 gets 1
    idx = np.array([[0], [1], [0], [2], [0], [1], [2], [0], [1], [3], [2], [0]])
    C = O.capacity(g["T"], g["E"], g["k"], g["CF"])
    d = O.dispatch(idx, g["E"], C)
    assert d["counts_routed"].tolist() == [5, 3, 3, 1]
    assert d["counts_routed"][0] - d["counts_kept"][0] == g["hot_expert_dropped"]
    assert C - d["counts_kept"][3] == g["cold_expert_idle_slots"]
    dropped = [t for t in range(12) if d["slot_row"][t] < 0]
    assert dropped == [7, 11]                        # the last two of expert 0, in token order
    assert d["n_dropped"] == 2
    assert d["offsets"].tolist() == [0, 3, 6, 9, 10]
    assert d["row_token"].tolist() == [0, 2, 4, 1, 5, 8, 3, 6, 10, 9]


def pin_dispatch_large_example(O):
    """T=4096, E=64, k=8, CF=1.25: C=640; 900 assignments drop 260, 300 leave 340 slots idle."""
    g = golden("capacity_examples.json")["large"]
    T, E, k = g["T"], g["E"], g["k"]
    rng = _rng(4)
    idx = np.zeros((T, k), dtype=np.int64)
    for t in range(T):
        fixed = []
        if t < g["hot_expert_assignments"]:
            fixed.append(0)
        if t < g["cold_expert_assignments"]:
            fixed.append(1)
        rest = rng.choice(np.arange(2, E), size=k - len(fixed), replace=False)
        row = np.concatenate([fixed, rest])
        rng.shuffle(row)
        idx[t] = row
    C = O.capacity(T, E, k, g["CF"])
    d = O.dispatch(idx, E, C)
    assert d["counts_routed"][0] == 900 and d["counts_routed"][1] == 300
    assert d["counts_routed"][0] - d["counts_kept"][0] == g["hot_expert_dropped"]
    assert C - d["counts_kept"][1] == g["cold_expert_idle_slots"]


def _dispatch_loop(idx, E, C, priority):
    """Pure-Python slot filling, one pair at a time (brute force for tiny inputs)."""
    T, k = idx.shape
    pairs = ([(t, j) for j in range(k) for t in range(T)] if priority == 0
             else [(t, j) for t in range(T) for j in range(k)])
    fill = [0] * E
    slot = {}
    for (t, j) in pairs:
        e = int(idx[t, j])
        slot[(t, j)] = fill[e]
        fill[e] += 1
    kept = [min(c, C) for c in fill]
    off = [0]
    for c in kept:
        off.append(off[-1] + c)
    slot_row = [-1] * (T * k)
    row_token = [None] * off[-1]
    for (t, j), s in slot.items():
        if s < C:
            r = off[int(idx[t, j])] + s
            slot_row[t * k + j] = r
            row_token[r] = t
    return fill, kept, off, slot_row, row_token


def pin_dispatch_bruteforce(O):
    rng = _rng(5)
    for (T, E, k, C) in ((9, 3, 2, 2), (20, 5, 3, 4), (16, 4, 4, 16), (1, 1, 1, 1), (30, 6, 1, 3), (7, 8, 8, 1)):
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
        for pr in (0, 1):
            d = O.dispatch(idx, E, C, pr)
            fill, kept, off, slot_row, row_token = _dispatch_loop(idx, E, C, pr)
            assert d["counts_routed"].tolist() == fill
            assert d["counts_kept"].tolist() == kept
            assert d["offsets"].tolist() == off
            assert d["slot_row"].tolist() == slot_row, (T, E, k, C, pr)
            assert d["row_token"].tolist() == row_token


def pin_dispatch_invariants(O):
    """Counts add up, slot_row is a bijection onto [0, A), rows point back at their token,
    and under choice-major priority the kept pairs of every expert precede its dropped ones."""
    rng = _rng(6)
    T, E, k = 300, 10, 3
    p = np.arange(1, E + 1, dtype=float) ** -1.2
    p /= p.sum()
    idx = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)])
    C = O.capacity(T, E, k, 1.0)
    d = O.dispatch(idx, E, C, 0)
    A = int(d["offsets"][-1])
    assert d["counts_kept"].sum() == T * k - d["n_dropped"] == A
    assert d["counts_routed"].sum() == T * k
    kept = d["slot_row"][d["slot_row"] >= 0]
    assert sorted(kept.tolist()) == list(range(A))
    for pair in range(T * k):
        r = d["slot_row"][pair]
        if r >= 0:
            t, j = divmod(pair, k)
            assert d["row_token"][r] == t
            e = idx[t, j]
            assert d["offsets"][e] <= r < d["offsets"][e + 1]
    assert np.all(np.diff(d["offsets"]) >= 0)
    for e in range(E):
        ks = [(j, t) for t in range(T) for j in range(k) if idx[t, j] == e and d["slot_row"][t * k + j] >= 0]
        ds = [(j, t) for t in range(T) for j in range(k) if idx[t, j] == e and d["slot_row"][t * k + j] < 0]
        if ks and ds:
            assert max(ks) < min(ds)
    assert d["n_dropped"] > 0      # the skewed draw must overflow somebody for this to test anything


# ---------------------------------------------------------------- experts / combine

def _small_layer(rng, T, h, E, k, d_e, std=0.3):
    return _inputs(U=rng.normal(size=(T, h)), W_r=rng.normal(size=(h, E)) * std, b_r=None,
                   W_noise=None, eps=None,
                   W_gate=rng.normal(size=(E, d_e, h)) * std, W_up=rng.normal(size=(E, d_e, h)) * std,
                   W_down=rng.normal(size=(E, h, d_e)) * std)


def pin_textbook_dense_swiglu(O):
    """E=1, k=1 reduces to a dense SwiGLU FFN plus the residual (torch's silu and matmul)."""
    import torch
    rng = _rng(7)
    T, h, d_e = 13, 6, 10
    inp = _small_layer(rng, T, h, 1, 1, d_e)
    res = O.layer_forward(inp, T=T, h=h, E=1, k=1, d_e=d_e, score_fn=O.SOFTMAX, renorm=True,
                          capacity_factor=0.0)
    U = torch.tensor(inp.U)
    Wg, Wu, Wd = (torch.tensor(x[0]) for x in (inp.W_gate, inp.W_up, inp.W_down))
    ref = U + torch.nn.functional.linear(torch.nn.functional.silu(torch.nn.functional.linear(U, Wg))
                                         * torch.nn.functional.linear(U, Wu), Wd)
    assert np.allclose(res["out"], ref.numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(res["gate"], 1.0)


def pin_dense_bruteforce(O):
    """Unbounded capacity: every expert on every token, masked by the gates, equals the routed path."""
    import torch
    rng = _rng(8)
    for (T, h, E, k, d_e, fn, rn) in ((17, 8, 5, 2, 12, 0, True), (11, 6, 4, 3, 7, 1, True),
                                      (9, 5, 6, 1, 4, 0, False)):
        inp = _small_layer(rng, T, h, E, k, d_e)
        res = O.layer_forward(inp, T=T, h=h, E=E, k=k, d_e=d_e, score_fn=fn, renorm=rn,
                              capacity_factor=0.0)
        assert res["n_dropped"] == 0
        G = np.zeros((T, E))
        for t in range(T):
            for j in range(k):
                G[t, res["idx"][t, j]] = res["gate"][t, j]
        U = torch.tensor(inp.U)
        out = U.clone()
        for e in range(E):
            Wg, Wu, Wd = (torch.tensor(x[e]) for x in (inp.W_gate, inp.W_up, inp.W_down))
            y = torch.nn.functional.linear(torch.nn.functional.silu(U @ Wg.T) * (U @ Wu.T), Wd)
            out += torch.tensor(G[:, e])[:, None] * y
        assert np.allclose(res["out"], out.numpy(), rtol=1e-12, atol=1e-12)


def pin_zero_experts_and_drops(O):
    """Zero down-projection gives out == U exactly; a token whose pairs all drop keeps U exactly."""
    rng = _rng(9)
    T, h, E, k, d_e = 40, 8, 4, 2, 6
    inp = _small_layer(rng, T, h, E, k, d_e)
    inp.W_down = np.zeros_like(inp.W_down)
    res = O.layer_forward(inp, T=T, h=h, E=E, k=k, d_e=d_e, score_fn=0, renorm=True, capacity_factor=1.0)
    assert np.array_equal(res["out"], inp.U)
    inp = _small_layer(rng, T, h, E, k, d_e)
    res = O.layer_forward(inp, T=T, h=h, E=E, k=k, d_e=d_e, score_fn=0, renorm=True,
                          capacity_factor=0.0, capacity_override=2)
    sr = res["slot_row"].reshape(T, k)
    all_dropped = np.all(sr < 0, axis=1)
    assert all_dropped.sum() > 0
    assert np.array_equal(res["out"][all_dropped], inp.U[all_dropped])
    assert not np.allclose(res["out"][~all_dropped], inp.U[~all_dropped])


def pin_sampled_matches_full(O):
    rng = _rng(10)
    T, h, E, k, d_e = 50, 8, 6, 2, 12
    inp = _small_layer(rng, T, h, E, k, d_e)
    res = O.layer_forward(inp, T=T, h=h, E=E, k=k, d_e=d_e, score_fn=0, renorm=True, capacity_factor=1.0)
    toks = [0, 7, 21, 49]
    smp = O.sampled_outputs(inp, toks, res["idx"], res["gate"], res["slot_row"], k)
    assert np.allclose(smp["out"], res["out"][toks], rtol=1e-12, atol=1e-12)
    for row, y in smp["Y"].items():
        assert np.allclose(y, res["Y"][row], rtol=1e-12, atol=1e-12)


def pin_sampled_shared_and_fp8_match_full(O):
    """sampled_outputs with shared experts, with the FP8 up-projection, and with both, equals
    layer_forward's out and Y rows, row by row, on a small case with drops (dropped tokens
    sampled too)."""
    rng = _rng(12)
    T, h, E, k, d_e, d_s = 60, 16, 6, 2, 12, 10
    inp = _small_layer(rng, T, h, E, k, d_e)
    shared = (rng.normal(size=(2, d_s, h)) * 0.3, rng.normal(size=(2, d_s, h)) * 0.3,
              rng.normal(size=(2, h, d_s)) * 0.3)
    for kw in (dict(shared=shared), dict(fp8=True), dict(shared=shared, fp8=True)):
        res = O.layer_forward(inp, T=T, h=h, E=E, k=k, d_e=d_e, score_fn=0, renorm=True, capacity_factor=0.8,
                              **kw)
        assert res["n_dropped"] > 0
        sr = np.asarray(res["slot_row"]).reshape(T, k)
        dropped = [int(t) for t in np.nonzero(np.any(sr < 0, axis=1))[0][:3]]
        toks = sorted(set([0, 9, 31, T - 1] + dropped))
        smp = O.sampled_outputs(inp, toks, res["idx"], res["gate"], res["slot_row"], k, **kw)
        assert np.allclose(smp["out"], res["out"][toks], rtol=1e-12, atol=1e-12), kw.keys()
        assert smp["Y"], kw.keys()
        for row, y in smp["Y"].items():
            assert np.allclose(y, res["Y"][row], rtol=1e-12, atol=1e-12), kw.keys()


# ---------------------------------------------------------------- statistics

def pin_aux_balance(O):
    """E * sum f P == 1 at perfect balance; == E when all load and all probability sit on one expert."""
    g = golden("aux_balance.json")
    for E, k in ((4, 1), (8, 2), (64, 6)):
        T = E * 10
        counts = np.full(E, T * k // E)
        s = np.full((T, E), 1.0 / E)
        st = O.load_stats(counts, s, T, k, O.SOFTMAX)
        assert abs(st["aux"] - g["value_at_balance"]) < 1e-12
        assert abs(st["maxvio"]) < 1e-12
    E, T = 8, 20
    counts = np.zeros(E)
    counts[3] = T
    s = np.zeros((T, E))
    s[:, 3] = 1.0
    assert abs(O.load_stats(counts, s, T, 1, O.SOFTMAX)["aux"] - E) < 1e-12


def pin_stats_sums(O):
    """sum f = 1; sum P = 1 for softmax and for normalised sigmoid scores; MaxVio of (2,1,1,0) is 1."""
    rng = _rng(11)
    T, E, k = 30, 7, 2
    H = rng.normal(size=(T, E))
    for fn in (O.SOFTMAX, O.SIGMOID):
        r = O.route(H, k, fn, True)
        d = O.dispatch(r["idx"], E, T)
        st = O.load_stats(d["counts_routed"], r["s"], T, k, fn)
        assert abs(st["f"].sum() - 1) < 1e-12
        assert abs(st["P"].sum() - 1) < 1e-12
    st = O.load_stats(np.array([2, 1, 1, 0]), np.full((4, 4), 0.25), 4, 1, O.SOFTMAX)
    assert abs(st["maxvio"] - 1.0) < 1e-15


def pin_sigmoid_P_normalised(O):
    """Sigmoid P_i averages s_i / sum_j s_j: two tokens, sigmoid scores (1/2, 1/2) and (3/4, 1/4)."""
    H = np.array([[0.0, 0.0], [math.log(3.0), -math.log(3.0)]])
    s = O.scores(H, O.SIGMOID)
    st = O.load_stats(np.array([1, 1]), s, 2, 1, O.SIGMOID)
    assert np.allclose(st["P"], [(0.5 + 0.75) / 2, (0.5 + 0.25) / 2], atol=1e-15)


# ---------------------------------------------------------------- router z-loss

def pin_z_loss_closed_forms(O):
    """Constant logits c over E experts: LSE = c + ln E, so L_z = (c + ln E)^2; the z-loss section's
    rounding example row (ten logits of 128, one of 128.5) has LSE = 128 + ln(10 + e^0.5); a mean
    over tokens, not a sum."""
    for c, E in ((0.0, 8), (-3.0, 64), (2.5, 1)):
        H = np.full((5, E), c)
        assert abs(O.router_z_loss(H) - (c + math.log(E)) ** 2) < 1e-10
    g = golden("softmax_bf16_example.json")
    row = np.array([g["logits"]], dtype=np.float64)
    lse = 128.0 + math.log(10.0 + math.exp(0.5))
    assert abs(O.router_z_loss(row) - lse ** 2) < 1e-8
    two = np.vstack([row, np.zeros((1, 11))])
    assert abs(O.router_z_loss(two) - (lse ** 2 + math.log(11.0) ** 2) / 2) < 1e-8
    assert O.router_z_loss(np.zeros((0, 4))) == 0.0


def pin_z_loss_library_logsumexp(O):
    """Against scipy's logsumexp on random logits of several scales (library routine)."""
    from scipy.special import logsumexp
    rng = _rng(23)
    for scale in (0.1, 3.0, 40.0):
        H = rng.normal(size=(50, 13)) * scale
        want = float(np.mean(logsumexp(H, axis=1) ** 2))
        assert abs(O.router_z_loss(H) - want) <= 1e-12 * max(1.0, want)


def pin_z_loss_gradient_formula(O):
    """The section's gradient, dL_z/dH_{t,k} = (2/T) LSE(H_t) softmax(H_t)_k, against central
    differences of the oracle's L_z."""
    rng = _rng(29)
    H = rng.normal(size=(4, 6))
    T = H.shape[0]
    eps = 1e-6
    lse = np.log(np.exp(H).sum(axis=1))
    sm = np.exp(H) / np.exp(H).sum(axis=1, keepdims=True)
    for t, j in ((0, 0), (2, 5), (3, 1)):
        Hp, Hm = H.copy(), H.copy()
        Hp[t, j] += eps
        Hm[t, j] -= eps
        fd = (O.router_z_loss(Hp) - O.router_z_loss(Hm)) / (2 * eps)
        assert abs(fd - 2.0 / T * lse[t] * sm[t, j]) < 1e-7


# ---------------------------------------------------------------- loss-free balancing bias

def pin_loss_free_selection_example(O):
    """Selection on s + b, gates from s: scores (.5, .4, .3) with b = (-.2, 0, .15) give keys
    (.3, .4, .45); top-1 is expert 2 with gate s_2 = .3 (1 after renormalising); top-2 is (2, 1)
    with renormalised gates (3/7, 4/7)."""
    # softmax(log(s / sum s)) = s / sum s; the logits pass through float32, hence the 1e-7
    s = np.array([[0.5, 0.4, 0.3]])
    H = np.log(s / s.sum())
    b = np.array([-0.2, 0.0, 0.15]) / s.sum()
    r1 = O.route(H, 1, O.SOFTMAX, False, sel_bias=b)
    assert r1["idx"].tolist() == [[2]]
    assert abs(r1["gate"][0, 0] - 0.3 / s.sum()) < 1e-7
    assert abs(O.route(H, 1, O.SOFTMAX, True, sel_bias=b)["gate"][0, 0] - 1.0) < 1e-12
    r2 = O.route(H, 2, O.SOFTMAX, True, sel_bias=b)
    assert r2["idx"].tolist() == [[2, 1]]
    assert np.allclose(r2["gate"], [[3 / 7, 4 / 7]], atol=1e-7)
    assert O.route(H, 1, O.SOFTMAX, False)["idx"].tolist() == [[0]]  # without the bias: expert 0


def pin_loss_free_zero_bias_and_gates(O):
    """A zero bias selects exactly what the logits select; any bias leaves the gate of a selected
    expert equal to its (renormalised) score."""
    rng = _rng(31)
    H = rng.normal(size=(40, 12))
    for fn in (O.SOFTMAX, O.SIGMOID):
        plain = O.route(H, 3, fn, True)
        zero = O.route(H, 3, fn, True, sel_bias=np.zeros(12))
        assert np.array_equal(plain["idx"], zero["idx"])
        b = rng.normal(size=12) * 0.3
        biased = O.route(H, 3, fn, False, sel_bias=b)
        sel = np.take_along_axis(biased["s"], biased["idx"].astype(np.int64), axis=1)
        assert np.allclose(biased["gate"], sel, atol=0)
        key = biased["s"] + b
        brute = np.argsort(-key, axis=1, kind="stable")[:, :3]
        assert np.array_equal(biased["idx"], brute)


def pin_group_limited_example(O):
    """Group-limited routing worked by hand (sigmoid, 8 experts in 4 groups of 2, 2 groups kept,
    k = 4 so each group is scored on its 2 best affinities): the group scores are
    s(3)+s(-2) = 1.072, s(2.9)+s(2.8) = 1.891, 2 s(0) = 1.0 and s(1)+s(2.95) = 1.681, so groups
    1 and 3 are kept and the top-4 is (7, 2, 3, 6), leaving out expert 0, the highest logit,
    which plain top-4 ranks first."""
    H = np.array([[3.0, -2.0, 2.9, 2.8, 0.0, 0.0, 1.0, 2.95]])
    r = O.route(H, 4, O.SIGMOID, True, n_group=4, topk_group=2)
    assert r["idx"].tolist() == [[7, 2, 3, 6]]
    assert O.route(H, 4, O.SIGMOID, True)["idx"].tolist() == [[0, 7, 2, 3]]
    sel = np.array([1.0 / (1.0 + math.exp(-v)) for v in (2.95, 2.9, 2.8, 1.0)])
    assert np.allclose(r["gate"][0], sel / sel.sum(), rtol=0, atol=1e-7)


def pin_group_limited_special_cases(O):
    """Keeping every group, or a single group, or groups of one expert with topk_group = k, all
    select exactly the plain top-k."""
    rng = _rng(33)
    H = rng.normal(size=(60, 16)) * 1.5
    for fn in (O.SOFTMAX, O.SIGMOID):
        plain = O.route(H, 4, fn, True)["idx"]
        for n_group, topk_group in ((4, 4), (1, 1), (16, 4), (2, 2)):
            r = O.route(H, 4, fn, True, n_group=n_group, topk_group=topk_group)
            assert np.array_equal(r["idx"], plain), (fn, n_group, topk_group)


def _group_limited_bruteforce(key, aff, n_group, topk_group, k):
    """Per token: every topk_group-subset of groups scored by the sum of its groups' r best
    affinities, the best subset kept; then every k-subset of the kept experts, the one with
    the largest key sum selected, listed by decreasing key.  (Continuous random values: no ties.)"""
    T, E = key.shape
    S, r = E // n_group, k // topk_group
    out = []
    for t in range(T):
        gscore = []
        for q in range(n_group):
            vals = sorted((aff[t, q * S + i] for i in range(S)), reverse=True)
            gscore.append(sum(vals[:r]))
        best = max(itertools.combinations(range(n_group), topk_group), key=lambda c: sum(gscore[q] for q in c))
        experts = [e for e in range(E) if e // S in best]
        sel = max(itertools.combinations(experts, k), key=lambda c: sum(key[t, e] for e in c))
        out.append(sorted(sel, key=lambda e: -key[t, e]))
    return np.array(out, dtype=np.int64)


def pin_group_limited_bruteforce(O):
    """Group-limited top-k against the subset brute force, with and without a selection bias."""
    rng = _rng(34)
    for E, n_group, topk_group, k, fn, bias in ((12, 4, 2, 4, O.SIGMOID, False), (8, 4, 2, 2, O.SOFTMAX, False),
                                                (12, 3, 1, 2, O.SOFTMAX, True), (16, 4, 3, 3, O.SIGMOID, True),
                                                (16, 8, 2, 4, O.SIGMOID, True)):
        H = rng.normal(size=(40, E)) * 2.0
        b = rng.normal(size=E) * 0.1 if bias else None
        H32 = np.asarray(H, dtype=np.float32).astype(np.float64)
        s = O.scores(H32, fn)
        key = H32 if b is None else s + b
        want = _group_limited_bruteforce(key, s if b is None else key, n_group, topk_group, k)
        r = O.route(H, k, fn, True, b, n_group, topk_group)
        assert np.array_equal(r["idx"], want), (E, n_group, topk_group, k)
        groups = np.asarray(r["idx"]) // (E // n_group)
        assert all(len(set(g)) <= topk_group for g in groups.tolist())


def _e4m3_probe_values():
    """Every E4M3 grid value, every midpoint between neighbours (ties), points just either side
    of each midpoint, and log-uniform random values, with both signs."""
    grid = [0.0] + [k * 2.0 ** -9 for k in range(1, 8)]
    for e in range(-6, 9):
        grid += [(1 + m / 8.0) * 2.0 ** e for m in range(8)]
    grid = np.array(sorted(v for v in grid if v <= 448.0))
    mids = (grid[1:] + grid[:-1]) / 2
    rnd = np.exp(_rng(41).uniform(np.log(2.0 ** -12), np.log(448.0), size=4000))
    v = np.concatenate([grid, mids, mids * (1 + 2.0 ** -20), mids * (1 - 2.0 ** -20), rnd])
    return grid, np.concatenate([v, -v])


def pin_e4m3_rounding_against_torch(O):
    """E4M3 rounding and bit codes equal torch's float8_e4m3fn cast (round to nearest even) on
    every grid value, every tie, both sides of every tie and random values."""
    import torch
    _, v = _e4m3_probe_values()
    t = torch.tensor(v, dtype=torch.float64).to(torch.float8_e4m3fn)
    assert np.array_equal(O.e4m3_round(v), t.to(torch.float64).numpy())
    assert np.array_equal(O.e4m3_bits(O.e4m3_round(v)), t.view(torch.uint8).numpy())


def pin_e4m3_grid(O):
    """The format's facts: 127 non-negative finite values, largest 448, smallest normal 2^-6,
    smallest subnormal 2^-9; half the smallest subnormal rounds to zero (tie to even)."""
    grid, _ = _e4m3_probe_values()
    dense = np.concatenate([np.linspace(0, 448, 200001), grid])
    vals = np.unique(O.e4m3_round(dense))
    assert len(vals) == 127 and vals.max() == 448.0 and vals[1] == 2.0 ** -9
    assert 2.0 ** -6 in vals and O.e4m3_round(2.0 ** -10) == 0.0 and O.e4m3_round(1.5 * 2.0 ** -10) == 2.0 ** -9
    assert O.e4m3_round(1000.0) == 448.0


def pin_pow2_scale_exponents(O):
    """The scale 2^s is the smallest power of two with amax <= 448 * 2^s: worked values and a
    brute-force minimality check."""
    got = O.pow2_scale_exponents(np.array([448.0, 449.0, 1.0, 0.0, 896.0, 897.0, 3.0, 0.75]))
    assert got.tolist() == [0, 1, -8, -127, 1, 2, -7, -9]
    amax = np.exp(_rng(42).uniform(-30, 30, size=2000))
    s = O.pow2_scale_exponents(amax)
    assert np.all(amax <= 448.0 * 2.0 ** s.astype(float))
    assert np.all((amax > 448.0 * 2.0 ** (s - 1.0)) | (s == -127))


def pin_fp8_rows_on_grid_and_bounded(O):
    """Quantised rows: codes are E4M3 values within +-448, the row maximum uses the top binade,
    and each dequantised entry is within half an E4M3 step (2^-4 relative, or 2^-10 * 2^s in the
    subnormal range) of the input; fp8_weights applies exactly that to every expert row."""
    A = _rng(43).normal(size=(30, 200)) * np.exp(_rng(44).uniform(-5, 5, size=(30, 1)))
    codes, s = O.quantize_rows_fp8(A)
    assert np.array_equal(O.e4m3_round(codes), codes) and np.abs(codes).max() <= 448.0
    assert np.all(np.abs(codes).max(axis=1) >= 224.0)
    deq = O.dequantize_rows_fp8(codes, s)
    bound = np.maximum(np.abs(A) * 2.0 ** -4, 2.0 ** -10 * 2.0 ** s[:, None].astype(float))
    assert np.all(np.abs(deq - A) <= bound)
    W = A.reshape(3, 10, 200)
    assert np.array_equal(O.fp8_weights(W), deq.reshape(3, 10, 200))


def pin_fp8_layer_lossless_on_grid(O):
    """When every token row and every gate/up weight row is exactly representable after its
    power-of-two scaling (entries in {0, +-1, +-2, +-3} with a 3 in each row; weights in
    {+-1/4, +-1/2, +-3/4} with a 3/4 in each row), the FP8 layer equals the unquantised one."""
    rng = _rng(45)
    T, h, E, k, d_e = 40, 16, 4, 2, 12
    U = rng.integers(-3, 4, size=(T, h)).astype(float)
    U[:, 0] = 3.0
    def wq(shape):
        w = rng.choice([-0.75, -0.5, -0.25, 0.25, 0.5, 0.75], size=shape)
        w[..., 0] = 0.75
        return w
    inp = _inputs(U=U, W_r=rng.normal(size=(h, E)) * 0.3, b_r=None, W_noise=None, eps=None,
                  W_gate=wq((E, d_e, h)), W_up=wq((E, d_e, h)), W_down=rng.normal(size=(E, h, d_e)) * 0.1)
    kw = dict(T=T, h=h, E=E, k=k, d_e=d_e, score_fn=O.SOFTMAX, renorm=True, capacity_factor=1.0)
    a, b = O.layer_forward(inp, **kw), O.layer_forward(inp, fp8=True, **kw)
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["act"], b["act"])
    assert np.array_equal(b["U_s"], np.full(T, -7))
    assert np.array_equal(O.dequantize_rows_fp8(b["U_codes"], b["U_s"]), U)


def pin_fp8_layer_is_the_composition_of_its_pinned_parts(O):
    """The FP8 layer on random (off-grid) inputs equals the unquantised path applied to the
    dequantised token rows (quantize_rows_fp8 / dequantize_rows_fp8) and to fp8_weights of W_gate
    and W_up, both pinned above against torch's E4M3 cast; and it differs from the unquantised layer."""
    rng = _rng(46)
    T, h, E, k, d_e = 40, 16, 4, 2, 12
    inp = _small_layer(rng, T, h, E, k, d_e)
    kw = dict(T=T, h=h, E=E, k=k, d_e=d_e, score_fn=O.SOFTMAX, renorm=True, capacity_factor=1.0)
    q = O.layer_forward(inp, fp8=True, **kw)
    X = O.dequantize_rows_fp8(*O.quantize_rows_fp8(inp.U))[q["row_token"]]
    Y, act = O.expert_ffn(X, q["offsets"], O.fp8_weights(inp.W_gate), O.fp8_weights(inp.W_up), inp.W_down, d_e)
    assert np.array_equal(q["act"], act) and np.array_equal(q["Y"], Y)
    assert np.array_equal(q["out"], O.combine(inp.U, Y, q["slot_row"], q["gate"], k))
    assert not np.allclose(q["act"], O.layer_forward(inp, **kw)["act"], rtol=1e-3, atol=0)


def pin_balance_bias_update(O):
    """e_i = mean(c) - c_i; an overloaded expert's bias drops by u, an underloaded one rises by u,
    one exactly at the mean keeps its bias."""
    b = np.array([0.1, -0.2, 0.0, 0.3])
    nb = O.balance_bias_update(b, [10, 5, 0, 5], 0.01)
    assert np.allclose(nb, [0.09, -0.2, 0.01, 0.3], atol=1e-15)


def pin_balance_bias_feedback(O):
    """The section's illustration: 6 experts, 2400 random tokens a step, top-1, u = 0.01.  Experts
    of unequal popularity start far from balance; the sign updates pull every load toward the
    mean, so MaxVio falls by a large factor."""
    rng = _rng(37)
    E, T = 6, 2400
    pop = np.linspace(-0.6, 0.6, E)
    b = np.zeros(E)

    def step(b):
        s = O.scores(rng.normal(size=(T, E)) * 0.3 + pop, O.SIGMOID)
        idx = O.topk_select(s + b, 1)
        return np.bincount(idx[:, 0], minlength=E)

    c0 = step(b)
    vio0 = (c0.max() - c0.mean()) / c0.mean()
    for _ in range(300):
        b = O.balance_bias_update(b, step(b), 0.01)
    vio = np.mean([(c.max() - c.mean()) / c.mean() for c in (step(b) for _ in range(20))])
    assert vio0 > 1.0 and vio < vio0 / 5


# ---------------------------------------------------------------- shared experts

def pin_shared_experts(O):
    """h' = u + sum_s FFN_s(u) + sum_i g_i FFN_i(u): zero shared weights change nothing; one
    routed expert (k = 1, gate 1) identical to one shared expert doubles the FFN term; the shared
    term equals torch's dense SwiGLU on every token."""
    import torch
    rng = _rng(41)
    T, h, d = 9, 6, 5
    U = rng.normal(size=(T, h))
    Wg, Wu, Wd = rng.normal(size=(1, d, h)), rng.normal(size=(1, d, h)), rng.normal(size=(h, d))[None]
    inp = _inputs(U=U, W_r=rng.normal(size=(h, 1)), b_r=None, W_noise=None, eps=None, W_gate=Wg, W_up=Wu,
                  W_down=Wd)
    kw = dict(T=T, h=h, E=1, k=1, d_e=d, score_fn=O.SOFTMAX, renorm=True, capacity_factor=0.0)
    base = O.layer_forward(inp, **kw)
    zero = O.layer_forward(inp, shared=(np.zeros_like(Wg), np.zeros_like(Wu), np.zeros_like(Wd)), **kw)
    assert np.allclose(zero["out"], base["out"], atol=0)
    same = O.layer_forward(inp, shared=(Wg, Wu, Wd), **kw)
    assert np.allclose(same["out"] - U, 2 * (base["out"] - U), rtol=1e-12, atol=1e-12)
    tU = torch.tensor(U)
    dense = (torch.nn.functional.silu(tU @ torch.tensor(Wg[0]).T) * (tU @ torch.tensor(Wu[0]).T)) @ torch.tensor(Wd[0]).T
    assert np.allclose(O.shared_ffn(U, Wg, Wu, Wd)[0], dense.numpy(), rtol=1e-12, atol=1e-12)
    two = O.shared_ffn(U, np.concatenate([Wg, Wg]), np.concatenate([Wu, Wu]), np.concatenate([Wd, -Wd]))
    assert np.allclose(two.sum(axis=0), 0, atol=1e-12)


# ---------------------------------------------------------------- router-side backward

def pin_aux_grad_worked_example(O):
    """The section's example: f = (.55, .25, .10, .10), s = (.4, .3, .2, .1): weighted mean load .325
    and logit gradients (x T) .090, -.0225, -.045, -.0225 for sum f P (aux_loss_grad carries E/T)."""
    g = golden("aux_grad_example.json")
    s = np.array(g["s"])
    f = np.array(g["f"])
    assert abs(float((f * s).sum()) - g["weighted_mean_load"]) < 1e-12
    H = np.log(s)[None, :]  # softmax(log s) = s, since s sums to 1
    E, T = 4, 1
    grad = O.aux_loss_grad(H, f, O.SOFTMAX) * T / E
    assert np.allclose(grad[0], g["grad_times_T"], atol=5e-8)  # H passes through no rounding here


def _fd(fun, X, i, j, eps=1e-6):
    Xp, Xm = X.copy(), X.copy()
    Xp[i, j] += eps
    Xm[i, j] -= eps
    return (fun(Xp) - fun(Xm)) / (2 * eps)


def pin_aux_grad_finite_differences(O):
    """aux_loss_grad against central differences of E * sum f P(H) with the load f held fixed, for
    softmax and for sigmoid (P from s' = s / sum s), including the sigmoid saturation factor."""
    rng = _rng(43)
    T, E = 5, 6
    H = rng.normal(size=(T, E)) * 1.5
    counts = np.array([7, 1, 0, 3, 2, 2])
    f = counts / counts.sum()
    for fn in (O.SOFTMAX, O.SIGMOID):
        def aux(Hx):
            return O.load_stats(counts, O.scores(Hx, fn), T, counts.sum() / T, fn)["aux"]
        G = O.aux_loss_grad(H, f, fn)
        for (i, j) in ((0, 0), (2, 3), (4, 5), (1, 2)):
            assert abs(_fd(aux, H, i, j) - G[i, j]) < 1e-7


def pin_gate_backward_finite_differences(O):
    """gate_backward against central differences of L(H) = sum_{t,j} w_{t,j} g_{t,j}(H) with the
    top-k set fixed, for softmax/sigmoid, with and without renormalisation."""
    rng = _rng(47)
    T, E, k = 4, 7, 3
    H = rng.normal(size=(T, E))
    idx = O.topk_select(H, k)
    w = rng.normal(size=(T, k))
    for fn in (O.SOFTMAX, O.SIGMOID):
        for renorm in (True, False):
            def L(Hx):
                return float((O.gates(O.scores(Hx, fn), idx, renorm) * w).sum())
            G = O.gate_backward(H, idx, w, fn, renorm)
            for (i, j) in ((0, int(idx[0, 0])), (1, int(idx[1, 2])), (3, 0), (2, 6), (2, int(idx[2, 1]))):
                assert abs(_fd(L, H, i, j) - G[i, j]) < 1e-7, (fn, renorm, i, j)


def pin_combine_and_z_backward(O):
    """combine_backward: d_gate = dO . Y[row] and dY = g dO (the section's delta^T FFN_i), checked
    by central differences of <dO, out>; a dropped pair gets zero.  z_loss_grad against differences
    of the oracle's L_z."""
    rng = _rng(53)
    T, h, k = 3, 4, 2
    U = rng.normal(size=(T, h))
    Y = rng.normal(size=(T * k, h))
    slot_row = np.array([0, 1, 2, -1, 4, 5])
    gate = rng.random((T, k))
    dO = rng.normal(size=(T, h))
    b = O.combine_backward(dO, Y, slot_row, gate, k)
    L_gate = lambda G: float((dO * O.combine(U, Y, slot_row, G, k)).sum())
    for (i, j) in ((0, 0), (1, 0), (2, 1)):
        assert abs(_fd(L_gate, gate, i, j) - b["d_gate"][i, j]) < 1e-7
    assert b["d_gate"][1, 1] == 0.0
    L_Y = lambda Yx: float((dO * O.combine(U, Yx, slot_row, gate, k)).sum())
    for (r, c) in ((0, 1), (2, 3), (5, 0), (3, 2)):
        assert abs(_fd(L_Y, Y, r, c) - b["dY"][r, c]) < 1e-7
    H = rng.normal(size=(4, 5))
    G = O.z_loss_grad(H)
    for (i, j) in ((0, 0), (3, 4), (2, 1)):
        assert abs(_fd(O.router_z_loss, H, i, j) - G[i, j]) < 1e-7


# ---------------------------------------------------------------- expert and dispatch backward

def pin_swiglu_backward_autograd(O):
    """swiglu_backward against torch autograd through torch's silu and matmul (float64), and
    SiLU'(0) = 1/2."""
    import torch
    rng = _rng(59)
    n, h, d = 5, 7, 6
    x, Wg, Wu, Wd, dy = (rng.normal(size=s) for s in ((n, h), (d, h), (d, h), (h, d), (n, h)))
    t = {k_: torch.tensor(v, requires_grad=True) for k_, v in dict(x=x, Wg=Wg, Wu=Wu, Wd=Wd).items()}
    y = (torch.nn.functional.silu(t["x"] @ t["Wg"].T) * (t["x"] @ t["Wu"].T)) @ t["Wd"].T
    (y * torch.tensor(dy)).sum().backward()
    b = O.swiglu_backward(x, Wg, Wu, Wd, dy)
    for mine, ref in (("dx", "x"), ("dW_gate", "Wg"), ("dW_up", "Wu"), ("dW_down", "Wd")):
        assert np.allclose(b[mine], t[ref].grad.numpy(), rtol=1e-10, atol=1e-12), mine
    z = O.swiglu_backward(np.zeros((1, 1)), np.ones((1, 1)), np.ones((1, 1)), np.ones((1, 1)), np.ones((1, 1)))
    assert z["dG"][0, 0] == 0.0  # Up = 0 at x = 0
    one = O.swiglu_backward(np.ones((1, 1)), np.zeros((1, 1)), np.ones((1, 1)), np.ones((1, 1)), np.ones((1, 1)))
    assert abs(one["dG"][0, 0] - 0.5) < 1e-15  # G = 0: SiLU'(0) = 1/2, Up = 1, d_act = 1


def pin_expert_and_dispatch_backward_segments(O):
    """The grouped backward equals the per-expert backward on each segment; an empty expert gets
    zero weight gradients; dispatch_backward adds each kept row's dX to its token once."""
    rng = _rng(61)
    E, h, d, T, k = 3, 5, 4, 6, 2
    idx = np.array([[0, 1], [1, 0], [0, 1], [1, 0], [0, 1], [1, 0]])
    disp = O.dispatch(idx, E, T)
    U = rng.normal(size=(T, h))
    X = O.permute(U, disp["row_token"])
    Wg, Wu, Wd = rng.normal(size=(E, d, h)), rng.normal(size=(E, d, h)), rng.normal(size=(E, h, d))
    dY = rng.normal(size=X.shape)
    g = O.expert_ffn_backward(X, disp["offsets"], Wg, Wu, Wd, dY, d)
    for e in range(E):
        lo, hi = disp["offsets"][e], disp["offsets"][e + 1]
        if hi > lo:
            b = O.swiglu_backward(X[lo:hi], Wg[e], Wu[e], Wd[e], dY[lo:hi])
            assert np.allclose(g["dW_gate"][e], b["dW_gate"]) and np.allclose(g["dX"][lo:hi], b["dx"])
        else:
            assert not g["dW_down"][e].any() and not g["dW_gate"][e].any()
    dO = rng.normal(size=(T, h))
    dU = O.dispatch_backward(dO, g["dX"], disp["slot_row"], k)
    want = dO.copy()
    for t in range(T):
        for j in range(k):
            want[t] += g["dX"][disp["slot_row"][t * k + j]]
    assert np.allclose(dU, want, atol=1e-12)


def _torch_layer_loss(t, fwd, dO, *, T, E, k, score_fn, renorm, w_aux, w_z, noisy):
    """The layer written with torch ops for autograd, routing decisions (idx, slots) fixed."""
    import torch
    H = t["U"] @ t["W_r"] + t["b_r"]
    if noisy:
        H = H + torch.tensor(fwd["eps"]) * torch.nn.functional.softplus(t["U"] @ t["W_noise"])
    s = torch.softmax(H, dim=1) if score_fn == 0 else torch.sigmoid(H)
    idx = torch.tensor(fwd["idx"], dtype=torch.int64)
    sel = torch.gather(s, 1, idx)
    g = sel / sel.sum(dim=1, keepdim=True) if renorm else sel
    out = t["U"].clone()
    sr = fwd["slot_row"].reshape(T, k)
    for tok in range(T):
        for j in range(k):
            if sr[tok, j] >= 0:
                e = int(idx[tok, j])
                u = t["U"][tok]
                y = (torch.nn.functional.silu(t["W_gate"][e] @ u) * (t["W_up"][e] @ u)) @ t["W_down"][e].T
                out[tok] = out[tok] + g[tok, j] * y
    if "W_gate_sh" in t:
        for i in range(t["W_gate_sh"].shape[0]):
            out = out + (torch.nn.functional.silu(t["U"] @ t["W_gate_sh"][i].T) *
                         (t["U"] @ t["W_up_sh"][i].T)) @ t["W_down_sh"][i].T
    loss = (out * torch.tensor(dO)).sum()
    f = torch.tensor(fwd["counts_routed"] / (T * k))
    sp = s / s.sum(dim=1, keepdim=True) if score_fn == 1 else s
    loss = loss + w_aux * E * (f * sp.mean(dim=0)).sum() + w_z * (torch.logsumexp(H, dim=1) ** 2).mean()
    return loss


def pin_layer_backward_autograd(O):
    """layer_backward against torch autograd of the layer written with torch ops (softplus, softmax /
    sigmoid, silu, matmul, logsumexp; float64), routing decisions held fixed: softmax+renorm with
    drops and the noisy router, and sigmoid with a shared expert."""
    import torch
    rng = _rng(67)
    T, h, E, k, d = 7, 5, 4, 2, 3
    for score_fn, renorm, noisy, shared, C in ((0, True, True, False, 3), (1, True, False, True, 0), (0, False, False, False, 0)):
        v = dict(U=rng.normal(size=(T, h)), W_r=rng.normal(size=(h, E)), b_r=rng.normal(size=E),
                 W_noise=rng.normal(size=(h, E)) if noisy else None, eps=rng.normal(size=(T, E)) if noisy else None,
                 W_gate=rng.normal(size=(E, d, h)), W_up=rng.normal(size=(E, d, h)), W_down=rng.normal(size=(E, h, d)))
        inp = _inputs(**v)
        if shared:
            inp.shared = (rng.normal(size=(1, d, h)), rng.normal(size=(1, d, h)), rng.normal(size=(1, h, d)))
        fwd = O.layer_forward(inp, T=T, h=h, E=E, k=k, d_e=d, score_fn=score_fn, renorm=renorm, capacity_factor=0.0,
                              capacity_override=C, shared=getattr(inp, "shared", None))
        fwd["eps"] = v["eps"]
        dO = rng.normal(size=(T, h))
        w_aux, w_z = 0.3, 0.2
        g = O.layer_backward(inp, fwd, dO, k=k, d_e=d, score_fn=score_fn, renorm=renorm, w_aux=w_aux, w_z=w_z)
        t = {n: torch.tensor(x, requires_grad=True) for n, x in v.items() if x is not None and n != "eps"}
        if shared:
            for n, x in zip(("W_gate_sh", "W_up_sh", "W_down_sh"), inp.shared):
                t[n] = torch.tensor(x, requires_grad=True)
        _torch_layer_loss(t, fwd, dO, T=T, E=E, k=k, score_fn=score_fn, renorm=renorm, w_aux=w_aux, w_z=w_z,
                          noisy=noisy).backward()
        pairs = [("dU", "U"), ("dW_r", "W_r"), ("db_r", "b_r"), ("dW_gate", "W_gate"), ("dW_up", "W_up"),
                 ("dW_down", "W_down")]
        if noisy:
            pairs.append(("dW_noise", "W_noise"))
        if shared:
            pairs += [("dW_gate_sh", "W_gate_sh"), ("dW_up_sh", "W_up_sh"), ("dW_down_sh", "W_down_sh")]
        for mine, ref in pairs:
            assert np.allclose(g[mine], t[ref].grad.numpy(), rtol=1e-6, atol=1e-6), (score_fn, renorm, mine)


ALL_PINS = [v for k_, v in sorted(globals().items()) if k_.startswith("pin_")]

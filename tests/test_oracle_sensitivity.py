"""Each plausible oracle mistake must be caught by at least one pin (CPU).

A mistake is planted in the oracle module (never in the library), all pins are
run against the planted oracle, and at least one must fail.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
import oracle_pins

O = oracle.moe_oracle
_orig = {name: getattr(O, name) for name in dir(O) if callable(getattr(O, name))}


def _gates_no_renorm(s, idx, renorm):
    return _orig["gates"](s, idx, False)


def _topk_ties_high(H32, k, allowed=None):
    E = H32.shape[1]
    rev = np.asarray(H32)[:, ::-1]
    if allowed is None:
        order = np.argsort(-rev, axis=1, kind="stable")
    else:
        order = np.lexsort((-rev, ~np.asarray(allowed, dtype=bool)[:, ::-1]), axis=-1)
    return (E - 1 - order[:, :k]).astype(np.int32)


def _topk_ignores_allowed(H32, k, allowed=None):
    return _orig["topk_select"](H32, k, None)


def _group_scores_best_only(aff, n_group, r):
    return _orig["group_scores"](aff, n_group, 1)


def _group_mask_strided(aff, n_group, topk_group, k):
    T, E = np.asarray(aff).shape
    perm = np.arange(E).reshape(E // n_group, n_group).T.reshape(-1)  # group q = experts q, q+n_group, ...
    inv = np.argsort(perm)
    m = _orig["group_limited_mask"](np.asarray(aff)[:, perm], n_group, topk_group, k)
    return m[:, inv]


def _route_groups_on_logits(H, k, fn, renorm, sel_bias=None, n_group=1, topk_group=1):
    r = _orig["route"](H, k, fn, renorm, sel_bias, 1, 1)
    if n_group > 1:
        allowed = _orig["group_limited_mask"](r["logits"], n_group, topk_group, k)
        r["idx"] = _orig["topk_select"](r["sel_key"], k, allowed)
        r["gate"] = _orig["gates"](r["s"], r["idx"], renorm)
    return r


def _capacity_floor(T, E, k, cf, override=0):
    if override > 0:
        return override
    if cf <= 0:
        return T
    return int(math.floor(Fraction(float(np.float32(cf))) * T * k / E))


def _capacity_without_k(T, E, k, cf, override=0):
    return _orig["capacity"](T, E, 1, cf, override)


def _silu_sign(x):
    return x / (1.0 + np.exp(x))


def _swiglu_swapped(x, Wg, Wu, Wd):
    return _orig["swiglu"](x, Wu, Wg, Wd)


def _combine_no_gate(U, Y, slot_row, gate, k):
    return _orig["combine"](U, Y, slot_row, np.ones_like(np.asarray(gate, dtype=float)), k)


def _dispatch_token_major(idx, E, C, priority=0):
    return _orig["dispatch"](idx, E, C, 1)


def _stats_unnormalised_sigmoid(counts, s, T, k, fn):
    return _orig["load_stats"](counts, s, T, k, O.SOFTMAX)


def _stats_f_over_T(counts, s, T, k, fn):
    return _orig["load_stats"](counts, s, T, 1, fn)


def _logits_no_bias(U, W_r, b_r=None, W_noise=None, eps=None):
    return _orig["router_logits"](U, W_r, None, W_noise, eps)


def _softplus_exp(x):
    return np.exp(x)


def _dispatch_offsets_routed(idx, E, C, priority=0):
    d = _orig["dispatch"](idx, E, C, priority)
    d["offsets"] = np.concatenate([[0], np.cumsum(d["counts_routed"])])
    return d


def _scores_softmax_no_shift_wrong_axis(H, fn):
    if fn == O.SOFTMAX:
        z = np.exp(H)
        return z / z.sum(axis=0, keepdims=True)
    return _orig["scores"](H, fn)


def _sigmoid_wrong_sign(H, fn):
    if fn == O.SIGMOID:
        return 1.0 / (1.0 + np.exp(H))
    return _orig["scores"](H, fn)


def _z_loss_no_square(H):
    H = np.asarray(H, dtype=np.float64)
    if H.shape[0] == 0:
        return 0.0
    m = H.max(axis=1)
    return float(np.mean(m + np.log(np.exp(H - m[:, None]).sum(axis=1))))


def _z_loss_sum_over_tokens(H):
    return _orig["router_z_loss"](H) * max(1, np.asarray(H).shape[0])


def _z_loss_max_not_lse(H):
    H = np.asarray(H, dtype=np.float64)
    return float(np.mean(H.max(axis=1) ** 2)) if H.shape[0] else 0.0


def _bias_update_wrong_sign(b, counts, u):
    c = np.asarray(counts, dtype=np.float64)
    return np.asarray(b, dtype=np.float64) + u * np.sign(c - c.mean())


def _route_gates_from_key(H, k, fn, renorm, sel_bias=None, n_group=1, topk_group=1):
    r = _orig["route"](H, k, fn, renorm, sel_bias, n_group, topk_group)
    if sel_bias is not None:
        r["gate"] = _orig["gates"](r["s"] + np.asarray(sel_bias, dtype=np.float64)[None, :], r["idx"], renorm)
    return r


def _route_ignores_bias(H, k, fn, renorm, sel_bias=None, n_group=1, topk_group=1):
    return _orig["route"](H, k, fn, renorm, None, n_group, topk_group)


def _combine_ignores_shared(U, Y, slot_row, gate, k, Y_shared=None):
    return _orig["combine"](U, Y, slot_row, gate, k, None)


def _aux_grad_no_mean_term(H, f, fn):
    s = O.scores(np.asarray(H, dtype=np.float64), fn)
    T, E = s.shape
    return E / T * s * np.asarray(f, dtype=np.float64)[None, :]


def _gate_backward_ignores_renorm(H, idx, d_gate, fn, renorm):
    return _orig["gate_backward"](H, idx, d_gate, fn, False)


def _z_grad_half(H):
    return 0.5 * _orig["z_loss_grad"](H)


def _combine_backward_no_gate(dO, Y, slot_row, gate, k):
    return _orig["combine_backward"](dO, Y, slot_row, np.ones_like(np.asarray(gate, dtype=float)), k)


def _swiglu_backward_sigmoid_only(x, Wg, Wu, Wd, dy):
    b = _orig["swiglu_backward"](x, Wg, Wu, Wd, dy)
    x64 = np.asarray(x, dtype=np.float64)
    G = x64 @ np.asarray(Wg, dtype=np.float64).T
    Up = x64 @ np.asarray(Wu, dtype=np.float64).T
    sg = 1.0 / (1.0 + np.exp(-G))
    b["dG"] = b["d_act"] * Up * sg  # drops the G (1 - s) term of SiLU'
    b["dx"] = b["dG"] @ np.asarray(Wg, dtype=np.float64) + b["dUp"] @ np.asarray(Wu, dtype=np.float64)
    b["dW_gate"] = b["dG"].T @ x64
    return b


def _dispatch_backward_no_residual(dO, dX, slot_row, k):
    return _orig["dispatch_backward"](np.zeros_like(np.asarray(dO, dtype=np.float64)), dX, slot_row, k)


def _router_input_backward_no_noise_factor(U, W_r, dH, W_noise=None, eps=None):
    r = _orig["router_input_backward"](U, W_r, dH, None, None)
    if W_noise is not None:
        dN = np.asarray(dH, dtype=np.float64) * np.asarray(eps, dtype=np.float64)  # softplus' dropped
        r["dU"] = r["dU"] + dN @ np.asarray(W_noise, dtype=np.float64).T
        r["dW_noise"] = np.asarray(U, dtype=np.float64).T @ dN
    return r


def _e4m3_ties_away(x):
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, E = np.frexp(a)
    q = np.ldexp(1.0, np.maximum(E - 1, -6) - 3)
    return np.copysign(np.minimum(np.floor(a / q + 0.5) * q, 448.0), x)


def _e4m3_flush_subnormals(x):
    r = _orig["e4m3_round"](x)
    return np.where(np.abs(r) < 2.0 ** -6, 0.0 * r, r)


def _scale_one_too_small(amax):
    return _orig["pow2_scale_exponents"](amax) - 1


def _fp8_weights_unquantised(W):
    return np.stack([np.asarray(W[e], dtype=np.float64) for e in range(W.shape[0])])


def _quantize_rows_scale_up(A):
    codes, s = _orig["quantize_rows_fp8"](A)
    return codes, s + 1


def _sampled_without_shared(inp, tokens, idx, gate, slot_row, k, shared=None, fp8=False):
    return _orig["sampled_outputs"](inp, tokens, idx, gate, slot_row, k, None, fp8)


def _sampled_fp8_weights_unquantised(inp, tokens, idx, gate, slot_row, k, shared=None, fp8=False):
    if not fp8:
        return _orig["sampled_outputs"](inp, tokens, idx, gate, slot_row, k, shared, False)
    # the token rows are quantised, the gate/up weights are not
    U_q = O.dequantize_rows_fp8(*O.quantize_rows_fp8(np.asarray(inp.U, dtype=np.float64)))
    sub = type(inp)(**dict(vars(inp), U=U_q))
    return _orig["sampled_outputs"](sub, tokens, idx, gate, slot_row, k, shared, False)


MUTANTS = {
    "sampled_shared_term_dropped": ("sampled_outputs", _sampled_without_shared),
    "sampled_fp8_weights_not_quantised": ("sampled_outputs", _sampled_fp8_weights_unquantised),
    "gates_not_renormalised": ("gates", _gates_no_renorm),
    "ties_to_higher_id": ("topk_select", _topk_ties_high),
    "capacity_floor": ("capacity", _capacity_floor),
    "capacity_without_k": ("capacity", _capacity_without_k),
    "silu_sign": ("silu", _silu_sign),
    "gate_up_swapped": ("swiglu", _swiglu_swapped),
    "combine_ignores_gates": ("combine", _combine_no_gate),
    "token_major_priority": ("dispatch", _dispatch_token_major),
    "sigmoid_P_unnormalised": ("load_stats", _stats_unnormalised_sigmoid),
    "f_normalised_by_T": ("load_stats", _stats_f_over_T),
    "bias_dropped": ("router_logits", _logits_no_bias),
    "noise_exp_not_softplus": ("softplus", _softplus_exp),
    "offsets_from_routed_counts": ("dispatch", _dispatch_offsets_routed),
    "softmax_over_tokens": ("scores", _scores_softmax_no_shift_wrong_axis),
    "sigmoid_sign": ("scores", _sigmoid_wrong_sign),
    "z_loss_not_squared": ("router_z_loss", _z_loss_no_square),
    "z_loss_summed_not_averaged": ("router_z_loss", _z_loss_sum_over_tokens),
    "z_loss_max_for_lse": ("router_z_loss", _z_loss_max_not_lse),
    "bias_update_wrong_sign": ("balance_bias_update", _bias_update_wrong_sign),
    "loss_free_gates_from_key": ("route", _route_gates_from_key),
    "loss_free_bias_ignored": ("route", _route_ignores_bias),
    "shared_experts_not_added": ("combine", _combine_ignores_shared),
    "group_mask_ignored": ("topk_select", _topk_ignores_allowed),
    "e4m3_ties_away_from_zero": ("e4m3_round", _e4m3_ties_away),
    "e4m3_subnormals_flushed": ("e4m3_round", _e4m3_flush_subnormals),
    "fp8_scale_one_binade_low": ("pow2_scale_exponents", _scale_one_too_small),
    "fp8_weights_not_quantised": ("fp8_weights", _fp8_weights_unquantised),
    "fp8_dequant_with_wrong_scale": ("quantize_rows_fp8", _quantize_rows_scale_up),
    "group_scored_on_best_expert_only": ("group_scores", _group_scores_best_only),
    "groups_strided_not_contiguous": ("group_limited_mask", _group_mask_strided),
    "groups_scored_on_logits": ("route", _route_groups_on_logits),
    "aux_grad_without_mean_load": ("aux_loss_grad", _aux_grad_no_mean_term),
    "gate_backward_ignores_renorm": ("gate_backward", _gate_backward_ignores_renorm),
    "z_grad_half": ("z_loss_grad", _z_grad_half),
    "combine_backward_ignores_gate": ("combine_backward", _combine_backward_no_gate),
    "silu_derivative_missing_term": ("swiglu_backward", _swiglu_backward_sigmoid_only),
    "dispatch_backward_drops_residual": ("dispatch_backward", _dispatch_backward_no_residual),
    "noise_branch_without_softplus_derivative": ("router_input_backward", _router_input_backward_no_noise_factor),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(O, attr, fn)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(O)
        except Exception:  # an assertion, or a shape error the mistake causes
            failed.append(pin.__name__)
    assert failed, f"planted mistake {name!r} passed every pin"

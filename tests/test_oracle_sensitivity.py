"""Each plausible oracle mistake must be caught by at least one pin (CPU).

A mistake is planted in a copy of the oracle's C++ source (oracle/moe_oracle.cpp, never the
library), the copy is compiled, and every pin runs against it in a subprocess
(oracle_mutant_runner.py); at least one pin must fail.  A mutant that crashes its subprocess
counts only through the pins it failed before the crash.  The unplanted source, compiled the same
way, must pass every pin (the control).
"""
import concurrent.futures as cf
import os
import subprocess
import sys
import tempfile

import pytest

import oracle_pins
from oracle import moe_oracle

HERE = os.path.dirname(os.path.abspath(__file__))
RUNNER = os.path.join(HERE, "oracle_mutant_runner.py")

# name -> [(text in moe_oracle.cpp, replacement)]; each text must occur exactly once
MUTANTS = {
    "gates_not_renormalised": [("gate[t * k + j] = renorm ? v / sum : v;", "gate[t * k + j] = v;")],
    "ties_to_higher_id": [("  if (key[a] != key[b]) return key[a] > key[b];\n  return a < b;",
                           "  if (key[a] != key[b]) return key[a] > key[b];\n  return a > b;")],
    "capacity_floor": [("long double q = std::ceil(num / E);\n  while (q > 0 && (q - 1) * E >= num) q -= 1;\n"
                        "  while (q * E < num) q += 1;", "long double q = std::floor(num / E);")],
    "capacity_without_k": [("static_cast<long double>(T * k)", "static_cast<long double>(T)")],
    "silu_sign": [("double silu(double x) { return x / (1.0 + std::exp(-x)); }",
                   "double silu(double x) { return x / (1.0 + std::exp(x)); }")],
    "gate_up_swapped": [("a[r * d + j] = silu(G) * Up;", "a[r * d + j] = silu(Up) * G;")],
    "combine_ignores_gates": [("o[c] += gate[t * k + j] * Y[row * h + c];", "o[c] += Y[row * h + c];")],
    "token_major_priority": [("    if (priority == CHOICE_MAJOR) {\n      j = static_cast<int>(p / T);",
                              "    if (false) {\n      j = static_cast<int>(p / T);")],
    "sigmoid_P_unnormalised": [("    if (fn == SIGMOID) {\n      S = 0.0;", "    if (false) {\n      S = 0.0;")],
    "f_normalised_by_T": [("f[e] = counts[e] / (static_cast<double>(T) * k);",
                           "f[e] = counts[e] / static_cast<double>(T);")],
    "bias_dropped": [("        if (b_r) acc += elem(b_r, b_dt, e);\n", "")],
    "noise_exp_not_softplus": [("double softplus(double x) { return std::max(x, 0.0) + std::log1p(std::exp(-std::fabs(x))); }",
                                "double softplus(double x) { return std::exp(x); }")],
    "offsets_from_routed_counts": [("offsets[e + 1] = offsets[e] + counts_kept[e];",
                                    "offsets[e + 1] = offsets[e] + counts_routed[e];")],
    "softmax_denominator_unshifted": [("    for (int e = 0; e < E; ++e) z += std::exp(H[e] - m);\n    for (int e = 0; e < E; ++e) s[e]",
                                       "    for (int e = 0; e < E; ++e) z += std::exp(H[e]);\n    for (int e = 0; e < E; ++e) s[e]")],
    "sigmoid_sign": [("double sigmoid(double x) { return 1.0 / (1.0 + std::exp(-x)); }",
                      "double sigmoid(double x) { return 1.0 / (1.0 + std::exp(x)); }")],
    "z_loss_not_squared": [("    sum += lse * lse;", "    sum += lse;")],
    "z_loss_summed_not_averaged": [("  return sum / T;", "  return sum;")],
    "z_loss_max_for_lse": [("    const double lse = m + std::log(z);\n    sum += lse * lse;",
                            "    const double lse = m;\n    sum += lse * lse;")],
    "bias_update_wrong_sign": [("const double err = mean - counts[e];", "const double err = counts[e] - mean;")],
    "loss_free_gates_from_key": [("orc_gates(T, E, k, s, idx, renorm, gate);",
                                  "orc_gates(T, E, k, sel_key, idx, renorm, gate);")],
    "loss_free_bias_ignored": [("sel_key[t * E + e] = sel_bias ? s[t * E + e] + sel_bias[e] : logits32[t * E + e];",
                                "sel_key[t * E + e] = logits32[t * E + e];")],
    "shared_experts_not_added": [("    for (int s = 0; s < n_s; ++s)\n      for (int c = 0; c < h; ++c) o[c] += Y_sh[(s * T + t) * h + c];\n", "")],
    "group_mask_ignored": [("orc_topk(T, E, sel_key, k, mask, idx);", "orc_topk(T, E, sel_key, k, nullptr, idx);")],
    "e4m3_ties_away_from_zero": [("std::nearbyint(a / quantum)", "std::floor(a / quantum + 0.5)")],
    "e4m3_subnormals_flushed": [("  return std::copysign(r, x);\n}",
                                 "  return std::copysign(r < std::ldexp(1.0, -6) ? 0.0 : r, x);\n}")],
    "fp8_scale_one_binade_low": [("return std::max<int64_t>(s, -127);", "return std::max<int64_t>(s, -127) - 1;")],
    "fp8_weights_not_quantised": [("      if (fp8_w) {\n        fp8_roundtrip_row(wg.data(), h);",
                                   "      if (false) {\n        fp8_roundtrip_row(wg.data(), h);")],
    "fp8_roundtrip_scale_wrong": [("row[i] = std::ldexp(e4m3_round(std::ldexp(row[i], -s)), s);",
                                   "row[i] = std::ldexp(e4m3_round(std::ldexp(row[i], -s)), s + 1);")],
    "fp8_dequant_with_wrong_scale": [("out[r * c + i] = std::ldexp(codes[r * c + i], static_cast<int>(s[r]));",
                                      "out[r * c + i] = std::ldexp(codes[r * c + i], static_cast<int>(s[r]) + 1);")],
    "group_scored_on_best_expert_only": [("gs[q] = sum_of_largest(aff + q * S, S, r);",
                                          "gs[q] = sum_of_largest(aff + q * S, S, 1);")],
    "groups_strided_not_contiguous": [("allowed[e] = keep[e / S];", "allowed[e] = keep[e % n_group];")],
    "groups_scored_on_logits": [("orc_group_limited_mask(T, E, sel_bias ? sel_key : s,",
                                 "orc_group_limited_mask(T, E, sel_bias ? sel_key : logits32,")],
    "aux_grad_without_mean_load": [("/ T * sp[e] * sat * (f[e] - mean);", "/ T * sp[e] * sat * f[e];")],
    "gate_backward_ignores_renorm": [("ds[e] += renorm ? (d_gate[t * k + j] - wg) / S : d_gate[t * k + j];",
                                      "ds[e] += d_gate[t * k + j];")],
    "z_grad_half": [("out[t * E + e] = 2.0 / T * lse * s[e];", "out[t * E + e] = 1.0 / T * lse * s[e];")],
    "combine_backward_ignores_gate": [("dY[row * h + c] = gate[t * k + j] * dO[t * h + c];",
                                       "dY[row * h + c] = dO[t * h + c];")],
    "silu_derivative_missing_term": [("dG[r * d + j] = da * Up * sg * (1.0 + G * (1.0 - sg));",
                                      "dG[r * d + j] = da * Up * sg;")],
    "dispatch_backward_drops_residual": [("double acc = dO[t * h + c];", "double acc = 0.0;")],
    "noise_branch_without_softplus_derivative": [("* elem(eps, eps_dt, t * E + e) * sigmoid(z);",
                                                  "* elem(eps, eps_dt, t * E + e);")],
    "sampled_shared_term_dropped": [("    for (int s = 0; s < n_s; ++s)\n      for (int c = 0; c < h; ++c) o[c] += Y_sh[(s * n + t) * h + c];\n", "")],
    "sampled_fp8_weights_not_quantised": [("expert_rows(n, h, d, xq.data(), Wg, wg_dt, wg_off, Wu, wu_dt, wu_off, Wd, wd_dt, wd_off, fp8_w, y, a);",
                                           "expert_rows(n, h, d, xq.data(), Wg, wg_dt, wg_off, Wu, wu_dt, wu_off, Wd, wd_dt, wd_off, 0, y, a);")],
    "router_weight_read_transposed": [("for (int c = 0; c < h; ++c) acc += u[c] * wr[static_cast<size_t>(c) * E + e];",
                                       "for (int c = 0; c < h; ++c) acc += u[c] * wr[static_cast<size_t>(e) * h + c];")],
    "logits_not_rounded_to_f32": [("  orc_round_f32(T * E, H, logits32);\n  orc_scores",
                                   "  for (int64_t i = 0; i < T * E; ++i) logits32[i] = H[i];\n  orc_scores")],
    "slot_row_without_offset": [("slot_row[pair] = offsets[e] + slot[pair];", "slot_row[pair] = slot[pair];")],
    "every_expert_uses_expert_0_gate": [("expert_rows(hi - lo, h, d, X + lo * h, Wg, wg_dt, e * hd,",
                                         "expert_rows(hi - lo, h, d, X + lo * h, Wg, wg_dt, 0,")],
    "shared_backward_dx_not_added": [("      for (int64_t j = 0; j < T * h; ++j) dU[j] += dx[j];\n", "")],
    "router_input_backward_db_zero": [("    for (int64_t t = 0; t < T; ++t) a += dH[t * E + e];\n    db_r[e] = a;",
                                       "    db_r[e] = a;")],
}


def _planted_source(edits) -> str:
    src = open(moe_oracle.SRC).read()
    for old, new in edits:
        n = src.count(old)
        assert n == 1, f"mutation anchor found {n} times: {old[:60]!r}"
        src = src.replace(old, new)
    return src


def _run(name, edits, workdir):
    cpp = os.path.join(workdir, f"{name}.cpp")
    with open(cpp, "w") as fh:
        fh.write(_planted_source(edits))
    lib = os.path.join(workdir, f"lib_{name}.so")
    moe_oracle.build(cpp, lib, force=True)
    env = dict(os.environ, OMP_NUM_THREADS="1")
    res = subprocess.run([sys.executable, RUNNER, lib], capture_output=True, text=True, timeout=600, env=env)
    failed = [ln.split()[1].rstrip(":") for ln in res.stdout.splitlines() if ln.startswith("FAILED")]
    passed = [ln.split()[1] for ln in res.stdout.splitlines() if ln.startswith("passed")]
    return dict(failed=failed, passed=passed, rc=res.returncode, stderr=res.stderr[-2000:])


@pytest.fixture(scope="module")
def outcomes():
    jobs = dict(MUTANTS, control=[])
    with tempfile.TemporaryDirectory() as workdir, cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        futs = {name: ex.submit(_run, name, edits, workdir) for name, edits in jobs.items()}
        return {name: f.result() for name, f in futs.items()}


def test_control_passes_every_pin(outcomes):
    r = outcomes["control"]
    assert r["rc"] == 0 and not r["failed"], r
    assert len(r["passed"]) == len(oracle_pins.ALL_PINS), r


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, outcomes):
    r = outcomes[name]
    assert r["failed"], f"planted mistake {name!r} passed every pin (rc {r['rc']}): {r['stderr']}"

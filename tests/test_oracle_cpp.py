"""Properties of the C++ oracle library itself (CPU): its results do not depend on the OpenMP
thread count, and its layer forward reports the wall time of every stage."""
import numpy as np

import oracle
from mixture_experts_layer_84_b300 import synth
from mixture_experts_layer_84_b300 import workloads as W

CASES = [
    W.Workload("noisy_groups_shared", T=90, h=24, E=8, k=2, d_e=20, dtype=W.BF16, score_fn=W.SOFTMAX, renorm=True,
               noisy=True, capacity_factor=0.9, bias="zipf", n_shared=1, d_shared=16, sel_bias="normal",
               n_group=4, topk_group=2),
    W.Workload("sigmoid_f32", T=70, h=16, E=6, k=3, d_e=12, dtype=W.F32, score_fn=W.SIGMOID, renorm=False,
               noisy=False, capacity_factor=1.1, priority=W.PRIORITY_TOKEN_MAJOR),
]


def _forward(w, inp, fp8=False):
    return oracle.layer_forward(inp, T=w.T, h=w.h, E=w.E, k=w.k, d_e=w.d_e, score_fn=w.score_fn, renorm=w.renorm,
                                capacity_factor=w.capacity_factor, capacity_override=w.capacity, priority=w.priority,
                                sel_bias=inp.sel_bias, shared=inp.shared, n_group=w.n_group,
                                topk_group=w.topk_group, fp8=fp8)


def test_results_do_not_depend_on_the_thread_count():
    default = oracle.threads()
    try:
        for w in CASES:
            inp = synth.generate(w, 0, "cpu")
            runs = []
            for n in (1, 3, max(2, default)):
                oracle.set_threads(n)
                runs.append(_forward(w, inp, fp8=w.dtype == W.BF16))
            for r in runs[1:]:
                for name, v in runs[0].items():
                    if isinstance(v, np.ndarray):
                        assert np.array_equal(v, r[name]), (w.name, name)
    finally:
        oracle.set_threads(default)


def test_layer_forward_reports_stage_seconds():
    w = CASES[0]
    r = _forward(w, synth.generate(w, 0, "cpu"))
    assert list(r["seconds"]) == list(oracle.STAGES)
    assert all(s >= 0.0 for s in r["seconds"].values())
    assert r["seconds"]["experts"] > 0.0

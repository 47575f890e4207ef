"""moe_dispatch against the oracle: counts, offsets, slots, drop mask, permutation and
the row copy, all bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_84_b300 import _lib as L
from mixture_experts_layer_84_b300 import synth
from mixture_experts_layer_84_b300 import workloads as W

pytestmark = pytest.mark.gpu

CM, TM = W.PRIORITY_CHOICE_MAJOR, W.PRIORITY_TOKEN_MAJOR

CASES = [
    # T, E, k, C (0 = unbounded), priority, zipf skew, h
    (4096, 64, 8, 640, CM, 0.0, 64),        # the capacity example's shape
    (12, 4, 1, 3, CM, 0.0, 64),
    (65536, 64, 6, 12288, CM, 0.0, 4096),   # full-size stress workload
    (65536, 64, 6, 2048, CM, 0.0, 256),     # literal ceil(CF*T/E) capacity on the same shape
    (16384, 128, 1, 128, CM, 1.1, 1024),    # Switch-like skew, heavy drops
    (4096, 256, 8, 0, CM, 0.5, 512),        # no capacity limit
    (777, 8, 2, 1, TM, 0.0, 64),
    (1000, 16, 16, 100, TM, 0.3, 128),      # k = E
    (1, 1, 1, 1, CM, 0.0, 8),
    (9000, 1024, 16, 50, CM, 1.0, 64),      # largest E and k
    (5000, 7, 3, 1500, TM, 2.0, 200),
    (4096, 256, 8, 0, CM, 0.5, 7168),       # 256-expert shape at its row width (14 KB rows)
    (2048, 8, 2, 640, CM, 0.0, 4096),       # Mixtral shape
    (64, 4, 2, 0, CM, 0.0, 53248),          # 104 KB rows: two do not fit one block, scatter kernel copies
    # more than 8192 ids but small chunk histograms: the placement blocks add the histograms up
    # themselves (no column scan), with 16-byte loads (k E = 16) and with scalar ones (k E = 10)
    (16384, 16, 1, 1100, CM, 0.8, 64),
    (12000, 5, 2, 2500, CM, 0.5, 64),
]


def run_dispatch(T, E, k, C, priority, idx, U, dtype=W.BF16):
    cfg = L.config(T, U.shape[1], E, k, 8, capacity=C if C > 0 else 0,
                   capacity_factor=0.0, priority=priority, dtype=dtype)
    b = dict(counts_routed=torch.full((E,), -5, dtype=torch.int32, device="cuda"),
             counts_kept=torch.full((E,), -5, dtype=torch.int32, device="cuda"),
             offsets=torch.full((E + 1,), -5, dtype=torch.int32, device="cuda"),
             slot_row=torch.full((T * k,), -5, dtype=torch.int32, device="cuda"),
             row_token=torch.full((T * k,), -5, dtype=torch.int32, device="cuda"),
             X=torch.zeros((T * k, cfg.h), dtype=U.dtype, device="cuda"),
             n_dropped=torch.full((1,), -5, dtype=torch.int64, device="cuda"))
    ws = L.new_workspace(cfg)
    L.moe_dispatch(cfg, U, idx, b["counts_routed"], b["counts_kept"], b["offsets"], b["slot_row"], b["row_token"],
                   b["X"], b["n_dropped"], ws)
    return cfg, b, ws


@pytest.mark.parametrize("T,E,k,C,priority,zipf,h", CASES)
def test_dispatch_bitexact(T, E, k, C, priority, zipf, h):
    idx = synth.random_routing(T, E, k, seed=T * 7 + E, zipf_s=zipf).cuda()
    U = synth.random_rows(T, h, seed=3, stream="U", device="cuda", dtype=torch.bfloat16)
    cfg, b, ws = run_dispatch(T, E, k, C, priority, idx, U)
    assert L.moe_get_device_status(ws) == 0
    Cap = C if C > 0 else T
    d = oracle.dispatch(idx.cpu().numpy(), E, Cap, priority)
    A = int(d["offsets"][-1])
    assert np.array_equal(b["counts_routed"].cpu().numpy(), d["counts_routed"])
    assert np.array_equal(b["counts_kept"].cpu().numpy(), d["counts_kept"])
    assert np.array_equal(b["offsets"].cpu().numpy(), d["offsets"])
    assert np.array_equal(b["slot_row"].cpu().numpy(), d["slot_row"])
    assert np.array_equal(b["row_token"][:A].cpu().numpy(), d["row_token"])
    assert int(b["n_dropped"].item()) == d["n_dropped"]
    # the permutation: every kept row is an exact copy of its token's row
    rt = b["row_token"][:A].long()
    assert torch.equal(b["X"][:A], U[rt])
    # rows past A are untouched
    assert torch.all(b["row_token"][A:] == -5)


def test_dispatch_fp32_rows():
    T, E, k, h = 513, 8, 2, 40
    idx = synth.random_routing(T, E, k, seed=11, zipf_s=0.5).cuda()
    U = synth.random_rows(T, h, seed=4, stream="U", device="cuda", dtype=torch.float32)
    cfg, b, ws = run_dispatch(T, E, k, 80, CM, idx, U, dtype=W.F32)
    d = oracle.dispatch(idx.cpu().numpy(), E, 80, CM)
    A = int(d["offsets"][-1])
    assert np.array_equal(b["slot_row"].cpu().numpy(), d["slot_row"])
    assert torch.equal(b["X"][:A], U[b["row_token"][:A].long()])


def test_dispatch_empty():
    T, E, k = 0, 8, 2
    idx = torch.empty((0, k), dtype=torch.int32, device="cuda")
    U = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    cfg, b, ws = run_dispatch(T, E, k, 0, CM, idx, U)
    assert L.moe_get_device_status(ws) == 0
    assert b["counts_routed"].tolist() == [0] * E and b["counts_kept"].tolist() == [0] * E
    assert b["offsets"].tolist() == [0] * (E + 1)
    assert int(b["n_dropped"].item()) == 0


def test_dispatch_out_of_range_ids_are_dropped_and_flagged():
    T, E, k, h = 300, 8, 2, 64
    idx = synth.random_routing(T, E, k, seed=5).cuda()
    idx[3, 0] = -1
    idx[10, 1] = E
    idx[299, 0] = 1 << 20
    U = synth.random_rows(T, h, seed=3, stream="U", device="cuda", dtype=torch.bfloat16)
    cfg, b, ws = run_dispatch(T, E, k, T, CM, idx, U)
    assert L.moe_get_device_status(ws) == L.MOE_DEV_BAD_EXPERT_ID
    assert L.moe_get_device_status(ws) == 0  # reading clears it
    sr = b["slot_row"].cpu().numpy()
    for (t, j) in ((3, 0), (10, 1), (299, 0)):
        assert sr[t * k + j] == -1
    assert int(b["counts_routed"].sum()) == T * k - 3
    assert int(b["n_dropped"].item()) == 3

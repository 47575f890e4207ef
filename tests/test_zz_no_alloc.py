"""moe_dispatch_noalloc: the dispatch entry point for callers that cannot allocate.

Some callers may not allocate device memory at all. Examples: a serving engine that reserves all
of its memory at start-up, or a plugin whose host framework offers no scratch allocator. For them,
moe_dispatch_noalloc keeps dispatch's one piece of scratch, the per-chunk expert histogram, in a
static device array inside the library, so it takes no workspace.

This test calls it through the C ABI and checks its results against the ordinary moe_dispatch
on the same inputs. It does so on two calls in a row with different shapes, because the second
call reuses the array the first one left behind. The integer outputs and the copied rows must be
identical. The file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

from mixture_experts_layer_84_b300 import _lib as L
from mixture_experts_layer_84_b300 import synth
from mixture_experts_layer_84_b300 import workloads as W

OUTPUTS = ("counts_routed", "counts_kept", "offsets", "slot_row", "row_token", "X", "n_dropped")


def _buffers(T, E, k, h, dtype):
    i32 = torch.int32
    return dict(counts_routed=torch.full((E,), -7, dtype=i32, device="cuda"),
                counts_kept=torch.full((E,), -7, dtype=i32, device="cuda"),
                offsets=torch.full((E + 1,), -7, dtype=i32, device="cuda"),
                slot_row=torch.full((T * k,), -7, dtype=i32, device="cuda"),
                row_token=torch.full((T * k,), -7, dtype=i32, device="cuda"),
                X=torch.zeros((T * k, h), dtype=dtype, device="cuda"),
                n_dropped=torch.full((1,), -7, dtype=torch.int64, device="cuda"))


def _args(b):
    return [b[n] for n in OUTPUTS]


# T, h, E, k, capacity (0: unbounded), priority, Zipf skew of the routing, dtype
CALLS = [
    (65536, 256, 64, 6, 2048, W.PRIORITY_CHOICE_MAJOR, 0.3, W.BF16),   # heavy drops, 96 chunks
    (9000, 64, 1024, 16, 50, W.PRIORITY_TOKEN_MAJOR, 1.0, W.F32),       # largest E and k, other layout
]


@pytest.mark.gpu
def test_noalloc_dispatch_matches_dispatch_on_two_calls_in_a_row():
    for n, (T, h, E, k, C, prio, zipf, dtype) in enumerate(CALLS):
        cfg = L.config(T, h, E, k, 8, capacity=C, capacity_factor=0.0, priority=prio, dtype=dtype)
        tdt = torch.bfloat16 if dtype == W.BF16 else torch.float32
        U = synth.random_rows(T, h, seed=n, stream="X", device="cuda", dtype=tdt)
        idx = synth.random_routing(T, E, k, seed=n, device="cuda", zipf_s=zipf)

        ref = _buffers(T, E, k, h, tdt)
        ws = L.new_workspace(cfg)
        L.moe_dispatch(cfg, U, idx, *_args(ref), ws)
        assert L.moe_get_device_status(ws) == 0

        got = _buffers(T, E, k, h, tdt)
        status = torch.full((1,), 99, dtype=torch.int32, device="cuda")
        L.moe_dispatch_noalloc(cfg, U, idx, *_args(got), status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0

        A = int(ref["offsets"][-1].item())
        assert int(ref["n_dropped"].item()) > 0  # both calls exercise the capacity limit
        for name in OUTPUTS:
            a, b = got[name], ref[name]
            if name in ("row_token", "X"):
                a, b = a[:A], b[:A]
            assert torch.equal(a, b), f"call {n}: {name} differs from moe_dispatch"


@pytest.mark.gpu
def test_noalloc_dispatch_without_a_status_word():
    """status = NULL: device-side errors go unreported, the results are still moe_dispatch's."""
    T, h, E, k = 5000, 128, 16, 2
    cfg = L.config(T, h, E, k, 8, capacity=400, capacity_factor=0.0, dtype=W.BF16)
    U = synth.random_rows(T, h, seed=7, stream="X", device="cuda", dtype=torch.bfloat16)
    idx = synth.random_routing(T, E, k, seed=7, device="cuda", zipf_s=0.8)
    ref = _buffers(T, E, k, h, torch.bfloat16)
    ws = L.new_workspace(cfg)
    L.moe_dispatch(cfg, U, idx, *_args(ref), ws)
    assert L.moe_get_device_status(ws) == 0
    got = _buffers(T, E, k, h, torch.bfloat16)
    L.moe_dispatch_noalloc(cfg, U, idx, *_args(got), None)
    torch.cuda.synchronize()
    A = int(ref["offsets"][-1].item())
    assert int(ref["n_dropped"].item()) > 0
    for name in OUTPUTS:
        a, b = got[name], ref[name]
        if name in ("row_token", "X"):
            a, b = a[:A], b[:A]
        assert torch.equal(a, b), f"{name} differs from moe_dispatch"


def test_noalloc_dispatch_rejects_sizes_beyond_its_static_scratch():
    # ceil(T*k / 4096) * E = 1025 * 1024 > 2^20 histogram entries: refused on the host, before any
    # CUDA call, so no pointer is needed
    cfg = L.config(1025 * 4096, 8, 1024, 1, 8, capacity_factor=1.0)
    st = L.lib.moe_dispatch_noalloc(ctypes.byref(cfg), *([None] * 10), None)
    assert st == L.MOE_ERR_UNSUPPORTED
    assert "static histogram" in L.lib.moe_last_error().decode()

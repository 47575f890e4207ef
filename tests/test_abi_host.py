"""The C ABI on the host: it loads, exports what include/moe.h declares, and its
host-only logic (capacity, workspace size, argument validation) is right.
No kernel is launched here."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import oracle
from mixture_experts_layer_84_b300 import _lib as L
from mixture_experts_layer_84_b300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src))
    return sorted(names)


def test_header_declarations_are_exported():
    decl = declared_functions()
    assert set(L.EXPORTS) <= set(decl)
    out = subprocess.run(["nm", "-D", "--defined-only", L.LIB_PATH], capture_output=True, text=True, check=True)
    exported = sorted(set(m.group(1) for m in re.finditer(r" T (moe_\w+)$", out.stdout, flags=re.M)))
    assert exported == decl
    for name in decl:
        assert hasattr(L.lib, name)


def test_version_and_status_strings():
    assert "sm_103a" in L.version()
    assert L.status_name(0) == "MOE_OK"
    assert L.status_name(1) == "MOE_ERR_INVALID_ARG"
    assert L.status_name(4) == "MOE_ERR_DEVICE"


def test_config_struct_layout():
    assert ctypes.sizeof(L.moe_config) == 8 + 4 * 15 + 4  # int64 T, 15 x 32-bit fields, tail padding
    assert ctypes.sizeof(L.moe_layer_args) == 32 * 8


@pytest.mark.parametrize("w", W.FULL + W.SMALL, ids=lambda w: w.name)
def test_capacity_matches_oracle_on_workloads(w):
    assert L.capacity(L.config_of(w)) == oracle.capacity(w.T, w.E, w.k, w.capacity_factor, w.capacity)


def test_capacity_worked_examples_and_random_factors():
    assert L.capacity(L.config(12, 8, 4, 1, 8, capacity_factor=1.0)) == 3
    assert L.capacity(L.config(4096, 8, 64, 8, 8, capacity_factor=1.25)) == 640
    assert L.capacity(L.config(16, 8, 4, 2, 8, capacity_factor=0.0)) == 16
    assert L.capacity(L.config(16, 8, 4, 2, 8, capacity_factor=1.0, capacity=5)) == 5
    assert L.capacity(L.config(0, 8, 4, 2, 8, capacity_factor=1.0)) == 0
    rng = np.random.default_rng(0)
    for _ in range(2000):
        T = int(rng.integers(1, 200000))
        E = int(rng.integers(1, 1025))
        k = int(rng.integers(1, min(E, 16) + 1))
        cf = float(np.float32(rng.choice([rng.uniform(0.01, 4.0), rng.integers(1, 9) / 4.0, 1.1, 1.3])))
        got = L.capacity(L.config(T, 8, E, k, 8, capacity_factor=cf))
        assert got == oracle.capacity(T, E, k, cf), (T, E, k, cf)


def test_workspace_size_grows_with_tokens():
    small = L.workspace_size(L.config_of(W.MIXTRAL_SMALL))
    big = L.workspace_size(L.config_of(W.MIXTRAL))
    assert 256 <= small < big
    noisy = L.workspace_size(L.config_of(W.SWITCH))
    quiet = L.workspace_size(L.config_of(W.SWITCH, noisy=False))
    assert noisy > quiet


@pytest.mark.parametrize("kw,status", [
    (dict(T=-1), L.MOE_ERR_INVALID_ARG),
    (dict(E=0), L.MOE_ERR_INVALID_ARG),
    (dict(k=0), L.MOE_ERR_INVALID_ARG),
    (dict(k=9, E=8), L.MOE_ERR_INVALID_ARG),
    (dict(E=2048, k=2), L.MOE_ERR_UNSUPPORTED),
    (dict(E=64, k=17), L.MOE_ERR_UNSUPPORTED),
    (dict(h=100), L.MOE_ERR_UNSUPPORTED),
    (dict(d_e=12), L.MOE_ERR_UNSUPPORTED),
    (dict(dtype=7), L.MOE_ERR_INVALID_ARG),
    (dict(score_fn=3), L.MOE_ERR_INVALID_ARG),
    (dict(priority=2), L.MOE_ERR_INVALID_ARG),
    (dict(capacity=-3), L.MOE_ERR_INVALID_ARG),
    (dict(capacity_factor=float("nan")), L.MOE_ERR_INVALID_ARG),
    (dict(T=2 ** 30, k=2), L.MOE_ERR_UNSUPPORTED),
    (dict(n_group=-1), L.MOE_ERR_INVALID_ARG),
    (dict(n_group=3, topk_group=1), L.MOE_ERR_INVALID_ARG),           # E = 8 not a multiple of 3
    (dict(n_group=4, topk_group=0), L.MOE_ERR_INVALID_ARG),
    (dict(n_group=4, topk_group=5), L.MOE_ERR_INVALID_ARG),
    (dict(E=16, k=3, n_group=4, topk_group=2), L.MOE_ERR_INVALID_ARG),  # k not a multiple of topk_group
    (dict(E=16, k=4, n_group=8, topk_group=1), L.MOE_ERR_INVALID_ARG),  # 1 group of 2 cannot hold k = 4
    (dict(E=128, n_group=64, topk_group=2), L.MOE_ERR_UNSUPPORTED),
])
def test_bad_configs_rejected(kw, status):
    base = dict(T=64, h=64, E=8, k=2, d_e=64)
    base.update(kw)
    T, h, E, k, d = (base.pop(n) for n in ("T", "h", "E", "k", "d_e"))
    cfg = L.config(T, h, E, k, d, **base)
    n = ctypes.c_size_t()
    assert L.lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == status
    assert L.lib.moe_last_error().decode()


def test_group_limited_configs_accepted():
    n = ctypes.c_size_t()
    for kw in (dict(n_group=0), dict(n_group=1), dict(n_group=8, topk_group=4), dict(n_group=32, topk_group=8)):
        cfg = L.config(4096, 7168, 256, 8, 2048, **kw)
        assert L.lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == L.MOE_OK, kw


def test_fp8_entry_points_reject_unsupported_configs_before_any_launch():
    assert ctypes.sizeof(L.moe_fp8_args) == 6 * 8
    for cfg, msg in ((L.config(64, 136, 8, 2, 64), "multiple of 16"),
                     (L.config(64, 128, 8, 2, 64, dtype=W.F32), "bf16")):
        assert L.lib.moe_dispatch_fp8(ctypes.byref(cfg), *([None] * 12)) == L.MOE_ERR_UNSUPPORTED
        assert msg in L.lib.moe_last_error().decode()
        assert L.lib.moe_expert_ffn_fp8(ctypes.byref(cfg), *([None] * 12)) == L.MOE_ERR_UNSUPPORTED
        assert L.lib.moe_layer_forward_fp8(ctypes.byref(cfg), None, None, None, None) == L.MOE_ERR_UNSUPPORTED
    assert L.lib.moe_quantize_fp8(4, 12, None, None, None, None) == L.MOE_ERR_UNSUPPORTED
    assert L.lib.moe_quantize_fp8(4, 16, None, None, None, None) == L.MOE_ERR_INVALID_ARG  # NULL src
    assert L.lib.moe_quantize_fp8(-1, 16, None, None, None, None) == L.MOE_ERR_INVALID_ARG


def test_null_pointers_rejected_before_any_launch():
    cfg = L.config(64, 64, 8, 2, 64, capacity_factor=1.0)
    st = L.lib.moe_route(ctypes.byref(cfg), None, None, None, None, None, None, None, None, None, None, None, None)
    assert st == L.MOE_ERR_INVALID_ARG
    assert "U is NULL" in L.lib.moe_last_error().decode()
    assert L.lib.moe_dispatch(ctypes.byref(cfg), *([None] * 11)) == L.MOE_ERR_INVALID_ARG
    assert L.lib.moe_expert_ffn(ctypes.byref(cfg), *([None] * 9)) == L.MOE_ERR_INVALID_ARG
    assert L.lib.moe_combine(ctypes.byref(cfg), *([None] * 13)) == L.MOE_ERR_INVALID_ARG
    assert L.lib.moe_layer_forward(ctypes.byref(cfg), None, None, None) == L.MOE_ERR_INVALID_ARG
    assert L.lib.moe_get_device_status(None, None, None) == L.MOE_ERR_INVALID_ARG


def test_misaligned_pointer_rejected():
    cfg = L.config(64, 64, 8, 2, 64, capacity_factor=1.0, dtype=W.BF16)
    fake = ctypes.c_void_p(0x1000 + 2)  # never dereferenced: validation fails first
    ok = ctypes.c_void_p(0x100000)
    st = L.lib.moe_route(ctypes.byref(cfg), fake, ok, None, None, None, None, None, None, ok, ok, ok, None)
    assert st == L.MOE_ERR_INVALID_ARG
    assert "aligned" in L.lib.moe_last_error().decode()


def test_binding_argument_counts_match_the_header():
    """Every ctypes signature in the binding takes as many arguments as include/*.h declares."""
    for f in os.listdir(os.path.join(ROOT, "include")):
        if not f.endswith(".h"):
            continue
        src = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", f)).read(), flags=re.S)
        for m in re.finditer(r"\b(moe_[a-z_0-9]+)\s*\(([^;{]*?)\)\s*;", src):
            name, args = m.group(1), m.group(2).strip()
            n = 0 if args in ("void", "") else len(args.split(","))
            argtypes = getattr(L.lib, name).argtypes
            assert argtypes is None and n == 0 or argtypes is not None and len(argtypes) == n, name

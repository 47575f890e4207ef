"""Seeded synthetic inputs for the MoE layer.

This module is shared by the tests, the benchmark and the oracle's checks.  It
holds no step of the method itself: only random draws with fixed
distributions, shapes and structure.

Recipe (every tensor has its own generator stream, derived from the seed):
  U ~ N(0, 1)                       [T, h]    activation dtype (bf16 by RNE)
  W_r, W_noise ~ N(0, 0.02)         [h, E]    activation dtype
  W_gate, W_up ~ N(0, 0.02)         [E, d_e, h]  (drawn expert by expert)
  W_down ~ N(0, 0.02)               [E, h, d_e]
  eps ~ N(0, 1)                     [T, E]    fp32 (noisy router only)
  b_r (per-expert logit bias)       [E]       fp32
      zipf:   b_e = 1.5 * ln p(e+1), p(r) = r^-1.1 / sum_{r'<=E} r'^-1.1
      normal: b_e ~ N(0, 0.5)
  sel_bias (loss-free selection)    [E]       fp32, normal: N(0, 0.05)
  W_gate_sh, W_up_sh ~ N(0, 0.02)   [n_shared, d_shared, h]  (shared experts)
  W_down_sh ~ N(0, 0.02)            [n_shared, h, d_shared]
Draws use torch's own generator on the device the tensors live on (Philox on
CUDA, Mersenne twister on the CPU), so a given seed yields one fixed set of
inputs per device type; a check always hands the oracle a copy of the exact
tensors the library saw.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

from .workloads import Workload

_MASK63 = (1 << 63) - 1

_STREAM = {
    "U": 1, "W_r": 2, "W_noise": 3, "eps": 4, "b_r": 5,
    "W_gate": 10, "W_up": 11, "W_down": 12,
    "redraw_U": 20, "redraw_eps": 21, "sel_bias": 6,
    "W_gate_sh": 13, "W_up_sh": 14, "W_down_sh": 15,
    "logits": 30, "routing": 31, "gates": 32, "Y": 33, "X": 34,
}


def _seed_of(seed: int, stream: str, sub: int = 0) -> int:
    s = (seed * 0x9E3779B97F4A7C15 + _STREAM[stream] * 0xBF58476D1CE4E5B9
         + sub * 0x94D049BB133111EB + 0x2545F4914F6CDD1D) & ((1 << 64) - 1)
    s ^= s >> 31
    return s & _MASK63


def generator(device, seed: int, stream: str, sub: int = 0) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(_seed_of(seed, stream, sub))
    return g


def normal(shape, std: float, seed: int, stream: str, device, dtype, sub: int = 0) -> torch.Tensor:
    g = generator(device, seed, stream, sub)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x if dtype == torch.float32 else x.to(dtype)


@dataclasses.dataclass
class LayerInputs:
    U: torch.Tensor
    W_r: torch.Tensor
    b_r: Optional[torch.Tensor]
    W_noise: Optional[torch.Tensor]
    eps: Optional[torch.Tensor]
    W_gate: Optional[torch.Tensor]
    W_up: Optional[torch.Tensor]
    W_down: Optional[torch.Tensor]
    sel_bias: Optional[torch.Tensor] = None
    W_gate_sh: Optional[torch.Tensor] = None
    W_up_sh: Optional[torch.Tensor] = None
    W_down_sh: Optional[torch.Tensor] = None

    @property
    def shared(self):
        """(W_gate_sh, W_up_sh, W_down_sh), or None without shared experts."""
        return None if self.W_gate_sh is None else (self.W_gate_sh, self.W_up_sh, self.W_down_sh)

    def to(self, device) -> "LayerInputs":
        return LayerInputs(**{f.name: (None if getattr(self, f.name) is None
                                       else getattr(self, f.name).to(device))
                              for f in dataclasses.fields(self)})


def logit_bias(w: Workload, seed: int, device) -> Optional[torch.Tensor]:
    if w.bias == "none":
        return None
    if w.bias == "zipf":
        z = sum(r ** -1.1 for r in range(1, w.E + 1))
        vals = [1.5 * (math.log(r ** -1.1) - math.log(z)) for r in range(1, w.E + 1)]
        return torch.tensor(vals, dtype=torch.float32, device=device)
    if w.bias == "normal":
        return normal((w.E,), 0.5, seed, "b_r", device, torch.float32)
    raise ValueError(f"unknown bias kind {w.bias!r}")


def generate(w: Workload, seed: int = 0, device="cpu", experts: bool = True) -> LayerInputs:
    """Draw one layer's inputs and weights on `device`."""
    dt = w.torch_dtype
    std = w.weight_std
    U = normal((w.T, w.h), 1.0, seed, "U", device, dt)
    W_r = normal((w.h, w.E), std, seed, "W_r", device, dt)
    b_r = logit_bias(w, seed, device)
    W_noise = eps = None
    if w.noisy:
        W_noise = normal((w.h, w.E), std, seed, "W_noise", device, dt)
        eps = normal((w.T, w.E), 1.0, seed, "eps", device, torch.float32)
    W_gate = W_up = W_down = None
    if experts:
        W_gate = torch.empty((w.E, w.d_e, w.h), dtype=dt, device=device)
        W_up = torch.empty((w.E, w.d_e, w.h), dtype=dt, device=device)
        W_down = torch.empty((w.E, w.h, w.d_e), dtype=dt, device=device)
        for e in range(w.E):  # expert by expert bounds the fp32 scratch of the draw
            W_gate[e] = normal((w.d_e, w.h), std, seed, "W_gate", device, dt, sub=e)
            W_up[e] = normal((w.d_e, w.h), std, seed, "W_up", device, dt, sub=e)
            W_down[e] = normal((w.h, w.d_e), std, seed, "W_down", device, dt, sub=e)
    sel_bias = normal((w.E,), 0.05, seed, "sel_bias", device, torch.float32) if w.sel_bias == "normal" else None
    if w.sel_bias not in ("none", "normal"):
        raise ValueError(f"unknown selection bias kind {w.sel_bias!r}")
    sh = [None, None, None]
    if experts and w.n_shared > 0:
        sh[0] = torch.empty((w.n_shared, w.d_shared, w.h), dtype=dt, device=device)
        sh[1] = torch.empty((w.n_shared, w.d_shared, w.h), dtype=dt, device=device)
        sh[2] = torch.empty((w.n_shared, w.h, w.d_shared), dtype=dt, device=device)
        for i in range(w.n_shared):
            sh[0][i] = normal((w.d_shared, w.h), std, seed, "W_gate_sh", device, dt, sub=i)
            sh[1][i] = normal((w.d_shared, w.h), std, seed, "W_up_sh", device, dt, sub=i)
            sh[2][i] = normal((w.h, w.d_shared), std, seed, "W_down_sh", device, dt, sub=i)
    return LayerInputs(U, W_r, b_r, W_noise, eps, W_gate, W_up, W_down, sel_bias, *sh)


def redraw_rows(inp: LayerInputs, rows: torch.Tensor, seed: int, attempt: int) -> None:
    """Replace the given token rows of U (and of eps) by fresh draws, in place."""
    if rows.numel() == 0:
        return
    dev = inp.U.device
    rows = rows.to(dev)
    n = int(rows.numel())
    inp.U[rows] = normal((n, inp.U.shape[1]), 1.0, seed, "redraw_U", dev, inp.U.dtype, sub=attempt)
    if inp.eps is not None:
        inp.eps[rows] = normal((n, inp.eps.shape[1]), 1.0, seed, "redraw_eps", dev,
                               torch.float32, sub=attempt)


def random_logits(T: int, E: int, seed: int, device="cpu", scale: float = 1.0,
                  tie_fraction: float = 0.25) -> torch.Tensor:
    """fp32 logits [T, E] with exact ties planted in a fraction of the rows.

    In a tied row a few entries are copied onto other positions, so the
    selection has to break equal values; the last rows (if T >= 4) are
    entirely constant.
    """
    g = generator("cpu", seed, "logits")
    x = torch.randn((T, E), generator=g, dtype=torch.float32) * scale
    n_tied = int(T * tie_fraction)
    if n_tied and E > 1:
        rows = torch.randperm(T, generator=g)[:n_tied]
        for r in rows.tolist():
            n_copy = int(torch.randint(1, max(2, E // 2), (1,), generator=g))
            src = torch.randint(0, E, (n_copy,), generator=g)
            dst = torch.randint(0, E, (n_copy,), generator=g)
            x[r, dst] = x[r, src]
    if T >= 4:
        x[-2:] = 0.5
    return x.to(device)


def random_routing(T: int, E: int, k: int, seed: int, device="cpu", zipf_s: float = 0.0) -> torch.Tensor:
    """idx [T, k] int32: k distinct experts per token, drawn without replacement.

    zipf_s = 0 gives uniform choices; zipf_s > 0 weights expert e by (e+1)^-s
    so that low-numbered experts are hot (and overflow their capacity).
    """
    g = generator("cpu", seed, "routing")
    w = torch.arange(1, E + 1, dtype=torch.float64) ** (-zipf_s)
    probs = (w / w.sum()).expand(T, E).contiguous()
    idx = torch.multinomial(probs, k, replacement=False, generator=g)
    return idx.to(torch.int32).to(device)


def random_gates(T: int, k: int, seed: int, device="cpu") -> torch.Tensor:
    g = generator("cpu", seed, "gates")
    return (torch.rand((T, k), generator=g, dtype=torch.float32) + 0.05).to(device)


def random_rows(n: int, h: int, seed: int, stream: str, device, dtype) -> torch.Tensor:
    return normal((n, h), 1.0, seed, stream, device, dtype)

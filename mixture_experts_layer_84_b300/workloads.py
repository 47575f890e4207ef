"""The synthetic MoE-layer workloads, in the pages' notation.

T tokens, hidden size h, E routed experts, top-k, expert intermediate size d_e,
capacity factor CF (<= 0 means no capacity limit), score function, whether the
selected gates are renormalised, whether the router is the noisy top-k router,
and the kind of per-expert logit bias that skews the load.

The shapes follow the model tables of "MoE 与专家并行" (hs-black.github.io/posts/
scaling-moe), section 细粒度专家与共享专家 (Mixtral 8x7B: 8 experts, top-2,
d_e 14336; DeepSeek-V3: 256 routed experts, top-8, d_e 2048) and the Switch
(k=1) / noisy top-k routers of its section 路由器：打分、top-k、加权求和.

Each full-size workload has a reduced twin with the same E, k, score function,
precision and capacity rule, small enough for the plain CPU oracle to finish in
seconds, while still spanning several 128-row tiles, ragged expert segments
and (for some) a ragged d_e tail.
"""
from __future__ import annotations

import dataclasses

SOFTMAX = 0
SIGMOID = 1
PRIORITY_CHOICE_MAJOR = 0
PRIORITY_TOKEN_MAJOR = 1
F32 = 0
BF16 = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    h: int
    E: int
    k: int
    d_e: int
    dtype: int            # F32 or BF16 (activations and weights)
    score_fn: int         # SOFTMAX or SIGMOID
    renorm: bool          # renormalise the k selected gates to sum 1
    noisy: bool           # noisy top-k router (logits + N(0,1)*softplus(U W_noise))
    capacity_factor: float  # <= 0: unbounded
    bias: str = "none"    # per-expert router logit bias: none | zipf | normal
    capacity: int = 0     # > 0 overrides the capacity formula
    priority: int = PRIORITY_CHOICE_MAJOR
    weight_std: float = 0.02
    n_shared: int = 0     # shared experts (every token, outside the router)
    d_shared: int = 0     # their intermediate size
    sel_bias: str = "none"  # loss-free selection bias: none | normal
    n_group: int = 0      # group-limited routing: experts in n_group contiguous groups (0 = off)
    topk_group: int = 0   # groups a token may use

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def torch_dtype(self):
        import torch
        return torch.float32 if self.dtype == F32 else torch.bfloat16

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == F32 else 2


# The five layer shapes.
TINY_FP32 = Workload("tiny_fp32", T=256, h=128, E=8, k=2, d_e=256, dtype=F32,
                     score_fn=SOFTMAX, renorm=True, noisy=False, capacity_factor=1.25)
MIXTRAL = Workload("mixtral_bf16", T=2048, h=4096, E=8, k=2, d_e=14336, dtype=BF16,
                   score_fn=SOFTMAX, renorm=True, noisy=False, capacity_factor=1.25)
SWITCH = Workload("switch_noisy_bf16", T=16384, h=1024, E=128, k=1, d_e=4096, dtype=BF16,
                  score_fn=SOFTMAX, renorm=False, noisy=True, capacity_factor=1.0, bias="zipf")
DSV3 = Workload("dsv3_bf16", T=4096, h=7168, E=256, k=8, d_e=2048, dtype=BF16,
                score_fn=SIGMOID, renorm=True, noisy=False, capacity_factor=0.0, bias="normal")
STRESS = Workload("stress_bf16", T=65536, h=4096, E=64, k=6, d_e=1408, dtype=BF16,
                  score_fn=SOFTMAX, renorm=True, noisy=False, capacity_factor=2.0)

FULL = [TINY_FP32, MIXTRAL, SWITCH, DSV3, STRESS]

# DeepSeek-V3's full MoE block: the DS-V3 shape plus its one shared expert (d = 2048), a
# loss-free balancing bias on the selection, and group-limited routing with its 8 groups of 32
# experts, 4 kept per token ("MoE 与专家并行", sections 细粒度专家与共享专家,
# 无辅助损失的负载均衡 and 设备受限与节点受限路由, the node limit M = 4 read as expert groups).
DSV3_SHARED = DSV3.replace(name="dsv3_shared_bf16", n_shared=1, d_shared=2048, sel_bias="normal",
                           n_group=8, topk_group=4)
DSV3_SHARED_SMALL = DSV3_SHARED.replace(name="dsv3_shared_small", T=600, h=512, d_e=256, d_shared=384)
EXTENDED = [DSV3_SHARED]

# Reduced twins (same routing rule and precision, oracle-sized).
MIXTRAL_SMALL = MIXTRAL.replace(name="mixtral_small", T=700, h=512, d_e=640)
SWITCH_SMALL = SWITCH.replace(name="switch_small", T=3000, h=256, d_e=384)
DSV3_SMALL = DSV3.replace(name="dsv3_small", T=600, h=512, d_e=256)
STRESS_SMALL = STRESS.replace(name="stress_small", T=3000, h=256, d_e=192)

SMALL = [TINY_FP32, MIXTRAL_SMALL, SWITCH_SMALL, DSV3_SMALL, STRESS_SMALL]

# Mixtral-shaped with a quarter of d_e: the same kernels and tiles with about
# 1 GB on the device, for detailed hardware-counter captures.
MIXTRAL_NARROW = MIXTRAL.replace(name="mixtral_narrow_bf16", d_e=3584)
# The Switch shape with a quarter of d_e (the same 128 segments of at most 128 tokens, 0.8 GB of
# expert weights) and the stress shape with 12288 tokens (segments of about 1150 rows, the CTA-pair
# row tiles, 3.5 GB on the device): small cases of those kernels for hardware-counter captures.
SWITCH_NARROW = SWITCH.replace(name="switch_narrow_bf16", d_e=1024)
STRESS_NARROW = STRESS.replace(name="stress_narrow_bf16", T=12288)
# The 256-expert shape with d_e = 64: the same router, dispatch and combine with 2 GB on the device.
DSV3_NARROW = DSV3.replace(name="dsv3_narrow_bf16", d_e=64)
NARROW = [MIXTRAL_NARROW, SWITCH_NARROW, STRESS_NARROW, DSV3_NARROW]

BY_NAME = {w.name: w for w in FULL + SMALL + EXTENDED + NARROW + [DSV3_SHARED_SMALL]}


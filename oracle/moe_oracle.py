"""Plain CPU oracle for the single-GPU MoE layer forward.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import or run this module; the library never does.  It
shares no code with the CUDA path: it is the method's definition written out
in float64 numpy, step by step, in the order and notation of the pages.

Sources (page title, section):
  [FFN]  "MoE 与专家并行" (hs-black.github.io/posts/scaling-moe), 从稠密 FFN 到 MoE:
         SwiGLU FFN(u) = W_down (SiLU(W_gate u) ⊙ W_up u);
         layer output h'_t = u_t + sum_i g_{i,t} FFN_i(u_t), g = 0 off the top-k.
  [RTR]  same page, 路由器：打分、top-k、加权求和: H = U W_r; score s = softmax or
         sigmoid of H; top-k set T_t; gates from the selected scores; the
         noisy top-k logits H_i = (x W_g)_i + N(0,1) * Softplus((x W_noise)_i);
         the single-GPU shapes listing (permute by expert, grouped FFN,
         index_add back into token order).
  [SCR]  same page, softmax 门控还是 sigmoid 门控: the scoring table (softmax
         then top-k without renormalisation; softmax then renormalise over the
         selected; top-k then softmax; sigmoid then renormalise) and the
         identity top-k-then-softmax == softmax-then-renormalise.
  [CAP]  same page, 专家容量与丢 token: C = ceil(CF * T * k / E); slots are
         filled in token order, overflow is dropped and takes the residual
         only; for top-k every token's first choice is placed before any
         second choice.
  [AUX]  same page, 负载均衡辅助损失：推导与梯度: f_i = fraction of assignments to
         expert i, P_i = (1/T) sum_t s_{i,t}, L_aux = alpha * E * sum_i f_i P_i
         (this oracle reports E * sum f_i P_i, i.e. alpha = 1); for sigmoid
         scores P_i uses s'_{i,t} = s_{i,t} / sum_j s_{j,t}.
  [VIO]  same page, 无辅助损失的负载均衡: MaxVio = (max_i Load_i - mean) / mean.
  [ZL]   same page, Router z-loss 与数值稳定: L_z = (1/T) sum_t (log sum_j e^{H_{t,j}})^2,
         the mean square of each token's log-sum-exp of its router logits.
  [SHR]  same page, 细粒度专家与共享专家 (shared expert isolation, the V3 form):
         h'_t = u_t + sum_{i<=N_s} FFN^(s)_i(u_t) + sum_{i<=N_r} g_{i,t} FFN^(r)_i(u_t);
         the shared experts take every token and bypass the router.
  [LFB]  same page, 无辅助损失的负载均衡: a per-expert bias b_i used only to choose
         the top-k (s_{i,t} + b_i), the gate stays s_{i,t}; after each batch
         e_i = mean(c) - c_i and b_i <- b_i + u * sign(e_i).
  [GRD]  same page, 路由器：打分、top-k、加权求和 (how the router learns): with the
         upstream gradient delta_t = dL/dh'_t, dL/dg_{i,t} = delta_t^T FFN_i(u_t) for
         the selected experts, then through dg/dH to the logits; section
         负载均衡辅助损失：推导与梯度 (梯度往哪推): f is a constant, and
         d(sum_i f_i P_i)/dH_{t,k} = (1/T) s_k (f_k - sum_i f_i s_i) for softmax,
         (1/T) s'_k (1 - s_k) (f_k - sum_i f_i s'_i) for sigmoid; section Router
         z-loss: dL_z/dH_{t,k} = (2/T) LSE(H_t) softmax(H_t)_k.
  [GRP]  same page, 设备受限与节点受限路由 (node-limited routing, the V3 form): a token
         may use the experts of at most M nodes, the nodes being ranked by the sum
         of the K_r/M highest affinities among their experts; the top-k is then
         taken over the experts of the chosen nodes only.  On one GPU the nodes
         become n_group equal, contiguous groups of experts (reading below).
  [FP8]  same page, 低精度通信: DeepSeek-V3 turns the activations that enter the MoE
         up-projection into FP8 before the dispatch, so that they feed the
         up-projection's FP8 forward as they are; the scaling factors are
         integral powers of 2; the combine stays BF16.
  [BWD]  same page, 专家计算：padding、block-sparse 与 grouped GEMM: the backward of
         the SwiGLU experts is grouped GEMMs too, one group for the input
         gradients and one for the weight gradients.

Readings where the pages are silent (the same readings the library follows):
  * selection is made on the float32 logits (softmax and sigmoid are strictly
    increasing, so this is the top-k of the scores without exp-rounding ties);
    ties go to the lower expert id, both for membership and for rank order;
  * the logits are rounded to float32 before selection and scoring (the
    library's logits are float32);
  * "no capacity limit" means C = T (an expert can receive each token once);
  * f_i counts the router's assignments before drops and is normalised by T*k;
  * a dropped assignment contributes nothing and the kept gates are not
    renormalised; rows inside an expert segment are in slot (priority) order;
  * group-limited routing ([GRP]) on one GPU: group q holds experts
    [q*E/n_group, (q+1)*E/n_group); a group's score is the sum of its
    r = k/topk_group highest affinities (the scores s, or s + b with a
    loss-free selection bias); the topk_group best groups are kept, ties to
    the lower group id; the top-k is then taken over the kept groups' experts
    only (by the usual selection key).  Group selection adds no gradient path;
  * FP8 ([FP8]) is E4M3 (finite, largest 448, round to nearest even).  Every
    token row of U and every row (output channel) of W_gate and W_up gets one
    power-of-two scale 2^s, s the smallest integer >= -127 with
    amax <= 448 * 2^s; codes = E4M3(x * 2^-s).  The up-projection (gate|up)
    multiplies the dequantised values codes * 2^s exactly; act, the down
    projection, the shared experts and the combine stay at the layer's
    precision (bf16).

Every function here is pinned by the `-m "not gpu"` tests (worked examples of
the pages, closed forms, invariants, brute force and textbook special cases).
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

SOFTMAX = 0
SIGMOID = 1
CHOICE_MAJOR = 0
TOKEN_MAJOR = 1


def f64(a) -> np.ndarray:
    """Exact float64 copy of a numpy array or (CPU/GPU) torch tensor of any float type."""
    if hasattr(a, "detach"):
        import torch
        a = a.detach().to("cpu")
        if a.dtype in (torch.bfloat16, torch.float16):
            a = a.to(torch.float32)
        a = a.numpy()
    return np.asarray(a, dtype=np.float64)


# --------------------------------------------------------------------------
# Router  [RTR]
# --------------------------------------------------------------------------

def softplus(x: np.ndarray) -> np.ndarray:
    """Softplus(x) = ln(1 + e^x), written in the overflow-free form."""
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


def router_logits(U, W_r, b_r=None, W_noise=None, eps=None) -> np.ndarray:
    """Router logits H = U W_r (+ per-expert bias) (+ noisy-top-k noise), float64.

    [RTR]: H = U W_r with W_r in R^{h x E}; the noisy router adds
    N(0,1) * Softplus(U W_noise), with the standard-normal draws eps [T, E]
    passed in.  The bias b_r [E] is an additive per-expert logit offset.
    """
    U = f64(U)
    H = U @ f64(W_r)
    if b_r is not None:
        H = H + f64(b_r)[None, :]
    if W_noise is not None:
        H = H + f64(eps) * softplus(U @ f64(W_noise))
    return H


def round_f32(H: np.ndarray) -> np.ndarray:
    """Round to float32 (returned as float64 holding float32 values)."""
    return np.asarray(H, dtype=np.float32).astype(np.float64)


def topk_select(H32: np.ndarray, k: int, allowed=None) -> np.ndarray:
    """Top-k expert ids per token, highest first, ties to the lower expert id.

    [RTR] step 2 (select the k highest); the stable sort keeps equal values in
    increasing expert order.  `allowed` [T, E] (group-limited routing) puts
    every allowed expert ahead of every other one, whatever the values.
    """
    key = -np.asarray(H32, dtype=np.float64)
    if allowed is None:
        order = np.argsort(key, axis=1, kind="stable")
    else:
        order = np.lexsort((key, ~np.asarray(allowed, dtype=bool)), axis=-1)  # lexsort is stable
    return order[:, :k].astype(np.int32)


def group_scores(aff: np.ndarray, n_group: int, r: int) -> np.ndarray:
    """[T, n_group]: each contiguous expert group's sum of its r highest affinities.  [GRP]"""
    aff = np.asarray(aff, dtype=np.float64)
    T, E = aff.shape
    grouped = -np.sort(-aff.reshape(T, n_group, E // n_group), axis=2)
    return grouped[:, :, :r].sum(axis=2)


def group_limited_mask(aff: np.ndarray, n_group: int, topk_group: int, k: int) -> np.ndarray:
    """[T, E] bool: the experts of each token's topk_group highest-scoring groups.

    [GRP]: groups ranked by the sum of their k/topk_group highest affinities,
    ties to the lower group id.
    """
    T, E = np.asarray(aff).shape
    gs = group_scores(aff, n_group, k // topk_group)
    best = np.argsort(-gs, axis=1, kind="stable")[:, :topk_group]
    chosen = np.zeros(gs.shape, dtype=bool)
    np.put_along_axis(chosen, best, True, axis=1)
    return np.repeat(chosen, E // n_group, axis=1)


def scores(H: np.ndarray, score_fn: int) -> np.ndarray:
    """Affinities s_{i,t}: softmax over the E experts or independent sigmoids.  [RTR] step 1, [SCR]."""
    H = np.asarray(H, dtype=np.float64)
    if score_fn == SOFTMAX:
        z = np.exp(H - H.max(axis=1, keepdims=True))
        return z / z.sum(axis=1, keepdims=True)
    if score_fn == SIGMOID:
        return 1.0 / (1.0 + np.exp(-H))
    raise ValueError("score_fn")


def gates(s: np.ndarray, idx: np.ndarray, renorm: bool) -> np.ndarray:
    """Gate values of the selected experts, [T, k].

    [SCR]: g_i = s_i / sum_{j in T_t} s_j when renormalised, g_i = s_i otherwise.
    """
    sel = np.take_along_axis(s, np.asarray(idx, dtype=np.int64), axis=1)
    if renorm:
        return sel / sel.sum(axis=1, keepdims=True)
    return sel


# --------------------------------------------------------------------------
# Capacity and dispatch  [CAP]
# --------------------------------------------------------------------------

def capacity(T: int, E: int, k: int, capacity_factor: float, override: int = 0) -> int:
    """C = ceil(CF * T * k / E), exact on the float32 value of CF; CF <= 0: C = T."""
    if override > 0:
        return int(override)
    if capacity_factor <= 0:
        return int(T)
    cf = Fraction(float(np.float32(capacity_factor)))
    return int(math.ceil(cf * T * k / E))


def priority_order(T: int, k: int, priority: int):
    """The (token, choice) pairs in the order their slots are filled.

    [CAP]: every token's first choice before any second choice (choice-major,
    tokens in order within a choice); token-major takes a token's choices
    together.
    """
    if priority == CHOICE_MAJOR:
        j, t = np.meshgrid(np.arange(k), np.arange(T), indexing="ij")
    elif priority == TOKEN_MAJOR:
        t, j = np.meshgrid(np.arange(T), np.arange(k), indexing="ij")
    else:
        raise ValueError("priority")
    return t.reshape(-1), j.reshape(-1)


def dispatch(idx: np.ndarray, E: int, C: int, priority: int = CHOICE_MAJOR) -> dict:
    """Capacity-limited assignment of (token, choice) pairs to expert slots.

    [CAP] + the permute of [RTR]'s shapes listing: walking the pairs in
    priority order, the n-th pair that chose expert e takes slot n of e; it is
    kept iff n < C.  Kept rows are packed expert by expert (offsets = the
    exclusive prefix sum of the kept counts) in slot order, so the row of a
    kept pair is offsets[e] + slot and row_token[row] is its token.
    Returns counts_routed [E], counts_kept [E], offsets [E+1], slot [T*k]
    (slot of pair t*k+j), slot_row [T*k] (-1 when dropped), row_token [A],
    n_dropped.
    """
    idx = np.asarray(idx, dtype=np.int64)
    T, k = idx.shape
    t_seq, j_seq = priority_order(T, k, priority)
    e_seq = idx[t_seq, j_seq]
    counts_routed = np.bincount(e_seq, minlength=E).astype(np.int64)
    # rank of each pair among the earlier pairs of the same expert (stable sort keeps priority order)
    grouped = np.argsort(e_seq, kind="stable")
    first = np.concatenate([[0], np.cumsum(counts_routed)[:-1]])
    rank = np.empty(T * k, dtype=np.int64)
    rank[grouped] = np.arange(T * k) - first[e_seq[grouped]]
    counts_kept = np.minimum(counts_routed, C)
    offsets = np.concatenate([[0], np.cumsum(counts_kept)]).astype(np.int64)
    pair = t_seq * k + j_seq
    slot = np.empty(T * k, dtype=np.int64)
    slot[pair] = rank
    kept = rank < C
    slot_row = np.full(T * k, -1, dtype=np.int64)
    slot_row[pair[kept]] = offsets[e_seq[kept]] + rank[kept]
    A = int(offsets[E])
    row_token = np.full(A, -1, dtype=np.int64)
    row_token[slot_row[pair[kept]]] = t_seq[kept]
    return dict(counts_routed=counts_routed, counts_kept=counts_kept, offsets=offsets,
                slot=slot, slot_row=slot_row, row_token=row_token,
                n_dropped=int(T * k - A), C=int(C))


def permute(U, row_token: np.ndarray) -> np.ndarray:
    """X = U[row_token]: the expert inputs, contiguous per expert.  [RTR] shapes listing."""
    return f64(U)[np.asarray(row_token, dtype=np.int64)]


# --------------------------------------------------------------------------
# Experts and combine  [FFN]
# --------------------------------------------------------------------------

def silu(x: np.ndarray) -> np.ndarray:
    """SiLU(x) = x * sigmoid(x)."""
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def swiglu(x, W_gate_e, W_up_e, W_down_e):
    """One expert on rows x [n, h]: returns (FFN(x) [n, h], the SiLU(gate)*up activation [n, d_e]).

    [FFN]: FFN(u) = W_down (SiLU(W_gate u) ⊙ W_up u), W_gate, W_up in R^{d_e x h},
    W_down in R^{h x d_e}.
    """
    x = f64(x)
    a = silu(x @ f64(W_gate_e).T) * (x @ f64(W_up_e).T)
    return a @ f64(W_down_e).T, a


def expert_ffn(X, offsets, W_gate, W_up, W_down, d_e: int):
    """Y = the grouped FFN over the expert segments of X (rows offsets[e]..offsets[e+1]).

    [RTR] shapes listing (grouped_ffn) with [FFN]'s expert.
    """
    X = f64(X)
    offsets = np.asarray(offsets, dtype=np.int64)
    E = len(offsets) - 1
    Y = np.zeros((X.shape[0], X.shape[1]))
    act = np.zeros((X.shape[0], d_e))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            Y[lo:hi], act[lo:hi] = swiglu(X[lo:hi], W_gate[e], W_up[e], W_down[e])
    return Y, act


# --------------------------------------------------------------------------
# FP8 dispatch and up-projection  [FP8]
# --------------------------------------------------------------------------

E4M3_MAX = 448.0


def e4m3_round(x) -> np.ndarray:
    """Nearest E4M3 value, ties to even, saturating at +-448.

    E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no
    infinities.  In the binade [2^e, 2^(e+1)), e >= -6, neighbours are
    2^(e-3) apart; below 2^-6 the subnormals are 2^-9 apart.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, E = np.frexp(a)                      # a = m 2^E, m in [0.5, 1): binade e = E - 1
    e = np.maximum(E - 1, -6)
    quantum = np.ldexp(1.0, e - 3)
    r = np.minimum(np.round(a / quantum) * quantum, E4M3_MAX)  # np.round: half to even
    return np.copysign(r, x)


def e4m3_bits(v) -> np.ndarray:
    """The 8-bit codes (sign | exponent field << 3 | mantissa) of E4M3 values."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, E = np.frexp(a)
    e = E - 1
    normal = a >= 2.0 ** -6
    field = np.where(normal, e + 7, 0)
    mant = np.where(normal, (np.ldexp(a, -np.where(normal, e, 0)) - 1.0) * 8.0, a * 2.0 ** 9)
    sign = np.signbit(v).astype(np.int64) << 7
    return (sign | (field.astype(np.int64) << 3) | mant.astype(np.int64)).astype(np.uint8)


def pow2_scale_exponents(amax) -> np.ndarray:
    """Per row, the smallest integer s >= -127 with amax <= 448 * 2^s (-127 when amax = 0).

    With amax = m 2^E, m in [0.5, 1), and 448 = 0.875 * 2^9: s = E - 9, plus 1 when m > 0.875.
    """
    amax = np.asarray(amax, dtype=np.float64)
    m, E = np.frexp(amax)
    s = E - 9 + (m > 0.875).astype(np.int64)
    return np.where(amax > 0, np.maximum(s, -127), -127).astype(np.int64)


def quantize_rows_fp8(A):
    """Row-wise E4M3 with one power-of-two scale per row: (codes [n, c], s [n]), A ~ codes * 2^s."""
    A = f64(A)
    amax = np.max(np.abs(A), axis=1) if A.shape[1] else np.zeros(A.shape[0])
    s = pow2_scale_exponents(amax)
    return e4m3_round(np.ldexp(A, -s[:, None])), s


def dequantize_rows_fp8(codes, s) -> np.ndarray:
    return np.ldexp(f64(codes), np.asarray(s, dtype=np.int64)[:, None])


def fp8_weights(W) -> np.ndarray:
    """[E, d, h] weights as the FP8 up-projection sees them: each row quantised and dequantised."""
    out = np.empty(tuple(W.shape), dtype=np.float64)
    for e in range(W.shape[0]):
        out[e] = dequantize_rows_fp8(*quantize_rows_fp8(W[e]))
    return out


def shared_ffn(U, W_gate_sh, W_up_sh, W_down_sh) -> np.ndarray:
    """Y_sh [N_s, T, h]: each shared expert's SwiGLU FFN on every token.  [SHR], [FFN]"""
    U = f64(U)
    n_s = len(W_gate_sh)
    Y = np.zeros((n_s,) + U.shape)
    for i in range(n_s):
        Y[i], _ = swiglu(U, W_gate_sh[i], W_up_sh[i], W_down_sh[i])
    return Y


def combine(U, Y, slot_row, gate, k: int, Y_shared=None) -> np.ndarray:
    """out_t = u_t + sum_s Y_shared[s, t] + sum_j g_{j,t} Y[row of (t, j)], kept pairs only, j ascending.

    [FFN] layer output with [RTR]'s index_add back into token order; a dropped
    pair adds nothing (its token keeps the residual only, [CAP]); [SHR] the
    shared experts' outputs enter with weight 1.
    """
    out = f64(U).copy()
    if Y_shared is not None:
        for ys in f64(Y_shared):
            out += ys
    T = out.shape[0]
    sr = np.asarray(slot_row, dtype=np.int64).reshape(T, k)
    g = f64(gate).reshape(T, k)
    Y = f64(Y)
    for j in range(k):
        m = sr[:, j] >= 0
        out[m] += g[m, j][:, None] * Y[sr[m, j]]
    return out


# --------------------------------------------------------------------------
# Load statistics  [AUX], [VIO]
# --------------------------------------------------------------------------

def load_stats(counts_routed, s: np.ndarray, T: int, k: int, score_fn: int) -> dict:
    """f_i, P_i, E * sum_i f_i P_i and MaxVio.  [AUX], [VIO]."""
    counts_routed = np.asarray(counts_routed, dtype=np.float64)
    E = counts_routed.shape[0]
    f = counts_routed / (T * k)
    sp = s / s.sum(axis=1, keepdims=True) if score_fn == SIGMOID else s
    P = sp.sum(axis=0) / T
    aux = E * float((f * P).sum())
    mean = counts_routed.mean()
    maxvio = float((counts_routed.max() - mean) / mean) if mean > 0 else 0.0
    return dict(f=f, P=P, aux=aux, maxvio=maxvio)


def router_z_loss(H) -> float:
    """L_z = (1/T) sum_t LSE(H_t)^2 with LSE(x) = log sum_j e^{x_j}.  [ZL]

    The log-sum-exp is taken in the max-shifted form m + log sum_j e^{x_j - m}.
    """
    H = np.asarray(H, dtype=np.float64)
    T = H.shape[0]
    if T == 0:
        return 0.0
    m = H.max(axis=1)
    lse = m + np.log(np.exp(H - m[:, None]).sum(axis=1))
    return float((lse ** 2).sum() / T)


# --------------------------------------------------------------------------
# The whole layer
# --------------------------------------------------------------------------

def balance_bias_update(b, counts_routed, u: float) -> np.ndarray:
    """One step of the loss-free balancing bias: e_i = mean(c) - c_i, b_i <- b_i + u * sign(e_i).  [LFB]"""
    c = np.asarray(counts_routed, dtype=np.float64)
    e = c.mean() - c
    return f64(b) + u * np.sign(e)


def route(H, k: int, score_fn: int, renorm: bool, sel_bias=None, n_group: int = 1, topk_group: int = 1) -> dict:
    """From logits to (idx, gates, scores): rounding to fp32, selection, scoring, gates.

    Without a selection bias the top-k is taken on the logits (the same order
    as on the scores).  With one ([LFB]) it is taken on s + b, while the gates
    still come from s; "sel_key" holds s + b.  With n_group > 1 the top-k is
    limited to the experts of the topk_group best groups ([GRP]), the groups
    being scored on the affinities s (s + b with a selection bias); "allowed"
    holds that [T, E] mask (None without groups).
    """
    H32 = round_f32(H)
    s = scores(H32, score_fn)
    key = H32 if sel_bias is None else s + f64(sel_bias)[None, :]
    allowed = None
    if n_group > 1:
        allowed = group_limited_mask(s if sel_bias is None else key, n_group, topk_group, k)
    idx = topk_select(key, k, allowed)
    return dict(logits=H32, idx=idx, s=s, gate=gates(s, idx, renorm), sel_key=key, allowed=allowed)


def layer_forward(inp, *, T, h, E, k, d_e, score_fn, renorm, capacity_factor,
                  capacity_override=0, priority=CHOICE_MAJOR, logits=None, sel_bias=None, shared=None,
                  n_group=1, topk_group=1, fp8=False) -> dict:
    """The full single-GPU MoE layer forward, stage by stage, in float64.

    `inp` carries U, W_r, b_r, W_noise, eps, W_gate, W_up, W_down (numpy or
    torch).  If `logits` is given the router GEMM is skipped and those logits
    are used as they are.  `sel_bias` [E] is the loss-free selection bias
    ([LFB]); `shared` = (W_gate_sh, W_up_sh, W_down_sh) adds shared experts
    ([SHR]); n_group > 1 limits each token to topk_group expert groups ([GRP]);
    fp8 runs the dispatch and the up-projection on E4M3 codes ([FP8]): X holds
    the dequantised token rows, and "U_codes", "U_s" the quantised U.
    """
    H = router_logits(inp.U, inp.W_r, inp.b_r, inp.W_noise, inp.eps) if logits is None else f64(logits)
    r = route(H, k, score_fn, renorm, sel_bias, n_group, topk_group)
    C = capacity(T, E, k, capacity_factor, capacity_override)
    d = dispatch(r["idx"], E, C, priority)
    extra = {}
    if fp8:
        codes, s_u = quantize_rows_fp8(inp.U)
        X = permute(dequantize_rows_fp8(codes, s_u), d["row_token"])
        Y, act = expert_ffn(X, d["offsets"], fp8_weights(inp.W_gate), fp8_weights(inp.W_up), inp.W_down, d_e)
        extra = dict(U_codes=codes, U_s=s_u)
    else:
        X = permute(inp.U, d["row_token"])
        Y, act = expert_ffn(X, d["offsets"], inp.W_gate, inp.W_up, inp.W_down, d_e)
    Y_sh = None if shared is None else shared_ffn(inp.U, *shared)
    out = combine(inp.U, Y, d["slot_row"], r["gate"], k, Y_sh)
    st = load_stats(d["counts_routed"], r["s"], T, k, score_fn)
    return dict(r, **d, X=X, act=act, Y=Y, Y_shared=Y_sh, out=out, z_loss=router_z_loss(r["logits"]), **st,
                **extra)


def sampled_outputs(inp, tokens, idx, gate, slot_row, k: int, shared=None, fp8=False) -> dict:
    """out rows (and the Y rows they use) for a sample of tokens.

    For full-size checks: X[row] = U[t] for a kept pair, so each needed Y row
    is one expert applied to one token row ([FFN]); out follows [FFN]'s layer
    output.  The sampled rows are grouped by expert so that each expert's
    weights are read (and widened to float64) once.
    With `shared` the shared experts' outputs ([SHR]) are added too; with
    `fp8` the experts see the E4M3 token rows and gate/up weights ([FP8]).
    Returns {"out": [n, h], "Y": {row: [h]}}.
    """
    tokens = [int(t) for t in tokens]
    idx = np.asarray(idx, dtype=np.int64)
    gate = f64(gate)
    sr = np.asarray(slot_row, dtype=np.int64).reshape(-1, k)
    U = {t: f64(inp.U[t]) for t in tokens}
    by_expert = {}
    for t in tokens:
        for j in range(k):
            if sr[t, j] >= 0:
                by_expert.setdefault(int(idx[t, j]), []).append((t, j))
    y_of = {}
    for e, pairs in sorted(by_expert.items()):
        x = np.stack([U[t] for t, _ in pairs])
        if fp8:
            x = dequantize_rows_fp8(*quantize_rows_fp8(x))
            y, _ = swiglu(x, dequantize_rows_fp8(*quantize_rows_fp8(inp.W_gate[e])),
                          dequantize_rows_fp8(*quantize_rows_fp8(inp.W_up[e])), inp.W_down[e])
        else:
            y, _ = swiglu(x, inp.W_gate[e], inp.W_up[e], inp.W_down[e])
        for (t, j), row in zip(pairs, y):
            y_of[(t, j)] = row
    outs, Yrows = [], {}
    sh = {}
    if shared is not None and tokens:
        ysh = shared_ffn(np.stack([U[t] for t in tokens]), *shared).sum(axis=0)
        sh = {t: ysh[i] for i, t in enumerate(tokens)}
    for t in tokens:
        acc = U[t].copy()
        if shared is not None:
            acc = acc + sh[t]
        for j in range(k):
            if sr[t, j] >= 0:
                Yrows[int(sr[t, j])] = y_of[(t, j)]
                acc = acc + gate[t, j] * y_of[(t, j)]
        outs.append(acc)
    return dict(out=np.stack(outs) if outs else np.zeros((0, 0)), Y=Yrows)


# --------------------------------------------------------------------------
# Backward of the router side  [GRD]
# --------------------------------------------------------------------------

def combine_backward(dO, Y, slot_row, gate, k: int) -> dict:
    """Backward of the combine for the upstream gradient dO [T, h].

    out_t = u_t + sum_j g_{t,j} Y[row(t,j)] gives, per kept pair,
    dL/dg_{t,j} = dO_t . Y[row] ([GRD]) and dL/dY[row] = g_{t,j} dO_t;
    dropped pairs get d_gate = 0.  Returns d_gate [T, k] and dY [A, h] (rows of Y).
    """
    dO, Y, g = f64(dO), f64(Y), f64(gate)
    T = dO.shape[0]
    sr = np.asarray(slot_row, dtype=np.int64).reshape(T, k)
    d_gate = np.zeros((T, k))
    dY = np.zeros_like(Y)
    for j in range(k):
        m = sr[:, j] >= 0
        rows = sr[m, j]
        d_gate[m, j] = np.einsum("th,th->t", dO[m], Y[rows])
        dY[rows] = g.reshape(T, k)[m, j][:, None] * dO[m]
    return dict(d_gate=d_gate, dY=dY)


def gate_backward(H32, idx, d_gate, score_fn: int, renorm: bool) -> np.ndarray:
    """dL/dH [T, E] from dL/dg through the gate definition ([SCR], [GRD]).

    softmax:  s = softmax(H); g_j = s_{i_j}, or s_{i_j} / sum_m s_{i_m} with renorm;
    sigmoid:  s = sigmoid(H); the same two forms.  The selection itself is
    not differentiated (the top-k set is held fixed).
    """
    H = np.asarray(H32, dtype=np.float64)
    T, E = H.shape
    idx = np.asarray(idx, dtype=np.int64)
    k = idx.shape[1]
    s = scores(H, score_fn)
    sel = np.take_along_axis(s, idx, axis=1)
    d_gate = f64(d_gate).reshape(T, k)
    # dL/ds_{i_j} (for the selected experts; the other scores do not enter g)
    if renorm:
        S = sel.sum(axis=1, keepdims=True)
        g = sel / S
        # g_j = s_j / S: dg_j/ds_m = (delta_jm - g_j) / S
        ds_sel = (d_gate - (d_gate * g).sum(axis=1, keepdims=True)) / S
    else:
        ds_sel = d_gate
    ds = np.zeros((T, E))
    np.add.at(ds, (np.repeat(np.arange(T), k), idx.reshape(-1)), ds_sel.reshape(-1))
    if score_fn == SOFTMAX:
        # ds_i/dH_k = s_i (delta_ik - s_k)
        return s * (ds - (ds * s).sum(axis=1, keepdims=True))
    return ds * s * (1.0 - s)


def aux_loss_grad(H32, f, score_fn: int) -> np.ndarray:
    """d(E * sum_i f_i P_i)/dH [T, E] with f held constant ([AUX], [GRD])."""
    H = np.asarray(H32, dtype=np.float64)
    T, E = H.shape
    f = np.asarray(f, dtype=np.float64)
    s = scores(H, score_fn)
    if score_fn == SOFTMAX:
        return E / T * s * (f[None, :] - (s * f[None, :]).sum(axis=1, keepdims=True))
    sp = s / s.sum(axis=1, keepdims=True)
    return E / T * sp * (1.0 - s) * (f[None, :] - (sp * f[None, :]).sum(axis=1, keepdims=True))


def z_loss_grad(H32) -> np.ndarray:
    """dL_z/dH [T, E] = (2/T) LSE(H_t) softmax(H_t) ([ZL])."""
    H = np.asarray(H32, dtype=np.float64)
    T = H.shape[0]
    m = H.max(axis=1, keepdims=True)
    lse = m + np.log(np.exp(H - m).sum(axis=1, keepdims=True))
    return 2.0 / T * lse * scores(H, SOFTMAX)


def router_backward(H32, idx, d_gate, f, score_fn: int, renorm: bool, w_aux: float = 0.0,
                    w_z: float = 0.0) -> np.ndarray:
    """dL/dH for L = (the loss through the gates) + w_aux * E sum f P + w_z * L_z."""
    dH = gate_backward(H32, idx, d_gate, score_fn, renorm)
    if w_aux:
        dH = dH + w_aux * aux_loss_grad(H32, f, score_fn)
    if w_z:
        dH = dH + w_z * z_loss_grad(H32)
    return dH


# --------------------------------------------------------------------------
# Backward of the experts and of the dispatch  [BWD], [FFN]
# --------------------------------------------------------------------------

def swiglu_backward(x, W_gate_e, W_up_e, W_down_e, dy) -> dict:
    """Gradients of y = W_down (SiLU(W_gate x) * W_up x) for rows x [n, h] and dL/dy [n, h].

    With G = x W_gate^T, Up = x W_up^T, s = sigmoid(G), a = G s Up:
      d_act = dy W_down, dW_down = dy^T a,
      dUp = d_act * G s, dG = d_act * Up * s (1 + G (1 - s)),
      dx = dG W_gate + dUp W_up, dW_gate = dG^T x, dW_up = dUp^T x.
    """
    x, Wg, Wu, Wd, dy = f64(x), f64(W_gate_e), f64(W_up_e), f64(W_down_e), f64(dy)
    G = x @ Wg.T
    Up = x @ Wu.T
    with np.errstate(over="ignore"):
        sg = 1.0 / (1.0 + np.exp(-G))
    silu_g = G * sg
    act = silu_g * Up
    d_act = dy @ Wd
    dUp = d_act * silu_g
    dG = d_act * Up * sg * (1.0 + G * (1.0 - sg))
    return dict(d_act=d_act, dG=dG, dUp=dUp, dx=dG @ Wg + dUp @ Wu, dW_gate=dG.T @ x, dW_up=dUp.T @ x,
                dW_down=dy.T @ act)


def expert_ffn_backward(X, offsets, W_gate, W_up, W_down, dY, d_e: int) -> dict:
    """The grouped backward over the expert segments: per row d_act, dG, dUp, dX; per expert
    dW_gate [E, d_e, h], dW_up [E, d_e, h], dW_down [E, h, d_e] (zero for an expert with no rows)."""
    X, dY = f64(X), f64(dY)
    offsets = np.asarray(offsets, dtype=np.int64)
    E = len(offsets) - 1
    A, h = X.shape
    out = dict(d_act=np.zeros((A, d_e)), dG=np.zeros((A, d_e)), dUp=np.zeros((A, d_e)), dX=np.zeros((A, h)),
               dW_gate=np.zeros((E, d_e, h)), dW_up=np.zeros((E, d_e, h)), dW_down=np.zeros((E, h, d_e)))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            b = swiglu_backward(X[lo:hi], W_gate[e], W_up[e], W_down[e], dY[lo:hi])
            out["d_act"][lo:hi], out["dG"][lo:hi], out["dUp"][lo:hi] = b["d_act"], b["dG"], b["dUp"]
            out["dX"][lo:hi] = b["dx"]
            out["dW_gate"][e], out["dW_up"][e], out["dW_down"][e] = b["dW_gate"], b["dW_up"], b["dW_down"]
    return out


def dispatch_backward(dO, dX, slot_row, k: int) -> np.ndarray:
    """dL/dU from the residual and the permute: dU_t = dO_t + sum_{kept j} dX[row(t, j)] (X = U[perm])."""
    dU = f64(dO).copy()
    T = dU.shape[0]
    sr = np.asarray(slot_row, dtype=np.int64).reshape(T, k)
    dX = f64(dX)
    for j in range(k):
        m = sr[:, j] >= 0
        dU[m] += dX[sr[m, j]]
    return dU


def router_input_backward(U, W_r, dH, W_noise=None, eps=None) -> dict:
    """Backward of the router linear H = U W_r + b_r (+ eps * softplus(U W_noise)) ([RTR]).

    dU = dH W_r^T (+ dN W_noise^T), dW_r = U^T dH, db_r = sum_t dH, dW_noise = U^T dN with
    dN = dH * eps * sigmoid(U W_noise) (softplus' = sigmoid).
    """
    U, W_r, dH = f64(U), f64(W_r), f64(dH)
    out = dict(dU=dH @ W_r.T, dW_r=U.T @ dH, db_r=dH.sum(axis=0), dW_noise=None)
    if W_noise is not None:
        with np.errstate(over="ignore"):
            sg = 1.0 / (1.0 + np.exp(-(U @ f64(W_noise))))
        dN = dH * f64(eps) * sg
        out["dU"] = out["dU"] + dN @ f64(W_noise).T
        out["dW_noise"] = U.T @ dN
    return out


def layer_backward(inp, fwd: dict, dO, *, k: int, d_e: int, score_fn: int, renorm: bool, w_aux: float = 0.0,
                   w_z: float = 0.0) -> dict:
    """Gradients of L = <dO, out> + w_aux E sum_i f_i P_i + w_z L_z through the whole layer, with
    the routing decisions (top-k set, slots, drops) held fixed.  `fwd` is layer_forward's result.
    [GRD], [BWD], [SHR], [RTR]
    """
    cb = combine_backward(dO, fwd["Y"], fwd["slot_row"], fwd["gate"], k)
    dH = router_backward(fwd["logits"], fwd["idx"], cb["d_gate"], fwd["f"], score_fn, renorm, w_aux, w_z)
    eb = expert_ffn_backward(fwd["X"], fwd["offsets"], inp.W_gate, inp.W_up, inp.W_down, cb["dY"], d_e)
    rb = router_input_backward(inp.U, inp.W_r, dH, inp.W_noise, inp.eps)
    dU = dispatch_backward(dO, eb["dX"], fwd["slot_row"], k) + rb["dU"]
    out = dict(dU=dU, d_gate=cb["d_gate"], dY=cb["dY"], dH=dH, dW_r=rb["dW_r"], db_r=rb["db_r"],
               dW_noise=rb["dW_noise"], **{n: eb[n] for n in ("d_act", "dG", "dUp", "dX", "dW_gate", "dW_up",
                                                              "dW_down")})
    shared = getattr(inp, "shared", None)
    if shared is not None:
        Wg, Wu, Wd = shared
        sh = [swiglu_backward(inp.U, Wg[i], Wu[i], Wd[i], dO) for i in range(len(Wg))]
        for b in sh:
            out["dU"] = out["dU"] + b["dx"]
        out["dW_gate_sh"] = np.stack([b["dW_gate"] for b in sh])
        out["dW_up_sh"] = np.stack([b["dW_up"] for b in sh])
        out["dW_down_sh"] = np.stack([b["dW_down"] for b in sh])
    return out


def group_margins(aff: np.ndarray, n_group: int, topk_group: int, k: int) -> np.ndarray:
    """Per token, the gap between the topk_group-th and the next group score (inf when every
    group is kept).  Used by the tests to keep group decisions away from ties."""
    if topk_group >= n_group:
        return np.full(np.asarray(aff).shape[0], np.inf)
    gs = -np.sort(-group_scores(aff, n_group, k // topk_group), axis=1)
    return gs[:, topk_group - 1] - gs[:, topk_group]


def topk_margins(H32: np.ndarray, k: int) -> np.ndarray:
    """Smallest gap between adjacent values among each row's k+1 largest logits.

    Used by the tests to keep end-to-end routing decisions away from ties:
    a token whose margin is below the threshold is redrawn.
    """
    s = -np.sort(-np.asarray(H32, dtype=np.float64), axis=1)[:, :k + 1]
    if s.shape[1] < 2:
        return np.full(s.shape[0], np.inf)
    return np.min(s[:, :-1] - s[:, 1:], axis=1)

"""CPU oracle for the routed MoE FFN layer forward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library and the library never calls it: a missing CUDA extension
is an error, never a fallback to this file.

Everything here is a plain, slow, literal restatement of the pages' formulas in
float64 with numpy (``@`` is numpy's float64 matrix product, used as a library
primitive).  Sources, cited by page title and section:

* [MM] "mega_moe" (Ascend CANN operator page), section "计算公式" (computation
  formula) with its sub-steps "EP Dispatch", "Expert Compute" (Linear1,
  SwiGLU, Linear2) and "Token Combine".
* [MG] "Megatron-LM 的 MoE 并行：以 DeepSeek-V4 为例": section "模型与入口"
  (the MoE output equation y_t = F_s(x_t) + sum_{e in I_t} g_{t,e} F_e(x_t)),
  section "路由与负载 / 路由张量" (affinity a = sqrt(softplus(l)), selection
  I_t = TopK(a + beta), mixing weight g = alpha * a / sum_{I_t} a),
  "路由与负载 / Hash 路由" (ids looked up from tid2eid; gating and weights
  kept), "AlltoAll 的前向 / 计数与重排" (per-expert counts, permutation with
  duplication, the four-token split example).
* [PD] "Megatron 分布式训练全维度并行技术文档", section "4.2 数学推导"
  (softmax gate G(x) = TopK(softmax(x W_gate))).
* [MM] again, section "计算过程", A8W8 scenario: per-token int8 activations,
  per-channel int8 weights, int32 products, dequantisation, per-row
  re-quantisation of the SwiGLU output.
* [MG] section "反向的通信" and [PD] section 4.7 "反向流程": the backward (un-permute
  backward, expert dgrad and wgrad, the k input gradients of a token summed,
  router backward; the top-k ids are constants, the selected experts' scores
  and mixing weights are differentiable).
* [MM] again, section "计算过程", MXFP scenario (the four stages: MX
  quantisation of the dispatched rows, GMM1 + SwiGLU + MX quantisation, GMM2,
  weighted combine) and section "约束说明" (group size 32, FLOAT8_E8M0
  scales, element types FLOAT8_E4M3FN / FLOAT8_E5M2 / FLOAT4_E2M1, the
  A8W8-FP, A8W4-FP and A4W4-FP scenarios, weight1 [E, 2I, H] with scales
  [E, 2I, ceil(H/64), 2], weight2 [E, H, I] with scales over I).

Readings taken where the pages are silent:
the score function is a parameter (sigmoid, sqrt-softplus, softmax); the k ids
of a token are listed by descending selection score, equal scores to the lower
expert id; rows inside an expert block follow ascending flat index t*k+j; the
gate half of Linear1's output is its first I columns; the shared expert has the
same width I and weight 1; an assignment whose id is outside [0, E) is dropped.

Parity status: routing ids, counts, permutation and the FFN/combine are pinned
by tests/test_oracle_pins.py (closed forms, brute force, the worked split
example, reductions to a dense FFN).  The MX functions are pinned against the
FP8 code tables and round-to-nearest-even conversion of torch's float8 types,
a hand-worked group, closed forms of the shared exponent and of the rounding
error, and a scalar brute-force layer.  The backward is pinned by central
finite differences of the oracle's forward (every parameter of tiny layers,
all three score functions, with and without renormalisation) and by torch's
float64 reverse-mode differentiation of a larger layer.  The absolute gate and output values for
the sigmoid and sqrt-softplus rules at the workload sizes rest on these same
formulas; the pages print no worked numbers for them.
"""
from __future__ import annotations

import numpy as np

SCORE_SIGMOID = 0
SCORE_SQRT_SOFTPLUS = 1
SCORE_SOFTMAX = 2

__all__ = [
    "bf16_to_f64", "round_to_bf16", "f64_to_bf16_bits",
    "router_logits", "affinity", "select_topk", "gates",
    "route", "route_from_logits", "route_hash",
    "dispatch", "swiglu_expert", "forward", "forward_tokens",
    "round_half_away", "quantize_rows_int8", "swiglu_expert_a8w8", "forward_a8w8_tokens",
    "SCORE_SIGMOID", "SCORE_SQRT_SOFTPLUS", "SCORE_SOFTMAX",
]


# ----------------------------------------------------------------------------- numbers
def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 values (exact widening)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def as_f64(w) -> np.ndarray:
    """bf16 bit patterns (uint16) decoded, any floating array as float64: the
    oracle's functions take either, so that a test can hand them real-valued
    parameters (finite differences)."""
    w = np.asarray(w)
    return bf16_to_f64(w) if w.dtype == np.uint16 else w.astype(np.float64)


def round_to_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even), returned
    as float64.  Direct rounding of the 52-bit fraction to 7 bits: no
    intermediate float32 step, so there is no double rounding."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    u = x.view(np.uint64)
    drop = np.uint64(45)  # 52 - 7 fraction bits are discarded
    half = np.uint64(1) << np.uint64(44)
    lsb = (u >> drop) & np.uint64(1)
    r = (u + (half - np.uint64(1)) + lsb) & ~((np.uint64(1) << drop) - np.uint64(1))
    return r.view(np.float64)


def f64_to_bf16_bits(x) -> np.ndarray:
    """float64 -> bf16 bit patterns, rounding to nearest even."""
    r = round_to_bf16(x).astype(np.float32)  # exact: r has 8 significant bits
    return (r.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def _silu(z):
    # [MM] conventions: SiLU(z) = z * sigma(z) = z / (1 + e^{-z})
    return z * _sigmoid(z)


# ----------------------------------------------------------------------------- routing
def router_logits(X_bits, Wg_bits) -> np.ndarray:
    """[MG] 路由张量: the gating linear maps [n, h] to [n, E] logits, l = X Wg."""
    return as_f64(X_bits) @ as_f64(Wg_bits)


def affinity(logits, score_fn: int) -> np.ndarray:
    """Affinity a[t, e] from the logits.

    sigmoid: a = 1 / (1 + exp(-l)).
    sqrt-softplus ([MG] 路由张量, V4 rule): a = sqrt(softplus(l)), with
      softplus(l) = log(1 + e^l) evaluated as max(l, 0) + log1p(e^{-|l|}).
    softmax ([PD] 4.2): a = softmax over the experts of the token's logits.
    """
    l = np.asarray(logits, dtype=np.float64)
    if score_fn == SCORE_SIGMOID:
        return _sigmoid(l)
    if score_fn == SCORE_SQRT_SOFTPLUS:
        return np.sqrt(np.maximum(l, 0.0) + np.log1p(np.exp(-np.abs(l))))
    if score_fn == SCORE_SOFTMAX:
        m = l.max(axis=-1, keepdims=True)
        p = np.exp(l - m)
        return p / p.sum(axis=-1, keepdims=True)
    raise ValueError(f"unknown score function {score_fn}")


def select_topk(scores, k: int) -> np.ndarray:
    """Per row, the k largest scores' column ids, listed by descending score;
    equal scores are listed (and kept) lower id first.  A stable sort of the
    negated scores gives exactly that order."""
    s = np.asarray(scores, dtype=np.float64)
    order = np.argsort(-s, axis=-1, kind="stable")
    return order[..., :k].astype(np.int32)


def gates(a, E_ids, alpha: float, renorm: bool) -> np.ndarray:
    """[MG] 路由张量: g_{t,e} = alpha * a_{t,e} / sum_{j in I_t} a_{t,j} taken at
    the selected ids with the raw (un-biased) affinity.  Without
    renormalisation (the softmax gate of [PD] 4.2) g = alpha * a at the ids.
    A zero denominator gives zero gates."""
    a_sel = np.take_along_axis(np.asarray(a, dtype=np.float64), E_ids.astype(np.int64), axis=-1)
    if not renorm:
        return alpha * a_sel
    den = a_sel.sum(axis=-1, keepdims=True)
    safe = np.where(den > 0, den, 1.0)
    return np.where(den > 0, alpha * a_sel / safe, 0.0)


def route_from_logits(logits, bias, score_fn: int, k: int, alpha: float, renorm: bool):
    """Selection and gates from given logits: a = score(l); I_t = TopK(a + beta)
    ([MG] 路由张量; beta is used for selection only); softmax selects on a alone
    ([PD] 4.2).  Returns (E_ids int32 [T,k], G float64 [T,k], a float64 [T,E])."""
    a = affinity(logits, score_fn)
    s = a
    if bias is not None:
        if score_fn == SCORE_SOFTMAX:
            raise ValueError("the softmax gate takes no selection bias")
        s = a + np.asarray(bias, dtype=np.float64)[None, :]
    E_ids = select_topk(s, k)
    return E_ids, gates(a, E_ids, alpha, renorm), a


def route(X_bits, Wg_bits, bias, score_fn: int, k: int, alpha: float, renorm: bool):
    """Router: logits, affinity, biased top-k selection, alpha-scaled gates.
    Returns (E_ids, G, logits)."""
    l = router_logits(X_bits, Wg_bits)
    E_ids, G, _ = route_from_logits(l, bias, score_fn, k, alpha, renorm)
    return E_ids, G, l


def route_hash(X_bits, Wg_bits, token_ids, tid2eid, score_fn: int, alpha: float, renorm: bool):
    """[MG] Hash 路由: the expert ids are the table row of the token id; the
    gating linear and the gate formula are unchanged.  Returns (E_ids, G, logits)."""
    tid2eid = np.asarray(tid2eid, dtype=np.int32)
    E_ids = tid2eid[np.asarray(token_ids, dtype=np.int64)]
    l = router_logits(X_bits, Wg_bits)
    a = affinity(l, score_fn)
    return E_ids.astype(np.int32), gates(a, E_ids, alpha, renorm), l


# ----------------------------------------------------------------------------- dispatch
def dispatch(E_ids, E: int):
    """[MM] EP Dispatch: expert e receives the rows of I_e stacked in a fixed
    order; row(i, k) is the unique position of token i in expert e_{i,k}'s block.
    [MG] 计数与重排: count[e] assignments per expert; the permutation groups the
    flat assignment list by expert, copying a token once per selection.

    Fixed order taken here: ascending flat index f = t*k + j inside each block.
    Returns counts [E], offsets [E+1] (exclusive prefix sum), perm [sum counts]
    (perm[p] = flat index at block row p) and inv [T*k] (inv[f] = p, or -1 for
    an id outside [0, E), which is dropped)."""
    flat = np.asarray(E_ids, dtype=np.int64).reshape(-1)
    valid = (flat >= 0) & (flat < E)
    counts = np.zeros(E, dtype=np.int64)
    for e in flat[valid]:
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    perm = np.empty(int(offsets[-1]), dtype=np.int64)
    fill = offsets[:-1].copy()
    inv = np.full(flat.shape[0], -1, dtype=np.int64)
    for f in range(flat.shape[0]):  # ascending f: the order inside each block
        if valid[f]:
            e = flat[f]
            perm[fill[e]] = f
            inv[f] = fill[e]
            fill[e] += 1
    return (counts.astype(np.int32), offsets.astype(np.int32),
            perm.astype(np.int32), inv.astype(np.int32))


# ----------------------------------------------------------------------------- experts
def swiglu_expert(X_rows64, W1e, W2e, act_round_bf16: bool = False) -> np.ndarray:
    """[MM] Expert Compute: H = X_e W1[e] ([N_e, 2I]); gate = H[:, :I],
    up = H[:, I:]; A = SiLU(gate) * up; Y_e = A W2[e].  W1e/W2e are bf16 bits.
    ``act_round_bf16`` rounds A to bf16 before Linear2 (off by default)."""
    W1 = as_f64(W1e)
    W2 = as_f64(W2e)
    I = W2.shape[0]
    Hm = X_rows64 @ W1
    A = _silu(Hm[:, :I]) * Hm[:, I:]
    if act_round_bf16:
        A = round_to_bf16(A)
    return A @ W2


def _get(w, e):
    return w(e) if callable(w) else w[e]


def forward_tokens(tokens, X_rows_bits, E_rows, G_rows, W1, W2, Ws1=None, Ws2=None,
                   act_round_bf16: bool = False, E: int | None = None) -> np.ndarray:
    """The layer output for a set of tokens, in float64 (no final rounding).

    [MG] 模型与入口: y_t = F_s(x_t) + sum_{e in I_t} g_{t,e} F_e(x_t).
    [MM] Token Combine: y_i = sum_k G[i,k] * Y_{e_{i,k}}[row(i,k), :].

    ``tokens`` only labels the rows (X_rows_bits[r] is token tokens[r]); each
    output row depends on its own token alone.  W1/W2 may be arrays indexed by
    expert or callables e -> bf16 bits, so that a caller can hand over experts
    one at a time (then ``E``, the expert count, must be given).  Ws1/Ws2
    (the shared expert, weight 1) may be None.
    """
    R = len(tokens)
    E_rows = np.asarray(E_rows, dtype=np.int64).reshape(R, -1)
    G_rows = np.asarray(G_rows, dtype=np.float64).reshape(R, -1)
    k = E_rows.shape[1]
    X64 = as_f64(X_rows_bits).reshape(R, -1)
    Hdim = X64.shape[1]
    if E is None:
        E = np.asarray(W1).shape[0]
    # dispatch the selected rows: the expert blocks of these tokens
    counts, offsets, perm, inv = dispatch(E_rows, E)
    Yp = np.zeros((perm.shape[0], Hdim), dtype=np.float64)
    for e in range(len(counts)):
        if counts[e] == 0:
            continue
        rows = perm[offsets[e]:offsets[e + 1]]
        Xe = X64[rows // k]
        Yp[offsets[e]:offsets[e + 1]] = swiglu_expert(Xe, _get(W1, e), _get(W2, e), act_round_bf16)
    # combine in j order
    Y = np.zeros((R, Hdim), dtype=np.float64)
    for j in range(k):
        f = np.arange(R) * k + j
        p = inv[f]
        ok = p >= 0
        Y[ok] += G_rows[ok, j:j + 1] * Yp[p[ok]]
    if Ws1 is not None:
        Y += swiglu_expert(X64, Ws1, Ws2, act_round_bf16)
    return Y


def forward(X_bits, E_ids, G, W1, W2, Ws1=None, Ws2=None, act_round_bf16: bool = False):
    """Whole-layer output: float64 Y [T, H] and its bf16 rounding (bits)."""
    T = np.asarray(X_bits).shape[0]
    Y = forward_tokens(np.arange(T), X_bits, E_ids, G, W1, W2, Ws1, Ws2, act_round_bf16,
                       E=np.asarray(W1).shape[0])
    return Y, f64_to_bf16_bits(Y)


# ----------------------------------------------------------------------------- backward
# [MG] 反向的通信: for an upstream gradient dL/dy_t the gradient flows through
# the selected experts' branches, the shared expert, and the router: the top-k
# ids are constants, the selected experts' continuous scores and mixing weights
# stay differentiable (hash layers included).  The backward runs the forward's
# dependencies in reverse: un-permute backward (one gradient row per
# assignment), expert dgrad and wgrad, the k expert input gradients of a token
# added (the permute duplicated the row), then router and input.  [PD] 4.7
# 反向流程 lists the same steps: d(w_e Y_e) = w_e dY, expert backward (dW_gate,
# dW_up, dW_down and the input gradient), router backward (dW_gate of the
# router).  Below, plain chain rule in float64.
def _silu_grad(z):
    """d/dz [z sigma(z)] = sigma(z) (1 + z (1 - sigma(z)))."""
    s = _sigmoid(z)
    return s * (1.0 + z * (1.0 - s))


def swiglu_expert_backward(X_rows64, W1e, W2e, dOut, round_bf16: bool = False, mass: bool = False):
    """Gradients of Y = (SiLU(X W1[:, :I]) * X W1[:, I:]) W2 for dL/dY = dOut
    ([n, H]): returns (dX [n, H], dW1 [H, 2I], dW2 [I, H], Y [n, H]).

    ``round_bf16`` rounds to bf16 where a path that keeps its tensors in bf16
    would: the pre-activations H (as used by the backward), the SwiGLU output
    A (used for Y and dW2), the incoming row gradient dOut and dH; every
    product and sum stays float64.  ``mass`` appends, for each of the four
    results, the sum of the magnitudes of the products of its last
    contraction (|dH| |W1|^T, |X|^T |dH|, |A|^T |dOut|, |A| |W2|): one
    rounding step of a bf16 operand moves a result by at most 2^-8 of it."""
    r = round_to_bf16 if round_bf16 else (lambda v: v)
    W1 = as_f64(W1e)
    W2 = as_f64(W2e)
    I = W2.shape[0]
    Hm = X_rows64 @ W1
    A = r(_silu(Hm[:, :I]) * Hm[:, I:])
    Hk = r(Hm)
    Hg, Hu = Hk[:, :I], Hk[:, I:]
    dOut = r(dOut)
    dA = dOut @ W2.T
    dH = r(np.concatenate([dA * Hu * _silu_grad(Hg), dA * _silu(Hg)], axis=1))
    out = (dH @ W1.T, X_rows64.T @ dH, A.T @ dOut, A @ W2)
    if mass:
        aH, aA, aO = np.abs(dH), np.abs(A), np.abs(dOut)
        out += (aH @ np.abs(W1).T, np.abs(X_rows64).T @ aH, aA.T @ aO, aA @ np.abs(W2))
    return out


def affinity_backward(logits, da, score_fn: int) -> np.ndarray:
    """dL/dl from dL/da for a = score(l), elementwise (sigmoid: a (1 - a);
    sqrt-softplus: sigma(l) / (2 a)) or through the softmax Jacobian
    (a (da - sum(a da)))."""
    l = np.asarray(logits, dtype=np.float64)
    a = affinity(l, score_fn)
    if score_fn == SCORE_SIGMOID:
        return da * a * (1.0 - a)
    if score_fn == SCORE_SQRT_SOFTPLUS:
        return da * _sigmoid(l) / (2.0 * a)
    if score_fn == SCORE_SOFTMAX:
        return a * (da - (a * da).sum(axis=-1, keepdims=True))
    raise ValueError(f"unknown score function {score_fn}")


def gates_backward(a, E_ids, dG, alpha: float, renorm: bool) -> np.ndarray:
    """dL/da [T, E] from dL/dg [T, k] for the gates of ``gates``: with
    renormalisation g_j = alpha a_j / S, S = sum_i a_i over the selected ids,
    so dL/da_i = (alpha / S)(dG_i - sum_j dG_j a_j / S); without, alpha dG.
    Zero where S = 0 and at the experts not selected."""
    a = np.asarray(a, dtype=np.float64)
    ids = np.asarray(E_ids, dtype=np.int64)
    dG = np.asarray(dG, dtype=np.float64)
    a_sel = np.take_along_axis(a, ids, axis=-1)
    if renorm:
        S = a_sel.sum(axis=-1, keepdims=True)
        safe = np.where(S > 0, S, 1.0)
        da_sel = np.where(S > 0, alpha / safe * (dG - (dG * a_sel).sum(axis=-1, keepdims=True) / safe), 0.0)
    else:
        da_sel = alpha * dG
    da = np.zeros_like(a)
    for j in range(ids.shape[1]):
        np.add.at(da, (np.arange(a.shape[0]), ids[:, j]), da_sel[:, j])
    return da


def backward(X_bits, Wg_bits, E_ids, dY, W1, W2, Ws1, Ws2, score_fn: int, alpha: float,
             renorm: bool, E: int | None = None, round_bf16: bool = False,
             mass: bool = False, weight_experts=None) -> dict:
    """Gradients of the layer for upstream dY [T, H] at the routing E_ids (from
    the top-k or the hash table; held constant).  W1/W2 arrays or callables
    e -> weights; Ws1/Ws2 may be None.  Returns float64 arrays: dX [T, H],
    dWg [H, E], dW1 [E, H, 2I], dW2 [E, I, H], dWs1, dWs2 (or None), dG [T, k]
    (the mixing-weight gradient <dY_t, Y_e(x_t)>) and dlogits [T, E].
    ``round_bf16``: as in swiglu_expert_backward, and the logit gradient is
    rounded to bf16 before its two products (dWg, the router part of dX).
    ``mass``: also "mass_<name>" for dX, dWg, dW1, dW2, dWs1, dWs2 and dG, the
    sums of product magnitudes of each result's last contractions.
    ``weight_experts``: if given, dW1 and dW2 (and their masses) are dicts
    holding only these experts (full-size checks of a few experts)."""
    X = as_f64(X_bits)
    Wg = as_f64(Wg_bits)
    ids = np.asarray(E_ids, dtype=np.int64)
    T, k = ids.shape
    dY = np.asarray(dY, dtype=np.float64)
    if E is None:
        E = np.asarray(W1).shape[0]
    l = X @ Wg
    a = affinity(l, score_fn)
    G = gates(a, ids.astype(np.int32), alpha, renorm)
    counts, offsets, perm, inv = dispatch(ids, E)
    dX = np.zeros_like(X)
    dG = np.zeros((T, k))
    dW1 = dW2 = None
    m = {"dX": np.zeros_like(X), "dG": np.zeros((T, k))} if mass else None
    keep = None if weight_experts is None else set(int(e) for e in weight_experts)
    if keep is not None:
        dW1, dW2 = {}, {}
        if mass:
            m["dW1"], m["dW2"] = {}, {}
    for e in range(E):
        if counts[e] == 0 and keep is None and dW1 is not None:
            continue
        W1e, W2e = _get(W1, e), _get(W2, e)
        if dW1 is None:
            dW1 = np.zeros((E,) + np.shape(W1e))
            dW2 = np.zeros((E,) + np.shape(W2e))
            if mass:
                m["dW1"], m["dW2"] = np.zeros_like(dW1), np.zeros_like(dW2)
        if keep is not None and e in keep:
            dW1[e], dW2[e] = np.zeros(np.shape(W1e)), np.zeros(np.shape(W2e))
            if mass:
                m["dW1"][e], m["dW2"][e] = np.zeros_like(dW1[e]), np.zeros_like(dW2[e])
        if counts[e] == 0:
            continue
        f = perm[offsets[e]:offsets[e + 1]]     # flat assignment ids t * k + j
        t, j = f // k, f % k
        # un-permute backward: the assignment's gradient row is g_{t,j} dY_t
        res = swiglu_expert_backward(X[t], W1e, W2e, G[t, j][:, None] * dY[t], round_bf16, mass)
        dXe, Ye = res[0], res[3]
        if keep is None or e in keep:
            dW1[e], dW2[e] = res[1], res[2]
        dG[t, j] = (dY[t] * Ye).sum(axis=1)
        np.add.at(dX, t, dXe)                    # the k dgrads of a token add up
        if mass:
            np.add.at(m["dX"], t, res[4])
            if keep is None or e in keep:
                m["dW1"][e], m["dW2"][e] = res[5], res[6]
            m["dG"][t, j] = (np.abs(dY[t]) * res[7]).sum(axis=1)
    dWs1 = dWs2 = None
    if Ws1 is not None:
        res = swiglu_expert_backward(X, Ws1, Ws2, dY, round_bf16, mass)
        dXs, dWs1, dWs2 = res[:3]
        dX += dXs
        if mass:
            m["dX"] += res[4]
            m["dWs1"], m["dWs2"] = res[5], res[6]
    dl = affinity_backward(l, gates_backward(a, ids, dG, alpha, renorm), score_fn)
    dlr = round_to_bf16(dl) if round_bf16 else dl
    dX += dlr @ Wg.T
    out = {"dX": dX, "dWg": X.T @ dlr, "dW1": dW1, "dW2": dW2, "dWs1": dWs1, "dWs2": dWs2,
           "dG": dG, "dlogits": dl}
    if mass:
        m["dX"] += np.abs(dlr) @ np.abs(Wg).T
        m["dWg"] = np.abs(X).T @ np.abs(dlr)
        out.update({"mass_" + key: v for key, v in m.items()})
    return out


# ----------------------------------------------------------------------------- A8W8-INT
# [MM] 计算过程, A8W8 scenario: per-token int8 activations, per-channel int8
# weights, int8 x int8 -> int32 products, dequantisation by both scales, and
# the SwiGLU output re-quantised per row before Linear2.
def round_half_away(z) -> np.ndarray:
    """[MM] conventions: the nearest integer, halves away from zero (四舍五入).
    Evaluated in float64, where |z| + 0.5 is exact for any float32 z."""
    z = np.asarray(z, dtype=np.float64)
    return np.sign(z) * np.floor(np.abs(z) + 0.5)


def quantize_rows_int8(x, dtype=np.float64):
    """[MM] A8W8 EP Dispatch / Linear2: s_i = max|x_i| / 127 and
    q_i = round(x_i / s_i) in [-127, 127], evaluated in ``dtype``.  A row of
    zeros has s = 0 and codes 0.  Returns (q int32 [R, C], s dtype [R])."""
    x = np.asarray(x, dtype=dtype)
    amax = np.abs(x).max(axis=-1)
    s = (amax / dtype(127.0)).astype(dtype)
    safe = np.where(s > 0, s, dtype(1.0)).astype(dtype)
    q = round_half_away((x / safe[..., None]).astype(dtype))
    q = np.where(s[..., None] > 0, q, 0.0)
    return q.astype(np.int32), s


def swiglu_expert_a8w8(q_rows, sx_rows, W1q, S1, W2q, S2) -> np.ndarray:
    """[MM] A8W8 Expert Compute for one expert.  The weights are stored as the
    operator's weight1 [2I, H] and weight2 [H, I] (one row per output channel,
    the contraction contiguous), with one scale per output channel.
    C = Q W1q^T (int32, exact); H = (C * s^W1) * s^X; A = SiLU(H[:, :I]) *
    H[:, I:]; s^A, A8 = quantize(A) per row; D = A8 W2q^T (int32, exact);
    Y = (D * s^W2) * s^A."""
    C = np.asarray(q_rows, np.int64) @ np.asarray(W1q, np.int64).T
    Hm = (C.astype(np.float64) * np.asarray(S1, np.float64)[None, :]) * np.asarray(sx_rows, np.float64)[:, None]
    I = np.asarray(W2q).shape[1]
    A = _silu(Hm[:, :I]) * Hm[:, I:]
    A8, sA = quantize_rows_int8(A, np.float64)
    D = A8.astype(np.int64) @ np.asarray(W2q, np.int64).T
    return (D.astype(np.float64) * np.asarray(S2, np.float64)[None, :]) * sA[:, None]


def forward_a8w8_tokens(tokens, X_rows_bits, E_rows, G_rows, W1q, S1, W2q, S2, E: int) -> np.ndarray:
    """A8W8 layer output for a set of tokens, float64.  The token codes are
    decided in float32, as the kernel decides them; every later step is
    float64 with exact integer products.  W1q/W2q/S1/S2 may be arrays indexed
    by expert or callables e -> array."""
    R = len(tokens)
    E_rows = np.asarray(E_rows, dtype=np.int64).reshape(R, -1)
    G_rows = np.asarray(G_rows, dtype=np.float64).reshape(R, -1)
    k = E_rows.shape[1]
    x32 = bf16_to_f64(X_rows_bits).reshape(R, -1).astype(np.float32)
    q, sx = quantize_rows_int8(x32, np.float32)
    counts, offsets, perm, inv = dispatch(E_rows, E)
    Hdim = x32.shape[1]
    Yp = np.zeros((perm.shape[0], Hdim), dtype=np.float64)
    for e in range(E):
        if counts[e] == 0:
            continue
        rows = perm[offsets[e]:offsets[e + 1]] // k
        Yp[offsets[e]:offsets[e + 1]] = swiglu_expert_a8w8(
            q[rows], sx[rows], _get(W1q, e), _get(S1, e), _get(W2q, e), _get(S2, e))
    Y = np.zeros((R, Hdim), dtype=np.float64)
    for j in range(k):
        p = inv[np.arange(R) * k + j]
        ok = p >= 0
        Y[ok] += G_rows[ok, j:j + 1] * Yp[p[ok]]
    return Y


# ----------------------------------------------------------------------------- MXFP8 (A8W8-FP)
# [MM] 计算过程, MXFP scenario (dispatch_quant_mode 4): the token rows are
# quantised per group of 32 consecutive elements along the contraction with a
# shared power-of-two scale (FLOAT8_E8M0) and FP8 elements (FLOAT8_E4M3FN or
# FLOAT8_E5M2); the weights arrive quantised the same way (W1 [E, 2I, H] with
# scales over H, W2 [E, H, I] with scales over I, both stored K-contiguous);
# Linear1 and Linear2 multiply the dequantised operands; the SwiGLU output is
# re-quantised the same way before Linear2; the combine is unquantised.
#
# Readings (the pages name the operation Q_MX without spelling it out): the
# shared exponent follows the OCP Microscaling formats definition,
# X = floor(log2(max|v|)) - emax_elem, clamped to the E8M0 range [-127, 127]
# (a group of zeros gets X = -127); each element is v / 2^X rounded to the
# nearest FP8 value, ties to even mantissa, magnitudes beyond the largest
# finite value saturating to it; the sign of zero is kept.

# name -> (exponent bits, mantissa bits, exponent bias, largest finite value)
FP8_FORMATS = {
    "e4m3": (4, 3, 7, 448.0),      # FLOAT8_E4M3FN: no infinities, S.1111.111 is NaN
    "e5m2": (5, 2, 15, 57344.0),   # FLOAT8_E5M2: IEEE-style, exponent 11111 is Inf/NaN
    "e2m1": (2, 1, 1, 6.0),        # FLOAT4_E2M1: 4-bit, no infinities or NaN
}
MX_GROUP = 32


def _code_bits(fmt: str) -> int:
    eb, mb, _, _ = FP8_FORMATS[fmt]
    return 1 + eb + mb


def fp8_decode(codes, fmt: str) -> np.ndarray:
    """Value of each FP8 (or FP4) code from the format's definition (sign,
    biased exponent, mantissa; exponent field 0 is subnormal), float64."""
    eb, mb, bias, _ = FP8_FORMATS[fmt]
    nb = _code_bits(fmt)
    c = np.asarray(codes, dtype=np.int64) & ((1 << nb) - 1)
    sign = np.where(c >> (nb - 1), -1.0, 1.0)
    ef = (c >> mb) & ((1 << eb) - 1)
    mf = c & ((1 << mb) - 1)
    mag = np.where(ef == 0, mf / 2.0 ** mb * 2.0 ** (1 - bias),
                   (1.0 + mf / 2.0 ** mb) * 2.0 ** (ef.astype(np.float64) - bias))
    v = sign * mag
    if fmt == "e4m3":
        v = np.where((ef == 15) & (mf == 7), np.nan, v)
    elif fmt == "e5m2":
        v = np.where(ef == 31, np.where(mf == 0, sign * np.inf, np.nan), v)
    return v


def fp8_round(v, fmt: str) -> np.ndarray:
    """Nearest FP8 value to v (float64), ties to the even mantissa, magnitude
    saturated at the largest finite value.  The grid spacing at |v| is
    2^(e - mantissa_bits) with e = floor(log2|v|), never below the subnormal
    spacing 2^(1 - bias - mantissa_bits)."""
    eb, mb, bias, vmax = FP8_FORMATS[fmt]
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), vmax)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, 1 - bias)
    q = 2.0 ** (e - mb)
    r = np.minimum(np.round(a / q) * q, vmax)   # np.round: halves to even
    return np.copysign(r, v)


def fp8_encode(v, fmt: str) -> np.ndarray:
    """FP8 code (uint8) of fp8_round(v): the sign bit of v, then the code of
    the rounded magnitude found in the table of finite non-negative codes."""
    r = fp8_round(v, fmt)
    nb = _code_bits(fmt)
    pos = np.arange(1 << (nb - 1))
    vals = fp8_decode(pos, fmt)
    finite = np.isfinite(vals)
    pos, vals = pos[finite], vals[finite]          # ascending with the code
    mag = np.searchsorted(vals, np.abs(r))
    assert np.array_equal(vals[mag], np.abs(r)), "rounded value off the FP8 grid"
    return (pos[mag] | np.where(np.signbit(r), 1 << (nb - 1), 0)).astype(np.uint8)


def unpack_e2m1(packed) -> np.ndarray:
    """FLOAT4_E2M1 codes stored two per byte (element 2i in the low nibble,
    2i + 1 in the high nibble) -> one code per element along the last axis."""
    b = np.asarray(packed, dtype=np.uint8)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = b & 0x0F
    out[..., 1::2] = b >> 4
    return out


def e8m0_decode(codes) -> np.ndarray:
    """FLOAT8_E8M0 scale: 2^(code - 127); code 255 is NaN."""
    c = np.asarray(codes, dtype=np.int64)
    return np.where(c == 255, np.nan, 2.0 ** (c.astype(np.float64) - 127))


def mx_quantize(x, fmt: str, dtype=np.float64):
    """Q_MX over the last axis (its length a multiple of 32): per group of 32,
    X = floor(log2 max|v|) - emax_elem clamped to [-127, 127], elements
    fp8(v / 2^X).  The group maximum and its exponent are taken in ``dtype``
    (exact in either precision); v / 2^X is exact.  Returns (codes uint8
    [..., K], scale codes uint8 [..., K/32])."""
    eb, mb, bias, vmax = FP8_FORMATS[fmt]
    emax = int(np.floor(np.log2(vmax)))
    x = np.asarray(x, dtype=dtype)
    K = x.shape[-1]
    assert K % MX_GROUP == 0
    g = x.reshape(x.shape[:-1] + (K // MX_GROUP, MX_GROUP)).astype(np.float64)
    amax = np.abs(g).max(axis=-1)
    with np.errstate(divide="ignore"):
        ex = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))), -np.inf)
    X = np.clip(ex - emax, -127, 127)
    codes = fp8_encode(g / 2.0 ** X[..., None], fmt).reshape(x.shape)
    return codes, (X + 127).astype(np.uint8)


def mx_dequantize(codes, scales, fmt: str) -> np.ndarray:
    """DQ_MX: element value times the scale of its group of 32 along the last
    axis, float64."""
    v = fp8_decode(codes, fmt)
    s = np.repeat(e8m0_decode(scales), MX_GROUP, axis=-1)
    return v * s


def swiglu_expert_mx(xq, sx, W1q, S1, W2q, S2, fmt: str, wfmt: str | None = None) -> np.ndarray:
    """[MM] MXFP Expert Compute for one expert.  xq/sx: the expert's token
    rows quantised [m, H] / [m, H/32]; W1q [2I, H], S1 [2I, H/32]; W2q [H, I],
    S2 [H, I/32] (one code per element).  Z = DQ(xq) DQ(W1)^T; U = Z^(x) *
    sigma(Z^(x)) * Z^(y) with Z^(x) the first I columns; (Uq, SU) = Q_MX(U);
    O = DQ(Uq) DQ(W2)^T.  ``fmt`` is the activations' element type, ``wfmt``
    the weights' (default: the same; "e2m1" with "e4m3" activations is the
    pages' A8W4-FP scenario, "e2m1" for both A4W4-FP)."""
    wfmt = fmt if wfmt is None else wfmt
    Xd = mx_dequantize(xq, sx, fmt)
    W1d = mx_dequantize(W1q, S1, wfmt)
    Z = Xd @ W1d.T
    I = np.asarray(W2q).shape[1]
    U = _silu(Z[:, :I]) * Z[:, I:]
    Uq, SU = mx_quantize(U, fmt)
    return mx_dequantize(Uq, SU, fmt) @ mx_dequantize(W2q, S2, wfmt).T


def forward_mx_tokens(tokens, X_rows_bits, E_rows, G_rows, W1q, S1, W2q, S2, E: int,
                      fmt: str, wfmt: str | None = None) -> np.ndarray:
    """MXFP layer output for a set of tokens, float64 (the caller rounds to
    bf16).  The token rows are quantised once per token (a row's groups do
    not depend on which expert receives it, so quantising after the gather,
    as the pages order it, gives the same codes).  W1q/S1/W2q/S2 may be
    arrays indexed by expert or callables e -> array."""
    R = len(tokens)
    E_rows = np.asarray(E_rows, dtype=np.int64).reshape(R, -1)
    G_rows = np.asarray(G_rows, dtype=np.float64).reshape(R, -1)
    k = E_rows.shape[1]
    x = bf16_to_f64(X_rows_bits).reshape(R, -1)
    xq, sx = mx_quantize(x, fmt)
    counts, offsets, perm, inv = dispatch(E_rows, E)
    Hdim = x.shape[1]
    Yp = np.zeros((perm.shape[0], Hdim), dtype=np.float64)
    for e in range(E):
        if counts[e] == 0:
            continue
        rows = perm[offsets[e]:offsets[e + 1]] // k
        Yp[offsets[e]:offsets[e + 1]] = swiglu_expert_mx(
            xq[rows], sx[rows], _get(W1q, e), _get(S1, e), _get(W2q, e), _get(S2, e), fmt, wfmt)
    Y = np.zeros((R, Hdim), dtype=np.float64)
    for j in range(k):
        p = inv[np.arange(R) * k + j]
        ok = p >= 0
        Y[ok] += G_rows[ok, j:j + 1] * Yp[p[ok]]
    return Y


# ----------------------------------------------------------------------------- decision margins
# For the tests of a path that decides the activation codes of the quantised
# forms from float32 values, where this oracle decides them from float64
# values: if the exact SwiGLU output of an element lies within the float32
# path's error of a code boundary (or its group's maximum within that error of
# a power of two), the two may pick neighbouring codes.  The functions below
# bound, per output element, how far such decisions can move it.  They change
# none of the values computed above.
def _swiglu_with_bound(Z, dZ, I):
    """U = SiLU(Zx) * Zy and a bound dU on |U' - U| for any Z' within dZ of Z:
    SiLU(Zx + a) - SiLU(Zx) is at most (|SiLU'(Zx)| + |a| / 2) |a| (|SiLU''| <= 1/2),
    so |dU| <= (|SiLU'(Zx)| + dZx / 2) dZx (|Zy| + dZy) + |SiLU(Zx)| dZy."""
    Zx, Zy = Z[:, :I], Z[:, I:]
    dx, dy = dZ[:, :I], dZ[:, I:]
    U = _silu(Zx) * Zy
    dU = (np.abs(_silu_grad(Zx)) + 0.5 * dx) * dx * (np.abs(Zy) + dy) + np.abs(_silu(Zx)) * dy
    return U, dU


def _mx_decision_steps(U, dU, fmt: str) -> np.ndarray:
    """Per element of U [m, K]: the largest change of its Q_MX dequantised value
    (code times group scale) when the values move anywhere within dU, taking
    both the element's rounding and its group's shared exponent into account."""
    _, _, _, vmax = FP8_FORMATS[fmt]
    emax = int(np.floor(np.log2(vmax)))
    m, K = U.shape
    g = U.reshape(m, K // MX_GROUP, MX_GROUP)
    dg = dU.reshape(g.shape)

    def expo(amax):
        with np.errstate(divide="ignore"):
            ex = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))), -np.inf)
        return np.clip(ex - emax, -127, 127)[..., None]

    X = expo(np.abs(g).max(axis=-1))
    chosen = fp8_round(g / 2.0 ** X, fmt) * 2.0 ** X
    step = np.zeros_like(g)
    Xs = [X, expo(np.maximum(np.abs(g) - dg, 0.0).max(axis=-1)), expo((np.abs(g) + dg).max(axis=-1))]
    for Xa in Xs:
        for sgn in (-1.0, 1.0):
            alt = fp8_round((g + sgn * dg) / 2.0 ** Xa, fmt) * 2.0 ** Xa
            step = np.maximum(step, np.abs(alt - chosen))
    return step.reshape(m, K)


def swiglu_margin_mx(xq, sx, W1q, S1, W2q, S2, fmt: str, wfmt: str | None = None,
                     rel: float = 2.0 ** -12) -> np.ndarray:
    """Decision margin of swiglu_expert_mx's output [m, H]: sum over the
    activation elements of |largest change of the dequantised activation| x
    |Linear2 weight|, the activations moving within the float32 path's error:
    each pre-activation within rel times the sum of its products' magnitudes
    (a float32 accumulation of up to 2^13 exact products in blocks of 16
    stays within 2^-15 of that sum; rel leaves 8x)."""
    wfmt = fmt if wfmt is None else wfmt
    Xd = mx_dequantize(xq, sx, fmt)
    W1d = mx_dequantize(W1q, S1, wfmt)
    Z = Xd @ W1d.T
    dZ = rel * (np.abs(Xd) @ np.abs(W1d).T)
    I = np.asarray(W2q).shape[1]
    U, dU = _swiglu_with_bound(Z, dZ, I)
    return _mx_decision_steps(U, dU, fmt) @ np.abs(mx_dequantize(W2q, S2, wfmt)).T


def swiglu_margin_a8w8(q_rows, sx_rows, W1q, S1, W2q, S2, rel: float = 2.0 ** -18) -> np.ndarray:
    """Decision margin of swiglu_expert_a8w8's output [m, H]: sum over the
    activation elements of |largest change of code x row scale| x |Linear2
    weight (dequantised)|, the SwiGLU output moving within the float32 path's
    error (its integer products are exact; two dequantisation roundings and
    the SiLU evaluation stay within rel of each value) and the row scale
    within rel of itself."""
    C = np.asarray(q_rows, np.int64) @ np.asarray(W1q, np.int64).T
    Z = (C.astype(np.float64) * np.asarray(S1, np.float64)[None, :]) * np.asarray(sx_rows, np.float64)[:, None]
    I = np.asarray(W2q).shape[1]
    U, dU = _swiglu_with_bound(Z, rel * np.abs(Z), I)
    dU = dU + rel * np.abs(U)
    s = np.abs(U).max(axis=-1) / 127.0
    safe = np.where(s > 0, s, 1.0)[:, None]
    z = U / safe
    dz = dU / safe + rel * np.abs(z)
    q = round_half_away(z)
    step = np.maximum(np.abs(round_half_away(z - dz) - q), np.abs(round_half_away(z + dz) - q)) * safe
    step = np.where(s[:, None] > 0, step, 0.0)
    W2d = np.asarray(W2q, np.float64) * np.asarray(S2, np.float64)[:, None]
    return step @ np.abs(W2d).T


def _combine_margin(tokens, E_rows, G_rows, E, rows_margin):
    """Sum over a token's assignments of |gate| x its rows' margins."""
    R = len(tokens)
    E_rows = np.asarray(E_rows, dtype=np.int64).reshape(R, -1)
    G_rows = np.asarray(G_rows, dtype=np.float64).reshape(R, -1)
    k = E_rows.shape[1]
    counts, offsets, perm, inv = dispatch(E_rows, E)
    B = None
    for e in range(E):
        if counts[e] == 0:
            continue
        rows = perm[offsets[e]:offsets[e + 1]] // k
        Me = rows_margin(e, rows)
        if B is None:
            B = np.zeros((perm.shape[0], Me.shape[1]))
        B[offsets[e]:offsets[e + 1]] = Me
    out = None
    for j in range(k):
        p = inv[np.arange(R) * k + j]
        ok = p >= 0
        if B is None:
            break
        if out is None:
            out = np.zeros((R, B.shape[1]))
        out[ok] += np.abs(G_rows[ok, j:j + 1]) * B[p[ok]]
    return out


def margin_mx_tokens(tokens, X_rows_bits, E_rows, G_rows, W1q, S1, W2q, S2, E: int,
                     fmt: str, wfmt: str | None = None) -> np.ndarray:
    """Decision margin [R, H] of forward_mx_tokens' output (same arguments)."""
    R = len(tokens)
    x = bf16_to_f64(X_rows_bits).reshape(R, -1)
    xq, sx = mx_quantize(x, fmt)
    out = _combine_margin(tokens, E_rows, G_rows, E, lambda e, rows: swiglu_margin_mx(
        xq[rows], sx[rows], _get(W1q, e), _get(S1, e), _get(W2q, e), _get(S2, e), fmt, wfmt))
    return np.zeros((R, x.shape[1])) if out is None else out


def margin_a8w8_tokens(tokens, X_rows_bits, E_rows, G_rows, W1q, S1, W2q, S2, E: int) -> np.ndarray:
    """Decision margin [R, H] of forward_a8w8_tokens' output (same arguments)."""
    R = len(tokens)
    x32 = bf16_to_f64(X_rows_bits).reshape(R, -1).astype(np.float32)
    q, sx = quantize_rows_int8(x32, np.float32)
    out = _combine_margin(tokens, E_rows, G_rows, E, lambda e, rows: swiglu_margin_a8w8(
        q[rows], sx[rows], _get(W1q, e), _get(S1, e), _get(W2q, e), _get(S2, e)))
    return np.zeros((R, x32.shape[1])) if out is None else out

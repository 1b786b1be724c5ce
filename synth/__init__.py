"""Seeded synthetic inputs for the routed MoE FFN layer.

This module only draws numbers.  It holds none of the layer's arithmetic (no
routing, no FFN, no combine); the oracle under ``oracle/`` and the CUDA library
both consume what it returns, and neither is imported here.

Workloads (shapes follow the pages' own worked layers):

* ``c1`` tiny layer: T=128, H=256, E=8, top-2, I=128, sigmoid routing, bias 0.
* ``c2`` given-routing layer: T=4096, H=4096, E=32, top-8, I=1536; expert ids
  are k distinct uniform experts per token, gates are a softmax of k N(0,1)
  draws per token.
* ``c3`` V4-Pro-shaped layer: T=4096, H=7168, E=384, top-6, I=2048, one shared
  expert, sigmoid affinity, selection bias ~N(0, 0.1), alpha = 2.5, and a
  Zipf(1.1)-skewed expert load (see ``zipf_offsets``).
* ``c4`` hash-routed layer: the ``c3`` tensors, expert ids looked up in a
  seeded random ``tid2eid[128000, 6]`` table by uniform token ids.
* ``c5`` large-FFN layer: T=16384, H=8192, E=64, top-2, I=22016, softmax top-2.
* ``*s`` variants: the same recipes at sizes a CPU oracle finishes in seconds,
  still spanning several GEMM tiles with ragged tails.
* ``*_q`` variants: the A8W8-INT form of a workload -- int8 expert weights
  (codes ~ round(N(0, 40^2)) clipped to +-127) with per-output-channel fp32
  scales, no shared expert.

Value distributions: X ~ N(0,1); Wg and W1 (and the shared Ws1) ~ N(0, 1/H);
W2 (and Ws2) ~ N(0, 1/I).  Every floating-point tensor that the layer reads in
bf16 is rounded to bf16 with round-to-nearest-even before use.

Two back ends draw the same recipe: ``numpy`` (host arrays; bf16 carried as
uint16 bit patterns) for sizes the oracle can take whole, and ``torch`` (device
tensors) for the full-size workloads, whose weights (up to 69 GB) are too large
to draw on the host.  The two back ends use different generators and do not
produce the same numbers; a test always hands one drawing to both sides.
"""
from __future__ import annotations

import copy
import json
import math
import os

import numpy as np

__all__ = ["CONFIGS", "get_config", "make_inputs", "make_inputs_torch", "covering_tokens",
           "bf16_bits_from_f32", "f32_from_bf16_bits", "zipf_targets",
           "zipf_offsets"]

_HERE = os.path.dirname(os.path.abspath(__file__))

# score function codes shared by every layer of this repository's interface
SCORE_SIGMOID = 0
SCORE_SQRT_SOFTPLUS = 1
SCORE_SOFTMAX = 2
_SCORE_NAMES = {"sigmoid": SCORE_SIGMOID, "sqrt_softplus": SCORE_SQRT_SOFTPLUS,
                "softmax": SCORE_SOFTMAX}

_BASE = dict(shared=0, score="sigmoid", alpha=1.0, renorm=1, routing="topk",
             bias=False, skew=None, V=0, quant=None)

CONFIGS = {
    # --- the five workloads --------------------------------------------------
    "c1": dict(_BASE, T=128, H=256, E=8, k=2, I=128),
    "c2": dict(_BASE, T=4096, H=4096, E=32, k=8, I=1536, routing="given",
               score="softmax", renorm=0),
    "c3": dict(_BASE, T=4096, H=7168, E=384, k=6, I=2048, shared=1, alpha=2.5,
               bias=True, skew="zipf1.1"),
    "c4": dict(_BASE, T=4096, H=7168, E=384, k=6, I=2048, shared=1, alpha=2.5,
               bias=True, skew="zipf1.1", routing="hash", V=128000),
    "c5": dict(_BASE, T=16384, H=8192, E=64, k=2, I=22016, score="softmax",
               renorm=0),
    # --- oracle-sized variants of the same recipes ----------------------------
    "c1s": dict(_BASE, T=128, H=256, E=8, k=2, I=128),
    "c2s": dict(_BASE, T=333, H=512, E=12, k=4, I=320, routing="given",
                score="softmax", renorm=0),
    "c3s": dict(_BASE, T=257, H=448, E=40, k=6, I=192, shared=1, alpha=2.5,
                bias=True, skew="zipf1.1"),
    "c3s_sp": dict(_BASE, T=257, H=448, E=40, k=6, I=192, shared=1, alpha=2.5,
                   bias=True, score="sqrt_softplus"),
    "c4s": dict(_BASE, T=257, H=448, E=40, k=6, I=192, shared=1, alpha=2.5,
                bias=True, skew="zipf1.1", routing="hash", V=1000),
    "c5s": dict(_BASE, T=515, H=384, E=8, k=2, I=704, score="softmax",
                renorm=0),
}
# A8W8-INT variants ("mega_moe" page, A8W8 scenario): int8 expert weights with
# per-output-channel fp32 scales; no shared expert (the operator has none).
CONFIGS["c2s_q"] = dict(CONFIGS["c2s"], quant="a8w8")
CONFIGS["c3s_q"] = dict(CONFIGS["c3s"], shared=0, quant="a8w8")
CONFIGS["c5s_q"] = dict(CONFIGS["c5s"], quant="a8w8")
CONFIGS["c2_q"] = dict(CONFIGS["c2"], quant="a8w8")
# top-1 variant of the given-routing layer: the combine fuses into Linear2
CONFIGS["c2k1"] = dict(CONFIGS["c2"], k=1)
CONFIGS["c3_q"] = dict(CONFIGS["c3"], shared=0, quant="a8w8")
# MXFP forms: FP8 weight codes with E8M0 group scales (no shared expert).
# H and I are multiples of 128 (one block of 128 FP8 elements = 4 groups).
CONFIGS["c2s_mx"] = dict(CONFIGS["c2s"], I=384, quant="mx_e4m3")
CONFIGS["c3s_mx"] = dict(CONFIGS["c3s"], H=512, I=256, shared=0, quant="mx_e4m3")
CONFIGS["c3s_mx5"] = dict(CONFIGS["c3s"], H=512, I=256, shared=0, quant="mx_e5m2")
CONFIGS["c5s_mx"] = dict(CONFIGS["c5s"], I=640, quant="mx_e4m3")
CONFIGS["c2_mx"] = dict(CONFIGS["c2"], quant="mx_e4m3")
CONFIGS["c3_mx"] = dict(CONFIGS["c3"], shared=0, quant="mx_e4m3")
# MXFP4 weights: A8W4-FP (E4M3 activations) and A4W4-FP (E2M1 activations)
CONFIGS["c2s_mx4"] = dict(CONFIGS["c2s_mx"], quant="mx_e4m3_e2m1")
CONFIGS["c3s_mx4"] = dict(CONFIGS["c3s_mx"], quant="mx_e4m3_e2m1")
CONFIGS["c3s_mxa4"] = dict(CONFIGS["c3s_mx"], quant="mx_e2m1")
CONFIGS["c3s_mx54"] = dict(CONFIGS["c3s_mx"], quant="mx_e5m2_e2m1")
CONFIGS["c2_mx4"] = dict(CONFIGS["c2_mx"], quant="mx_e4m3_e2m1")
CONFIGS["c3_mx4"] = dict(CONFIGS["c3_mx"], quant="mx_e4m3_e2m1")
CONFIGS["c3_mxa4"] = dict(CONFIGS["c3_mx"], quant="mx_e2m1")
# V4-Pro expert shapes at a size one ncu capture can take (4.2 GB of weights,
# ~64 rows per expert as in c3, uniform load)
CONFIGS["c3p"] = dict(_BASE, T=512, H=7168, E=48, k=6, I=2048, shared=1, alpha=2.5, bias=True)
CONFIGS["c3p_mx"] = dict(CONFIGS["c3p"], shared=0, quant="mx_e4m3")
CONFIGS["c3p_q"] = dict(CONFIGS["c3p"], shared=0, quant="a8w8")
CONFIGS["c3p_mxa4"] = dict(CONFIGS["c3p"], shared=0, quant="mx_e2m1")
# the large-FFN layer's expert shapes and rows per expert (~512) at a size one
# ncu capture can take (4.3 GB of weights), with given routing (ids drawn as
# for c2): its Linear1 traffic ratio scales to c5
CONFIGS["c5p"] = dict(CONFIGS["c5"], T=1024, E=4, routing="given")
# parity cases of the large-FFN hidden size whose token rows exceed L2 (151 MB)
# with few, wide experts: the path that copies the rows into expert order and
# loads them by TMA; with and without a shared expert
CONFIGS["c5x"] = dict(CONFIGS["c5"], T=9216, E=8, I=256)
CONFIGS["c5x_sh"] = dict(CONFIGS["c5"], T=9216, E=8, I=256, shared=1)
# the V4-Pro router at full size with a token-sized FFN (I = 64): a workload
# whose routing kernels one ncu capture can take (1.1 GB of weights)
CONFIGS["c3r"] = dict(CONFIGS["c3"], I=64)
# the pages' own V4-Pro routing rule (sqrt-softplus affinity) at the c3 shapes
CONFIGS["c3_sp"] = dict(CONFIGS["c3"], score="sqrt_softplus", skew=None)
# the V4-Pro layer at the pages' own expert width f = 3072 (the model table of
# the Megatron DeepSeek-V4 page); the other recipes of c3 unchanged
CONFIGS["c3_f3072"] = dict(CONFIGS["c3"], I=3072)


def get_config(name_or_cfg, **overrides) -> dict:
    """Return a full config dict (a copy) for a workload name or a dict."""
    if isinstance(name_or_cfg, str):
        cfg = copy.deepcopy(CONFIGS[name_or_cfg])
        cfg["name"] = name_or_cfg
    else:
        cfg = dict(_BASE)
        cfg.update(name_or_cfg)
        cfg.setdefault("name", "custom")
    cfg.update(overrides)
    cfg["score_fn"] = _SCORE_NAMES[cfg["score"]]
    return cfg


# --------------------------------------------------------------------------- bf16
def bf16_bits_from_f32(x) -> np.ndarray:
    """float32 array -> bf16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def f32_from_bf16_bits(b) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------- skew
def zipf_targets(E: int, A: int, T: int, s: float = 1.1, seed: int = 77) -> np.ndarray:
    """Target assignment counts per expert: Zipf(s) over a seeded random rank
    order, clipped at T (a token picks an expert at most once), the clipped
    excess spread over the unclipped experts in proportion to their share."""
    rng = np.random.default_rng(seed)
    rank = rng.permutation(E)  # rank[e] = Zipf rank (0 = hottest) of expert e
    w = (rank + 1.0) ** (-s)
    tgt = w / w.sum() * A
    for _ in range(100):
        over = tgt > T
        if not over.any():
            break
        excess = (tgt[over] - T).sum()
        tgt[over] = T
        free = ~over & (tgt < T)
        tgt[free] += excess * tgt[free] / tgt[free].sum()
    return tgt


def zipf_offsets(cfg) -> np.ndarray | None:
    """Per-expert router logit offsets c_e that realise the Zipf load.

    The offsets enter the inputs only: X[:, 0] = 1 and Wg[0, e] = c_e, so the
    router's logit of expert e carries the extra term c_e.  They come from a
    table that ``synth/calibrate_skew.py`` writes once (it iterates the
    oracle's routing on seeded logits); ``None`` if the table lacks this shape.
    """
    path = os.path.join(_HERE, "skew_offsets.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        tab = json.load(f)
    key = f"E{cfg['E']}_k{cfg['k']}_{cfg['score']}_{cfg['skew']}"
    if key not in tab:
        return None
    return np.asarray(tab[key]["c"], dtype=np.float32)


# --------------------------------------------------------------------------- numpy
def _rng(seed: int, tensor_id: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(tensor_id)])


def _normal_bf16(seed, tid, shape, std) -> np.ndarray:
    x = _rng(seed, tid).standard_normal(size=shape, dtype=np.float32) * np.float32(std)
    return bf16_bits_from_f32(x)


# int8 weights: codes drawn as round(N(0, 40^2)) clipped to [-127, 127] and a
# per-output-channel scale near std / 40 (times U(0.75, 1.25)), so that
# code * scale has the spread of the bf16 weights of the same layer.  Layout
# [E, N, K]: one row per output channel, the contraction contiguous (the
# operator's weight1 [E, 2I, H] and weight2 [E, H, I]); scales [E, N].
_CODE_STD = 40.0


def _int8_weights(seed, tid, shape, std):
    rng = _rng(seed, 100 + tid)
    codes = np.clip(np.rint(rng.standard_normal(size=shape, dtype=np.float32) * _CODE_STD), -127, 127)
    scales = (std / _CODE_STD) * rng.uniform(0.75, 1.25, size=(shape[0], shape[1]))
    return codes.astype(np.int8), scales.astype(np.float32)


# MX weights (FP8 element codes, E8M0 group scales), drawn as bytes: a random
# sign bit and a magnitude code from a rounded normal in code space centred on
# the code of 1.0 (E4M3: 0x38, eight codes per octave; E5M2: 0x3C, four per
# octave), clipped to the finite codes; group scale codes 2^floor(log2 std)
# or half of it.  Layout [E, N, K] with scales [E, N, K/32] (K contiguous).
# FLOAT4_E2M1 weights (the A8W4-FP and A4W4-FP forms): magnitude code from a
# rounded N(4.5, 1.5) over the eight codes (values 0 .. 6, mostly 2 and 3), a
# random sign, two codes per byte with the even element in the low nibble;
# group scales 2^floor(log2(std / 2.5)) or half of it.
# quant name -> (activation format, weight format, code-space centre, width, top code)
_MX_FORMS = {"mx_e4m3": ("e4m3", "e4m3", 56.0, 8.0, 126), "mx_e5m2": ("e5m2", "e5m2", 60.0, 4.0, 123),
             "mx_e4m3_e2m1": ("e4m3", "e2m1", 4.5, 1.5, 7), "mx_e5m2_e2m1": ("e5m2", "e2m1", 4.5, 1.5, 7),
             "mx_e2m1": ("e2m1", "e2m1", 4.5, 1.5, 7)}


def mx_format(quant) -> str | None:
    """Activation element format ('e4m3', 'e5m2', 'e2m1') of an MX workload, else None."""
    return _MX_FORMS[quant][0] if quant in _MX_FORMS else None


def mx_weight_format(quant) -> str | None:
    """Weight element format of an MX workload, else None."""
    return _MX_FORMS[quant][1] if quant in _MX_FORMS else None


def _mx_scale_code(std, wfmt="e4m3") -> int:
    return 127 + int(math.floor(math.log2(std / 2.5 if wfmt == "e2m1" else std)))


def _pack_nibbles(codes):
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def _mx_weights(seed, tid, shape, std, quant):
    """Codes [.., K] (E2M1: packed [.., K/2]) and E8M0 scales [.., K/32]."""
    rng = _rng(seed, 200 + tid)
    _, wfmt, c0, w, top = _MX_FORMS[quant]
    mag = np.clip(np.rint(rng.standard_normal(size=shape, dtype=np.float32) * w + c0), 0, top)
    sbit = 3 if wfmt == "e2m1" else 7
    sign = rng.integers(0, 2, size=shape, dtype=np.uint8) << sbit
    s0 = _mx_scale_code(std, wfmt)
    scales = rng.integers(s0 - 1, s0 + 1, size=shape[:-1] + (shape[-1] // 32,), dtype=np.int32)
    codes = mag.astype(np.uint8) | sign
    if wfmt == "e2m1":
        codes = _pack_nibbles(codes)
    return codes, scales.astype(np.uint8)


def _distinct_rows(rng: np.random.Generator, n: int, E: int, k: int) -> np.ndarray:
    """n rows of k distinct experts each, a uniform random k-subset per row in
    random order: the first k of a random permutation (random sort keys)."""
    out = np.empty((n, k), dtype=np.int32)
    for r0 in range(0, n, 4096):
        keys = rng.random((min(4096, n - r0), E))
        out[r0:r0 + keys.shape[0]] = np.argsort(keys, axis=1, kind="stable")[:, :k]
    return out


def make_inputs(name_or_cfg, seed: int = 1234, **overrides) -> dict:
    """Host (numpy) drawing of one workload.  bf16 tensors are uint16 bits."""
    cfg = get_config(name_or_cfg, **overrides)
    T, H, E, k, I = cfg["T"], cfg["H"], cfg["E"], cfg["k"], cfg["I"]
    d = {"cfg": cfg}
    X = _rng(seed, 1).standard_normal(size=(T, H), dtype=np.float32)
    Wg = _rng(seed, 2).standard_normal(size=(H, E), dtype=np.float32) * np.float32(1.0 / math.sqrt(H))
    c = zipf_offsets(cfg) if cfg.get("skew") else None
    if c is not None and T > 0:
        X[:, 0] = 1.0
        Wg[0, :] = c
    d["X"] = bf16_bits_from_f32(X)
    d["Wg"] = bf16_bits_from_f32(Wg)
    d["bias"] = (_rng(seed, 3).standard_normal(size=E, dtype=np.float32) * np.float32(0.1)
                 if cfg["bias"] else None)
    if cfg.get("quant") == "a8w8":
        d["W1"], d["S1"] = _int8_weights(seed, 4, (E, 2 * I, H), 1.0 / math.sqrt(H))
        d["W2"], d["S2"] = _int8_weights(seed, 5, (E, H, I), 1.0 / math.sqrt(I))
    elif mx_format(cfg.get("quant")):
        d["W1"], d["S1"] = _mx_weights(seed, 4, (E, 2 * I, H), 1.0 / math.sqrt(H), cfg["quant"])
        d["W2"], d["S2"] = _mx_weights(seed, 5, (E, H, I), 1.0 / math.sqrt(I), cfg["quant"])
    else:
        d["W1"] = _normal_bf16(seed, 4, (E, H, 2 * I), 1.0 / math.sqrt(H))
        d["W2"] = _normal_bf16(seed, 5, (E, I, H), 1.0 / math.sqrt(I))
    if cfg["shared"]:
        d["Ws1"] = _normal_bf16(seed, 6, (H, 2 * I), 1.0 / math.sqrt(H))
        d["Ws2"] = _normal_bf16(seed, 7, (I, H), 1.0 / math.sqrt(I))
    else:
        d["Ws1"] = d["Ws2"] = None
    if cfg["routing"] == "given":
        rng = _rng(seed, 8)
        d["E_ids"] = _distinct_rows(rng, T, E, k)
        z = _rng(seed, 9).standard_normal(size=(T, k))
        z = np.exp(z - z.max(axis=1, keepdims=True))
        d["G"] = (z / z.sum(axis=1, keepdims=True)).astype(np.float32)
    if cfg["routing"] == "hash":
        V = cfg["V"]
        d["tid2eid"] = _distinct_rows(_rng(seed, 10), V, E, k)
        d["token_ids"] = _rng(seed, 11).integers(0, V, size=T, dtype=np.int32)
    return d


def upstream_grad(T: int, H: int, seed: int = 1234) -> np.ndarray:
    """The upstream gradient dL/dY [T, H] of a backward step: N(0, 1) in bf16
    (uint16 bits)."""
    return _normal_bf16(seed, 12, (T, H), 1.0)


# --------------------------------------------------------------------------- torch
def make_inputs_torch(name_or_cfg, seed: int = 1234, device="cuda", token_seed=None,
                      weights: bool = True, **overrides) -> dict:
    """Device (torch) drawing of one workload, for sizes too large for the host.

    bf16 tensors are ``torch.bfloat16``; the conversion from the fp32 draw is
    torch's round-to-nearest-even.  Large weights are drawn one expert at a
    time so the fp32 temporary stays small.  ``token_seed`` (default: seed)
    draws the token-side tensors (X, given ids and gates, token ids) so that
    several batches can share one set of weights; ``weights=False`` skips the
    expert weights (router-only use).
    """
    import torch

    cfg = get_config(name_or_cfg, **overrides)
    T, H, E, k, I = cfg["T"], cfg["H"], cfg["E"], cfg["k"], cfg["I"]
    dev = torch.device(device)

    tseed = seed if token_seed is None else token_seed

    def gen(tid, token_side=False):
        g = torch.Generator(device=dev)
        g.manual_seed(int(tseed if token_side else seed) * 1000 + tid)
        return g

    def normal(tid, shape, std, per_slice=False):
        g = gen(tid)
        if per_slice:
            out = torch.empty(shape, dtype=torch.bfloat16, device=dev)
            for i in range(shape[0]):
                out[i] = (torch.randn(shape[1:], generator=g, device=dev) * std).to(torch.bfloat16)
            return out
        return (torch.randn(shape, generator=g, device=dev) * std).to(torch.bfloat16)

    d = {"cfg": cfg}
    X = torch.randn((T, H), generator=gen(1, True), device=dev)
    Wg = torch.randn((H, E), generator=gen(2), device=dev) * (1.0 / math.sqrt(H))
    c = zipf_offsets(cfg) if cfg.get("skew") else None
    if c is not None and T > 0:
        X[:, 0] = 1.0
        Wg[0, :] = torch.from_numpy(c).to(dev)
    d["X"] = X.to(torch.bfloat16)
    d["Wg"] = Wg.to(torch.bfloat16)
    del X, Wg
    # the selection bias is small and drawn on the host, identically in both
    # back ends: the skew offsets were calibrated against these values
    d["bias"] = (torch.from_numpy(_rng(seed, 3).standard_normal(size=E, dtype=np.float32)
                                  * np.float32(0.1)).to(dev) if cfg["bias"] else None)
    def int8_weights(tid, shape, std):
        g = gen(100 + tid)
        codes = torch.empty(shape, dtype=torch.int8, device=dev)
        for i in range(shape[0]):
            codes[i] = (torch.randn(shape[1:], generator=g, device=dev) * _CODE_STD).round_().clamp_(-127, 127).to(torch.int8)
        u = torch.rand((shape[0], shape[1]), generator=g, device=dev) * 0.5 + 0.75
        return codes, (u * (std / _CODE_STD)).float().contiguous()

    def mx_weights(tid, shape, std):
        g = gen(200 + tid)
        _, wfmt, c0, w, top = _MX_FORMS[cfg["quant"]]
        packed = wfmt == "e2m1"
        cshape = shape[:-1] + (shape[-1] // 2,) if packed else shape
        codes = torch.empty(cshape, dtype=torch.uint8, device=dev)
        for i in range(shape[0]):
            mag = (torch.randn(shape[1:], generator=g, device=dev) * w + c0).round_().clamp_(0, top)
            sign = torch.randint(0, 2, shape[1:], generator=g, device=dev, dtype=torch.int32) * (8 if packed else 128)
            c = mag.to(torch.int32) + sign
            if packed:
                c = c[..., 0::2] | (c[..., 1::2] << 4)
            codes[i] = c.to(torch.uint8)
        s0 = _mx_scale_code(std, wfmt)
        scales = torch.randint(s0 - 1, s0 + 1, shape[:-1] + (shape[-1] // 32,), generator=g,
                               device=dev, dtype=torch.int32).to(torch.uint8)
        return codes, scales

    if weights and cfg.get("quant") == "a8w8":
        d["W1"], d["S1"] = int8_weights(4, (E, 2 * I, H), 1.0 / math.sqrt(H))
        d["W2"], d["S2"] = int8_weights(5, (E, H, I), 1.0 / math.sqrt(I))
    elif weights and mx_format(cfg.get("quant")):
        d["W1"], d["S1"] = mx_weights(4, (E, 2 * I, H), 1.0 / math.sqrt(H))
        d["W2"], d["S2"] = mx_weights(5, (E, H, I), 1.0 / math.sqrt(I))
    elif weights:
        d["W1"] = normal(4, (E, H, 2 * I), 1.0 / math.sqrt(H), per_slice=True)
        d["W2"] = normal(5, (E, I, H), 1.0 / math.sqrt(I), per_slice=True)
    else:
        d["W1"] = d["W2"] = None
    if cfg["shared"] and weights:
        d["Ws1"] = normal(6, (H, 2 * I), 1.0 / math.sqrt(H))
        d["Ws2"] = normal(7, (I, H), 1.0 / math.sqrt(I))
    else:
        d["Ws1"] = d["Ws2"] = None
    if cfg["routing"] == "given":
        g = gen(8, True)
        keys = torch.rand((T, E), generator=g, device=dev)
        d["E_ids"] = keys.topk(k, dim=1).indices.to(torch.int32).contiguous()
        z = torch.randn((T, k), generator=gen(9, True), device=dev)
        d["G"] = torch.softmax(z, dim=1).float().contiguous()
    if cfg["routing"] == "hash":
        V = cfg["V"]
        keys = torch.rand((V, E), generator=gen(10), device=dev)
        d["tid2eid"] = keys.topk(k, dim=1).indices.to(torch.int32).contiguous()
        d["token_ids"] = torch.randint(0, V, (T,), generator=gen(11, True), device=dev, dtype=torch.int32)
    return d


# --------------------------------------------------------------------------- samples
def covering_tokens(ids, E: int, n_min: int, n_extra: int = 0, seed: int = 5) -> np.ndarray:
    """Sorted indices of a seeded token sample that reaches every expert some
    token is routed to: for each expert in turn, the first token in a seeded
    random order that is routed to it, unless a token already taken reaches
    it; then random tokens up to n_min; then n_extra more random tokens.
    ``ids`` [T, k] are the tokens' expert ids (ids outside [0, E) reach no
    expert)."""
    ids = np.asarray(ids)
    rng = np.random.default_rng(seed)
    T = ids.shape[0]
    order = rng.permutation(T)
    pos = np.empty(T, np.int64)
    pos[order] = np.arange(T)
    taken = np.zeros(T, bool)
    for e in range(E):
        hit = np.nonzero((ids == e).any(axis=1))[0]
        if hit.size and not taken[hit].any():
            taken[hit[np.argmin(pos[hit])]] = True

    def fill(want):
        free = order[~taken[order]]
        taken[free[:max(0, min(want, T) - int(taken.sum()))]] = True
    fill(n_min)
    fill(int(taken.sum()) + n_extra)
    return np.nonzero(taken)[0]

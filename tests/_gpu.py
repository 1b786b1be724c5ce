"""Helpers for the GPU parity tests: move seeded inputs to the device, run the
library through its C ABI, fetch tensors back for the oracle, and the output
tolerance."""
from __future__ import annotations

import numpy as np
import torch

import mixture_experts_ffn_route_gb300 as moe

DEV = torch.device("cuda:0")

# Y tolerance: the layer's stated bar, max |err| <= 2e-2 * RMS(Y_ref) with
# fp32 accumulation and bf16 I/O, where Y_ref is the oracle's output rounded
# once to bf16 (round to nearest even) and the oracle rounds where the path
# keeps low-precision numbers between its kernels (the SwiGLU rows in bf16;
# the quantised forms quantise their activations).
#
# One exception is counted, not absorbed: the GPU sums in another order than
# the oracle, so where the exact output lies within a few 1e-7 of a bf16
# rounding boundary the two round it to neighbouring bf16 values.  On the
# largest outputs one unit in the last place (2^-7 of the value's binade) can
# exceed 2e-2 RMS.  An element beyond the bar passes only if it is exactly such
# a neighbour (|err| <= the bar + one ulp of Y_ref), and such elements may be
# at most Y_FLIP_FRACTION of the output (a real defect moves many elements, by
# more than one ulp).  How often the two roundings part grows with the float32
# accumulation error, i.e. with the contraction length: the most seen is
# 1.4e-4 of the outputs on the large-FFN layer (K = 22016 in Linear2) and
# 6e-4 in the A8W8 form, whose Linear2 rows are kept in bf16.
Y_RTOL_RMS = 2e-2
Y_FLIP_FRACTION = 1e-3
# Against the exact (unrounded-intermediate) oracle the error RMS stays under
# this fraction of RMS: the bf16 SwiGLU rows contribute about 2^-9 / sqrt(3)
# of RMS, the final rounding about 2^-9 / sqrt(3) of each element.
Y_EXACT_RMS_ERR = 3e-3
# (case, max|err|/RMS, elements beyond the bar (one-ulp flips), elements,
# max|err|/RMS vs the exact oracle or None, beyond the bar vs the exact oracle)
Y_STATS = []
# Gates: g = alpha * a_e / sum a (or a softmax value) from fp32 tensor-core
# logits.  d(log g) is a difference of logit errors weighted by slopes <= 1, so
# |dg/g| <= 2 max|dl|; the router tests hold |dl| (score space) under 1e-4,
# hence a relative tolerance of 2e-4.
G_RTOL = 2e-4


def bf(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(DEV)


def host_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 device tensor -> uint16 host array of its bit patterns."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_device(d: dict) -> dict:
    """Host drawing (numpy; bf16 as uint16 bits) -> the same tensors on the GPU."""
    out = {"cfg": d["cfg"]}
    for key, v in d.items():
        if key == "cfg":
            continue
        if v is None or isinstance(v, torch.Tensor):
            out[key] = v
        elif v.dtype == np.uint16:
            out[key] = bf(v)
        else:
            out[key] = torch.from_numpy(np.ascontiguousarray(v)).to(DEV)
    return out


def to_host(dd: dict) -> dict:
    out = {"cfg": dd["cfg"]}
    for key, v in dd.items():
        if key == "cfg":
            continue
        if v is None:
            out[key] = None
        elif v.dtype == torch.bfloat16:
            out[key] = host_bits(v)
        else:
            out[key] = v.cpu().numpy()
    return out


def mixed_load_ids(T, E):
    """Top-2 expert ids [T, 2] under which some groups span several 128-row
    tiles and the rest one partial tile: expert 0 takes the first min(T, 450)
    tokens, expert 3 the first 260 and every fifth token after 450, experts
    1-5 share the rest of column 0 and experts 6 to E-1 the rest of column 1.
    The grouped GEMMs then interleave dense and sparse groups in one launch."""
    assert E >= 12
    t = np.arange(T)
    first = np.where(t < 450, 0, 1 + t % 5)
    second = np.where(t < 260, 3, 6 + t % (E - 6))
    return np.stack([first, second], axis=1).astype(np.int32)


def params(cfg, **kw):
    c = dict(cfg)
    c.update(kw)
    return moe.params_from_config(c)


def run_route(p, dd, ws):
    T, k = p.T, p.k
    E_ids = torch.full((T, k), -7, dtype=torch.int32, device=DEV)
    G = torch.full((T, k), float("nan"), dtype=torch.float32, device=DEV)
    if dd["cfg"]["routing"] == "hash":
        moe.moe_route(p, dd["X"], dd["Wg"], None, dd["token_ids"], dd["tid2eid"], dd["cfg"]["V"],
                      E_ids, G, ws)
    else:
        moe.moe_route(p, dd["X"], dd["Wg"], dd.get("bias"), None, None, 0, E_ids, G, ws)
    return E_ids, G


def run_forward(p, dd, E_ids, G, ws, Y=None):
    if Y is None:
        Y = torch.full((p.T, p.H), float("nan"), dtype=torch.bfloat16, device=DEV)
    moe.moe_forward(p, dd["X"], E_ids, G, dd["W1"], dd["W2"], dd.get("Ws1"), dd.get("Ws2"), Y, ws)
    return Y


def _rne_bf16(y):
    """float64 -> nearest bf16 value (ties to even), as float64."""
    import oracle
    return oracle.round_to_bf16(np.asarray(y, dtype=np.float64))


def bf16_ulp(v):
    """Spacing of the bf16 values at |v| (8 significant bits): 2^(floor(log2|v|) - 7)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 7), 2.0 ** -133)


def check_y(Y_gpu, Y_ref, what="", Y_exact=None, slack=None):
    """Assert |y - bf16(Y_ref)| <= 2e-2 * RMS(bf16(Y_ref)) element by element,
    apart from counted one-ulp rounding flips (see Y_FLIP_FRACTION).

    Y_ref: the oracle's float64 output with the path's intermediate rounding
    points.  slack (optional, per element): the oracle's bound on what its
    activation-code decisions that sit within the GPU's float32 rounding of a
    decision boundary can move the element (quantised forms); it adds to the
    bar.  Y_exact (optional): the oracle without intermediate rounding; the
    error against its bf16 rounding is recorded and its RMS held under
    Y_EXACT_RMS_ERR of RMS.  Returns max|err|/RMS."""
    y = Y_gpu.float().cpu().numpy().astype(np.float64) if isinstance(Y_gpu, torch.Tensor) else Y_gpu
    assert np.isfinite(y).all(), f"{what}: non-finite output"
    ref = _rne_bf16(Y_ref)
    rms = float(np.sqrt((ref ** 2).mean()))
    err = np.abs(y - ref)
    allow = Y_RTOL_RMS * rms + (0.0 if slack is None else np.asarray(slack))
    beyond = err > allow
    flips = beyond & (err <= allow + bf16_ulp(ref) * (1 + 1e-9))
    hard = beyond & ~flips
    ratio = float(err.max() / rms) if rms > 0 else float(err.max())
    x_ratio = x_beyond = None
    if Y_exact is not None:
        xref = _rne_bf16(Y_exact)
        xrms = float(np.sqrt((xref ** 2).mean()))
        xerr = np.abs(y - xref)
        x_ratio = float(xerr.max() / xrms)
        x_beyond = int((xerr > Y_RTOL_RMS * xrms).sum())
    n_flip = int(flips.sum())
    Y_STATS.append((what, ratio, n_flip, int(err.size), x_ratio, x_beyond))
    assert not hard.any(), (
        f"{what}: {int(hard.sum())} of {err.size} elements beyond the bar by more than one ulp "
        f"(max|err|/RMS = {ratio:.3e})")
    assert n_flip <= max(2, Y_FLIP_FRACTION * err.size), (
        f"{what}: {n_flip} of {err.size} one-ulp flips beyond the bar")
    if Y_exact is not None:
        xe = np.sqrt(((y - xref) ** 2).mean())
        assert xe <= Y_EXACT_RMS_ERR * xrms, f"{what}: error RMS vs the exact oracle {xe / xrms:.3e}"
    return ratio


def check_y_layer(Y_gpu, what, X, ids, G, W1, W2, Ws1=None, Ws2=None):
    """check_y for the bf16 forward of a whole small layer: the oracle with
    the SwiGLU rows rounded to bf16 (the path's one intermediate rounding
    point) sets the bar; the exact oracle is compared as well."""
    import oracle
    Y_r, _ = oracle.forward(X, ids, G, W1, W2, Ws1, Ws2, act_round_bf16=True)
    Y_x, _ = oracle.forward(X, ids, G, W1, W2, Ws1, Ws2)
    return check_y(Y_gpu, Y_r, what, Y_exact=Y_x)


def check_gates(G_gpu, G_ref, what=""):
    g = G_gpu.cpu().numpy().astype(np.float64) if isinstance(G_gpu, torch.Tensor) else G_gpu
    np.testing.assert_allclose(g, G_ref, rtol=G_RTOL, atol=1e-7, err_msg=what)

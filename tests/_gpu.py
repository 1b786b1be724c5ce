"""Helpers for the GPU parity tests: move seeded inputs to the device, run the
library through its C ABI, fetch tensors back for the oracle, and the output
tolerance."""
from __future__ import annotations

import numpy as np
import torch

import mixture_experts_ffn_route_gb300 as moe

DEV = torch.device("cuda:0")

# Y tolerance.  The layer's stated bar is max |err| <= 2e-2 * RMS(Y_ref) with
# fp32 accumulation and bf16 I/O.  The bf16 output format alone rounds each
# element by up to 2^-8 of its magnitude, which exceeds 2e-2 * RMS on the
# largest elements of a Gaussian-like output, so the bound is applied to the
# error beyond that rounding: |y - y_ref| <= 2e-2 * RMS(Y_ref) + 2^-8 |y_ref|.
Y_RTOL_RMS = 2e-2
Y_OUT_ULP = 2.0 ** -8
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


def check_y(Y_gpu, Y_ref, what=""):
    """Assert the output tolerance; return (max|err|/RMS, worst err/allowance)."""
    y = Y_gpu.float().cpu().numpy().astype(np.float64) if isinstance(Y_gpu, torch.Tensor) else Y_gpu
    assert np.isfinite(y).all(), f"{what}: non-finite output"
    rms = float(np.sqrt((Y_ref ** 2).mean()))
    err = np.abs(y - Y_ref)
    allow = Y_RTOL_RMS * rms + Y_OUT_ULP * np.abs(Y_ref)
    worst = float((err / allow).max())
    assert worst <= 1.0, (f"{what}: worst |err|/allowance = {worst:.3f} "
                          f"(max|err|/RMS = {err.max() / rms:.3e})")
    return float(err.max() / rms), worst


def check_gates(G_gpu, G_ref, what=""):
    g = G_gpu.cpu().numpy().astype(np.float64) if isinstance(G_gpu, torch.Tensor) else G_gpu
    np.testing.assert_allclose(g, G_ref, rtol=G_RTOL, atol=1e-7, err_msg=what)

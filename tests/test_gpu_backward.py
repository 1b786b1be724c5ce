"""Parity of the layer backward (moe_forward_train + moe_backward) with the
oracle's float64 chain rule: input, weight, router and mixing-weight
gradients for top-k (sigmoid, sqrt-softplus, softmax) and hash routing, with
and without the shared expert, and sampled tokens / experts at full size."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_route_gb300 as moe
import oracle
import synth
from _gpu import DEV, bf, host_bits, params, run_route, to_device

pytestmark = pytest.mark.gpu

# Gradient tolerance, against the oracle rounding to bf16 where the path keeps
# bf16 tensors (pre-activations, SwiGLU output, gate-scaled row gradients, dH,
# logit gradient).  The GPU holds those intermediates in fp32 before rounding
# them and the oracle in float64, so a value sitting near a bf16 rounding
# boundary can round to the neighbouring bf16 number on one side; each such
# flip moves the products it enters by at most 2^-8 of themselves (one more
# 2^-8 for a flip inside the SwiGLU derivative).  Hence three conditions:
#   every element:      |err| <= 2e-2 RMS(ref) + 2^-7 mass   (mass: the sum of
#                       the magnitudes of the products of the last contraction)
#   all but 0.1%:       |err| <= 2e-2 RMS(ref)   (+ 2^-8 |ref| for bf16 dX)
#   the whole tensor:   RMS(err) <= 1e-2 RMS(ref)
# A wrong index, sign or term moves whole tiles by O(RMS) and fails the last
# two.  The distance of the rounded oracle from the exact float64 gradient,
# the cost of bf16 operands, is bounded separately below.
RTOL_RMS = 2e-2
FLIP_FRACTION = 1e-3
RMS_ERR = 1e-2
# RMS distance of the rounded oracle from the exact gradient, relative to the
# exact gradient's RMS: five rounding points, each 2^-9 / sqrt(3)
EXACT_RMS = 5 * 2.0 ** -9 / 3 ** 0.5


def _check(got, ref, name, mass, bf16_out=False):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, name
    assert np.all(np.isfinite(got)), name
    rms = np.sqrt((ref ** 2).mean())
    err = np.abs(got - ref)
    tight = RTOL_RMS * rms + (2.0 ** -8 * np.abs(ref) if bf16_out else 0.0)
    assert np.all(err <= tight + 2.0 ** -7 * np.asarray(mass)), (name, "loose", float(err.max()), float(rms))
    frac = float((err > tight).mean())
    assert frac <= FLIP_FRACTION, (name, "tight fraction", frac)
    assert np.sqrt((err ** 2).mean()) <= RMS_ERR * rms, (name, "rms", float(np.sqrt((err ** 2).mean())), float(rms))


@pytest.fixture(scope="module", autouse=True)
def _lib(built_lib):
    moe.lib()
    torch.cuda.set_device(DEV)


def _run(p, dd, E_ids, G, dY):
    c = dd["cfg"]
    T, H, E, k, I = c["T"], c["H"], c["E"], c["k"], c["I"]
    ws = moe.alloc_workspace_train(p, DEV)
    Y = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    moe.moe_forward_train(p, dd["X"], E_ids, G, dd["W1"], dd["W2"], dd["Ws1"], dd["Ws2"], Y, ws)
    f32 = lambda *s: torch.full(s, float("nan"), dtype=torch.float32, device=DEV)  # noqa: E731
    out = {"dX": torch.full((T, H), float("nan"), dtype=torch.bfloat16, device=DEV),
           "dWg": f32(H, E), "dW1": f32(E, H, 2 * I), "dW2": f32(E, I, H), "dG": f32(T, k)}
    if c["shared"]:
        out["dWs1"], out["dWs2"] = f32(H, 2 * I), f32(I, H)
    else:
        out["dWs1"] = out["dWs2"] = None
    moe.moe_backward(p, dd["X"], dd["Wg"], E_ids, G, dd["W1"], dd["W2"], dd["Ws1"], dd["Ws2"], dY,
                     out["dX"], out["dWg"], out["dW1"], out["dW2"], out["dWs1"], out["dWs2"], out["dG"], ws)
    moe.moe_sync_status(ws)
    return out


# c5s at T = 1040 averages 260 routed rows per expert (several row tiles each)
@pytest.mark.parametrize("name,T", [("c1s", None), ("c3s", None), ("c3s_sp", None), ("c4s", None),
                                    ("c5s", None), ("c5s", 1040)])
def test_backward_matches_oracle(name, T):
    h = synth.make_inputs(name, **({"T": T} if T else {}))
    c = h["cfg"]
    dd = to_device(h)
    p = params(c)
    ws_r = moe.alloc_workspace(p, DEV)
    E_ids, G = run_route(p, dd, ws_r)
    moe.moe_sync_status(ws_r)
    dYb = synth.upstream_grad(c["T"], c["H"])
    out = _run(p, dd, E_ids, G, bf(dYb))
    ids = E_ids.cpu().numpy()
    dY = oracle.bf16_to_f64(dYb)
    ref = oracle.backward(h["X"], h["Wg"], ids, dY, h["W1"], h["W2"], h["Ws1"], h["Ws2"], c["score_fn"],
                          c["alpha"], c["renorm"], round_bf16=True, mass=True)
    exact = oracle.backward(h["X"], h["Wg"], ids, dY, h["W1"], h["W2"], h["Ws1"], h["Ws2"], c["score_fn"],
                            c["alpha"], c["renorm"])
    _check(out["dX"].float().cpu().numpy(), ref["dX"], name + " dX", ref["mass_dX"], bf16_out=True)
    for key in ("dWg", "dW1", "dW2", "dG") + (("dWs1", "dWs2") if c["shared"] else ()):
        got = out[key].cpu().numpy()
        _check(got, ref[key], f"{name} {key}", ref["mass_" + key])
        # against the exact gradient.  Each of the five bf16 rounding points
        # moves its operand by a relative error of RMS 2^-9 / sqrt(3); a
        # gradient depends on at most five of them with sensitivities of order
        # one, so the rounded oracle's distance d = ref - exact has RMS at most
        # EXACT_RMS (tests/test_oracle_pins.py checks this on the CPU).  The
        # GPU is within the parity tolerance of ref, so element by element
        # |got - exact| <= |d| + 2e-2 RMS + 2^-7 mass, and in RMS the two add.
        d = np.abs(ref[key] - exact[key])
        rms = np.sqrt((exact[key] ** 2).mean())
        e = np.abs(got - exact[key])
        assert np.all(e <= d + RTOL_RMS * np.sqrt((ref[key] ** 2).mean()) + 2.0 ** -7 * ref["mass_" + key]), \
            (name, key, "exact, per element")
        assert np.sqrt((e ** 2).mean()) <= (EXACT_RMS + RMS_ERR) * rms, (name, key, "exact, RMS")


def test_backward_is_deterministic():
    h = synth.make_inputs("c3s")
    c = h["cfg"]
    dd = to_device(h)
    p = params(c)
    ws_r = moe.alloc_workspace(p, DEV)
    E_ids, G = run_route(p, dd, ws_r)
    dY = bf(synth.upstream_grad(c["T"], c["H"]))
    a = _run(p, dd, E_ids, G, dY)
    b = _run(p, dd, E_ids, G, dY)
    for key in ("dX", "dWg", "dW1", "dW2", "dWs1", "dWs2", "dG"):
        assert torch.equal(a[key].view(torch.int16) if key == "dX" else a[key],
                           b[key].view(torch.int16) if key == "dX" else b[key]), key


@pytest.mark.parametrize("name", ["c3", "c5x_sh"])
def test_backward_full_size_sampled(name):
    """V4-Pro shapes, and the large-FFN hidden size with token rows beyond L2
    (whose forward loads them by TMA from a copy in expert order): dX of
    sampled tokens (each token's input gradient depends on its own path only)
    and the weight gradients of two experts (all of their rows)."""
    dd = synth.make_inputs_torch(name, device=DEV)
    c = dd["cfg"]
    T, H, E, k = c["T"], c["H"], c["E"], c["k"]
    p = params(c)
    ws_r = moe.alloc_workspace(p, DEV)
    E_ids, G = run_route(p, dd, ws_r)
    moe.moe_sync_status(ws_r)
    dYb = synth.upstream_grad(T, H)
    out = _run(p, dd, E_ids, G, bf(dYb))
    ids = E_ids.cpu().numpy()
    hX = host_bits(dd["X"])
    Wg = host_bits(dd["Wg"])
    dY = oracle.bf16_to_f64(dYb)
    W1 = lambda e: host_bits(dd["W1"][e])  # noqa: E731
    W2 = lambda e: host_bits(dd["W2"][e])  # noqa: E731
    Ws1, Ws2 = host_bits(dd["Ws1"]), host_bits(dd["Ws2"])
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([[0, T - 1], rng.choice(T, 4, replace=False)]))
    ref = oracle.backward(hX[rows], Wg, ids[rows], dY[rows], W1, W2, Ws1, Ws2, c["score_fn"], c["alpha"],
                          c["renorm"], E=E, round_bf16=True, mass=True, weight_experts=[])
    _check(out["dX"][torch.from_numpy(rows).to(DEV)].float().cpu().numpy(), ref["dX"], f"{name} dX",
           ref["mass_dX"], bf16_out=True)
    _check(out["dG"].cpu().numpy()[rows], ref["dG"], f"{name} dG", ref["mass_dG"])
    counts = np.bincount(ids.reshape(-1), minlength=E)
    for e in [int(np.argmin(np.where(counts > 0, counts, 1 << 30))), int(np.argsort(counts)[E // 2])]:
        toks = np.where((ids == e).any(axis=1))[0]
        r = oracle.backward(hX[toks], Wg, ids[toks], dY[toks], W1, W2, None, None, c["score_fn"], c["alpha"],
                            c["renorm"], E=E, round_bf16=True, mass=True, weight_experts=[e])
        _check(out["dW1"][e].cpu().numpy(), r["dW1"][e], f"{name} dW1[{e}] ({len(toks)} rows)", r["mass_dW1"][e])
        _check(out["dW2"][e].cpu().numpy(), r["dW2"][e], f"{name} dW2[{e}]", r["mass_dW2"][e])

"""Parity of the MX forms (FP8 / FP4 codes with E8M0 group scales, the MXFP
scenario of the "mega_moe" page: A8W8-FP, A8W4-FP, A4W4-FP) with the oracle's
restatement: the token quantisation bit-exact, the layer output within the Y
tolerance."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_route_gb300 as moe
import oracle
import synth
from _gpu import DEV, bf, check_y, host_bits, mixed_load_ids, params, run_route, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(built_lib):
    moe.lib()
    torch.cuda.set_device(DEV)


def _fmt(cfg):
    return synth.mx_format(cfg["quant"])


def _wfmt(cfg):
    return synth.mx_weight_format(cfg["quant"])


def _codes(w, wfmt):
    """Weight codes as the oracle takes them: one code per element."""
    return oracle.unpack_e2m1(w) if wfmt == "e2m1" else w


def _run(p, fmt, dd, E_ids, G, wfmt=None):
    ws = moe.alloc_workspace_mx(p, DEV)
    Y = torch.full((p.T, p.H), float("nan"), dtype=torch.bfloat16, device=DEV)
    moe.moe_forward_mx(p, moe.MX_FORMATS[fmt], dd["X"], E_ids, G, dd["W1"], dd["S1"], dd["W2"], dd["S2"], Y, ws,
                       wfmt=moe.MX_FORMATS[wfmt or fmt])
    moe.moe_sync_status(ws)
    return Y


def _quant_rows(fmt):
    """Rows of groups at magnitudes 2^-40 .. 2^40, a group of zeros, tiny values
    beside a large maximum (codes of signed zero), and a group whose scaled
    values are the exact midpoints between neighbouring FP8 values."""
    rng = np.random.default_rng(17)
    R, C = 67, 512
    x = rng.standard_normal((R, C // 32, 32)) * 2.0 ** rng.uniform(-40, 40, (R, C // 32, 1))
    x[1, 3] = 0.0
    x[2, 5] = rng.standard_normal(32) * 1e-9
    x[2, 5, 0] = 300.0
    grid = oracle.fp8_decode(np.arange(8 if fmt == "e2m1" else 128), fmt)
    grid = grid[np.isfinite(grid)]
    mids = (grid[:-1] + grid[1:]) / 2
    emax = {"e4m3": 8, "e5m2": 15, "e2m1": 2}[fmt]
    top = mids[(mids >= 1.0) & (mids < 2.0 ** emax)]
    g = rng.choice(top, 31)
    x[3, 0] = np.concatenate([[2.0 ** emax], g * rng.choice([-1, 1], 31)])   # shared exponent 0
    return oracle.f64_to_bf16_bits(x.reshape(R, C))


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2", "e2m1"])
def test_mx_token_quantisation_is_bit_exact(fmt):
    xb = _quant_rows(fmt)
    R, C = xb.shape
    X = bf(xb)
    Cb = C // 2 if fmt == "e2m1" else C
    Q = torch.full((R, Cb), 0xAB, dtype=torch.uint8, device=DEV)
    S = torch.full((R, C // 32), 0xAB, dtype=torch.uint8, device=DEV)
    moe.moe_quantize_mx(moe.MX_FORMATS[fmt], X, Q, S)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.mx_quantize(oracle.bf16_to_f64(xb).astype(np.float32), fmt, np.float32)
    assert np.array_equal(S.cpu().numpy(), s_ref)
    assert np.array_equal(_codes(Q.cpu().numpy(), fmt), q_ref)


@pytest.mark.parametrize("name", ["c2s_mx", "c3s_mx", "c3s_mx5", "c5s_mx", "c2s_mx4", "c3s_mx4", "c3s_mxa4",
                                  "c3s_mx54"])
def test_mx_forward_matches_oracle(name):
    h = synth.make_inputs(name)
    c = h["cfg"]
    dd = to_device(h)
    p = params(c)
    if c["routing"] == "given":
        ids, G = h["E_ids"], h["G"].astype(np.float64)
        E_ids, Gd = dd["E_ids"], dd["G"]
    else:
        ws_r = moe.alloc_workspace(p, DEV)
        E_ids, Gd = run_route(p, dd, ws_r)
        moe.moe_sync_status(ws_r)
        ids, _, _ = oracle.route(h["X"], h["Wg"], h["bias"], c["score_fn"], c["k"], c["alpha"], c["renorm"])
        assert np.array_equal(E_ids.cpu().numpy(), ids)
        G = Gd.cpu().numpy().astype(np.float64)
    Y = _run(p, _fmt(c), dd, E_ids, Gd, _wfmt(c))
    wf = _wfmt(c)
    Y_ref = oracle.forward_mx_tokens(np.arange(c["T"]), h["X"], ids, G, _codes(h["W1"], wf), h["S1"],
                                     _codes(h["W2"], wf), h["S2"], E=c["E"], fmt=_fmt(c), wfmt=wf)
    slack = oracle.margin_mx_tokens(np.arange(c["T"]), h["X"], ids, G, _codes(h["W1"], wf), h["S1"],
                                     _codes(h["W2"], wf), h["S2"], E=c["E"], fmt=_fmt(c), wfmt=wf)
    check_y(Y, Y_ref, name, slack=slack)


def test_mx_is_deterministic_and_rejects_a_shared_expert():
    h = synth.make_inputs("c2s_mx")
    dd = to_device(h)
    p = params(h["cfg"])
    Y1 = _run(p, "e4m3", dd, dd["E_ids"], dd["G"]).clone()
    Y2 = _run(p, "e4m3", dd, dd["E_ids"], dd["G"])
    assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))
    ps = params(h["cfg"], shared=1)
    ws = moe.alloc_workspace_mx(ps, DEV)
    with pytest.raises(moe.MoEError) as ex:
        moe.moe_forward_mx(ps, 0, dd["X"], dd["E_ids"], dd["G"], dd["W1"], dd["S1"], dd["W2"], dd["S2"],
                           torch.empty_like(dd["X"]), ws)
    assert ex.value.code == moe.MOE_ERR_UNSUPPORTED


@pytest.mark.parametrize("name,n_rows", [("c3_mx", 6), ("c2_mx", 6), ("c3_mx4", 4), ("c3_mxa4", 4)])
def test_mx_full_size_sampled(name, n_rows):
    dd = synth.make_inputs_torch(name, device=DEV)
    c = dd["cfg"]
    T, E = c["T"], c["E"]
    p = params(c)
    if c["routing"] == "given":
        E_ids, G = dd["E_ids"], dd["G"]
    else:
        ws_r = moe.alloc_workspace(p, DEV)
        E_ids, G = run_route(p, dd, ws_r)
        moe.moe_sync_status(ws_r)
    wf = _wfmt(c)
    Y = _run(p, _fmt(c), dd, E_ids, G, wf)
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([[0, T - 1], rng.choice(T, n_rows, replace=False)]))
    hX = host_bits(dd["X"])
    ids = E_ids.cpu().numpy()
    Gh = G.cpu().numpy().astype(np.float64)
    W1 = lambda e: _codes(dd["W1"][e].cpu().numpy(), wf)  # noqa: E731
    W2 = lambda e: _codes(dd["W2"][e].cpu().numpy(), wf)  # noqa: E731
    S1 = lambda e: dd["S1"][e].cpu().numpy()  # noqa: E731
    S2 = lambda e: dd["S2"][e].cpu().numpy()  # noqa: E731
    Y_ref = oracle.forward_mx_tokens(rows, hX[rows], ids[rows], Gh[rows], W1, S1, W2, S2, E=E, fmt=_fmt(c),
                                     wfmt=wf)
    slack = oracle.margin_mx_tokens(rows, hX[rows], ids[rows], Gh[rows], W1, S1, W2, S2, E=E, fmt=_fmt(c),
                                     wfmt=wf)
    check_y(Y[torch.from_numpy(rows).to(DEV)], Y_ref, name, slack=slack)


# Ragged and degenerate shapes (H and I multiples of 128, as the MX forms
# need): one token, k = E, every token on one expert (several 128-row tiles,
# the last partial, other experts empty), for FP8 and FP4 weights.
EDGE_MX = [
    dict(T=1, H=128, E=4, k=2, I=128),
    dict(T=17, H=256, E=5, k=5, I=128),
    dict(T=300, H=256, E=6, k=1, I=256, hot=True),
    dict(T=260, H=384, E=9, k=3, I=384),
    dict(T=700, H=256, E=12, k=2, I=256, mixed=True),
]


# mx_e2m1 takes the packed kind::mxf4 path where H and I are multiples of 256
# (the T=300 shape) and the spread kind::mxf8f6f4 path elsewhere
@pytest.mark.parametrize("quant", ["mx_e4m3", "mx_e4m3_e2m1", "mx_e2m1"])
@pytest.mark.parametrize("shape", EDGE_MX, ids=lambda s: "T{T}_H{H}_E{E}_k{k}_I{I}".format(**s))
def test_mx_edge_shapes(shape, quant):
    shape = dict(shape)
    hot = shape.pop("hot", False)
    mixed = shape.pop("mixed", False)
    h = synth.make_inputs(dict(shape, routing="given", score="softmax", renorm=0, quant=quant), seed=99)
    if hot:
        h["E_ids"][:] = 0
    if mixed:
        h["E_ids"][:] = mixed_load_ids(shape["T"], shape["E"])
    c = h["cfg"]
    dd = to_device(h)
    p = params(c)
    wf = _wfmt(c)
    Y = _run(p, _fmt(c), dd, dd["E_ids"], dd["G"], wf)
    Y_ref = oracle.forward_mx_tokens(np.arange(c["T"]), h["X"], h["E_ids"], h["G"].astype(np.float64),
                                     _codes(h["W1"], wf), h["S1"], _codes(h["W2"], wf), h["S2"], E=c["E"],
                                     fmt=_fmt(c), wfmt=wf)
    slack = oracle.margin_mx_tokens(np.arange(c["T"]), h["X"], h["E_ids"], h["G"].astype(np.float64),
                                     _codes(h["W1"], wf), h["S1"], _codes(h["W2"], wf), h["S2"], E=c["E"],
                                     fmt=_fmt(c), wfmt=wf)
    check_y(Y, Y_ref, f"{shape} {quant}", slack=slack)


def test_mx_with_no_tokens_writes_nothing():
    h = synth.make_inputs("c2s_mx")
    dd = to_device(h)
    p = params(h["cfg"], T=0)
    ws = moe.alloc_workspace_mx(p, DEV)
    Y = torch.full((4, h["cfg"]["H"]), 3.0, dtype=torch.bfloat16, device=DEV)
    moe.moe_forward_mx(p, 0, dd["X"], dd["E_ids"], dd["G"], dd["W1"], dd["S1"], dd["W2"], dd["S2"], Y, ws)
    moe.moe_sync_status(ws)
    assert (Y == 3.0).all()

"""Parity of the A8W8-INT forward (int8 weights with per-channel scales,
per-token int8 activations) with the oracle's A8W8 restatement."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_route_gb300 as moe
import oracle
import synth
from _gpu import DEV, check_y, host_bits, mixed_load_ids, params, run_route, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(built_lib):
    moe.lib()
    torch.cuda.set_device(DEV)


def _run(p, dd, E_ids, G):
    ws = moe.alloc_workspace_a8w8(p, DEV)
    Y = torch.full((p.T, p.H), float("nan"), dtype=torch.bfloat16, device=DEV)
    moe.moe_forward_a8w8(p, dd["X"], E_ids, G, dd["W1"], dd["S1"], dd["W2"], dd["S2"], Y, ws)
    moe.moe_sync_status(ws)
    return Y


@pytest.mark.parametrize("name", ["c2s_q", "c3s_q", "c5s_q"])
def test_a8w8_forward_matches_oracle(name):
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
        ids, G, _ = oracle.route(h["X"], h["Wg"], h["bias"], c["score_fn"], c["k"], c["alpha"], c["renorm"])
        assert np.array_equal(E_ids.cpu().numpy(), ids)
        G = Gd.cpu().numpy().astype(np.float64)
    Y = _run(p, dd, E_ids, Gd)
    Y_ref = oracle.forward_a8w8_tokens(np.arange(c["T"]), h["X"], ids, G, h["W1"], h["S1"], h["W2"],
                                       h["S2"], E=c["E"])
    slack = oracle.margin_a8w8_tokens(np.arange(c["T"]), h["X"], ids, G, h["W1"], h["S1"], h["W2"],
                                       h["S2"], E=c["E"])
    check_y(Y, Y_ref, name, slack=slack)


def test_a8w8_is_deterministic_and_rejects_a_shared_expert():
    h = synth.make_inputs("c2s_q")
    dd = to_device(h)
    p = params(h["cfg"])
    Y1 = _run(p, dd, dd["E_ids"], dd["G"]).clone()
    Y2 = _run(p, dd, dd["E_ids"], dd["G"])
    assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))
    ps = params(h["cfg"], shared=1)
    ws = moe.alloc_workspace_a8w8(ps, DEV)
    with pytest.raises(moe.MoEError) as ex:
        moe.moe_forward_a8w8(ps, dd["X"], dd["E_ids"], dd["G"], dd["W1"], dd["S1"], dd["W2"], dd["S2"],
                             torch.empty_like(dd["X"]), ws)
    assert ex.value.code == moe.MOE_ERR_UNSUPPORTED


@pytest.mark.parametrize("name,n_rows", [("c3_q", 6), ("c2_q", 6)])
def test_a8w8_full_size_sampled(name, n_rows):
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
    Y = _run(p, dd, E_ids, G)
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([[0, T - 1], rng.choice(T, n_rows, replace=False)]))
    hX = host_bits(dd["X"])
    ids = E_ids.cpu().numpy()
    Gh = G.cpu().numpy().astype(np.float64)
    W1 = lambda e: dd["W1"][e].cpu().numpy()  # noqa: E731
    W2 = lambda e: dd["W2"][e].cpu().numpy()  # noqa: E731
    S1 = lambda e: dd["S1"][e].cpu().numpy()  # noqa: E731
    S2 = lambda e: dd["S2"][e].cpu().numpy()  # noqa: E731
    Y_ref = oracle.forward_a8w8_tokens(rows, hX[rows], ids[rows], Gh[rows], W1, S1, W2, S2, E=E)
    slack = oracle.margin_a8w8_tokens(rows, hX[rows], ids[rows], Gh[rows], W1, S1, W2, S2, E=E)
    check_y(Y[torch.from_numpy(rows).to(DEV)], Y_ref, name, slack=slack)


# Ragged and degenerate shapes: one token, k = E, every token on one expert
# (several 128-token tiles, the last partial, other experts empty), H and I
# that are not multiples of 128 (partial channel tiles).
EDGE_Q = [
    dict(T=1, H=64, E=4, k=2, I=64),
    dict(T=17, H=128, E=5, k=5, I=192),
    dict(T=129, H=192, E=3, k=1, I=64),
    dict(T=300, H=128, E=6, k=1, I=320, hot=True),
    dict(T=260, H=320, E=9, k=3, I=448),
    dict(T=700, H=128, E=12, k=2, I=320, mixed=True),
]


@pytest.mark.parametrize("shape", EDGE_Q, ids=lambda s: "T{T}_H{H}_E{E}_k{k}_I{I}".format(**s))
def test_a8w8_edge_shapes(shape):
    shape = dict(shape)
    hot = shape.pop("hot", False)
    mixed = shape.pop("mixed", False)
    h = synth.make_inputs(dict(shape, routing="given", score="softmax", renorm=0, quant="a8w8"), seed=99)
    if hot:
        h["E_ids"][:] = 0
    if mixed:
        h["E_ids"][:] = mixed_load_ids(shape["T"], shape["E"])
    c = h["cfg"]
    dd = to_device(h)
    p = params(c)
    Y = _run(p, dd, dd["E_ids"], dd["G"])
    Y_ref = oracle.forward_a8w8_tokens(np.arange(c["T"]), h["X"], h["E_ids"], h["G"].astype(np.float64),
                                       h["W1"], h["S1"], h["W2"], h["S2"], E=c["E"])
    slack = oracle.margin_a8w8_tokens(np.arange(c["T"]), h["X"], h["E_ids"], h["G"].astype(np.float64),
                                       h["W1"], h["S1"], h["W2"], h["S2"], E=c["E"])
    check_y(Y, Y_ref, str(shape), slack=slack)


def test_a8w8_with_no_tokens_writes_nothing():
    h = synth.make_inputs("c3s_q")
    dd = to_device(h)
    p = params(h["cfg"], T=0)
    ws = moe.alloc_workspace_a8w8(p, DEV)
    Y = torch.full((4, h["cfg"]["H"]), 3.0, dtype=torch.bfloat16, device=DEV)
    moe.moe_forward_a8w8(p, dd["X"], dd["E_ids"] if "E_ids" in dd else dd["X"], dd["X"], dd["W1"], dd["S1"],
                         dd["W2"], dd["S2"], Y, ws)
    moe.moe_sync_status(ws)
    assert (Y == 3.0).all()
